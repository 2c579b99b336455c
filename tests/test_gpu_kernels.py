"""GPU parity of every libmoe call against the CPU oracle, through the C ABI.

Each call gets the same seeded inputs as the oracle function it is compared
with.  Integer outputs (top-k indices, cu_seqlens, the permutation, the MoD
selection) must match exactly; floating-point outputs within the normwise
relative tolerance of the storage type (1e-5 fp32, 2e-2 bf16).  Sizes span
several tiles and ragged tails (T not a multiple of the 256-token chunk, H and
H' not multiples of the GEMM tile widths)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from token_dispatch_gb300 import _lib as L
from token_dispatch_gb300 import layer, synth
from tests.gpu_util import (DEV, TDT, TOL, assert_close, check_topk, check_topk_exact, dev, gate_tol,
                            host_layer_inputs, to64)

pytestmark = pytest.mark.gpu

S = synth.MoEShape
SHAPES = [
    synth.TINY_F32,
    S("bf16_T1000_H384_E16_K4_Hp320", 1000, 384, 16, 4, 320, "bf16"),
    S("bf16_T777_H256_E64_K6_Hp192", 777, 256, 64, 6, 192, "bf16"),
    S("f32_T300_H64_E12_K3_Hp96", 300, 64, 12, 3, 96, "f32"),
]
# many experts: split over H into partials when the token tiles are few (T=300),
# one pass on CTA pairs of 256 x 256 tiles otherwise (ragged T=6600 with a
# half-empty last expert tile at E=384; E=1024)
ROUTE_ONLY = [S("bf16_T300_H128_E384_K8", 300, 128, 384, 8, 64, "bf16"),
              S("f32_T129_H32_E1024_K16", 129, 32, 1024, 16, 32, "f32"),
              S("bf16_T6600_H128_E384_K8", 6600, 128, 384, 8, 64, "bf16"),
              S("bf16_T4000_H256_E1024_K8", 4000, 256, 1024, 8, 64, "bf16")]
# bf16 routers with 8 or 16 experts and H a multiple of 512 take the one-launch
# streaming router: ragged token blocks of 8 to 64 tokens, fewer blocks than
# SMs, slices of H from 32 to 256 columns per warp
ROUTE_STREAM = [S("bf16_T2053_H1536_E8_K2", 2053, 1536, 8, 2, 64, "bf16"),
                S("bf16_T1000_H512_E16_K4", 1000, 512, 16, 4, 64, "bf16"),
                S("bf16_T5_H4096_E8_K1", 5, 4096, 8, 1, 64, "bf16"),
                S("bf16_T3001_H4096_E16_K16", 3001, 4096, 16, 16, 64, "bf16"),
                S("bf16_T4099_H512_E8_K3", 4099, 512, 8, 3, 64, "bf16"),
                S("bf16_T333_H1024_E8_K2", 333, 1024, 8, 2, 64, "bf16")]
CDT = {"f32": L.MOE_F32, "bf16": L.MOE_BF16}


@pytest.fixture(scope="module", autouse=True)
def built():
    from token_dispatch_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def ids(shapes):
    return [s.name for s in shapes]


def route_gpu(shape, x, wr, bias=None):
    T, E, K = x.shape[0], shape.E, shape.K
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, K), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, K), dtype=torch.float32, device=DEV)
    b = None if bias is None else torch.from_numpy(bias).to(DEV)
    nbytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE, T, shape.H, E, K, 0)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=DEV)
    L.moe_route(dev(x), dev(wr), b, T, shape.H, E, K, CDT[shape.dtype], logits, idx, gate, ws, nbytes)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), idx.cpu().numpy(), gate.cpu().numpy()


@pytest.mark.parametrize("shape", SHAPES + ROUTE_ONLY + ROUTE_STREAM, ids=ids(SHAPES + ROUTE_ONLY + ROUTE_STREAM))
def test_route_matches_oracle(shape):
    x, wr = synth.router_inputs(shape)
    bias = synth.expert_bias(shape.E, 0.7, expert=1)
    logits, idx, gate = route_gpu(shape, x, wr, bias)
    r_logits, r_p, r_idx, r_gate = O.route(x.ref, wr.ref, shape.K, bias.astype(np.float64))
    tol = 1e-5 if shape.dtype == "f32" else 1e-5  # fp32 accumulation in both storage types
    assert_close(logits, r_logits, tol, "logits")
    logit_err = float(np.max(np.abs(logits - r_logits)))
    check_topk_exact(idx, logits, shape.K)
    n_amb = check_topk(idx, r_logits, shape.K, logit_err)
    assert n_amb == 0, f"{n_amb} rows differ from the fp64 selection"
    same = (idx == r_idx).all(axis=1)
    assert_close(gate[same], r_gate[same], gate_tol(logit_err), "gate")


# every router form: streaming (E = 8 / 16), tcgen05 with the fused epilogue
# (E <= 64, one H range), tcgen05 split over H + softmax kernel (E = 384), FFMA (fp32)
VARIANT_SHAPES = [S("bf16_T1000_H512_E8_K2", 1000, 512, 8, 2, 64, "bf16"),
                  S("bf16_T777_H1024_E16_K4", 777, 1024, 16, 4, 64, "bf16"),
                  S("bf16_T777_H256_E64_K6", 777, 256, 64, 6, 64, "bf16"),
                  S("bf16_T300_H128_E384_K8", 300, 128, 384, 8, 64, "bf16"),
                  S("f32_T300_H64_E12_K3", 300, 64, 12, 3, 64, "f32")]
FLAGS = {"renorm": 1, "bias_select": 2, "both": 3}


@pytest.mark.parametrize("flags", list(FLAGS), ids=list(FLAGS))
@pytest.mark.parametrize("shape", VARIANT_SHAPES, ids=ids(VARIANT_SHAPES))
def test_route_variants_match_oracle(shape, flags):
    """Mixtral-style renormalised gates and the selection-only bias, against
    the oracle's route(renorm=..., bias_select_only=...)."""
    fl = FLAGS[flags]
    renorm, select = bool(fl & L.MOE_ROUTE_RENORM), bool(fl & L.MOE_ROUTE_BIAS_SELECT)
    T, E, K = shape.T, shape.E, shape.K
    x, wr = synth.router_inputs(shape)
    bias = (np.random.default_rng(11).standard_normal(E) * 0.5).astype(np.float32)  # shifts every expert
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, K), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, K), dtype=torch.float32, device=DEV)
    nbytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE, T, shape.H, E, K, 0)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=DEV)
    L.moe_route_ex(dev(x), dev(wr), torch.from_numpy(bias).to(DEV), T, shape.H, E, K, CDT[shape.dtype], fl, logits,
                   idx, gate, ws, nbytes)
    torch.cuda.synchronize()
    r_logits, r_p, r_idx, r_gate = O.route(x.ref, wr.ref, K, bias.astype(np.float64), renorm=renorm,
                                           bias_select_only=select)
    logits, idx, gate = logits.cpu().numpy(), idx.cpu().numpy(), gate.cpu().numpy()
    assert_close(logits, r_logits, 1e-5, "logits")
    err = float(np.max(np.abs(logits - r_logits)))
    r_sel = r_logits + (bias.astype(np.float64)[None, :] if select else 0.0)
    check_topk_exact(idx, logits, K, bias if select else None)
    n_amb = check_topk(idx, r_sel, K, err)
    assert n_amb == 0, f"{n_amb} rows differ from the fp64 selection"
    same = (idx == r_idx).all(axis=1)
    assert_close(gate[same], r_gate[same], gate_tol(err), "gate")
    if renorm:
        assert np.allclose(gate.sum(axis=1), 1.0, atol=1e-5)
    # the gate of every chosen expert, chosen or not by the oracle, is its own probability
    q = np.take_along_axis(r_p, idx.astype(np.int64), axis=1)
    if renorm:
        q = q / q.sum(axis=1, keepdims=True)
    assert_close(gate, q, gate_tol(err), "gate of the GPU's choice")


@pytest.mark.parametrize("dtype,E,K,H", [("f32", 8, 2, 64), ("bf16", 16, 4, 64), ("bf16", 384, 8, 64),
                                         ("f32", 64, 6, 64), ("bf16", 8, 2, 512), ("bf16", 16, 5, 1024),
                                         ("bf16", 64, 6, 64), ("bf16", 40, 3, 2048)])
def test_route_integer_inputs_select_exactly(dtype, E, K, H):
    """Small-integer x and W make every logit exact in fp32 on both sides, with
    many ties: the selection (tie -> lowest expert) must then match exactly."""
    T = 700
    rng = np.random.default_rng(E)
    x = synth.store(rng.integers(-2, 3, size=(T, H)).astype(np.float64), dtype)
    wr = synth.store(rng.integers(-1, 2, size=(H, E)).astype(np.float64), dtype)
    shape = S("int_route", T, H, E, K, 64, dtype)
    logits, idx, gate = route_gpu(shape, x, wr)
    r_logits, _, r_idx, r_gate = O.route(x.ref, wr.ref, K)
    assert np.array_equal(logits.astype(np.float64), r_logits)
    assert np.array_equal(idx, r_idx)
    assert_close(gate, r_gate, 1e-6, "gate")


def test_route_ties_pick_lowest_expert():
    shape = S("f32_ties", 64, 16, 8, 3, 16, "f32")
    x = synth.store(np.zeros((64, 16)), "f32")
    wr = synth.store(np.zeros((16, 8)), "f32")
    bias = np.array([0, 1, 1, 0, 1, 0, 0, 1], np.float32)
    logits, idx, gate = route_gpu(shape, x, wr, bias)
    assert (idx == np.array([1, 2, 4])).all()
    p1 = math.e / (4 * math.e + 4)
    assert np.allclose(gate, p1, rtol=1e-6)


@pytest.mark.parametrize("E,K", [(300, 7), (384, 8), (1000, 16)])
def test_route_many_experts_ties_and_infinities(E, K):
    """Warp top-K over many experts per lane: logits from the bias alone, with
    runs of equal values, +-0 and -inf entries, so that whole rounds are
    decided by the lowest expert index and the last picks fall on -inf."""
    T = 40
    shape = S(f"f32_T{T}_E{E}_K{K}_ties", T, 16, E, K, 16, "f32")
    x = synth.store(np.zeros((T, 16)), "f32")
    wr = synth.store(np.zeros((16, E)), "f32")
    rng = np.random.default_rng(11)
    bias = np.full(E, -np.inf, np.float32)
    n_fin = {300: 4, 384: 12, 1000: 40}[E]  # fewer finite values than K for E=300
    pos = rng.choice(E, n_fin, replace=False)
    bias[pos] = rng.choice(np.array([-1.5, 0.0, -0.0, 2.25], np.float32), n_fin)
    logits, idx, gate = route_gpu(shape, x, wr, bias)
    ref = np.broadcast_to(bias.astype(np.float64), (T, E))
    assert np.array_equal(idx, O.topk_experts(ref, K))
    p = np.exp(ref - ref.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    assert np.allclose(gate, np.take_along_axis(p, idx, axis=1), rtol=1e-6, atol=0)


def oracle_idx(shape, T=None):
    x, wr = synth.router_inputs(shape, tokens=T)
    return x, wr, O.topk_experts(O.router_logits(x.ref, wr.ref), shape.K)


@pytest.mark.parametrize("shape", SHAPES + ROUTE_ONLY, ids=ids(SHAPES + ROUTE_ONLY))
def test_dispatch_is_bit_exact(shape):
    x, wr, idx = oracle_idx(shape)
    T, H, E, K = shape.T, shape.H, shape.E, shape.K
    cu, dst, src, xs_ref = O.dispatch(x.ref, idx, E)
    b = layer.MoEBuffers(T, H, E, K, shape.Hp, shape.dtype, DEV, backward=False)
    L.moe_dispatch(dev(x), torch.from_numpy(idx).to(DEV), T, H, E, K, CDT[shape.dtype], b.cu, b.dst_row,
                   b.src_tok, b.xs, b.ws_dispatch, b.ws_dispatch_bytes)
    assert L.moe_last_device_error() == L.MOE_OK
    assert np.array_equal(b.cu.cpu().numpy(), cu)
    assert np.array_equal(b.dst_row.cpu().numpy(), dst)
    assert np.array_equal(b.src_tok.cpu().numpy(), src)
    assert np.array_equal(to64(b.xs), xs_ref)  # a pure copy: bit-exact


def test_dispatch_skewed_all_tokens_to_one_expert():
    T, H, E, K = 1030, 64, 32, 2
    idx = np.stack([np.zeros(T, np.int32), 1 + (np.arange(T) % (E - 1))], axis=1).astype(np.int32)
    x = synth.store(synth.normal(5, 1, T * H).reshape(T, H), "bf16")
    cu, dst, src, xs_ref = O.dispatch(x.ref, idx, E)
    b = layer.MoEBuffers(T, H, E, K, 64, "bf16", DEV, backward=False)
    L.moe_dispatch(dev(x), torch.from_numpy(idx).to(DEV), T, H, E, K, L.MOE_BF16, b.cu, b.dst_row, b.src_tok,
                   b.xs, b.ws_dispatch, b.ws_dispatch_bytes)
    assert np.array_equal(b.cu.cpu().numpy(), cu)
    assert np.array_equal(b.dst_row.cpu().numpy(), dst)
    assert np.array_equal(to64(b.xs), xs_ref)


@pytest.mark.parametrize("T,E,K", [(65536, 1024, 8), (8192, 384, 8), (16384, 64, 6), (16385, 64, 6),
                                   (7000, 1024, 16), (300, 1000, 3), (1, 8, 2)])
def test_dispatch_count_tables_small_and_large(T, E, K):
    """Both ways the chunk counts are scanned: tables of at most 8192 entries
    summed by every placing CTA, larger ones (65536 tokens x 1024 experts: a
    256 x 1024 table) by the column-scan launch.  Skewed (Zipf-like) expert
    choices, a ragged last chunk; index maps and rows bit-exact."""
    rng = np.random.default_rng(T + E)
    w = 1.0 / np.arange(1, E + 1) ** 1.1
    w /= w.sum()
    idx = np.stack([rng.choice(E, K, replace=False, p=w) for _ in range(T)]).astype(np.int32)
    H = 64
    x = synth.store(rng.standard_normal((T, H)), "bf16")
    cu, dst, src, xs_ref = O.dispatch(x.ref, idx, E)
    b = layer.MoEBuffers(T, H, E, K, 64, "bf16", DEV, backward=False)
    L.moe_dispatch(dev(x), torch.from_numpy(idx).to(DEV), T, H, E, K, L.MOE_BF16, b.cu, b.dst_row, b.src_tok,
                   b.xs, b.ws_dispatch, b.ws_dispatch_bytes)
    assert L.moe_last_device_error() == L.MOE_OK
    assert np.array_equal(b.cu.cpu().numpy(), cu)
    assert np.array_equal(b.dst_row.cpu().numpy(), dst)
    assert np.array_equal(b.src_tok.cpu().numpy(), src)
    assert np.array_equal(to64(b.xs), xs_ref)


def test_dispatch_out_of_range_expert_sets_bounds_error():
    T, H, E, K = 40, 64, 8, 2
    idx = np.stack([np.arange(T) % E, (np.arange(T) + 1) % E], axis=1).astype(np.int32)
    idx[7, 1] = E + 3
    x = synth.store(np.ones((T, H)), "f32")
    b = layer.MoEBuffers(T, H, E, K, 64, "f32", DEV, backward=False)
    assert L.moe_last_device_error() == L.MOE_OK
    L.moe_dispatch(dev(x), torch.from_numpy(idx).to(DEV), T, H, E, K, L.MOE_F32, b.cu, b.dst_row, b.src_tok,
                   b.xs, b.ws_dispatch, b.ws_dispatch_bytes)
    assert L.moe_last_device_error() == L.MOE_ERR_DEVICE_BOUNDS
    assert b.dst_row.cpu().numpy()[15] == -1
    assert int(b.cu[-1]) == T * K - 1
    assert L.moe_last_device_error() == L.MOE_OK  # cleared by the read


@pytest.mark.parametrize("shape", SHAPES, ids=ids(SHAPES))
def test_expert_ffn_matches_oracle(shape):
    x, wr, wg, wu, wd = host_layer_inputs(shape)
    idx = O.topk_experts(O.router_logits(x.ref, wr.ref), shape.K)
    cu, dst, src, xs_ref = O.dispatch(x.ref, idx, shape.E)
    act_ref, h_ref = O.expert_ffn(xs_ref, cu, wg.ref, wu.ref, wd.ref)
    R, H, Hp = shape.R, shape.H, shape.Hp
    xs = synth.store(xs_ref, shape.dtype)
    act = torch.empty((R, Hp), dtype=TDT[shape.dtype], device=DEV)
    h = torch.empty((R, H), dtype=TDT[shape.dtype], device=DEV)
    L.moe_expert_ffn(dev(xs), torch.from_numpy(cu).to(DEV), R, dev(wg), dev(wu), dev(wd), shape.E, H, Hp,
                     CDT[shape.dtype], act, h)
    torch.cuda.synchronize()
    assert_close(to64(act), act_ref, TOL[shape.dtype], "act")
    assert_close(to64(h), h_ref, TOL[shape.dtype], "h")


SPLIT_SHAPES = [S("bf16_T1000_H320_E4_K2_Hp320", 1000, 320, 4, 2, 320, "bf16"),
                S("bf16_T3000_H256_E8_K2_Hp1408", 3000, 256, 8, 2, 1408, "bf16"),
                # ~300 rows per expert: the last pair tile of every expert holds
                # rows of the leader CTA only
                S("bf16_T1200_H256_E8_K2_Hp320", 1200, 256, 8, 2, 320, "bf16")]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=ids(SPLIT_SHAPES))
def test_expert_ffn_tail_split_matches_oracle(shape):
    """With its workspace the down projection runs its last round of tiles as
    two K halves on two CTA pairs whose fp32 partials meet in the workspace
    (at these sizes every tile: there are fewer tiles than half the pairs; K =
    H' of 5 and 22 blocks, split 2 + 3 and 11 + 11).  The workspace starts
    as garbage (the call zeroes its counters itself); h matches the oracle and
    comes out bit for bit the same on a second call; act does not depend on
    the workspace (only the down projection splits); h without the workspace
    agrees within the bf16 tolerance."""
    x, wr, wg, wu, wd = host_layer_inputs(shape)
    idx = O.topk_experts(O.router_logits(x.ref, wr.ref), shape.K)
    cu, dst, src, xs_ref = O.dispatch(x.ref, idx, shape.E)
    act_ref, h_ref = O.expert_ffn(xs_ref, cu, wg.ref, wu.ref, wd.ref)
    R, H, Hp, E = shape.R, shape.H, shape.Hp, shape.E
    xs, cu_d = dev(synth.store(xs_ref, shape.dtype)), torch.from_numpy(cu).to(DEV)
    n = L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN, shape.T, H, E, shape.K, Hp)
    ws = torch.full((n,), 0x7F, dtype=torch.uint8, device=DEV)
    outs = []
    for use_ws in (True, True, False):
        act = torch.empty((R, Hp), dtype=TDT[shape.dtype], device=DEV)
        h = torch.empty((R, H), dtype=TDT[shape.dtype], device=DEV)
        L.moe_expert_ffn(xs, cu_d, R, dev(wg), dev(wu), dev(wd), E, H, Hp, CDT[shape.dtype], act, h,
                         ws if use_ws else None, n if use_ws else 0)
        outs.append((act, h))
    torch.cuda.synchronize()
    assert L.moe_last_device_error() == L.MOE_OK
    (act1, h1), (act2, h2), (act3, h3) = outs
    assert_close(to64(act1), act_ref, TOL[shape.dtype], "act")
    assert_close(to64(h1), h_ref, TOL[shape.dtype], "h (split)")
    assert torch.equal(h1, h2) and torch.equal(act1, act2)
    assert torch.equal(act1, act3)
    assert_close(to64(h3), h_ref, TOL[shape.dtype], "h (whole tiles)")


GATHER_SHAPES = [S("bf16_T1000_H384_E16_K4_Hp320", 1000, 384, 16, 4, 320, "bf16"),
                 S("bf16_T2048_H512_E8_K2_Hp768", 2048, 512, 8, 2, 768, "bf16"),
                 S("bf16_T777_H256_E64_K6_Hp192", 777, 256, 64, 6, 192, "bf16"),
                 S("bf16_T3_H128_E8_K2_Hp64", 3, 128, 8, 2, 64, "bf16"),
                 S("f32_T300_H64_E12_K3_Hp96", 300, 64, 12, 3, 96, "f32")]


@pytest.mark.parametrize("shape", GATHER_SHAPES, ids=ids(GATHER_SHAPES))
def test_expert_ffn_gather_equals_ffn_on_dispatched_rows(shape):
    """The gate/up GEMM reading the rows of x by src_tok gives bit for bit what
    the FFN gives on the expert-sorted rows dispatch writes (the same operands
    in the same order; the saved [g | u] too, and the same split of the down
    projection's last round when both get the workspace), and matches the
    oracle; dispatch without xs writes the same index maps.  Ragged experts and
    tiles (T not a multiple of 128, some experts without rows for T=3), several
    rounds of pair tiles and more K blocks than pipeline stages (T=2048)."""
    x, wr, wg, wu, wd = host_layer_inputs(shape)
    T, H, E, K, Hp, R = shape.T, shape.H, shape.E, shape.K, shape.Hp, shape.R
    idx = O.topk_experts(O.router_logits(x.ref, wr.ref), K)
    cu, dst, src, xs_ref = O.dispatch(x.ref, idx, E)
    act_ref, h_ref = O.expert_ffn(xs_ref, cu, wg.ref, wu.ref, wd.ref)
    b = layer.MoEBuffers(T, H, E, K, Hp, shape.dtype, DEV, backward=False)
    xd, idx_d = dev(x), torch.from_numpy(idx).to(DEV)
    L.moe_dispatch(xd, idx_d, T, H, E, K, CDT[shape.dtype], b.cu, b.dst_row, b.src_tok, b.xs, b.ws_dispatch,
                   b.ws_dispatch_bytes)
    bf = shape.dtype == "bf16"
    act1 = torch.empty((R, Hp), dtype=TDT[shape.dtype], device=DEV)
    h1 = torch.empty((R, H), dtype=TDT[shape.dtype], device=DEV)
    gu1 = torch.empty((R, 2 * Hp), dtype=TDT[shape.dtype], device=DEV) if bf else None
    nws = L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN, T, H, E, K, Hp) if bf else 0
    ws = torch.full((max(nws, 1),), 0x7F, dtype=torch.uint8, device=DEV)
    L.moe_expert_ffn_ex(b.xs, b.cu, R, dev(wg), dev(wu), dev(wd), E, H, Hp, CDT[shape.dtype], act1, gu1, h1,
                        ws if bf else None, nws)
    cu2 = torch.full_like(b.cu, -9)
    dst2 = torch.full_like(b.dst_row, -9)
    src2 = torch.full_like(b.src_tok, -9)
    L.moe_dispatch(None, idx_d, T, H, E, K, CDT[shape.dtype], cu2, dst2, src2, None, b.ws_dispatch,
                   b.ws_dispatch_bytes)
    act2 = torch.empty_like(act1)
    h2 = torch.empty_like(h1)
    gu2 = torch.empty_like(gu1) if bf else None
    ws.fill_(0x7F)  # stale partials and counters: the call zeroes what it uses
    L.moe_expert_ffn_gather(xd, src2, T, cu2, R, dev(wg), dev(wu), dev(wd), E, H, Hp, CDT[shape.dtype], act2, gu2,
                            h2, ws if bf else None, nws)
    torch.cuda.synchronize()
    assert L.moe_last_device_error() == L.MOE_OK
    for a_, b_ in ((b.cu, cu2), (b.dst_row, dst2), (b.src_tok, src2)):
        assert torch.equal(a_, b_)
    assert torch.equal(act1, act2) and torch.equal(h1, h2)
    if bf:
        assert torch.equal(gu1, gu2)
    assert_close(to64(act2), act_ref, TOL[shape.dtype], "act")
    assert_close(to64(h2), h_ref, TOL[shape.dtype], "h")


def test_expert_ffn_gather_out_of_range_row_sets_bounds_error():
    shape = S("bf16_T40_H128_E8_K2_Hp64", 40, 128, 8, 2, 64, "bf16")
    x, wr, wg, wu, wd = host_layer_inputs(shape)
    T, H, E, K, Hp, R = shape.T, shape.H, shape.E, shape.K, shape.Hp, shape.R
    cu = torch.from_numpy(np.array([0, R] + [R] * (E - 1), np.int32)).to(DEV)
    src = torch.arange(R, dtype=torch.int32, device=DEV) % T
    src[5] = T + 100
    act = torch.empty((R, Hp), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    assert L.moe_last_device_error() == L.MOE_OK
    L.moe_expert_ffn_gather(dev(x), src, T, cu, R, dev(wg), dev(wu), dev(wd), E, H, Hp, L.MOE_BF16, act, None, h)
    assert L.moe_last_device_error() == L.MOE_ERR_DEVICE_BOUNDS
    assert L.moe_last_device_error() == L.MOE_OK


def test_expert_ffn_empty_and_single_row_experts():
    shape = S("bf16_sparse", 5, 128, 8, 1, 128, "bf16")
    x = synth.normal_stored(3, 1, (5, 128), 1.0, "bf16")
    wg, wu, wd = synth.expert_weights_host(shape, seed=3)
    idx = np.array([[3], [3], [6], [0], [3]], np.int32)  # experts 1,2,4,5,7 empty
    cu, dst, src, xs_ref = O.dispatch(x.ref, idx, 8)
    act_ref, h_ref = O.expert_ffn(xs_ref, cu, wg.ref, wu.ref, wd.ref)
    act = torch.empty((5, 128), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((5, 128), dtype=torch.bfloat16, device=DEV)
    L.moe_expert_ffn(dev(synth.store(xs_ref, "bf16")), torch.from_numpy(cu).to(DEV), 5, dev(wg), dev(wu),
                     dev(wd), 8, 128, 128, L.MOE_BF16, act, h)
    torch.cuda.synchronize()
    assert_close(to64(h), h_ref, 2e-2, "h")
    # with the workspace: the one tile of each non-empty expert splits along K
    # (H' = 128: two K blocks, one per half)
    n = L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN, 5, 128, 8, 1, 128)
    ws = torch.full((n,), 0x5A, dtype=torch.uint8, device=DEV)
    h2 = torch.empty_like(h)
    L.moe_expert_ffn(dev(synth.store(xs_ref, "bf16")), torch.from_numpy(cu).to(DEV), 5, dev(wg), dev(wu),
                     dev(wd), 8, 128, 128, L.MOE_BF16, act, h2, ws, n)
    torch.cuda.synchronize()
    assert L.moe_last_device_error() == L.MOE_OK
    assert_close(to64(h2), h_ref, 2e-2, "h (split)")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("variant", ["plain", "scaled_residual_outrow"])
def test_combine_matches_oracle(dtype, variant):
    rng = np.random.default_rng(7)
    T, K, H = 333, 3, 200 if dtype == "f32" else 256
    R = T * K
    h = synth.store(rng.standard_normal((R, H)), dtype)
    gate = rng.random((T, K)).astype(np.float32)
    dst = rng.permutation(R).astype(np.int32)
    kw, gk = {}, {}
    n_out = T
    if variant != "plain":
        n_out = 2 * T
        scale = rng.standard_normal(T).astype(np.float32)
        out = np.sort(rng.choice(n_out, T, replace=False)).astype(np.int32)
        res = synth.store(rng.standard_normal((n_out, H)), dtype)
        kw = dict(row_scale=scale.astype(np.float64), residual=res.ref, out_row=out, n_out=n_out)
        gk = dict(row_scale=torch.from_numpy(scale).to(DEV), residual=dev(res), out_row=torch.from_numpy(out).to(DEV))
    ref = O.combine(h.ref, gate.astype(np.float64), dst, **kw)
    y = torch.zeros((n_out, H), dtype=TDT[dtype], device=DEV)
    if variant != "plain":
        y.copy_(gk["residual"])  # rows not written by any token keep the residual
    L.moe_combine(dev(h), torch.from_numpy(gate).to(DEV), torch.from_numpy(dst).to(DEV), gk.get("row_scale"),
                  gk.get("residual"), gk.get("out_row"), T, H, K, CDT[dtype], y)
    torch.cuda.synchronize()
    assert_close(to64(y), ref, TOL[dtype], "y")


def test_combine_of_dispatch_with_unit_gates_is_K_times_x():
    for K in (1, 2, 4, 8, 6):
        T, E, H = 513, 16, 128
        x = synth.store(synth.normal(11, K, T * H).reshape(T, H), "bf16")
        idx = np.stack([np.random.default_rng(K).choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
        b = layer.MoEBuffers(T, H, E, K, 64, "bf16", DEV, backward=False)
        L.moe_dispatch(dev(x), torch.from_numpy(idx).to(DEV), T, H, E, K, L.MOE_BF16, b.cu, b.dst_row, b.src_tok,
                       b.xs, b.ws_dispatch, b.ws_dispatch_bytes)
        ones = torch.ones((T, K), dtype=torch.float32, device=DEV)
        y = torch.empty((T, H), dtype=torch.float32, device=DEV)
        # identity expert: combine the dispatched rows, accumulate in fp32 (f32 view of bf16 rows)
        xs32 = b.xs.float()
        L.moe_combine(xs32, ones, b.dst_row, None, None, None, T, H, K, L.MOE_F32, y)
        torch.cuda.synchronize()
        want = K * x.ref
        got = y.cpu().numpy().astype(np.float64)
        if K in (1, 2, 4, 8):
            assert np.array_equal(got, want)
        else:
            assert np.max(np.abs(got - want) / np.maximum(np.abs(want), 1e-30)) <= 2 ** -22


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_permute_bwd_matches_oracle(dtype):
    rng = np.random.default_rng(9)
    T, K, H = 301, 4, 128
    R, n_out = T * K, 2 * T
    h = synth.store(rng.standard_normal((R, H)), dtype)
    dy = synth.store(rng.standard_normal((n_out, H)), dtype)
    dxs = synth.store(rng.standard_normal((R, H)), dtype)
    gate = rng.random((T, K)).astype(np.float32)
    dst = rng.permutation(R).astype(np.int32)
    scale = rng.standard_normal(T).astype(np.float32)
    out = rng.choice(n_out, T, replace=False).astype(np.int32)
    dh_r, dg_r, ds_r, dx_r = O.permute_bwd(dy.ref, h.ref, gate.astype(np.float64), dst, dxs.ref,
                                           row_scale=scale.astype(np.float64), out_row=out)
    dh = torch.zeros((R, H), dtype=TDT[dtype], device=DEV)
    dg = torch.empty((T, K), dtype=torch.float32, device=DEV)
    ds = torch.empty((T,), dtype=torch.float32, device=DEV)
    dx = torch.empty((T, H), dtype=TDT[dtype], device=DEV)
    L.moe_permute_bwd(dev(dy), dev(h), torch.from_numpy(gate).to(DEV), torch.from_numpy(dst).to(DEV),
                      torch.from_numpy(scale).to(DEV), torch.from_numpy(out).to(DEV), dev(dxs), T, H, K,
                      CDT[dtype], dh, dg, ds, dx)
    torch.cuda.synchronize()
    tol = 1e-5 if dtype == "f32" else 2e-2
    assert_close(to64(dh), dh_r, tol, "dh")
    assert_close(dg.cpu().numpy(), dg_r, 1e-5, "d_gate")
    assert_close(ds.cpu().numpy(), ds_r, 1e-5, "d_scale")
    assert_close(to64(dx), dx_r, tol, "dx")


@pytest.mark.parametrize("shape", SHAPES + ROUTE_ONLY[:1], ids=ids(SHAPES + ROUTE_ONLY[:1]))
def test_route_bwd_softmax_topk_matches_oracle(shape):
    T, H, E, K = shape.T, shape.H, shape.E, shape.K
    x, wr = synth.router_inputs(shape)
    logits = (x.ref @ wr.ref).astype(np.float32)  # an fp32 logits input shared by both sides
    idx = O.topk_experts(logits.astype(np.float64), K)
    d_gate = np.random.default_rng(4).standard_normal((T, K)).astype(np.float32)
    dl_r, dw_r, dx_r = O.route_bwd_softmax_topk(d_gate.astype(np.float64), logits.astype(np.float64), idx,
                                                x.ref, wr.ref)
    dx0 = synth.store(np.random.default_rng(5).standard_normal((T, H)), shape.dtype)
    dl = torch.empty((T, E), dtype=torch.float32, device=DEV)
    dw = torch.empty((H, E), dtype=torch.float32, device=DEV)
    dx = dev(dx0).clone()
    nbytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, T, H, E, K, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK, torch.from_numpy(d_gate).to(DEV), torch.from_numpy(logits).to(DEV),
                    torch.from_numpy(idx).to(DEV), dev(x), dev(wr), T, H, E, K, CDT[shape.dtype], dl, dw, dx, ws,
                    nbytes)
    torch.cuda.synchronize()
    assert_close(dl.cpu().numpy(), dl_r, 1e-5, "d_logits")
    assert_close(dw.cpu().numpy(), dw_r, 1e-5, "dw_router")
    assert_close(to64(dx), dx0.ref + dx_r, TOL[shape.dtype], "dx (accumulated)")
    # overwrite mode
    L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | L.MOE_ROUTE_DX_WRITE, torch.from_numpy(d_gate).to(DEV),
                    torch.from_numpy(logits).to(DEV), torch.from_numpy(idx).to(DEV), dev(x), dev(wr), T, H, E, K,
                    CDT[shape.dtype], None, None, dx, ws, nbytes)
    torch.cuda.synchronize()
    assert_close(to64(dx), dx_r, TOL[shape.dtype], "dx (written)")


@pytest.mark.parametrize("shape", SHAPES + ROUTE_ONLY[:1], ids=ids(SHAPES + ROUTE_ONLY[:1]))
def test_route_bwd_renorm_matches_oracle(shape):
    """Backward of renormalised gates: only the chosen logits get a gradient."""
    T, H, E, K = shape.T, shape.H, shape.E, shape.K
    x, wr = synth.router_inputs(shape)
    logits = (x.ref @ wr.ref).astype(np.float32)
    idx = O.topk_experts(logits.astype(np.float64), K)
    d_gate = np.random.default_rng(6).standard_normal((T, K)).astype(np.float32)
    dl_r, dw_r, dx_r = O.route_bwd_softmax_topk(d_gate.astype(np.float64), logits.astype(np.float64), idx,
                                                x.ref, wr.ref, renorm=True)
    dl = torch.empty((T, E), dtype=torch.float32, device=DEV)
    dw = torch.empty((H, E), dtype=torch.float32, device=DEV)
    dx = torch.empty((T, H), dtype=TDT[shape.dtype], device=DEV)
    nbytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, T, H, E, K, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | L.MOE_ROUTE_GATE_RENORM | L.MOE_ROUTE_DX_WRITE,
                    torch.from_numpy(d_gate).to(DEV), torch.from_numpy(logits).to(DEV), torch.from_numpy(idx).to(DEV),
                    dev(x), dev(wr), T, H, E, K, CDT[shape.dtype], dl, dw, dx, ws, nbytes)
    torch.cuda.synchronize()
    dl_g = dl.cpu().numpy()
    assert_close(dl_g, dl_r, 1e-5, "d_logits")
    assert (dl_g[dl_r == 0] == 0).all()
    assert_close(dw.cpu().numpy(), dw_r, 1e-5, "dw_router")
    assert_close(to64(dx), dx_r, TOL[shape.dtype], "dx")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_route_bwd_linear_matches_oracle(dtype):
    T, H = 700, 256
    rng = np.random.default_rng(6)
    x = synth.store(rng.standard_normal((T, H)), dtype)
    w = synth.store(rng.standard_normal(H) / 16, dtype)
    ds = rng.standard_normal(T).astype(np.float32)
    dw_r, dx_r = O.route_bwd_linear(ds.astype(np.float64), x.ref, w.ref)
    nbytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, T, H, 1, 1, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    dw = torch.empty((H,), dtype=torch.float32, device=DEV)
    dx = torch.zeros((T, H), dtype=TDT[dtype], device=DEV)
    L.moe_route_bwd(L.MOE_ROUTE_MOD_LINEAR, torch.from_numpy(ds).to(DEV), None, None, dev(x), dev(w), T, H, 1, 1,
                    CDT[dtype], None, dw, dx, ws, nbytes)
    torch.cuda.synchronize()
    assert_close(dw.cpu().numpy(), dw_r, 1e-5, "dw_mod")
    assert_close(to64(dx), dx_r, TOL[dtype], "dx")


# bf16 routers with 8 or 16 experts take the one-pass streaming backward:
# slices of H with idle threads (H=1536), several slices (H=4096, 6144), fewer
# tokens than CTAs (T=5), several 256-token chunks per CTA (T=40000), ragged
# token ranges everywhere
ROUTE_BWD_STREAM = [(2053, 1536, 8, 2), (1000, 512, 16, 4), (5, 4096, 8, 1), (3001, 4096, 16, 16),
                    (40000, 1024, 8, 2), (777, 6144, 8, 3)]


@pytest.mark.parametrize("T,H,E,K", ROUTE_BWD_STREAM, ids=[f"T{t}_H{h}_E{e}_K{k}" for t, h, e, k in ROUTE_BWD_STREAM])
def test_route_bwd_stream_matches_oracle(T, H, E, K):
    """All outputs together (dx accumulated), then dx alone (written), then dW
    alone, with plain and renormalised gates."""
    shape = S(f"bf16_T{T}_H{H}_E{E}_K{K}", T, H, E, K, 64, "bf16")
    x, wr = synth.router_inputs(shape)
    logits = (x.ref @ wr.ref).astype(np.float32)
    idx = O.topk_experts(logits.astype(np.float64), K)
    d_gate = np.random.default_rng(7).standard_normal((T, K)).astype(np.float32)
    dx0 = synth.store(np.random.default_rng(8).standard_normal((T, H)), "bf16")
    nbytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, T, H, E, K, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    g_d, l_d, i_d = (torch.from_numpy(a).to(DEV) for a in (d_gate, logits, idx))
    x_d, w_d = dev(x), dev(wr)
    for renorm in (False, True):
        dl_r, dw_r, dx_r = O.route_bwd_softmax_topk(d_gate.astype(np.float64), logits.astype(np.float64), idx,
                                                    x.ref, wr.ref, renorm=renorm)
        flags = L.MOE_ROUTE_SOFTMAX_TOPK | (L.MOE_ROUTE_GATE_RENORM if renorm else 0)
        dl = torch.empty((T, E), dtype=torch.float32, device=DEV)
        dw = torch.empty((H, E), dtype=torch.float32, device=DEV)
        dx = dev(dx0).clone()
        L.moe_route_bwd(flags, g_d, l_d, i_d, x_d, w_d, T, H, E, K, L.MOE_BF16, dl, dw, dx, ws, nbytes)
        torch.cuda.synchronize()
        assert_close(dl.cpu().numpy(), dl_r, 1e-5, "d_logits")
        assert_close(dw.cpu().numpy(), dw_r, 1e-5, "dw_router")
        assert_close(to64(dx), dx0.ref + dx_r, TOL["bf16"], "dx (accumulated)")
        dx.fill_(7)
        L.moe_route_bwd(flags | L.MOE_ROUTE_DX_WRITE, g_d, l_d, i_d, x_d, w_d, T, H, E, K, L.MOE_BF16, None, None,
                        dx, ws, nbytes)
        torch.cuda.synchronize()
        assert_close(to64(dx), dx_r, TOL["bf16"], "dx (written)")
        dw.fill_(7)
        L.moe_route_bwd(flags, g_d, l_d, i_d, x_d, w_d, T, H, E, K, L.MOE_BF16, None, dw, None, ws, nbytes)
        torch.cuda.synchronize()
        assert_close(dw.cpu().numpy(), dw_r, 1e-5, "dw_router (alone)")
    assert L.moe_last_device_error() == L.MOE_OK


@pytest.mark.parametrize("T,H", [(20000, 2048), (3, 768), (1000, 4096), (513, 8192)])
def test_route_bwd_linear_stream_matches_oracle(T, H):
    """The MoD score backward (E = 1) on the streaming pass: several rows side by
    side (H=2048), idle threads (H=768), one row per CTA (4096) and two slices
    (8192)."""
    rng = np.random.default_rng(9)
    x = synth.store(rng.standard_normal((T, H)), "bf16")
    w = synth.store(rng.standard_normal(H) / 16, "bf16")
    ds = rng.standard_normal(T).astype(np.float32)
    dx0 = synth.store(rng.standard_normal((T, H)), "bf16")
    dw_r, dx_r = O.route_bwd_linear(ds.astype(np.float64), x.ref, w.ref)
    nbytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, T, H, 1, 1, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    dw = torch.empty((H,), dtype=torch.float32, device=DEV)
    dl = torch.empty((T,), dtype=torch.float32, device=DEV)
    dx = dev(dx0).clone()
    L.moe_route_bwd(L.MOE_ROUTE_MOD_LINEAR, torch.from_numpy(ds).to(DEV), None, None, dev(x), dev(w), T, H, 1, 1,
                    L.MOE_BF16, dl, dw, dx, ws, nbytes)
    torch.cuda.synchronize()
    assert np.array_equal(dl.cpu().numpy(), ds)
    assert_close(dw.cpu().numpy(), dw_r, 1e-5, "dw_mod")
    assert_close(to64(dx), dx0.ref + dx_r.reshape(T, H), TOL["bf16"], "dx (accumulated)")


# all but the last run the one-launch form (the CTAs' rows fit in shared memory;
# (3, 1000) puts sequence boundaries inside CTAs; (4, 8192) gives a CTA 215-216
# rows, more than its eight row groups of 16, so the last group takes the rest);
# rows of H = 8192 do not fit and take the two-launch form
@pytest.mark.parametrize("B,Lseq,C,H,dtype", [(4, 2048, 1024, 128, "bf16"), (3, 1000, 333, 64, "f32"),
                                              (2, 8192, 100, 64, "bf16"), (4, 8192, 3000, 64, "bf16"),
                                              (1, 7, 7, 64, "f32"), (2, 64, 0, 64, "f32"),
                                              (2, 2048, 700, 8192, "bf16")])
def test_mod_select_matches_oracle(B, Lseq, C, H, dtype):
    n = B * Lseq
    x = synth.store(synth.normal(2, 1, n * H).reshape(n, H), dtype)
    w = synth.store(synth.normal(2, 2, H) / math.sqrt(H), dtype)
    score = torch.empty(n, dtype=torch.float32, device=DEV)
    sel = torch.empty(max(B * C, 1), dtype=torch.int32, device=DEV)
    sel_score = torch.empty(max(B * C, 1), dtype=torch.float32, device=DEV)
    mask = torch.empty(n, dtype=torch.uint8, device=DEV)
    x_sel = torch.empty((max(B * C, 1), H), dtype=TDT[dtype], device=DEV)
    y = torch.full((n, H), float("nan"), dtype=TDT[dtype], device=DEV)
    L.mod_select(dev(x), dev(w), B, Lseq, H, C, CDT[dtype], score, sel, sel_score, mask, x_sel, y)
    torch.cuda.synchronize()
    s_ref = O.mod_scores(x.ref, w.ref)
    s_gpu = score.cpu().numpy()
    assert_close(s_gpu, s_ref, 1e-5, "score")
    sel_r, mask_r = O.mod_select(s_ref, B, Lseq, C)
    mask_g = mask.cpu().numpy()
    # exact on the GPU's own scores: the oracle's select run on them
    sel_x, mask_x = O.mod_select(s_gpu.astype(np.float64), B, Lseq, C)
    assert np.array_equal(mask_g, mask_x)
    if C:
        assert np.array_equal(sel.cpu().numpy()[:B * C], (np.arange(B)[:, None] * Lseq + sel_x).reshape(-1))
    n_amb = check_mod_selection(mask_g, mask_r, s_ref, B, Lseq, C, float(np.max(np.abs(s_gpu - s_ref))))
    flat_g = sel.cpu().numpy()[:B * C]
    # whatever was selected: sel lists exactly the masked tokens, ascending per sequence
    assert np.array_equal(np.sort(flat_g), np.nonzero(mask_g)[0])
    if C:
        assert (np.diff(flat_g.reshape(B, C), axis=1) > 0).all()
        assert np.array_equal(sel_score.cpu().numpy()[:B * C], s_gpu[flat_g])
        assert np.array_equal(to64(x_sel)[:B * C], x.ref[flat_g])
    if n_amb == 0 and C:
        flat_r = (np.arange(B)[:, None] * Lseq + sel_r).reshape(-1)
        assert np.array_equal(flat_g, flat_r)
    yv = to64(y)
    keep = mask_g == 0
    assert np.array_equal(yv[keep], x.ref[keep])
    assert np.isnan(yv[~keep]).all()  # selected rows are left for the combine


def check_mod_selection(mask_g, mask_r, s_ref, B, Lseq, C, err):
    """GPU and oracle selections may differ only at near-ties of the C-th score."""
    n = 0
    for b in range(B):
        seg = slice(b * Lseq, (b + 1) * Lseq)
        assert mask_g[seg].sum() == C
        diff = np.nonzero(mask_g[seg] != mask_r[seg])[0]
        if len(diff):
            kth = np.sort(s_ref[seg])[::-1][C - 1]
            assert all(abs(s_ref[b * Lseq + p] - kth) <= 2 * err + 1e-12 for p in diff)
            n += len(diff)
    return n


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_mod_select_integer_scores_select_exactly(dtype):
    """Integer x and w_mod give exact scores with many ties: the capacity top-C
    (tie -> lower position) must match the oracle exactly."""
    B, Lseq, C, H = 3, 1500, 600, 64
    rng = np.random.default_rng(3)
    n = B * Lseq
    x = synth.store(rng.integers(-2, 3, size=(n, H)).astype(np.float64), dtype)
    w = synth.store(rng.integers(-1, 2, size=H).astype(np.float64), dtype)
    score = torch.empty(n, dtype=torch.float32, device=DEV)
    sel = torch.empty(B * C, dtype=torch.int32, device=DEV)
    mask = torch.empty(n, dtype=torch.uint8, device=DEV)
    L.mod_select(dev(x), dev(w), B, Lseq, H, C, CDT[dtype], score, sel, None, mask, None, None)
    torch.cuda.synchronize()
    s_ref = O.mod_scores(x.ref, w.ref)
    assert np.array_equal(score.cpu().numpy().astype(np.float64), s_ref)
    sel_r, mask_r = O.mod_select(s_ref, B, Lseq, C)
    assert np.array_equal(mask.cpu().numpy(), mask_r)
    assert np.array_equal(sel.cpu().numpy(), (np.arange(B)[:, None] * Lseq + sel_r).reshape(-1))


@pytest.mark.parametrize("flags", [0, 1, 3], ids=["plain", "renorm", "renorm_bias_select"])
def test_tiny_fp32_layer_end_to_end(flags):
    """The tiny fp32 layer (T=256, H=128, E=8, K=2, H'=256): forward plus the
    gate/dispatch backward through the C ABI, max relative error <= 1e-5; also
    with the Mixtral-style renormalised gates and a selection-only bias."""
    shape = synth.TINY_F32
    T, H, E, K, Hp = shape.T, shape.H, shape.E, shape.K, shape.Hp
    x, wr, wg, wu, wd = host_layer_inputs(shape)
    dy = synth.upstream_grad(shape, T, H)
    dxs = synth.upstream_grad(shape, T * K, H, seed=2, stream=synth.S_DXS)
    bias = (np.random.default_rng(12).standard_normal(E) * 0.3).astype(np.float32) if flags & 2 else None
    b = layer.MoEBuffers(T, H, E, K, Hp, "f32", DEV)
    xd, wrd = dev(x), dev(wr)
    bd = None if bias is None else torch.from_numpy(bias).to(DEV)
    layer.moe_forward(b, xd, wrd, bd, dev(wg), dev(wu), dev(wd), route_flags=flags)
    layer.moe_backward(b, xd, wrd, dev(dy), dev(dxs), route_flags=flags)
    assert L.moe_last_device_error() == L.MOE_OK
    f = O.moe_forward(x.ref, wr.ref, wg.ref, wu.ref, wd.ref, K, None if bias is None else bias.astype(np.float64),
                      renorm=bool(flags & 1), bias_select_only=bool(flags & 2))
    g = O.moe_backward(f, dy.ref, dxs.ref, x.ref, wr.ref, renorm=bool(flags & 1))
    assert np.array_equal(b.idx.cpu().numpy(), f["idx"])
    assert np.array_equal(b.cu.cpu().numpy(), f["cu"])
    assert np.array_equal(b.dst_row.cpu().numpy(), f["dst_row"])
    assert np.array_equal(b.src_tok.cpu().numpy(), f["src_tok"])
    for name, gpu, ref in [("logits", b.logits, f["logits"]), ("gate", b.gate, f["gate"]), ("act", b.act, f["act"]),
                           ("h", b.h, f["h"]), ("y", b.y, f["y"]), ("dh", b.dh, g["dh"]),
                           ("d_gate", b.d_gate, g["d_gate"]), ("d_logits", b.d_logits, g["d_logits"]),
                           ("dw_router", b.dw_router, g["dw_router"]), ("dx", b.dx, g["dx"])]:
        assert_close(to64(gpu), ref, 1e-5, name)


def test_outputs_are_deterministic():
    shape = SHAPES[1]
    x, wr, wg, wu, wd = host_layer_inputs(shape)
    outs = []
    for _ in range(2):
        b = layer.MoEBuffers(shape.T, shape.H, shape.E, shape.K, shape.Hp, shape.dtype, DEV)
        xd, wrd = dev(x), dev(wr)
        layer.moe_forward(b, xd, wrd, None, dev(wg), dev(wu), dev(wd))
        dy = dev(synth.upstream_grad(shape, shape.T, shape.H))
        dxs = dev(synth.upstream_grad(shape, shape.R, shape.H, seed=2, stream=synth.S_DXS))
        layer.moe_backward(b, xd, wrd, dy, dxs)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (b.logits, b.idx, b.dst_row, b.act, b.h, b.y, b.dx, b.dw_router)])
    for a, c in zip(*outs):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                           c.view(torch.uint8) if c.dtype == torch.bfloat16 else c)


def test_zero_tokens_is_a_no_op():
    E, K, H = 8, 2, 64
    cu = torch.full((E + 1,), -5, dtype=torch.int32, device=DEV)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    w = torch.zeros((E, H, 64), dtype=torch.float32, device=DEV)
    L.moe_dispatch(None, None, 0, H, E, K, L.MOE_F32, cu, None, None, None, ws, 256)
    assert (cu.cpu() == 0).all()
    L.moe_route(None, torch.zeros((H, E), device=DEV), None, 0, H, E, K, L.MOE_F32, None, None, None)
    L.moe_combine(None, None, None, None, None, None, 0, H, K, L.MOE_F32, None)
    L.moe_expert_ffn(None, cu, 0, w, w, w, E, H, 64, L.MOE_F32, None, None)
    # the router backward of no tokens: dW_r is all zeros, on both bf16 designs
    # (the one-pass stream for E = 8, the tensor-core GEMMs for E = 64) and fp32
    for E_, dt in [(8, L.MOE_BF16), (64, L.MOE_BF16), (8, L.MOE_F32)]:
        nb = L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, 0, H, E_, K, 0)
        wsb = torch.empty(max(nb, 256), dtype=torch.uint8, device=DEV)
        dw = torch.full((H, E_), 7.0, device=DEV)
        L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK, None, None, None, None, None, 0, H, E_, K, dt, None, dw, None,
                        wsb, nb)
        torch.cuda.synchronize()
        assert (dw.cpu() == 0).all()
    assert L.moe_last_device_error() == L.MOE_OK


def test_bounded_wait_times_out_and_the_context_survives():
    """Failure detection without a fault: a kernel waits on a barrier nothing
    arrives at; its bounded wait gives up after ~1 ms, the device error word
    reports MOE_ERR_TIMEOUT, reading it clears it, and the next calls run."""
    assert L.moe_last_device_error() == L.MOE_OK
    L.moe_check_wait_timeout(2_000_000)
    assert L.moe_last_device_error() == L.MOE_ERR_TIMEOUT
    assert L.moe_last_device_error() == L.MOE_OK
    shape = SHAPES[1]
    x, wr = synth.router_inputs(shape)
    logits, idx, gate = route_gpu(shape, x, wr)
    r_logits = O.router_logits(x.ref, wr.ref)
    assert_close(logits, r_logits, 1e-5, "logits after the timeout")
    assert L.moe_last_device_error() == L.MOE_OK
