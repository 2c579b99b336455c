"""GPU parity of the expert FFN backward through the C ABI: moe_expert_ffn_ex
(which also keeps the SwiGLU pre-activations g and u) and moe_expert_ffn_bwd,
against the oracle's expert_ffn / expert_ffn_bwd on the same bf16-rounded
inputs.  Row counts per expert are ragged: empty experts, a single row, exact
and inexact multiples of the 64-row K block of the weight-gradient GEMMs, H'
that is not a multiple of the 256-wide N tile, and experts whose last 256-row
tile of a CTA pair holds at most 128 rows (the peer CTA's rows all past the
expert's end, 64 or 128 exactly)."""
import numpy as np
import pytest
import torch

import oracle as O
from token_dispatch_gb300 import _lib as L
from token_dispatch_gb300 import synth
from tests.gpu_util import DEV, assert_close, dev, to64

pytestmark = pytest.mark.gpu

TOL = 2e-2  # bf16 storage of the inputs, of g/u, act and of dg/du; fp32 accumulation

CASES = [
    (4, 128, 192, [70, 0, 130, 33]),
    (3, 256, 128, [1, 64, 200]),
    (8, 128, 256, [0, 0, 0, 300, 0, 0, 0, 5]),
    (2, 192, 320, [129, 127]),
    (6, 128, 320, [1, 63, 64, 65, 128, 356]),
    (2, 256, 192, [384, 200]),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from token_dispatch_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def inputs(E, H, Hp, counts, seed):
    rng = np.random.default_rng(seed)
    R = int(sum(counts))
    cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    xs = synth.store(rng.standard_normal((R, H)), "bf16")
    wg = synth.store(rng.standard_normal((E, H, Hp)) / np.sqrt(H), "bf16")
    wu = synth.store(rng.standard_normal((E, H, Hp)) / np.sqrt(H), "bf16")
    wd = synth.store(rng.standard_normal((E, H, Hp)) / np.sqrt(Hp), "bf16")
    dh = synth.store(rng.standard_normal((R, H)), "bf16")
    return R, cu, xs, wg, wu, wd, dh


@pytest.mark.parametrize("E,H,Hp,counts", CASES, ids=[f"E{c[0]}_H{c[1]}_Hp{c[2]}" for c in CASES])
def test_expert_ffn_backward_matches_oracle(E, H, Hp, counts):
    R, cu, xs, wg, wu, wd, dh = inputs(E, H, Hp, counts, seed=E * 1000 + H)
    cu_d = torch.from_numpy(cu).to(DEV)
    act = torch.empty((R, Hp), dtype=torch.bfloat16, device=DEV)
    gu = torch.empty((R, 2 * Hp), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    L.moe_expert_ffn_ex(dev(xs), cu_d, R, dev(wg), dev(wu), dev(wd), E, H, Hp, L.MOE_BF16, act, gu, h)
    torch.cuda.synchronize()
    act_r, h_r = O.expert_ffn(xs.ref, cu, wg.ref, wu.ref, wd.ref)
    e_of = O.expert_of_row(cu, np.arange(R))
    g_r = np.einsum("rh,rhj->rj", xs.ref, wg.ref[e_of])
    u_r = np.einsum("rh,rhj->rj", xs.ref, wu.ref[e_of])
    gu_g = to64(gu)
    assert_close(gu_g[:, :Hp], g_r, TOL, "g")
    assert_close(gu_g[:, Hp:], u_r, TOL, "u")
    assert_close(to64(act), act_r, TOL, "act")
    assert_close(to64(h), h_r, TOL, "h")

    dxs = torch.full((R, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    dws = [torch.full((E, H, Hp), float("nan"), dtype=torch.float32, device=DEV) for _ in range(3)]
    nbytes = L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN_BWD, R, H, E, 1, Hp)
    assert nbytes >= R * 2 * Hp * 2
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=DEV)
    L.moe_expert_ffn_bwd(dev(xs), cu_d, R, dev(wg), dev(wu), dev(wd), E, H, Hp, L.MOE_BF16, gu, act, dev(dh), dxs,
                         dws[0], dws[1], dws[2], ws, nbytes)
    assert L.moe_last_device_error() == L.MOE_OK
    dxs_r, dwg_r, dwu_r, dwd_r = O.expert_ffn_bwd(xs.ref, cu, wg.ref, wu.ref, wd.ref, dh.ref)
    assert_close(to64(dxs), dxs_r, TOL, "dxs")
    for name, got, ref in [("dw_gate", dws[0], dwg_r), ("dw_up", dws[1], dwu_r), ("dw_down", dws[2], dwd_r)]:
        g = got.cpu().numpy().astype(np.float64)
        assert not np.isnan(g).any(), name
        for e in range(E):
            if counts[e] == 0:
                assert (g[e] == 0).all(), (name, e)
        assert_close(g, ref, TOL, name)


def test_expert_ffn_backward_alignment_of_saved_activations():
    """[g | u] and the workspace at 16-byte but not 32-byte aligned addresses
    (the SwiGLU backward then moves them as 16-byte vectors instead of 32-byte
    ones): the same bits as with 256-byte aligned buffers."""
    E, H, Hp, counts = 4, 128, 192, [70, 0, 130, 33]
    R, cu, xs, wg, wu, wd, dh = inputs(E, H, Hp, counts, seed=11)
    cu_d = torch.from_numpy(cu).to(DEV)
    nbytes = L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN_BWD, R, H, E, 1, Hp)
    outs = []
    for off in (0, 8):  # bf16 elements: 0 or 16 bytes past a 256-byte aligned base
        act = torch.empty((R, Hp), dtype=torch.bfloat16, device=DEV)
        gu_buf = torch.empty(R * 2 * Hp + 16, dtype=torch.bfloat16, device=DEV)
        gu = gu_buf[off:off + R * 2 * Hp].view(R, 2 * Hp)
        h = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
        L.moe_expert_ffn_ex(dev(xs), cu_d, R, dev(wg), dev(wu), dev(wd), E, H, Hp, L.MOE_BF16, act, gu, h)
        ws_buf = torch.empty(nbytes + 64, dtype=torch.uint8, device=DEV)
        ws = ws_buf[2 * off:2 * off + nbytes]
        dxs = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
        dws = [torch.empty((E, H, Hp), dtype=torch.float32, device=DEV) for _ in range(3)]
        L.moe_expert_ffn_bwd(dev(xs), cu_d, R, dev(wg), dev(wu), dev(wd), E, H, Hp, L.MOE_BF16, gu, act, dev(dh),
                             dxs, dws[0], dws[1], dws[2], ws, nbytes)
        torch.cuda.synchronize()
        assert L.moe_last_device_error() == L.MOE_OK
        outs.append((dxs, dws))
    (dxs0, dws0), (dxs1, dws1) = outs
    assert torch.equal(dxs0, dxs1)
    for a_, b_ in zip(dws0, dws1):
        assert torch.equal(a_, b_)


def test_expert_ffn_backward_without_rows_zeroes_weight_gradients():
    E, H, Hp = 3, 128, 128
    z = torch.zeros(1, dtype=torch.bfloat16, device=DEV)
    cu = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    w = torch.zeros((E, H, Hp), dtype=torch.bfloat16, device=DEV)
    dws = [torch.full((E, H, Hp), float("nan"), dtype=torch.float32, device=DEV) for _ in range(3)]
    L.moe_expert_ffn_bwd(z, cu, 0, w, w, w, E, H, Hp, L.MOE_BF16, z, z, z, None, dws[0], dws[1], dws[2], None, 0)
    torch.cuda.synchronize()
    for d in dws:
        assert (d == 0).all()


FULL = [synth.MIXTRAL_BF16, synth.FINEGRAINED_BF16]


@pytest.mark.parametrize("shape", FULL, ids=[s.name for s in FULL])
def test_full_workload_training_backward_sampled(shape):
    """The whole training backward of a full-size layer in the benchmark's launch
    configuration (layer.moe_forward with g/u kept, layer.moe_train_backward), on
    the oracle's routing; the oracle recomputes sampled rows of dxs and sampled
    elements of the three weight gradients one by one."""
    from token_dispatch_gb300 import layer
    T, H, E, K, Hp = shape.T, shape.H, shape.E, shape.K, shape.Hp
    R = T * K
    rng = np.random.default_rng(3)
    x, wr = synth.router_inputs(shape)
    wg, wu, wd = synth.expert_weights_device(shape, DEV)
    r_idx = O.topk_experts(O.router_logits(x.ref, wr.ref), K)
    cu, dst, src = O.permutation(r_idx, E)
    b = layer.MoEBuffers(T, H, E, K, Hp, "bf16", DEV, backward=True, train=True)
    xd = x.host.to(DEV)
    # forward on the oracle's choice of experts (gates: the GPU's own)
    layer.moe_forward(b, xd, wr.host.to(DEV), None, wg, wu, wd)
    L.moe_dispatch(xd, torch.from_numpy(r_idx).to(DEV), T, H, E, K, L.MOE_BF16, b.cu, b.dst_row, b.src_tok, b.xs,
                   b.ws_dispatch, b.ws_dispatch_bytes)
    L.moe_expert_ffn_ex(b.xs, b.cu, R, wg, wu, wd, E, H, Hp, L.MOE_BF16, b.act, b.gu, b.h)
    dh = synth.upstream_grad(shape, R, H, seed=4)
    b.dh.copy_(dh.host.to(DEV))
    L.moe_expert_ffn_bwd(b.xs, b.cu, R, wg, wu, wd, E, H, Hp, L.MOE_BF16, b.gu, b.act, b.dh, b.dxs, b.dw_gate,
                         b.dw_up, b.dw_down, b.ws_ffn_bwd, b.ws_ffn_bwd_bytes)
    assert L.moe_last_device_error() == L.MOE_OK
    assert np.array_equal(b.cu.cpu().numpy(), cu)
    assert np.array_equal(b.dst_row.cpu().numpy(), dst)

    xs_rows = x.ref[src]  # the oracle's dispatched rows
    dxs_g = to64(b.dxs)
    got = {"dg": [], "du": [], "dd": []}
    ref = {"dg": [], "du": [], "dd": []}
    dxs_got, dxs_ref = [], []
    for e in sorted({0, E // 2, E - 1}):
        lo, hi = int(cu[e]), int(cu[e + 1])
        if hi == lo:
            continue
        wg_e, wu_e, wd_e = (synth.weights_to_host(w, [e])[0] for w in (wg, wu, wd))
        X, D = xs_rows[lo:hi], dh.ref[lo:hi]
        # dxs on sampled rows of e
        rows = np.unique(np.r_[lo, hi - 1, rng.integers(lo, hi, size=6)]) - lo
        dx_r = O.expert_swiglu_bwd(X[rows], wg_e, wu_e, wd_e, D[rows])[0]
        dxs_got.append(dxs_g[lo + rows])
        dxs_ref.append(dx_r)
        # weight gradients on sampled (h, j): the column j of g, u, da over all rows of e
        hs, js = rng.integers(0, H, size=12), rng.integers(0, Hp, size=12)
        for h_, j_ in zip(hs, js):
            g = X @ wg_e[:, j_]
            u = X @ wu_e[:, j_]
            s = 1.0 / (1.0 + np.exp(-g))
            da = D @ wd_e[:, j_]
            dg = da * u * s * (1.0 + g * (1.0 - s))
            du = da * g * s
            ref["dg"].append(X[:, h_] @ dg)
            ref["du"].append(X[:, h_] @ du)
            ref["dd"].append(D[:, h_] @ (g * s * u))
            got["dg"].append(float(b.dw_gate[e, h_, j_]))
            got["du"].append(float(b.dw_up[e, h_, j_]))
            got["dd"].append(float(b.dw_down[e, h_, j_]))
    assert_close(np.concatenate(dxs_got), np.concatenate(dxs_ref), TOL, "dxs (sampled rows)")
    for k, name in [("dg", "dw_gate"), ("du", "dw_up"), ("dd", "dw_down")]:
        assert_close(np.array(got[k]), np.array(ref[k]), TOL, name + " (sampled)")


def test_layer_training_step_end_to_end():
    """layer.moe_forward + layer.moe_train_backward on a small bf16 layer against
    the oracle chain: forward, permute_bwd (dh, d_gate), expert_ffn_bwd (dxs and
    the weight gradients), then the dispatch adjoint and the router backward."""
    from tests.gpu_util import host_layer_inputs
    from token_dispatch_gb300 import layer
    shape = synth.MoEShape("bf16_T1000_H384_E16_K4_Hp320", 1000, 384, 16, 4, 320, "bf16")
    T, H, E, K, Hp = shape.T, shape.H, shape.E, shape.K, shape.Hp
    x, wr, wg, wu, wd = host_layer_inputs(shape)
    dy = synth.upstream_grad(shape, T, H)
    b = layer.MoEBuffers(T, H, E, K, Hp, "bf16", DEV, backward=True, train=True)
    xd, wrd = dev(x), dev(wr)
    wgd, wud, wdd = dev(wg), dev(wu), dev(wd)
    layer.moe_forward(b, xd, wrd, None, wgd, wud, wdd)
    layer.moe_train_backward(b, xd, wrd, wgd, wud, wdd, dev(dy))
    assert L.moe_last_device_error() == L.MOE_OK
    f = O.moe_forward(x.ref, wr.ref, wg.ref, wu.ref, wd.ref, K)
    assert np.array_equal(b.idx.cpu().numpy(), f["idx"])
    dh_r, d_gate_r, _, _ = O.permute_bwd(dy.ref, f["h"], f["gate"], f["dst_row"])
    dxs_r, dwg_r, dwu_r, dwd_r = O.expert_ffn_bwd(f["xs"], f["cu"], wg.ref, wu.ref, wd.ref, dh_r)
    g = O.moe_backward(f, dy.ref, dxs_r, x.ref, wr.ref)
    for name, gpu, ref, tol in [("dh", b.dh, dh_r, TOL), ("d_gate", b.d_gate, d_gate_r, TOL),
                                ("dxs", b.dxs, dxs_r, TOL), ("dw_gate", b.dw_gate, dwg_r, TOL),
                                ("dw_up", b.dw_up, dwu_r, TOL), ("dw_down", b.dw_down, dwd_r, TOL),
                                ("dx", b.dx, g["dx"], TOL), ("dw_router", b.dw_router, g["dw_router"], TOL)]:
        assert_close(to64(gpu), ref, tol, name)
