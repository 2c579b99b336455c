"""Parity at the full layer workloads, in the launch configuration the benchmark
times: the Mixtral-shaped layer (T=8192, H=4096, E=8, K=2, H'=14336), the
fine-grained layer (T=16384, H=2048, E=64, K=6, H'=1408), the expert-parallel
benchmark shapes on one GPU (T=8192, E=384, H=7168, K=8, H'=2048) and the
MoD + MoE layer (4 x 2048 tokens, 50% capacity, E=16, K=2, H'=5632).

Checked exactly: top-k indices (up to genuine near-ties), cu_seqlens, the
permutation, the dispatched rows, the MoD selection, and the expert FFN with
the dispatch gather fused into its operand load against the FFN on the
dispatched rows (bit for bit).  Checked on every output
element: router logits and gates, combine, gate/dispatch backward.  Checked on
sampled rows (the oracle computes them one by one): the expert FFN (first, last
and random rows of sampled experts) and the layer output y of sampled tokens."""
import numpy as np
import pytest
import torch

import oracle as O
from token_dispatch_gb300 import _lib as L
from token_dispatch_gb300 import layer, synth
from tests.gpu_util import DEV, TDT, assert_close, check_topk, check_topk_exact, gate_tol, near_tie_rows, to64
from tests.test_gpu_kernels import check_mod_selection

pytestmark = pytest.mark.gpu

WL = [synth.MIXTRAL_BF16, synth.FINEGRAINED_BF16, synth.EPBENCH_BF16]
# Rows whose GPU top-K differs from the float64 top-K on these seeds.  The GPU
# selects exactly on its own fp32 logits (asserted); a row can still differ from
# the float64 selection where its K-th and (K+1)-th logits lie within the fp32
# accumulation error.  Over H = 7168 that error reaches 9e-5 and one of the
# E=384 layer's 8192 rows is such a tie; the other workloads have none.
AMBIGUOUS_ROWS = {synth.MIXTRAL_BF16.name: 0, synth.FINEGRAINED_BF16.name: 0, synth.EPBENCH_BF16.name: 1}
BWD = {synth.MIXTRAL_BF16.name, synth.FINEGRAINED_BF16.name}


@pytest.fixture(scope="module", autouse=True)
def built():
    from token_dispatch_gb300 import build
    build.build()


def sample_rows(cu, experts, rng, n_rand=16):
    rows = []
    for e in experts:
        lo, hi = int(cu[e]), int(cu[e + 1])
        if hi > lo:
            rows += [lo, hi - 1] + rng.integers(lo, hi, size=min(n_rand, hi - lo)).tolist()
    return np.unique(np.array(rows, np.int64))


@pytest.mark.parametrize("shape", WL, ids=[s.name for s in WL])
def test_full_workload_forward_and_backward(shape):
    T, H, E, K, Hp = shape.T, shape.H, shape.E, shape.K, shape.Hp
    R = T * K
    rng = np.random.default_rng(0)
    x, wr = synth.router_inputs(shape)
    wg, wu, wd = synth.expert_weights_device(shape, DEV)
    xd, wrd = x.host.to(DEV), wr.host.to(DEV)
    b = layer.MoEBuffers(T, H, E, K, Hp, "bf16", DEV, backward=shape.name in BWD)

    # ---- full GPU forward, as the benchmark runs it
    layer.moe_forward(b, xd, wrd, None, wg, wu, wd)
    assert L.moe_last_device_error() == L.MOE_OK

    # ---- router: every logit, indices up to near-ties, gates
    r_logits, r_p, r_idx, r_gate = O.route(x.ref, wr.ref, K)
    g_logits = b.logits.cpu().numpy()
    assert_close(g_logits, r_logits, 1e-5, "logits")
    g_idx = b.idx.cpu().numpy()
    logit_err = float(np.max(np.abs(g_logits - r_logits)))
    check_topk_exact(g_idx, g_logits, K)
    n_amb = check_topk(g_idx, r_logits, K, logit_err)
    n_near = near_tie_rows(r_logits, K, logit_err)
    print(f"{shape.name}: rows differing from the fp64 selection {n_amb}, "
          f"near-tie rows (K-th/K+1-th gap < 4x logit error {logit_err:.2e}) {n_near}")
    # every differing row is a genuine near-tie (checked above); their count on
    # these seeds is pinned so that a change shows
    assert n_amb == AMBIGUOUS_ROWS[shape.name], f"{n_amb} rows differ from the fp64 selection"
    same = (g_idx == r_idx).all(axis=1)
    assert_close(b.gate.cpu().numpy()[same], r_gate[same], gate_tol(logit_err), "gate")

    # ---- dispatch on the oracle's indices: bit-exact
    cu, dst, src, _ = O.dispatch(np.zeros((T, 1)), r_idx, E)
    b2 = layer.MoEBuffers(T, H, E, K, Hp, "bf16", DEV, backward=False)
    L.moe_dispatch(xd, torch.from_numpy(r_idx).to(DEV), T, H, E, K, L.MOE_BF16, b2.cu, b2.dst_row, b2.src_tok,
                   b2.xs, b2.ws_dispatch, b2.ws_dispatch_bytes)
    assert np.array_equal(b2.cu.cpu().numpy(), cu)
    assert np.array_equal(b2.dst_row.cpu().numpy(), dst)
    assert np.array_equal(b2.src_tok.cpu().numpy(), src)
    rows_chk = rng.integers(0, R, size=512)
    assert np.array_equal(to64(b2.xs[torch.from_numpy(rows_chk).to(DEV)]), x.ref[src[rows_chk]])
    # the layer's own dispatch, of its own indices: bit-exact
    cu_g, dst_g, src_g = O.permutation(g_idx, E)
    assert np.array_equal(b.cu.cpu().numpy(), cu_g)
    assert np.array_equal(b.dst_row.cpu().numpy(), dst_g)
    assert np.array_equal(b.src_tok.cpu().numpy(), src_g)

    # ---- expert FFN on sampled rows of sampled experts (same routing as the oracle)
    L.moe_expert_ffn(b2.xs, b2.cu, R, wg, wu, wd, E, H, Hp, L.MOE_BF16, b2.act, b2.h)
    torch.cuda.synchronize()
    experts = sorted(set([0, E - 1] + rng.choice(E, size=min(E, 6), replace=False).tolist()))
    rows = sample_rows(cu, experts, rng)
    e_of = O.expert_of_row(cu, rows)
    act_g = to64(b2.act[torch.from_numpy(rows).to(DEV)])
    h_g = to64(b2.h[torch.from_numpy(rows).to(DEV)])
    act_r = np.zeros_like(act_g)
    h_r = np.zeros_like(h_g)
    for e in experts:
        sel = e_of == e
        if not sel.any():
            continue
        we = [synth.weights_to_host(w, [e])[0] for w in (wg, wu, wd)]
        act_r[sel], h_r[sel] = O.expert_swiglu(x.ref[src[rows[sel]]], *we)
    assert_close(act_g, act_r, 2e-2, "act (sampled rows)")
    assert_close(h_g, h_r, 2e-2, "h (sampled rows)")
    # the dispatch gather fused into the gate/up operand load (index maps only,
    # rows read from x by src_tok): bit for bit the FFN on the dispatched rows
    cu3 = torch.empty_like(b2.cu)
    dst3 = torch.empty_like(b2.dst_row)
    src3 = torch.empty_like(b2.src_tok)
    L.moe_dispatch(xd, torch.from_numpy(r_idx).to(DEV), T, H, E, K, L.MOE_BF16, cu3, dst3, src3, None,
                   b2.ws_dispatch, b2.ws_dispatch_bytes)
    act3 = torch.empty_like(b2.act)
    h3 = torch.empty_like(b2.h)
    L.moe_expert_ffn_gather(xd, src3, T, cu3, R, wg, wu, wd, E, H, Hp, L.MOE_BF16, act3, None, h3)
    torch.cuda.synchronize()
    assert L.moe_last_device_error() == L.MOE_OK
    assert torch.equal(act3, b2.act) and torch.equal(h3, b2.h)
    del act3, h3

    # ---- layer output y of sampled tokens: sum_k gate * expert(x)
    toks = rng.choice(np.nonzero(same)[0], size=24 if E <= 64 else 6, replace=False)
    y_r = np.zeros((len(toks), H))
    cache = {}
    for i, t in enumerate(toks):
        for k in range(K):
            e = int(r_idx[t, k])
            if e not in cache:
                cache[e] = [synth.weights_to_host(w, [e])[0] for w in (wg, wu, wd)]
            _, hr = O.expert_swiglu(x.ref[t:t + 1], *cache[e])
            y_r[i] += r_gate[t, k] * hr[0]
        if len(cache) > 12:
            cache.clear()
    y_g = to64(b.y[torch.from_numpy(toks).to(DEV)])
    assert_close(y_g, y_r, 2e-2, "y (sampled tokens)")

    if shape.name not in BWD:
        return
    # ---- backward on every element, with synthetic h / dy / dxs inputs
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    hs = torch.randn((R, H), generator=g, device=DEV).to(torch.bfloat16)
    dy = torch.randn((T, H), generator=g, device=DEV).to(torch.bfloat16)
    dxs = torch.randn((R, H), generator=g, device=DEV).to(torch.bfloat16)
    gate32 = r_gate.astype(np.float32)
    L.moe_permute_bwd(dy, hs, torch.from_numpy(gate32).to(DEV), torch.from_numpy(dst).to(DEV), None, None, dxs,
                      T, H, K, L.MOE_BF16, b.dh, b.d_gate, None, b.dx)
    torch.cuda.synchronize()
    hs64, dy64, dxs64 = to64(hs), to64(dy), to64(dxs)
    dh_r, dg_r, _, dx_r = O.permute_bwd(dy64, hs64, gate32.astype(np.float64), dst, dxs64)
    assert_close(to64(b.dh), dh_r, 2e-2, "dh")
    assert_close(b.d_gate.cpu().numpy(), dg_r, 1e-5, "d_gate")
    assert_close(to64(b.dx), dx_r, 2e-2, "dx (dispatch part)")

    dgate = rng.standard_normal((T, K)).astype(np.float32)
    logits32 = r_logits.astype(np.float32)
    dl_r, dw_r, dxr_r = O.route_bwd_softmax_topk(dgate.astype(np.float64), logits32.astype(np.float64), r_idx,
                                                 x.ref, wr.ref)
    L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | L.MOE_ROUTE_DX_WRITE, torch.from_numpy(dgate).to(DEV),
                    torch.from_numpy(logits32).to(DEV), torch.from_numpy(r_idx).to(DEV), xd, wrd, T, H, E, K,
                    L.MOE_BF16, b.d_logits, b.dw_router, b.dx, b.ws_bwd, b.ws_bwd_bytes)
    torch.cuda.synchronize()
    assert_close(b.d_logits.cpu().numpy(), dl_r, 1e-5, "d_logits")
    assert_close(b.dw_router.cpu().numpy(), dw_r, 1e-5, "dw_router")
    assert_close(to64(b.dx), dxr_r, 2e-2, "dx (router part)")


def test_mod_workload_forward_and_route_backward():
    """MoD + MoE: 4 x 2048 tokens, capacity 1024 per sequence, E=16, K=2, H'=5632."""
    shape = synth.MOD_BF16
    B, Lq, C, H, E, K, Hp = shape.mod_B, shape.mod_L, shape.mod_C, shape.H, shape.E, shape.K, shape.Hp
    n = B * Lq
    rng = np.random.default_rng(1)
    x, wr = synth.router_inputs(shape, tokens=n)
    wmod = synth.mod_weight(shape)
    wg, wu, wd = synth.expert_weights_device(shape, DEV)
    xd = x.host.to(DEV)
    m = layer.MoDBuffers(B, Lq, C, H, E, K, Hp, "bf16", DEV)
    layer.mod_forward(m, xd, wmod.host.to(DEV), wr.host.to(DEV), wg, wu, wd)
    assert L.moe_last_device_error() == L.MOE_OK

    s_g = m.score.cpu().numpy()
    s_r = O.mod_scores(x.ref, wmod.ref)
    assert_close(s_g, s_r, 1e-5, "score")
    sel_o, mask_o = O.mod_select(s_r, B, Lq, C)
    # exact on the GPU's own scores
    sel_x, mask_x = O.mod_select(s_g.astype(np.float64), B, Lq, C)
    assert np.array_equal(m.mask.cpu().numpy(), mask_x)
    assert np.array_equal(m.sel.cpu().numpy(), (np.arange(B)[:, None] * Lq + sel_x).reshape(-1))
    err = float(np.max(np.abs(s_g - s_r)))
    n_amb = check_mod_selection(m.mask.cpu().numpy(), mask_o, s_r, B, Lq, C, err)
    assert n_amb == 0, f"{n_amb} near-tie positions"
    flat = (np.arange(B)[:, None] * Lq + sel_o).reshape(-1)
    assert np.array_equal(m.sel.cpu().numpy(), flat)
    assert np.array_equal(to64(m.x_sel), x.ref[flat])

    # unselected rows pass through unchanged
    keep = np.nonzero(mask_o == 0)[0]
    pick = rng.choice(keep, 256, replace=False)
    assert np.array_equal(to64(m.y[torch.from_numpy(pick).to(DEV)]), x.ref[pick])

    # selected rows: y = x + s * MoE(x) on sampled tokens (oracle routing of x_sel)
    xs_ref = x.ref[flat]
    r_logits, _, r_idx, r_gate = O.route(xs_ref, wr.ref, K)
    g_logits = m.moe.logits.cpu().numpy()
    logit_err = float(np.max(np.abs(g_logits - r_logits)))
    check_topk_exact(m.moe.idx.cpu().numpy(), g_logits, K)
    n_amb = check_topk(m.moe.idx.cpu().numpy(), r_logits, K, logit_err)
    print(f"MoD experts: rows differing from the fp64 selection {n_amb}, "
          f"near-tie rows {near_tie_rows(r_logits, K, logit_err)}")
    assert n_amb == 0, f"{n_amb} rows differ from the fp64 selection"
    same = (m.moe.idx.cpu().numpy() == r_idx).all(axis=1)
    toks = rng.choice(np.nonzero(same)[0], 16, replace=False)
    cache = {}
    y_r = np.zeros((len(toks), H))
    for i, j in enumerate(toks):
        acc = np.zeros(H)
        for k in range(K):
            e = int(r_idx[j, k])
            if e not in cache:
                cache[e] = [synth.weights_to_host(w, [e])[0] for w in (wg, wu, wd)]
            _, hr = O.expert_swiglu(xs_ref[j:j + 1], *cache[e])
            acc += r_gate[j, k] * hr[0]
        y_r[i] = x.ref[flat[j]] + s_r[flat[j]] * acc
    y_g = to64(m.y[torch.from_numpy(flat[toks]).to(DEV)])
    assert_close(y_g, y_r, 2e-2, "y (selected, sampled)")

    # route backward with the expert outputs held fixed, on inputs both sides
    # share: synthetic expert rows h, the oracle's gates, rows and scores
    Ts = B * C
    g = torch.Generator(device=DEV)
    g.manual_seed(3)
    hs = torch.randn((Ts * K, H), generator=g, device=DEV).to(torch.bfloat16)
    dy = torch.randn((n, H), generator=g, device=DEV).to(torch.bfloat16)
    _, dst_r, _ = O.permutation(r_idx, E)
    s_sel = s_r[flat].astype(np.float32)
    gate32 = r_gate.astype(np.float32)
    d_score = torch.empty(Ts, dtype=torch.float32, device=DEV)
    d_gate = torch.empty((Ts, K), dtype=torch.float32, device=DEV)
    L.moe_permute_bwd(dy, hs, torch.from_numpy(gate32).to(DEV), torch.from_numpy(dst_r).to(DEV),
                      torch.from_numpy(s_sel).to(DEV), torch.from_numpy(flat.astype(np.int32)).to(DEV), None,
                      Ts, H, K, L.MOE_BF16, None, d_gate, d_score, None)
    dw_mod = torch.empty(H, dtype=torch.float32, device=DEV)
    dx_sel = torch.zeros((Ts, H), dtype=torch.bfloat16, device=DEV)
    L.moe_route_bwd(L.MOE_ROUTE_MOD_LINEAR, d_score, None, None, m.x_sel, wmod.host.to(DEV), Ts, H, 1, 1,
                    L.MOE_BF16, None, dw_mod, dx_sel, m.ws_lin, m.ws_lin_bytes)
    torch.cuda.synchronize()
    _, dg_r, ds_r, _ = O.permute_bwd(to64(dy), to64(hs), gate32.astype(np.float64), dst_r, None,
                                     row_scale=s_sel.astype(np.float64), out_row=flat)
    assert_close(d_score.cpu().numpy(), ds_r, 1e-5, "d_score")
    assert_close(d_gate.cpu().numpy(), dg_r, 1e-5, "d_gate")
    dw_mod_r, dx_r = O.route_bwd_linear(ds_r, xs_ref, wmod.ref)
    assert_close(dw_mod.cpu().numpy(), dw_mod_r, 1e-5, "dw_mod")
    assert_close(to64(dx_sel), dx_r, 2e-2, "dx (MoD router)")
    # the composed backward of the layer, as the benchmark runs it on the
    # forward's own buffers, element by element against the oracle fed those
    # same buffers (h, gates, rows, scores, logits, indices, selected rows)
    layer.mod_route_backward(m, wr.host.to(DEV), wmod.host.to(DEV), dy)
    assert L.moe_last_device_error() == L.MOE_OK
    mb = m.moe
    h64, gate64, dst_g = to64(mb.h), mb.gate.cpu().numpy().astype(np.float64), mb.dst_row.cpu().numpy()
    ssel64, sel_g = m.sel_score.cpu().numpy().astype(np.float64), m.sel.cpu().numpy()
    xsel64 = to64(m.x_sel)
    dh_c, dg_c, ds_c, _ = O.permute_bwd(to64(dy), h64, gate64, dst_g, None, row_scale=ssel64, out_row=sel_g)
    dl_c, dwr_c, dxr_c = O.route_bwd_softmax_topk(dg_c, mb.logits.cpu().numpy().astype(np.float64),
                                                  mb.idx.cpu().numpy(), xsel64, wr.ref)
    dwm_c, dxm_c = O.route_bwd_linear(ds_c, xsel64, wmod.ref)
    assert_close(to64(mb.dh), dh_c, 2e-2, "composed dh")
    assert_close(mb.d_gate.cpu().numpy(), dg_c, 1e-5, "composed d_gate")
    assert_close(m.d_score.cpu().numpy(), ds_c, 1e-5, "composed d_score")
    assert_close(mb.d_logits.cpu().numpy(), dl_c, 1e-5, "composed d_logits")
    assert_close(mb.dw_router.cpu().numpy(), dwr_c, 1e-5, "composed dw_router")
    assert_close(m.dw_mod.cpu().numpy(), dwm_c, 1e-5, "composed dw_mod")
    assert_close(to64(mb.dx), dxr_c + dxm_c, 2e-2, "composed dx")
