"""Pins of the CPU oracle against what the mathematics fixes independently of it:
brute force on tiny inputs, closed forms, invariants and central finite
differences.  Each check is chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand, an unstable order)
fails at least one of them.  CPU only."""
import itertools
import math

import numpy as np
import pytest

import oracle as O
from token_dispatch_gb300 import synth

RNG = np.random.default_rng(12345)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# ---------------------------------------------------------------- softmax ---

def test_softmax_rows_sum_to_one_before_topk():
    p = O.softmax_experts(rand(64, 37, scale=5.0))
    assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert (p > 0).all()


def test_softmax_two_experts_is_logistic():
    l = rand(200, 2, scale=3.0)
    p = O.softmax_experts(l)
    sig = 1.0 / (1.0 + np.exp(-(l[:, 0] - l[:, 1])))
    assert np.allclose(p[:, 0], sig, rtol=1e-14, atol=0)


def test_softmax_shift_invariant_and_large_logits():
    l = rand(16, 9)
    assert np.allclose(O.softmax_experts(l), O.softmax_experts(l + 1000.0), rtol=1e-12)
    big = O.softmax_experts(np.array([[1000.0, 0.0, -1000.0]]))
    assert np.isfinite(big).all() and abs(big[0, 0] - 1.0) < 1e-15


def test_softmax_ratio_is_exp_difference():
    l = rand(10, 6)
    p = O.softmax_experts(l)
    assert np.allclose(p[:, 1] / p[:, 4], np.exp(l[:, 1] - l[:, 4]), rtol=1e-12)


# ------------------------------------------------------------------ top-k ---

def brute_topk(row, K):
    """Among all K-subsets: maximum logit sum, then the lexicographically smallest
    ascending index tuple; reported by decreasing logit, then increasing index."""
    best = None
    for sub in itertools.combinations(range(len(row)), K):
        key = (-sum(row[i] for i in sub), sub)
        if best is None or key < best:
            best = key
    chosen = best[1]
    return sorted(chosen, key=lambda i: (-row[i], i))


@pytest.mark.parametrize("E,K", [(4, 1), (5, 2), (6, 3), (8, 2), (7, 7)])
def test_topk_matches_brute_force_with_ties(E, K):
    # small integer logits force many ties
    l = RNG.integers(-2, 3, size=(60, E)).astype(np.float64)
    idx = O.topk_experts(l, K)
    for t in range(l.shape[0]):
        assert list(idx[t]) == brute_topk(list(l[t]), K), (t, l[t])


def test_topk_all_equal_rows_pick_lowest_indices():
    idx = O.topk_experts(np.zeros((3, 9)), 4)
    assert (idx == np.arange(4)[None, :]).all()


def test_topk_E_equals_K_takes_every_expert():
    l = rand(20, 5)
    idx = O.topk_experts(l, 5)
    assert (np.sort(idx, axis=1) == np.arange(5)).all()
    # ordered by decreasing logit
    assert (np.diff(np.take_along_axis(l, idx.astype(np.int64), axis=1), axis=1) <= 0).all()


def test_route_gate_is_probability_of_chosen_expert():
    x, w = rand(30, 12), rand(12, 8, scale=0.3)
    logits, p, idx, gate = O.route(x, w, 3)
    for t in range(30):
        for k in range(3):
            e = idx[t, k]
            assert gate[t, k] == p[t, e]
    # logits are x.W: check one entry by an explicit sum
    assert math.isclose(logits[7, 5], sum(x[7, h] * w[h, 5] for h in range(12)), rel_tol=1e-13)


def test_route_bias_shifts_only_its_expert():
    x, w = rand(10, 6), rand(6, 4)
    b = np.array([0.0, 2.5, 0.0, 0.0])
    l0 = O.router_logits(x, w)
    l1 = O.router_logits(x, w, b)
    assert np.array_equal(l1[:, [0, 2, 3]], l0[:, [0, 2, 3]])
    assert np.allclose(l1[:, 1] - l0[:, 1], 2.5)


def test_route_renorm_gates_sum_to_one_and_keep_ratios():
    """Mixtral-style renormalisation: the K gates of a token sum to 1 and keep
    the ratios of the chosen probabilities; K = 1 gives 1; K = E changes nothing."""
    r = np.random.default_rng(701)
    x, w = r.standard_normal((25, 10)), r.standard_normal((10, 6)) * 0.7
    _, p, idx, g0 = O.route(x, w, 3)
    _, _, idx_r, g = O.route(x, w, 3, renorm=True)
    assert np.array_equal(idx, idx_r)
    assert np.allclose(g.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(g[:, 0] / g[:, 2], g0[:, 0] / g0[:, 2], rtol=1e-13)
    assert np.array_equal(O.route(x, w, 1, renorm=True)[3], np.ones((25, 1)))
    _, p6, i6, g6 = O.route(x, w, 6, renorm=True)
    assert np.allclose(g6, np.take_along_axis(p6, i6.astype(np.int64), axis=1), rtol=1e-13)


def test_route_renorm_ignores_the_experts_not_chosen():
    """Renormalised gates depend only on the chosen logits: lowering every
    unchosen logit (keeping it below the K-th) leaves them as they are, while
    the plain gates grow."""
    l = np.random.default_rng(702).standard_normal((40, 7))
    K = 3
    idx = O.topk_experts(l, K)
    chosen = np.zeros_like(l, dtype=bool)
    np.put_along_axis(chosen, idx.astype(np.int64), True, axis=1)
    l2 = np.where(chosen, l, l - 3.0)
    x = np.eye(7)
    a = O.route(l, x, K, renorm=True)
    b = O.route(l2, x, K, renorm=True)
    assert np.array_equal(a[2], b[2])
    assert np.allclose(a[3], b[3], rtol=1e-13)
    assert (O.route(l2, x, K)[3] > O.route(l, x, K)[3]).all()


def test_route_bias_select_only_moves_choice_not_gates():
    """With the bias used for selection only, idx is the brute-force top-K of
    logits + bias (ties -> lower expert) while logits and gates are unbiased."""
    T, E, K = 60, 5, 2
    r = np.random.default_rng(703)
    x = r.integers(-2, 3, size=(T, 4)).astype(np.float64)
    w = r.integers(-1, 2, size=(4, E)).astype(np.float64)
    b = np.array([0.0, 1.0, -1.0, 2.0, 0.0])
    logits, p, idx, gate = O.route(x, w, K, b, bias_select_only=True)
    l0 = x @ w
    assert np.array_equal(logits, l0)
    assert np.allclose(p, O.softmax_experts(l0), rtol=1e-14)
    for t in range(T):
        sel = l0[t] + b
        best = max(itertools.combinations(range(E), K),
                   key=lambda c: (sorted((sel[e] for e in c), reverse=True), [-e for e in c]))
        order = sorted(best, key=lambda e: (-sel[e], e))
        assert list(idx[t]) == order
        assert np.array_equal(gate[t], p[t, order])


# ----------------------------------------------- histogram / cu_seqlens ---

def test_histogram_and_cu_seqlens_by_counting():
    E, T, K = 11, 97, 3
    idx = np.stack([RNG.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    counts = O.expert_histogram(idx, E)
    brute = [sum(1 for t in range(T) for k in range(K) if idx[t, k] == e) for e in range(E)]
    assert list(counts) == brute
    cu = O.cu_seqlens(counts)
    assert cu[0] == 0 and cu[-1] == T * K
    assert (np.diff(cu) == counts).all() and (np.diff(cu) >= 0).all()


def test_maxvio_definition():
    assert O.maxvio(np.array([4, 4, 4, 4]), 8, 2, 4) == 0.0
    # every token sends one of its K picks to expert 0: load T, maxvio E/K - 1
    assert math.isclose(O.maxvio(np.array([8, 3, 3, 2]), 8, 2, 4), 4 / 2 - 1)


# ----------------------------------------------------------- permutation ---

def make_idx(T, E, K, seed=0):
    r = np.random.default_rng(seed)
    return np.stack([r.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,K", [(1, 1, 1), (13, 4, 2), (50, 8, 3), (40, 16, 6), (9, 3, 3)])
def test_permutation_is_stable_sort_by_expert(T, E, K):
    idx = make_idx(T, E, K, seed=T)
    cu, dst, src = O.permutation(idx, E)
    # brute force: stable sort of (expert, token) pairs in (t, k) order
    pairs = sorted(((idx[t, k], t, k) for t in range(T) for k in range(K)), key=lambda p: (p[0], p[1]))
    for row, (e, t, k) in enumerate(pairs):
        assert dst[t * K + k] == row
        assert src[row] == t
        assert cu[e] <= row < cu[e + 1]
    # bijection
    assert sorted(dst.tolist()) == list(range(T * K))
    assert all(src[dst[j]] == j // K for j in range(T * K))


def test_dispatch_gathers_rows():
    T, E, K, H = 20, 5, 2, 7
    x = rand(T, H)
    idx = make_idx(T, E, K, seed=3)
    cu, dst, src, xs = O.dispatch(x, idx, E)
    for t in range(T):
        for k in range(K):
            assert np.array_equal(xs[dst[t * K + k]], x[t])


@pytest.mark.parametrize("K", [1, 2, 3, 6, 8])
def test_combine_of_dispatch_with_unit_gates_is_K_times_x(K):
    T, E, H = 31, 9, 5
    x = rand(T, H)
    idx = make_idx(T, E, K, seed=K)
    cu, dst, src, xs = O.dispatch(x, idx, E)
    y = O.combine(xs, np.ones((T, K)), dst)  # identity expert: h = xs
    assert np.allclose(y, K * x, rtol=1e-15, atol=0)


def test_combine_weights_residual_and_out_rows():
    T, K, H = 4, 2, 3
    h = rand(T * K, H)
    gate = rand(T, K)
    dst = np.array([3, 0, 5, 1, 2, 7, 6, 4], np.int32)
    scale = rand(T)
    res = rand(10, H)
    out = np.array([9, 2, 5, 0], np.int32)
    y = O.combine(h, gate, dst, row_scale=scale, residual=res, out_row=out, n_out=10)
    for t in range(T):
        want = res[out[t]] + scale[t] * (gate[t, 0] * h[dst[2 * t]] + gate[t, 1] * h[dst[2 * t + 1]])
        assert np.allclose(y[out[t]], want, rtol=1e-14)
    untouched = [r for r in range(10) if r not in out]
    assert np.array_equal(y[untouched], res[untouched])


# ------------------------------------------------------------- experts ---

def test_silu_special_values_and_odd_part():
    z = rand(1000, scale=4.0)
    # silu(z) - silu(-z) = z exactly in exact arithmetic (z*s(z) + z*s(-z) = z)
    assert np.allclose(O.silu(z) - O.silu(-z), z, rtol=1e-12, atol=1e-14)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert math.isclose(O.silu(np.array([50.0]))[0], 50.0, rel_tol=1e-15)
    assert abs(O.silu(np.array([-50.0]))[0]) < 1e-19


def test_single_expert_equals_dense_swiglu_mlp_by_loops():
    """E = 1, K = 1: the layer is a dense SwiGLU MLP, evaluated here with explicit
    scalar loops (no matrix routine)."""
    T, H, Hp = 3, 4, 5
    x = rand(T, H)
    wr = rand(H, 1)
    wg, wu, wd = rand(1, H, Hp), rand(1, H, Hp), rand(1, H, Hp)
    out = O.moe_forward(x, wr, wg, wu, wd, K=1)
    assert np.allclose(out["gate"], 1.0)
    for t in range(T):
        a = []
        for j in range(Hp):
            g = sum(x[t, i] * wg[0, i, j] for i in range(H))
            u = sum(x[t, i] * wu[0, i, j] for i in range(H))
            a.append(g / (1.0 + math.exp(-g)) * u)
        for i in range(H):
            want = sum(a[j] * wd[0, i, j] for j in range(Hp))
            assert math.isclose(out["y"][t, i], want, rel_tol=1e-12, abs_tol=1e-13)


def test_expert_rows_are_independent_and_use_their_own_expert():
    T, E, K, H, Hp = 25, 4, 2, 6, 8
    x = rand(T, H)
    wr = rand(H, E)
    wg, wu, wd = rand(E, H, Hp), rand(E, H, Hp), rand(E, H, Hp)
    f = O.moe_forward(x, wr, wg, wu, wd, K)
    e_of = O.expert_of_row(f["cu"], np.arange(T * K))
    for r in range(T * K):
        e = e_of[r]
        a, hr = O.expert_swiglu(f["xs"][r:r + 1], wg[e], wu[e], wd[e])
        assert np.allclose(hr[0], f["h"][r], rtol=1e-13)
        assert np.allclose(a[0], f["act"][r], rtol=1e-13)
        assert e == f["idx"][f["src_tok"][r]][list(f["dst_row"][f["src_tok"][r] * K:(f["src_tok"][r] + 1) * K]).index(r)]


def test_E_equals_K_is_dense_softmax_mixture():
    """E = K: every token visits every expert; y = sum_e p_e * expert_e(x)."""
    T, E, H, Hp = 6, 3, 4, 5
    x = rand(T, H)
    wr = rand(H, E)
    wg, wu, wd = rand(E, H, Hp), rand(E, H, Hp), rand(E, H, Hp)
    f = O.moe_forward(x, wr, wg, wu, wd, K=E)
    p = O.softmax_experts(x @ wr)
    want = np.zeros((T, H))
    for e in range(E):
        g = x @ wg[e]
        u = x @ wu[e]
        want += p[:, [e]] * ((g * (1 / (1 + np.exp(-g))) * u) @ wd[e].T)
    assert np.allclose(f["y"], want, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------ finite differences ---

def central_diff(f, theta, i, h_rel=1e-6):
    th = theta.copy().reshape(-1)
    h = h_rel * max(1.0, abs(th[i]))
    th[i] += h
    fp = f(th.reshape(theta.shape))
    th[i] -= 2 * h
    fm = f(th.reshape(theta.shape))
    return (fp - fm) / (2 * h)


def topk_margin(logits, K):
    s = np.sort(logits, axis=1)[:, ::-1]
    return (s[:, K - 1] - s[:, K]).min() if logits.shape[1] > K else np.inf


@pytest.mark.parametrize("T,H,E,K", [(8, 16, 4, 2), (6, 10, 8, 3), (5, 7, 5, 5)])
def test_route_backward_matches_central_differences(T, H, E, K):
    x, w = rand(T, H), rand(H, E, scale=0.5)
    d_gate = rand(T, K)
    logits, p, idx, gate = O.route(x, w, K)
    assert topk_margin(logits, K) > 1e-3

    def loss_w(wv):
        l = O.router_logits(x, wv)
        pp = O.softmax_experts(l)
        assert np.array_equal(O.topk_experts(l, K), idx)
        return float((d_gate * np.take_along_axis(pp, idx.astype(np.int64), axis=1)).sum())

    def loss_x(xv):
        l = O.router_logits(xv, w)
        pp = O.softmax_experts(l)
        assert np.array_equal(O.topk_experts(l, K), idx)
        return float((d_gate * np.take_along_axis(pp, idx.astype(np.int64), axis=1)).sum())

    def loss_l(lv):
        pp = O.softmax_experts(lv)
        return float((d_gate * np.take_along_axis(pp, idx.astype(np.int64), axis=1)).sum())

    d_logits, dw, dx = O.route_bwd_softmax_topk(d_gate, logits, idx, x, w)
    for i in range(logits.size):
        assert math.isclose(central_diff(loss_l, logits, i), d_logits.reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)
    for i in range(w.size):
        assert math.isclose(central_diff(loss_w, w, i), dw.reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)
    for i in range(x.size):
        assert math.isclose(central_diff(loss_x, x, i), dx.reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)


@pytest.mark.parametrize("T,E,K", [(6, 5, 2), (4, 8, 3), (5, 4, 4), (3, 6, 1)])
def test_route_backward_renorm_matches_central_differences(T, E, K):
    """Renormalised gates: the gradient w.r.t. every logit (chosen or not)."""
    r = np.random.default_rng(710 + T * E + K)
    l = r.standard_normal((T, E))
    d_gate = r.standard_normal((T, K))
    idx = O.topk_experts(l, K)
    assert topk_margin(l, K) > 1e-3

    def loss_l(lv):
        q = np.take_along_axis(O.softmax_experts(lv), idx.astype(np.int64), axis=1)
        return float((d_gate * q / q.sum(axis=1, keepdims=True)).sum())

    d_logits, _, _ = O.route_bwd_softmax_topk(d_gate, l, idx, np.zeros((T, 1)), np.zeros((1, E)), renorm=True)
    for i in range(l.size):
        assert math.isclose(central_diff(loss_l, l, i), d_logits.reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)
    chosen = np.zeros_like(l, dtype=bool)
    np.put_along_axis(chosen, idx.astype(np.int64), True, axis=1)
    assert (d_logits[~chosen] == 0).all()


def test_expert_ffn_backward_matches_central_differences():
    """dL/d(xs, Wg, Wu, Wd) for L = sum(dh * h) with h the grouped SwiGLU FFN, on
    three experts one of which has no rows."""
    r = np.random.default_rng(720)
    E, H, Hp = 3, 5, 4
    cu = np.array([0, 3, 3, 7])
    xs = r.standard_normal((7, H))
    wg, wu, wd = r.standard_normal((E, H, Hp)), r.standard_normal((E, H, Hp)), r.standard_normal((E, H, Hp))
    dh = r.standard_normal((7, H))

    def loss(xs_, wg_, wu_, wd_):
        return float((dh * O.expert_ffn(xs_, cu, wg_, wu_, wd_)[1]).sum())

    dxs, dwg, dwu, dwd = O.expert_ffn_bwd(xs, cu, wg, wu, wd, dh)
    assert (dwg[1] == 0).all() and (dwu[1] == 0).all() and (dwd[1] == 0).all()
    for arr, grad, f in [(xs, dxs, lambda v: loss(v, wg, wu, wd)), (wg, dwg, lambda v: loss(xs, v, wu, wd)),
                         (wu, dwu, lambda v: loss(xs, wg, v, wd)), (wd, dwd, lambda v: loss(xs, wg, wu, v))]:
        for i in range(arr.size):
            assert math.isclose(central_diff(f, arr, i), grad.reshape(-1)[i], rel_tol=1e-6, abs_tol=1e-8)


def test_expert_backward_single_row_by_hand():
    """One row, one expert, H = H' = 1: every gradient written out with scalars."""
    x, g_w, u_w, d_w, dy = 0.7, -1.3, 0.4, 2.1, -0.6
    g, u = x * g_w, x * u_w
    s = 1.0 / (1.0 + math.exp(-g))
    dsilu = s + g * s * (1.0 - s)  # derivative of g * s(g)
    da = dy * d_w
    dxs, dwg, dwu, dwd = O.expert_ffn_bwd(np.array([[x]]), np.array([0, 1]), np.array([[[g_w]]]),
                                          np.array([[[u_w]]]), np.array([[[d_w]]]), np.array([[dy]]))
    assert math.isclose(dwd[0, 0, 0], dy * g * s * u, rel_tol=1e-14)
    assert math.isclose(dwg[0, 0, 0], x * da * u * dsilu, rel_tol=1e-14)
    assert math.isclose(dwu[0, 0, 0], x * da * g * s, rel_tol=1e-14)
    assert math.isclose(dxs[0, 0], da * u * dsilu * g_w + da * g * s * u_w, rel_tol=1e-14)


def test_route_backward_E_equals_K_is_softmax_jacobian():
    """With every expert selected the gradient is J^T g with J = diag(p) - p p^T."""
    T, E = 7, 5
    l = rand(T, E)
    idx = O.topk_experts(l, E)
    d_gate = rand(T, E)
    d_logits, _, _ = O.route_bwd_softmax_topk(d_gate, l, idx, np.zeros((T, 1)), np.zeros((1, E)))
    p = O.softmax_experts(l)
    for t in range(T):
        g = np.zeros(E)
        g[idx[t]] = d_gate[t]
        J = np.diag(p[t]) - np.outer(p[t], p[t])
        assert np.allclose(d_logits[t], J.T @ g, rtol=1e-12, atol=1e-15)


def test_permute_backward_matches_central_differences():
    T, K, H, n_out = 5, 2, 4, 8
    R = T * K
    h = rand(R, H)
    gate = rand(T, K)
    dst = RNG.permutation(R).astype(np.int32)
    scale = rand(T)
    out = RNG.choice(n_out, T, replace=False).astype(np.int32)
    res = rand(n_out, H)
    dy = rand(n_out, H)
    dxs = rand(R, H)

    def L(hh=h, gg=gate, ss=scale):
        y = O.combine(hh, gg, dst, row_scale=ss, residual=res, out_row=out, n_out=n_out)
        return float((dy * y).sum())

    dh, d_gate, d_scale, dx = O.permute_bwd(dy, h, gate, dst, dxs, row_scale=scale, out_row=out)
    for i in range(h.size):
        assert math.isclose(central_diff(lambda v: L(hh=v), h, i), dh.reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)
    for i in range(gate.size):
        assert math.isclose(central_diff(lambda v: L(gg=v), gate, i), d_gate.reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)
    for i in range(scale.size):
        assert math.isclose(central_diff(lambda v: L(ss=v), scale, i), d_scale[i], rel_tol=1e-7, abs_tol=1e-9)

    # dx is the adjoint of the dispatch gather xs = x[src_tok]: <dxs, xs(x)> differentiated in x
    src = np.empty(R, np.int64)
    src[dst] = np.arange(R) // K
    x = rand(T, H)

    def L2(xv):
        return float((dxs * O.gather_rows(xv, src)).sum())

    for i in range(x.size):
        assert math.isclose(central_diff(L2, x, i), dx.reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)


def test_layer_backward_chain_matches_central_differences():
    """dL/dx through gate+dispatch for L = <dy, y> + <dxs, xs>, with the expert
    outputs h held fixed (the expert FFN backward is not part of this path)."""
    T, H, E, K = 6, 8, 4, 2
    x, wr = rand(T, H), rand(H, E, scale=0.5)
    f = O.moe_forward(x, wr, rand(E, H, 3), rand(E, H, 3), rand(E, H, 3), K)
    assert topk_margin(f["logits"], K) > 1e-3
    dy, dxs = rand(T, H), rand(T * K, H)
    b = O.moe_backward(f, dy, dxs, x, wr)
    h_fixed = f["h"]

    def L(xv):
        logits, p, idx, gate = O.route(xv, wr, K)
        assert np.array_equal(idx, f["idx"])
        _, dst, src, xs = O.dispatch(xv, idx, E)
        y = O.combine(h_fixed, gate, dst)
        return float((dy * y).sum() + (dxs * xs).sum())

    for i in range(x.size):
        assert math.isclose(central_diff(L, x, i), b["dx"].reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)


# ------------------------------------------------------------------- MoD ---

def brute_mod_select(score_row, C):
    order = sorted(range(len(score_row)), key=lambda i: (-score_row[i], i))
    return sorted(order[:C])


def test_mod_select_brute_force_with_ties():
    B, L, C = 3, 17, 6
    s = RNG.integers(-3, 4, size=B * L).astype(np.float64)
    sel, mask = O.mod_select(s, B, L, C)
    for b in range(B):
        assert list(sel[b]) == brute_mod_select(list(s[b * L:(b + 1) * L]), C)
    assert mask.sum() == B * C
    assert all(mask[b * L + p] == 1 for b in range(B) for p in sel[b])


def test_mod_full_capacity_is_moe_with_score_scaled_residual():
    B, L, H, E, K, Hp = 2, 6, 5, 3, 2, 4
    x = rand(B * L, H)
    wmod, wr = rand(H), rand(H, E)
    wg, wu, wd = rand(E, H, Hp), rand(E, H, Hp), rand(E, H, Hp)
    m = O.mod_forward(x, wmod, wr, wg, wu, wd, B, L, C=L, K=K)
    plain = O.moe_forward(x, wr, wg, wu, wd, K)
    s = x @ wmod
    assert np.allclose(m["y"], x + s[:, None] * plain["y"], rtol=1e-12, atol=1e-13)


def test_mod_zero_capacity_is_identity():
    B, L, H = 2, 5, 4
    x = rand(B * L, H)
    sel, mask = O.mod_select(O.mod_scores(x, rand(H)), B, L, 0)
    assert sel.shape == (B, 0) and mask.sum() == 0
    y = O.combine(np.zeros((0, H)), np.zeros((0, 1)), np.zeros(0, np.int32), residual=x, n_out=B * L)
    assert np.array_equal(y, x)


def test_mod_route_backward_matches_central_differences():
    T, H = 7, 5
    x, w = rand(T, H), rand(H)
    M, dy = rand(T, H), rand(T, H)   # MoE output held fixed; upstream gradient
    ds = (dy * M).sum(axis=1)        # d/ds of <dy, x + s*M>

    def L(wv):
        return float((dy * (x + (x @ wv)[:, None] * M)).sum())

    dw, dx = O.route_bwd_linear(ds, x, w)
    for i in range(H):
        assert math.isclose(central_diff(L, w, i), dw[i], rel_tol=1e-7, abs_tol=1e-9)

    def Lx(xv):
        return float((dy * ((xv @ w)[:, None] * M)).sum())

    for i in range(x.size):
        assert math.isclose(central_diff(Lx, x, i), dx.reshape(-1)[i], rel_tol=1e-7, abs_tol=1e-9)


# -------------------------------------------------------- input generator ---

def test_generator_is_chunking_independent_and_normal():
    a = synth.normal(0, 1, 10000)
    b = np.concatenate([synth.normal(0, 1, 4000), synth.normal(0, 1, 6000, start=4000)])
    assert np.array_equal(a, b)
    c = synth.normal(0, 1, 10000, chunk=777)
    assert np.array_equal(a, c)
    assert abs(a.mean()) < 0.05 and abs(a.std() - 1) < 0.05
    assert not np.array_equal(a, synth.normal(0, 2, 10000))


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 0.0], np.float64)
    got = synth.bf16_bits_to_f64(synth.round_bf16_bits(vals))
    # 1+2^-8 is halfway between 1 and 1+2^-7: ties to even (1.0); 1+3*2^-8 -> 1+2^-6
    assert list(got) == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 0.0]
