"""CPU oracle for the MoE / MoD layer hot path.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, float64 statement of
what the layer computes.  Only the tests, the package's ``smoke()`` check and the
benchmark's CPU-baseline leg may import it; the product path never does, and it
shares no code with the CUDA library.

Sources (web pages, cited by title and section):
  [FW]  "PyTorch MoE/MoD Training Framework: custom CUDA kernels, DeepSpeed and
        7x speed-up on T4" (ai-manual.ru), section "What's in the box": routing
        and gating = softmax over experts plus top-k selection in one launch;
        dispatch and combine = moving tokens between experts; a backward through
        the sparse operations for gating and dispatch; and the paragraph on
        Mixture-of-Depths (part of the tokens skips the layer entirely).
  [EP]  "Moonshot AI released MoonEP: Mixture-of-Experts training without GPU
        idle time" (dzen.guru), section "Step-by-step": one contiguous weight
        tensor [E(+B), H, H'] per expert projection, experts addressed purely by
        row index; dispatch returns cu_seqlens marking which expert rows are
        active; section "What problem it solves": the maxvio skew metric.
  [T4]  "MoE on T4: how to find and remove bottlenecks in training"
        (ai-manual.ru), table "RMSNorm, RoPE, SwiGLU": SwiGLU = three matrix
        products.

The pages print no formulas, so each function below writes out the plain
definition of the step.  Readings where the pages are silent:
  * top-k selects on the logits (monotone in the softmax), ties -> lower expert
    index, output ordered by decreasing logit then increasing index;
  * the gate is the full-softmax probability of the chosen expert (no
    renormalisation after top-k: the rows of the softmax sum to one before top-k);
  * rows of one expert segment are ordered by token index (stable);
  * cu_seqlens has E+1 entries (no preload pool on one GPU), cu[0]=0, cu[E]=T*K;
  * the down projection is stored [E, H, H'] like the others and applied as a.Wd[e]^T;
  * SwiGLU: a = silu(xs.Wg[e]) * (xs.Wu[e]), silu(z) = z / (1 + exp(-z)), no biases;
  * combine is the gate-weighted sum, written as a gather over each token's K rows;
  * MoD: score s = x.w_mod, per sequence the C highest scores run the layer (ties
    -> lower position), y = x + s * MoE(x) on those tokens and y = x elsewhere.

Every input is a float64 array holding the values in their storage type; nothing
is rounded inside the oracle.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# Routing: router GEMM, softmax over experts, top-k   [FW "What's in the box"]
# ----------------------------------------------------------------------------


def router_logits(x, w_router, bias=None):
    """logits[t, e] = sum_h x[t, h] * W_r[h, e] (+ bias[e])."""
    logits = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64)
    if bias is not None:
        logits = logits + np.asarray(bias, np.float64)[None, :]
    return logits


def softmax_experts(logits):
    """p[t, :] = softmax over the expert axis (max subtracted first)."""
    z = logits - logits.max(axis=1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=1, keepdims=True)


def topk_experts(logits, K):
    """The K experts with the largest logits per token.

    Order experts by decreasing logit, equal logits by increasing expert index,
    and keep the first K (a stable sort on the negated logits does exactly this).
    Returns int32 [T, K]."""
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :K].astype(np.int32)


def route(x, w_router, K, bias=None, renorm=False, bias_select_only=False):
    """Router forward: logits, softmax p, top-k idx, gate = p[idx].

    Two variants of the gate a drop-in for a Mixtral-style sparse MoE block
    needs [FW "How it looks in practice": the framework's block replaces the
    Mixtral one]:
      renorm            gate[t, k] = p[idx[t,k]] / sum_k' p[idx[t,k']], the top-k
                        weights rescaled to sum to 1 (the Mixtral block's routing);
      bias_select_only  the bias shifts only which experts are chosen
                        (idx = top-K of x W_r + bias); logits, p and the gate stay
                        those of x W_r (bias-based load balancing without an
                        auxiliary loss).
    """
    if bias_select_only and bias is not None:
        logits = router_logits(x, w_router)
        select = logits + np.asarray(bias, np.float64)[None, :]
    else:
        logits = router_logits(x, w_router, bias)
        select = logits
    p = softmax_experts(logits)
    idx = topk_experts(select, K)
    gate = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    if renorm:
        gate = gate / gate.sum(axis=1, keepdims=True)
    return logits, p, idx, gate


def maxvio(counts, T, K, E):
    """Router skew [EP "What problem it solves"]: max_e load_e / (T*K/E) - 1."""
    return float(np.max(counts) / (T * K / E) - 1.0)


# ----------------------------------------------------------------------------
# Dispatch: histogram, prefix sum -> cu_seqlens, permutation, gather
#   [FW "What's in the box"; EP "Step-by-step": contiguous rows, cu_seqlens]
# ----------------------------------------------------------------------------


def expert_histogram(idx, E):
    """count[e] = number of (t, k) with idx[t, k] == e."""
    counts = np.zeros(E, dtype=np.int64)
    for e in idx.reshape(-1):
        counts[e] += 1
    return counts


def cu_seqlens(counts):
    """Exclusive prefix sum with the total appended: cu[0]=0, cu[e+1]=cu[e]+count[e]."""
    cu = np.zeros(len(counts) + 1, dtype=np.int64)
    for e, c in enumerate(counts):
        cu[e + 1] = cu[e] + c
    return cu.astype(np.int32)


def permutation(idx, E):
    """Stable counting sort of the routed pairs by expert.

    dst_row[t*K + k] is the row of pair (t, k) in the expert-sorted buffer: the
    expert's segment start plus the number of earlier tokens that chose the same
    expert.  src_tok[row] is the token that fills that row."""
    T, K = idx.shape
    cu = cu_seqlens(expert_histogram(idx, E))
    fill = cu[:-1].astype(np.int64).copy()
    dst_row = np.empty(T * K, dtype=np.int32)
    src_tok = np.empty(T * K, dtype=np.int32)
    for t in range(T):
        for k in range(K):
            e = idx[t, k]
            row = fill[e]
            fill[e] += 1
            dst_row[t * K + k] = row
            src_tok[row] = t
    return cu, dst_row, src_tok


def gather_rows(x, src_tok):
    """xs[row, :] = x[src_tok[row], :]."""
    return np.asarray(x)[np.asarray(src_tok, np.int64)]


def dispatch(x, idx, E):
    cu, dst_row, src_tok = permutation(idx, E)
    return cu, dst_row, src_tok, gather_rows(x, src_tok)


# ----------------------------------------------------------------------------
# Grouped SwiGLU expert FFN   [EP "Step-by-step" (weights); T4 SwiGLU table]
# ----------------------------------------------------------------------------


def silu(z):
    return z / (1.0 + np.exp(-z))


def expert_swiglu(xs_rows, wg_e, wu_e, wd_e):
    """One expert on its rows: a = silu(X Wg) * (X Wu); h = a Wd^T."""
    g = xs_rows @ wg_e
    u = xs_rows @ wu_e
    a = silu(g) * u
    return a, a @ wd_e.T


def expert_ffn(xs, cu, w_gate, w_up, w_down):
    """Rows [cu[e], cu[e+1]) of xs go through expert e.  Returns act [R,H'], h [R,H]."""
    R = xs.shape[0]
    E, H, Hp = w_gate.shape
    act = np.zeros((R, Hp))
    h = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(cu[e]), int(cu[e + 1])
        if hi > lo:
            act[lo:hi], h[lo:hi] = expert_swiglu(xs[lo:hi], w_gate[e], w_up[e], w_down[e])
    return act, h


def expert_swiglu_bwd(xs_rows, wg_e, wu_e, wd_e, dh_rows):
    """Backward of one expert on its rows, given dh = dL/dh for h = a Wd^T with
    a = silu(g) * u, g = X Wg, u = X Wu  [T4 "RMSNorm, RoPE, SwiGLU": SwiGLU is
    three matrix products; FW "What's in the box": the layer trains].
        da  = dh Wd                       dWd = dh^T a
        dg  = da * u * silu'(g),          silu'(g) = s(g) (1 + g (1 - s(g))), s = logistic
        du  = da * silu(g)
        dX  = dg Wg^T + du Wu^T           dWg = X^T dg,  dWu = X^T du
    Returns dX, dWg, dWu, dWd."""
    g = xs_rows @ wg_e
    u = xs_rows @ wu_e
    sg = 1.0 / (1.0 + np.exp(-g))
    a = g * sg * u
    da = dh_rows @ wd_e
    dg = da * u * sg * (1.0 + g * (1.0 - sg))
    du = da * g * sg
    dx = dg @ wg_e.T + du @ wu_e.T
    return dx, xs_rows.T @ dg, xs_rows.T @ du, dh_rows.T @ a


def expert_ffn_bwd(xs, cu, w_gate, w_up, w_down, dh):
    """Backward of expert_ffn: dxs [R,H] and the weight gradients dW_gate,
    dW_up, dW_down [E,H,H'] (zero for experts without rows)."""
    xs, dh = np.asarray(xs, np.float64), np.asarray(dh, np.float64)
    E, H, Hp = w_gate.shape
    dxs = np.zeros_like(xs)
    dwg, dwu, dwd = np.zeros((E, H, Hp)), np.zeros((E, H, Hp)), np.zeros((E, H, Hp))
    for e in range(E):
        lo, hi = int(cu[e]), int(cu[e + 1])
        if hi > lo:
            dxs[lo:hi], dwg[e], dwu[e], dwd[e] = expert_swiglu_bwd(xs[lo:hi], w_gate[e], w_up[e], w_down[e],
                                                                   dh[lo:hi])
    return dxs, dwg, dwu, dwd


def expert_of_row(cu, rows):
    """Expert e with cu[e] <= row < cu[e+1] for each row."""
    cu = np.asarray(cu, np.int64)
    return np.searchsorted(cu, np.asarray(rows, np.int64), side="right") - 1


# ----------------------------------------------------------------------------
# Combine   [FW "What's in the box"]
# ----------------------------------------------------------------------------


def combine(h, gate, dst_row, row_scale=None, residual=None, out_row=None, n_out=None):
    """y[o(t)] = residual[o(t)] + scale[t] * sum_k gate[t,k] * h[dst_row[t*K+k]].

    o(t) = out_row[t] if given, else t.  Rows of y not written by any token are
    residual (or zero without residual).  Plain MoE: scale = 1, no residual."""
    T, K = gate.shape
    H = h.shape[1]
    n = T if n_out is None else n_out
    y = np.zeros((n, H)) if residual is None else np.array(residual, dtype=np.float64, copy=True)
    for t in range(T):
        acc = np.zeros(H)
        for k in range(K):
            acc += gate[t, k] * h[dst_row[t * K + k]]
        s = 1.0 if row_scale is None else row_scale[t]
        o = t if out_row is None else out_row[t]
        y[o] = y[o] + s * acc
    return y


# ----------------------------------------------------------------------------
# Backward of gating and dispatch/combine   [FW "What's in the box", sparse backward]
# ----------------------------------------------------------------------------


def route_bwd_softmax_topk(d_gate, logits, idx, x, w_router, renorm=False):
    """Gradient through gate[t,k] = softmax(logits[t])[idx[t,k]].

    The selection is piecewise constant (no gradient through it); gradient reaches
    every logit through the softmax:
        dlogit[t, j] = p_j * (G_j - sum_k d_gate[t,k] * p[idx[t,k]]),
        G_j = d_gate[t,k] if j == idx[t,k] else 0.
    With renorm the gate is q_k = p[idx_k] / sum_k' p[idx_k'], which is the
    softmax of the chosen logits alone, so only they get a gradient:
        dlogit[t, idx_k] = q_k * (d_gate[t,k] - sum_k' d_gate[t,k'] * q_k'),
    and 0 for the other experts.
    Then dW_r = x^T dlogit and dx = dlogit W_r^T (the logit bias gets sum_t dlogit)."""
    p = softmax_experts(logits)
    T, E = logits.shape
    ix = idx.astype(np.int64)
    if renorm:
        q = np.take_along_axis(p, ix, axis=1)
        q = q / q.sum(axis=1, keepdims=True)
        inner = (d_gate * q).sum(axis=1, keepdims=True)
        d_logits = np.zeros((T, E))
        np.put_along_axis(d_logits, ix, q * (d_gate - inner), axis=1)
    else:
        G = np.zeros((T, E))
        np.put_along_axis(G, ix, d_gate, axis=1)
        inner = (d_gate * np.take_along_axis(p, ix, axis=1)).sum(axis=1, keepdims=True)
        d_logits = p * (G - inner)
    dw = np.asarray(x).T @ d_logits
    dx = d_logits @ np.asarray(w_router).T
    return d_logits, dw, dx


def route_bwd_linear(d_score, x, w):
    """Gradient through a scalar linear score s[t] = x[t] . w:
    dw = sum_t d_score[t] x[t], dx[t] = d_score[t] * w."""
    d = np.asarray(d_score).reshape(-1)
    return np.asarray(x).T @ d, np.outer(d, w)


def permute_bwd(dy, h, gate, dst_row, dxs=None, row_scale=None, out_row=None):
    """Adjoint of ``combine`` (and of the dispatch gather for dx).

    With g(t) = dy[o(t)] and s_t the row scale:
        dh[dst_row[t*K+k]] = s_t * gate[t,k] * g(t)
        d_gate[t,k]        = s_t * <g(t), h[dst_row[t*K+k]]>
        d_scale[t]         = sum_k gate[t,k] * <g(t), h[dst_row[t*K+k]]>
        dx[t]              = sum_k dxs[dst_row[t*K+k]]     (adjoint of xs = x[src_tok])"""
    T, K = gate.shape
    H = h.shape[1]
    dh = np.zeros_like(h, dtype=np.float64)
    d_gate = np.zeros((T, K))
    d_scale = np.zeros(T)
    dx = np.zeros((T, H)) if dxs is not None else None
    for t in range(T):
        o = t if out_row is None else out_row[t]
        s = 1.0 if row_scale is None else row_scale[t]
        g = dy[o]
        for k in range(K):
            r = dst_row[t * K + k]
            dot = float(g @ h[r])
            dh[r] = s * gate[t, k] * g
            d_gate[t, k] = s * dot
            d_scale[t] += gate[t, k] * dot
            if dxs is not None:
                dx[t] += dxs[r]
    return dh, d_gate, d_scale, dx


# ----------------------------------------------------------------------------
# Mixture-of-Depths capacity router   [FW MoD paragraph]
# ----------------------------------------------------------------------------


def mod_scores(x, w_mod):
    """s[t] = x[t] . w_mod."""
    return np.asarray(x, np.float64) @ np.asarray(w_mod, np.float64)


def mod_select(score, B, L, C):
    """Per sequence b, the C positions with the highest score (equal scores -> the
    lower position).  Returns sel int32 [B, C] (positions ascending) and mask [B*L]."""
    s = np.asarray(score).reshape(B, L)
    sel = np.empty((B, C), dtype=np.int32)
    mask = np.zeros(B * L, dtype=np.uint8)
    for b in range(B):
        order = np.argsort(-s[b], kind="stable")[:C]
        sel[b] = np.sort(order)
        mask[b * L + sel[b]] = 1
    return sel, mask


# ----------------------------------------------------------------------------
# Layer compositions
# ----------------------------------------------------------------------------


def moe_forward(x, w_router, w_gate, w_up, w_down, K, bias=None, renorm=False, bias_select_only=False):
    """route -> dispatch -> grouped SwiGLU experts -> combine (gate options as in route)."""
    E = w_router.shape[1]
    logits, p, idx, gate = route(x, w_router, K, bias, renorm=renorm, bias_select_only=bias_select_only)
    cu, dst_row, src_tok, xs = dispatch(x, idx, E)
    act, h = expert_ffn(xs, cu, w_gate, w_up, w_down)
    y = combine(h, gate, dst_row)
    return dict(logits=logits, p=p, idx=idx, gate=gate, cu=cu, dst_row=dst_row,
                src_tok=src_tok, xs=xs, act=act, h=h, y=y)


def moe_backward(fwd, dy, dxs, x, w_router, renorm=False):
    """Gate and dispatch/combine backward given dy and a dxs for the expert inputs."""
    dh, d_gate, _, dx_disp = permute_bwd(dy, fwd["h"], fwd["gate"], fwd["dst_row"], dxs)
    d_logits, dw, dx_r = route_bwd_softmax_topk(d_gate, fwd["logits"], fwd["idx"], x, w_router, renorm=renorm)
    return dict(dh=dh, d_gate=d_gate, d_logits=d_logits, dw_router=dw, dx=dx_disp + dx_r)


def mod_forward(x, w_mod, w_router, w_gate, w_up, w_down, B, L, C, K):
    """MoD front end around the MoE: the selected tokens get x + s * MoE(x), the
    others pass through unchanged."""
    score = mod_scores(x, w_mod)
    sel, mask = mod_select(score, B, L, C)
    flat = (np.arange(B)[:, None] * L + sel).reshape(-1)
    x_sel = np.asarray(x)[flat]
    inner = moe_forward(x_sel, w_router, w_gate, w_up, w_down, K)
    y = combine(inner["h"], inner["gate"], inner["dst_row"], row_scale=score[flat],
                residual=x, out_row=flat, n_out=x.shape[0])
    return dict(score=score, sel=sel, mask=mask, flat=flat, x_sel=x_sel, inner=inner, y=y)
