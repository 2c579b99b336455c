"""Helpers shared by the GPU parity tests: device copies, error metrics and the
top-k comparison that tolerates only genuine near-ties."""
import numpy as np
import torch

import oracle as O
from token_dispatch_gb300 import synth

DEV = "cuda:0"
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}
# Tolerances on the normwise relative error max|gpu - ref| / max|ref|:
# 1e-5 for the fp32 layer, 2e-2 for bf16 storage against the oracle fed the
# same bf16-rounded inputs.
TOL = {"f32": 1e-5, "bf16": 2e-2}


def dev(stored):
    return stored.host.to(DEV)


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy() if t.dtype != torch.bfloat16 else \
        t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def rel_err(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    den = np.max(np.abs(ref))
    num = np.max(np.abs(gpu - ref))
    return float(num / den) if den > 0 else float(num)


def assert_close(gpu, ref, tol, what=""):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{what}: normwise relative error {e:.3e} > {tol:.1e}"
    return e


def gate_tol(logit_err):
    """Bound for the gates given the logits' absolute error d: since
    d(log p_j)/d(l_i) = [i==j] - p_i, a perturbation of every logit by at most d
    changes each p_j by at most 2d relative (to first order), so the normwise
    relative gate error is at most 2d; 1e-6 covers fp32 exp/divide rounding."""
    return 2.0 * logit_err + 1e-6


def check_topk(gpu_idx, ref_logits, K, logit_err, max_frac=1e-3):
    """Rows whose GPU top-K differs from the oracle's must be near-ties: every
    chosen expert's exact logit is within 2*logit_err of the K-th largest exact
    logit.  Returns the number of such rows (also bounded by max_frac)."""
    ref_idx = np.argsort(-ref_logits, axis=1, kind="stable")[:, :K]
    bad = np.where((gpu_idx != ref_idx).any(axis=1))[0]
    for t in bad:
        kth = np.sort(ref_logits[t])[::-1][K - 1]
        chosen = ref_logits[t, gpu_idx[t]]
        assert len(set(gpu_idx[t].tolist())) == K
        assert chosen.min() >= kth - 2 * logit_err - 1e-12, (t, chosen, kth, logit_err)
        # order inside the row: non-increasing by exact logits up to the bound
        assert (np.diff(chosen) <= 2 * logit_err + 1e-12).all()
    assert len(bad) <= max(1, int(max_frac * len(ref_idx))), f"{len(bad)} ambiguous rows"
    return len(bad)


def check_topk_exact(gpu_idx, gpu_logits, K, sel_bias=None, what="top-k"):
    """Exact index parity on the GPU's own logits: the oracle's top-K (value
    descending, lowest expert first on ties) run on the fp32 logits the GPU
    emitted must give the GPU's indices bit for bit.  With a selection-only
    bias the selection value is the fp32 sum logit + bias, rounded to nearest
    even exactly as the kernels add it; numpy's float32 add rounds the same way."""
    key = np.asarray(gpu_logits, np.float32)
    if sel_bias is not None:
        key = key + np.asarray(sel_bias, np.float32)[None, :]
    ref = O.topk_experts(key.astype(np.float64), K)
    bad = np.nonzero((np.asarray(gpu_idx) != ref).any(axis=1))[0]
    assert len(bad) == 0, f"{what}: {len(bad)} rows differ from the top-K of the GPU's logits, first {bad[:5]}"


def near_tie_rows(ref_logits, K, logit_err):
    """Rows whose K-th and (K+1)-th exact logits lie within 4x the logit error:
    the only rows where the fp32 and the fp64 selections may legitimately differ."""
    E = ref_logits.shape[1]
    if K >= E:
        return 0
    srt = -np.sort(-ref_logits, axis=1)
    return int(np.count_nonzero(srt[:, K - 1] - srt[:, K] < 4 * logit_err))


def host_layer_inputs(shape, T=None, seed=0, bias=None):
    """Small-size inputs drawn on the host (all tensors), as Stored pairs."""
    x, wr = synth.router_inputs(shape, seed=seed, tokens=T)
    wg, wu, wd = synth.expert_weights_host(shape, seed=seed)
    return x, wr, wg, wu, wd
