"""Benchmark of the MoE / MoD layer hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--bias-target MAXVIO|none] [--train]
                    [--eager] [--e2e-eager]

A step is one pass of the layer over one batch of synthetic input:
  * Mixtral-shaped and fine-grained layers: router GEMM + softmax/top-K,
    dispatch (histogram, cu_seqlens, permutation, gather), grouped SwiGLU
    expert FFN, combine, then the gate/dispatch backward (moe_permute_bwd +
    moe_route_bwd) with a synthetic expert-input gradient;
  * expert-parallel benchmark shapes (E=384): the forward only;
  * MoD + MoE: mod_select, the MoE forward on the selected tokens with the
    score-scaled residual combine, then the route backward of both routers.
The default workload is the Mixtral-shaped bf16 layer (4 x 2048 tokens, H=4096,
E=8, K=2, H'=14336) with the router skewed to maxvio 0.2 by an expert-0 logit
bias from tests/golden/skew_bias.json.

`value` times replays of the whole step captured once as a CUDA graph through
the library's entry points (the host issues one launch per step); the per-call
split comes from the same calls launched one by one, each bracketed by CUDA
events, and that loop's step time is reported as `eager_ms_per_step`
(`--eager` takes `value` from it instead).  The end-to-end figure replays one
CUDA graph per iteration holding the next step's host-to-device copies, this
step's calls and the previous step's device-to-host copies (`--e2e-eager`
issues the copies and the calls from the host, call by call, instead).

Multi-GPU runs (torchrun) are replicas: every rank processes its own batch with
no data-path collective; `value` is all ranks' tokens over the slowest rank's
time ("scaling": "weak").

`--impl reference` times the CPU oracle (float64, numpy) on the host cores on a
bounded sample of the same workload per step; under torchrun only rank 0 runs.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one
# moe_expert_ffn call, both GEMM launches, from one ncu capture per workload of
# the kernels as they stand; a workload without a capture reports null
FFN_DRAM_BYTES = {
    # (workload, rows gathered by the FFN): DRAM bytes read + written by the
    # gate/up and down GEMMs of one moe_expert_ffn call (ncu dram__bytes_read.sum
    # + dram__bytes_write.sum of the two CTA-pair kernels, one launch each, full
    # size, with the tail-split workspace; at the Mixtral shape the figure moves
    # by +-5% between captures with the L2 hit rate)
    ("mixtral_bf16_T8192_H4096_E8_K2_Hp14336", False): 3252134912 + 463967488 + 3088918016 + 128402432,
    ("finegrained_bf16_T16384_H2048_E64_K6_Hp1408", False): 1157933568 + 266742016 + 646429952 + 372195840,
    ("epbench_bf16_T8192_H7168_E384_K8_Hp2048", False): 25055941632 + 269882368 + 11618349824 + 934911232,
    ("mod_bf16_B4_L2048_C1024_H2048_E16_K2_Hp5632", False): 772024064 + 84482304 + 486685952 + 23238400,
}
DEFAULT_WORKLOAD = "mixtral_bf16_T8192_H4096_E8_K2_Hp14336"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--bias-target", default="auto",
                   help="router skew (maxvio) from tests/golden/skew_bias.json; 'none' for the natural "
                        "router; 'auto' = 0.2 where the table has it")
    p.add_argument("--cpu-sample-tokens", type=int, default=None)
    p.add_argument("--eager", action="store_true",
                   help="take `value` from the calls launched one by one instead of CUDA-graph replays of the step")
    p.add_argument("--graph", action="store_true", help="(the default) time CUDA-graph replays of the step")
    p.add_argument("--e2e-eager", action="store_true",
                   help="end-to-end loop launches every call from the host instead of replaying a captured graph")
    p.add_argument("--train", action="store_true",
                   help="time the full training step (expert backward and weight gradients included; bf16)")
    p.add_argument("--route-flags", type=int, default=0,
                   help="moe_route_ex gate options: 1 renormalise the top-k gates, 2 bias for selection only")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-tail-split", action="store_true",
                   help="run the down projection's last round as whole tiles (no expert FFN workspace)")
    p.add_argument("--fused-gather", action="store_true",
                   help="the forward's dispatch writes only the index maps and the gate/up GEMM gathers the rows "
                        "of x itself (moe_expert_ffn_gather) instead of reading the rows dispatch wrote")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(times_ms, device):
    """The slowest rank's times (each rank timed the same number of steps of its
    own batch): one all-reduce(max) over the process group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(times_ms, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def whole_job_tokens_per_s(tokens_per_rank, world, ms_per_step):
    """Replicas: every rank processes its own tokens_per_rank tokens per step, so
    the job's rate is all ranks' tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def mode_of(shape):
    from token_dispatch_gb300 import synth
    if shape.mod_B:
        return "mod"
    if shape.name == synth.EPBENCH_BF16.name:
        return "fwd"
    return "fwd_bwd"


METRICS = {"fwd_bwd": "MoE layer tokens/s (fwd + gate/dispatch bwd)",
           "train": "MoE layer tokens/s (fwd + full bwd incl. expert weight gradients)",
           "fwd": "MoE layer tokens/s (fwd)",
           "mod": "MoD+MoE layer tokens/s (fwd + route bwd)"}


def skew_bias(shape, target):
    """(bias [E] or None, table entry or None, target used)."""
    path = os.path.join(ROOT, "tests", "golden", "skew_bias.json")
    with open(path) as fh:
        table = json.load(fh)
    entries = table.get(shape.name, {})
    if target in (None, "none"):
        return None, None, None
    if target == "auto":
        if "0.2" not in entries:
            return None, None, None
        target = "0.2"
    key = f"{float(target):g}"
    entry = entries[key]
    from token_dispatch_gb300 import synth
    return synth.expert_bias(shape.E, entry["beta"], expert=0), entry, float(key)


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        # raw samples: a scratch file (the JSON line carries their summary)
        self.path = os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                f = [c.strip() for c in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def algorithmic_bytes(shape, mode=None):
    """Minimum HBM bytes each HBM-bound call must move (read + write), from its
    definition: b = storage bytes, R = T*K rows; indices, gates and scores are 4
    bytes.  For the MoD workload T is the selected tokens (B*C)."""
    T, H, E, K = shape.T, shape.H, shape.E, shape.K
    R = T * K
    b = 2 if shape.dtype == "bf16" else 4
    out = {
        # x, W_r in; logits, idx, gate out
        "route": T * H * b + H * E * b + T * E * 4 + 2 * T * K * 4,
        # idx in; x in once; xs, dst_row, src_tok, cu out
        "dispatch": T * K * 4 + T * H * b + R * H * b + 2 * R * 4 + (E + 1) * 4,
        # the same without the rows (the expert FFN gathers them): latency-bound
        "dispatch_maps": T * K * 4 + 2 * R * 4 + (E + 1) * 4,
        # h, gate, dst_row in; y out (MoD: also the score and the residual rows)
        "combine": R * H * b + T * K * 4 + R * 4 + T * H * b + (T * (H * b + 8) if shape.mod_B else 0),
        # dy, h, dxs, gate, dst_row in; dh, dx, d_gate out
        "permute_bwd": T * H * b + 3 * R * H * b + T * H * b + T * K * 4 + R * 4 + T * K * 4,
        # d_gate, logits, idx, x, W_r in; d_logits, dW out; dx read + written
        "route_bwd": T * K * 4 + T * E * 4 + T * K * 4 + T * H * b + H * E * b + T * E * 4 + H * E * 4
                     + 2 * T * H * b,
    }
    if mode == "train":
        # dh, d_gate only (dy, h, gate, dst_row in); then dx = sum_k dxs[row]
        out["permute_bwd"] = T * H * b + R * H * b + R * H * b + T * K * 4 + R * 4 + T * K * 4
        out["dispatch_bwd"] = R * H * b + T * H * b + T * K * 4 + R * 4
    if shape.mod_B:
        n = shape.mod_B * shape.mod_L
        # x read once, w_mod; score, mask, sel, sel_score out; x_sel and the skip rows written
        out["mod_select"] = n * H * b + H * b + n * 4 + n + 2 * T * 4 + T * H * b + (n - T) * H * b
        # MoD route backward: dy (selected rows), h in; dh, d_gate, d_score out (no dxs)
        out["permute_bwd"] = T * H * b + 2 * R * H * b + T * K * 4 + R * 4 + T * K * 4 + T * 4 + T * 4
        out["route_bwd"] = out["route_bwd"]
        out["mod_route_bwd"] = T * 4 + T * H * b + H * b + H * 4 + 2 * T * H * b
    return out


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# --------------------------------------------------------------------------- ours

def build_inputs(shape, dev, rank, bias_np):
    """Routing inputs from the host generator (each rank its own batch), expert
    weights and the synthetic upstream gradients drawn on the device."""
    import torch
    from token_dispatch_gb300 import synth
    mode = mode_of(shape)
    n_tok = shape.mod_B * shape.mod_L if shape.mod_B else shape.T
    tdt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    x, wr = synth.router_inputs(shape, seed=rank, tokens=n_tok)
    wg, wu, wd = synth.expert_weights_device(shape, dev, seed=0)
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    inp = dict(x=x, wr=wr, wg=wg, wu=wu, wd=wd, bias=bias_np, mode=mode, n_tok=n_tok)
    if mode == "fwd_bwd":
        inp["dy"] = torch.randn((shape.T, shape.H), generator=g, device=dev).to(tdt)
        inp["dxs"] = torch.randn((shape.R, shape.H), generator=g, device=dev).to(tdt)
    elif mode == "mod":
        inp["wmod"] = synth.mod_weight(shape, seed=rank)
        inp["dy"] = torch.randn((n_tok, shape.H), generator=g, device=dev).to(tdt)
    return inp


def make_step(shape, inp, dev, stream, route_flags=0, fused=True, tail_split=True):
    """(call names, step(x, dy, dxs, marks) -> None, buffers, outputs for the host).
    fused: the forward's dispatch writes only the index maps and the expert FFN
    gathers the rows of x in its gate/up operand load (not for the training
    step, whose expert backward reads the expert-sorted rows)."""
    import torch
    from token_dispatch_gb300 import _lib as L
    from token_dispatch_gb300 import layer
    bwd_renorm = L.MOE_ROUTE_GATE_RENORM if route_flags & L.MOE_ROUTE_RENORM else 0
    T, H, E, K, Hp = shape.T, shape.H, shape.E, shape.K, shape.Hp
    R = T * K
    mode = inp["mode"]
    wr_d = inp["wr"].host.to(dev)
    bias_d = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).to(dev)
    wg, wu, wd = inp["wg"], inp["wu"], inp["wd"]

    if mode in ("fwd_bwd", "fwd", "train"):
        b = layer.MoEBuffers(T, H, E, K, Hp, shape.dtype, dev, backward=(mode != "fwd"), train=(mode == "train"))
        fws, fwsb = (b.ws_ffn, b.ws_ffn_bytes) if tail_split else (None, 0)
        calls = [
            ("route", lambda xi, dyi, dxsi: L.moe_route_ex(xi, wr_d, bias_d, T, H, E, K, b.cdt, route_flags, b.logits,
                                                          b.idx, b.gate, b.ws_route, b.ws_route_bytes,
                                                          stream=stream)),
            ("dispatch_maps" if fused else "dispatch",
             lambda xi, dyi, dxsi: L.moe_dispatch(xi, b.idx, T, H, E, K, b.cdt, b.cu, b.dst_row, b.src_tok,
                                                  None if fused else b.xs, b.ws_dispatch, b.ws_dispatch_bytes,
                                                  stream=stream)),
            ("expert_ffn", (lambda xi, dyi, dxsi: L.moe_expert_ffn_gather(xi, b.src_tok, T, b.cu, R, wg, wu, wd, E, H,
                                                                         Hp, b.cdt, b.act, None, b.h, fws, fwsb,
                                                                         stream=stream))
             if fused else
             (lambda xi, dyi, dxsi: L.moe_expert_ffn(b.xs, b.cu, R, wg, wu, wd, E, H, Hp, b.cdt, b.act, b.h,
                                                     fws, fwsb, stream=stream))),
            ("combine", lambda xi, dyi, dxsi: L.moe_combine(b.h, b.gate, b.dst_row, None, None, None, T, H, K, b.cdt,
                                                           b.y, stream=stream)),
        ]
        outs = [b.y]
        if mode == "train":
            calls[2] = ("expert_ffn", lambda xi, dyi, dxsi: L.moe_expert_ffn_ex(b.xs, b.cu, R, wg, wu, wd, E, H, Hp,
                                                                              b.cdt, b.act, b.gu, b.h, fws, fwsb,
                                                                              stream=stream))
            calls += [
                ("permute_bwd", lambda xi, dyi, dxsi: L.moe_permute_bwd(dyi, b.h, b.gate, b.dst_row, None, None,
                                                                       None, T, H, K, b.cdt, b.dh, b.d_gate, None,
                                                                       None, stream=stream)),
                ("expert_ffn_bwd", lambda xi, dyi, dxsi: L.moe_expert_ffn_bwd(
                    b.xs, b.cu, R, wg, wu, wd, E, H, Hp, b.cdt, b.gu, b.act, b.dh, b.dxs, b.dw_gate, b.dw_up,
                    b.dw_down, b.ws_ffn_bwd, b.ws_ffn_bwd_bytes, stream=stream)),
                ("dispatch_bwd", lambda xi, dyi, dxsi: L.moe_permute_bwd(None, None, b.gate, b.dst_row, None, None,
                                                                        b.dxs, T, H, K, b.cdt, None, None, None,
                                                                        b.dx, stream=stream)),
                ("route_bwd", lambda xi, dyi, dxsi: L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | bwd_renorm, b.d_gate,
                                                                   b.logits, b.idx, xi, wr_d, T, H, E, K, b.cdt,
                                                                   b.d_logits, b.dw_router, b.dx, b.ws_bwd,
                                                                   b.ws_bwd_bytes, stream=stream)),
            ]
            outs = [b.y, b.dx, b.dw_router]
        if mode == "fwd_bwd":
            calls += [
                ("permute_bwd", lambda xi, dyi, dxsi: L.moe_permute_bwd(dyi, b.h, b.gate, b.dst_row, None, None,
                                                                       dxsi, T, H, K, b.cdt, b.dh, b.d_gate, None,
                                                                       b.dx, stream=stream)),
                ("route_bwd", lambda xi, dyi, dxsi: L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | bwd_renorm, b.d_gate,
                                                                   b.logits,
                                                                   b.idx, xi, wr_d, T, H, E, K, b.cdt, b.d_logits,
                                                                   b.dw_router, b.dx, b.ws_bwd, b.ws_bwd_bytes,
                                                                   stream=stream)),
            ]
            outs = [b.y, b.dx, b.dw_router]
        return calls, b, outs, b.cu

    # MoD + MoE
    Bq, Lq, C = shape.mod_B, shape.mod_L, shape.mod_C
    m = layer.MoDBuffers(Bq, Lq, C, H, E, K, Hp, shape.dtype, dev)
    b = m.moe
    fws, fwsb = (b.ws_ffn, b.ws_ffn_bytes) if tail_split else (None, 0)
    wmod_d = inp["wmod"].host.to(dev)
    calls = [
        ("mod_select", lambda xi, dyi, dxsi: L.mod_select(xi, wmod_d, Bq, Lq, H, C, m.cdt, m.score, m.sel,
                                                         m.sel_score, m.mask, m.x_sel, m.y, stream=stream)),
        ("route", lambda xi, dyi, dxsi: L.moe_route(m.x_sel, wr_d, bias_d, T, H, E, K, b.cdt, b.logits, b.idx,
                                                   b.gate, b.ws_route, b.ws_route_bytes, stream=stream)),
        ("dispatch_maps" if fused else "dispatch",
         lambda xi, dyi, dxsi: L.moe_dispatch(m.x_sel, b.idx, T, H, E, K, b.cdt, b.cu, b.dst_row, b.src_tok,
                                              None if fused else b.xs, b.ws_dispatch, b.ws_dispatch_bytes,
                                              stream=stream)),
        ("expert_ffn", (lambda xi, dyi, dxsi: L.moe_expert_ffn_gather(m.x_sel, b.src_tok, T, b.cu, R, wg, wu, wd, E,
                                                                     H, Hp, b.cdt, b.act, None, b.h, fws, fwsb,
                                                                     stream=stream))
         if fused else
         (lambda xi, dyi, dxsi: L.moe_expert_ffn(b.xs, b.cu, R, wg, wu, wd, E, H, Hp, b.cdt, b.act, b.h,
                                                 fws, fwsb, stream=stream))),
        ("combine", lambda xi, dyi, dxsi: L.moe_combine(b.h, b.gate, b.dst_row, m.sel_score, xi, m.sel, T, H, K,
                                                       b.cdt, m.y, stream=stream)),
        ("permute_bwd", lambda xi, dyi, dxsi: L.moe_permute_bwd(dyi, b.h, b.gate, b.dst_row, m.sel_score, m.sel,
                                                               None, T, H, K, b.cdt, b.dh, b.d_gate, m.d_score,
                                                               None, stream=stream)),
        ("route_bwd", lambda xi, dyi, dxsi: L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | L.MOE_ROUTE_DX_WRITE,
                                                           b.d_gate, b.logits, b.idx, m.x_sel, wr_d, T, H, E, K,
                                                           b.cdt, b.d_logits, b.dw_router, b.dx, b.ws_bwd,
                                                           b.ws_bwd_bytes, stream=stream)),
        ("mod_route_bwd", lambda xi, dyi, dxsi: L.moe_route_bwd(L.MOE_ROUTE_MOD_LINEAR, m.d_score, None, None,
                                                               m.x_sel, wmod_d, T, H, 1, 1, b.cdt, None, m.dw_mod,
                                                               b.dx, m.ws_lin, m.ws_lin_bytes, stream=stream)),
    ]
    return calls, m, [m.y, m.dw_mod, b.dw_router], b.cu


def run_ours(args, shape, rank, world, local):
    import torch
    from token_dispatch_gb300 import _lib as L

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    T, H, E, K, Hp = shape.T, shape.H, shape.E, shape.K, shape.Hp
    R = T * K
    bias_np, bias_entry, target = skew_bias(shape, args.bias_target)
    inp = build_inputs(shape, dev, rank, bias_np)
    if args.train:
        if inp["mode"] not in ("fwd_bwd", "fwd") or shape.dtype != "bf16":
            raise SystemExit("--train needs a bf16 MoE workload")
        inp["mode"] = "train"
        inp.pop("dxs", None)  # the expert backward produces dxs
    mode = inp["mode"]
    n_tok = inp["n_tok"]
    x_h = inp["x"].host.pin_memory()
    x_d = x_h.to(dev)
    dy_d, dxs_d = inp.get("dy"), inp.get("dxs")
    stream = torch.cuda.Stream(device=dev)
    fused = args.fused_gather and mode != "train"
    calls, bufs, outs, cu = make_step(shape, inp, dev, stream, args.route_flags, fused, not args.no_tail_split)
    names = [n for n, _ in calls]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another: the write-back of the
        # dirty lines happens here, not inside the next timed step
        flush.fill_(1)
        flush_rd.sum()

    def step(xi, dyi, dxsi, ev=None):
        for j, (_, fn) in enumerate(calls):
            if ev is not None:
                ev[j].record(stream)
            fn(xi, dyi, dxsi)
        if ev is not None:
            ev[len(calls)].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(x_d, dy_d, dxs_d)
            flush_l2()
        # kernels each call launches (the library counts its own launches)
        n_launch = {}
        for name, fn in calls:
            c0 = L.moe_kernel_launches()
            fn(x_d, dy_d, dxs_d)
            n_launch[name] = L.moe_kernel_launches() - c0
    st = L.moe_last_device_error(stream)
    if st != L.MOE_OK:
        raise RuntimeError(f"device error after warm-up: {L.moe_status_str(st)}")
    counts = np.diff(cu.cpu().numpy().astype(np.int64))
    maxvio = float(counts.max() / (R / E) - 1.0)

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    nc = len(calls)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nc + 1)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    launches0 = L.moe_kernel_launches()
    with torch.cuda.stream(stream):
        # the first timed step follows a flush like every other one, so the
        # host has enqueued it before the device reaches its first event
        flush_l2()
        for i in range(args.steps):
            step(x_d, dy_d, dxs_d, evs[i])
            flush_l2()  # between timed steps, outside the step's events
    torch.cuda.synchronize(dev)
    barrier()
    launches = L.moe_kernel_launches() - launches0
    step_ms = [evs[i][0].elapsed_time(evs[i][nc]) for i in range(args.steps)]
    call_ms = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
               for j, n in enumerate(names)}
    ms = statistics.mean(step_ms)
    eager_ms = ms

    if fused:
        # the step's dispatch writes index maps only; the row-materialising
        # dispatch (what a caller without the fused FFN runs) is timed on its
        # own, on the step's routing, for its HBM roofline
        b_moe = bufs.moe if hasattr(bufs, "moe") else bufs
        d_in = bufs.x_sel if hasattr(bufs, "moe") else x_d
        dev_ = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            flush_l2()
            for i in range(args.steps):
                dev_[i][0].record(stream)
                L.moe_dispatch(d_in, b_moe.idx, b_moe.T, b_moe.H, b_moe.E, b_moe.K, b_moe.cdt, b_moe.cu,
                               b_moe.dst_row, b_moe.src_tok, b_moe.xs, b_moe.ws_dispatch, b_moe.ws_dispatch_bytes,
                               stream=stream)
                dev_[i][1].record(stream)
                flush_l2()
        torch.cuda.synchronize(dev)
        call_ms["dispatch"] = statistics.mean(a.elapsed_time(c) for a, c in dev_)
        c0 = L.moe_kernel_launches()
        L.moe_dispatch(d_in, b_moe.idx, b_moe.T, b_moe.H, b_moe.E, b_moe.K, b_moe.cdt, b_moe.cu, b_moe.dst_row,
                       b_moe.src_tok, b_moe.xs, b_moe.ws_dispatch, b_moe.ws_dispatch_bytes, stream=stream)
        n_launch["dispatch"] = L.moe_kernel_launches() - c0

    # The fixed cost of a call as the events see it: n back-to-back launches of
    # a one-element kernel between two events (each repetition after an L2
    # flush, so the host is ahead of the device as in the timed steps; the
    # fastest of 10).  A call of B bytes in n launches can at best take
    # floor(n) + B / peak.
    with torch.cuda.stream(stream):
        tiny = torch.zeros(1, device=dev)
    launch_floor_ms = {}
    for n in sorted(set(n_launch.values())):
        pairs = []
        with torch.cuda.stream(stream):
            for _ in range(10):
                flush_l2()
                a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(n):
                    tiny.add_(1)
                c.record(stream)
                pairs.append((a, c))
        torch.cuda.synchronize(dev)
        launch_floor_ms[n] = min(a.elapsed_time(c) for a, c in pairs)

    def capture(xi, dyi, dxsi):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            step(xi, dyi, dxsi)
        return g

    if not args.eager:
        # the whole step as one CUDA graph: the library's launches are recorded
        # once (counted here) and replayed with no host work per kernel
        n0 = L.moe_kernel_launches()
        graph_main = capture(x_d, dy_d, dxs_d)
        per_step = L.moe_kernel_launches() - n0
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):  # untimed replays first
                graph_main.replay()
                flush_l2()
        barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            flush_l2()
            for i in range(args.steps):
                gev[i][0].record(stream)
                graph_main.replay()
                gev[i][1].record(stream)
                flush_l2()
        torch.cuda.synchronize(dev)
        barrier()
        ms = statistics.mean(a.elapsed_time(b) for a, b in gev)
        launches = per_step * args.steps

    # End to end through the public API: every step copies its inputs from pinned
    # host memory and its results back.  Inputs are double-buffered: the next
    # step's host-to-device copies run on a copy stream while this step computes.
    # Results are read back to pinned host memory on a third stream while the
    # next step computes: from a second set of layer buffers used on alternate
    # steps (graph iterations), or, issued from the host (--e2e-eager), after a
    # device copy into a double-buffered staging area.  The timed region ends
    # when the last step's results are on the host.
    srcs = [x_h] + ([dy_d.cpu().pin_memory()] if dy_d is not None else []) + \
        ([dxs_d.cpu().pin_memory()] if dxs_d is not None else [])
    bufs_in = [[torch.empty_like(h, device=dev) for h in srcs] for _ in range(2)]
    host_out = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs] for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    # every transfer is cut into pieces on several streams, so several copy
    # engines move a step's inputs (and results) at once
    N_COPY = 4
    h2d_sub = [torch.cuda.Stream(device=dev) for _ in range(N_COPY)]
    d2h_sub = [torch.cuda.Stream(device=dev) for _ in range(N_COPY)]

    def split_copy(pairs, lead, subs):
        # pairs of (destination, source); pieces on the sub-streams after `lead`,
        # joined back into `lead`
        start = torch.cuda.Event()
        start.record(lead)
        for j, sub in enumerate(subs):
            sub.wait_event(start)
            with torch.cuda.stream(sub):
                for dst, src in pairs:
                    n = dst.numel()
                    a, b = n * j // len(subs), n * (j + 1) // len(subs)
                    if b > a:
                        dst.view(-1)[a:b].copy_(src.view(-1)[a:b], non_blocking=True)
            done = torch.cuda.Event()
            done.record(sub)
            lead.wait_event(done)
    e2e_steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def join(side):
        # the step's stream waits for everything issued so far on `side`
        ev = torch.cuda.Event()
        ev.record(side)
        stream.wait_event(ev)

    if not args.e2e_eager:
        # One CUDA graph per iteration (built once per input slot and position):
        # the next step's inputs go up on the copy streams, this step's calls
        # run through the public entry points into the slot's own layer
        # buffers, and the previous step's results go down from the other
        # slot's buffers, all three concurrent inside the graph; consecutive
        # graphs on the step's stream run one after the other, so step i+1
        # reads inputs loaded in iteration i and step i's results are read back
        # in iteration i+1, before iteration i+2 overwrites them.
        calls_b, _, outs_b, _ = make_step(shape, inp, dev, stream, args.route_flags, fused,
                                          not args.no_tail_split)
        slot_calls, slot_outs = [calls, calls_b], [outs, outs_b]

        def iteration_graph(slot, load_next, read_prev):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                fork = torch.cuda.Event()
                fork.record(stream)
                if load_next:
                    copy_stream.wait_event(fork)
                    split_copy(list(zip(bufs_in[1 - slot], srcs)), copy_stream, h2d_sub)
                if read_prev:
                    d2h_stream.wait_event(fork)
                    split_copy(list(zip(host_out[1 - slot], slot_outs[1 - slot])), d2h_stream, d2h_sub)
                ins = bufs_in[slot] + [None, None]
                for _, fn in slot_calls[slot]:
                    fn(ins[0], ins[1], ins[2])
                if load_next:
                    join(copy_stream)
                if read_prev:
                    join(d2h_stream)
            return g
        keys = [(i % 2, i + 1 < e2e_steps, i >= 1) for i in range(e2e_steps)]
        graphs = {k: iteration_graph(*k) for k in sorted(set(keys))}
        torch.cuda.synchronize(dev)
        e0.record(stream)
        copy_stream.wait_event(e0)
        split_copy(list(zip(bufs_in[0], srcs)), copy_stream, h2d_sub)  # step 0's inputs
        join(copy_stream)
        with torch.cuda.stream(stream):
            for k in keys:
                graphs[k].replay()
        last = (e2e_steps - 1) % 2
        tail = torch.cuda.Event()
        tail.record(stream)
        d2h_stream.wait_event(tail)
        split_copy(list(zip(host_out[last], slot_outs[last])), d2h_stream, d2h_sub)  # the last results
        join(d2h_stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    else:
        stage_out = [[torch.empty_like(o) for o in outs] for _ in range(2)]
        loaded = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        staged = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]

        def load(i):
            slot = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(consumed[slot])  # step i-2 no longer reads this slot
                split_copy(list(zip(bufs_in[slot], srcs)), copy_stream, h2d_sub)
                loaded[slot].record(copy_stream)

        torch.cuda.synchronize(dev)
        e0.record(stream)
        copy_stream.wait_event(e0)
        d2h_stream.wait_event(e0)
        load(0)
        for i in range(e2e_steps):
            if i + 1 < e2e_steps:
                load(i + 1)
            slot = i % 2
            stream.wait_event(loaded[slot])
            with torch.cuda.stream(stream):
                ins = bufs_in[slot] + [None, None]
                step(ins[0], ins[1], ins[2])
                consumed[slot].record(stream)
                if i >= 2:
                    stream.wait_event(read_back[slot])  # step i-2's results are on the host
                for d, st in zip(outs, stage_out[slot]):
                    st.copy_(d, non_blocking=True)
                staged[slot].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(staged[slot])
                split_copy(list(zip(host_out[slot], stage_out[slot])), d2h_stream, d2h_sub)
                read_back[slot].record(d2h_stream)
        stream.wait_event(read_back[(e2e_steps - 1) % 2])
        e1.record(stream)
        torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    clk = clocks.stop()
    h2d = sum(h.numel() * h.element_size() for h in srcs)
    d2h = sum(h.numel() * h.element_size() for h in host_out[0])

    if world > 1:
        ms, e2e_ms = max_over_ranks([ms, e2e_ms], dev)

    peaks, peak_src = measured_peaks()
    ffn_flops = 6.0 * R * H * Hp
    ffn_s = call_ms["expert_ffn"] * 1e-3
    b_el = 2 if shape.dtype == "bf16" else 4
    # the pair's minimum DRAM bytes: every expert's three projections once, xs
    # read, the SwiGLU output written and read back, h written
    ffn_bytes = 3 * E * H * Hp * b_el + (T if fused else R) * H * b_el + 2 * R * Hp * b_el + R * H * b_el
    if mode == "train":
        # forward also writes [g | u]; backward: 12 R H H' FLOP; reads dh, the
        # three projections, [g | u], act, xs; writes and reads back [dg | du];
        # writes dxs and the three fp32 weight gradients
        ffn_flops += 12.0 * R * H * Hp
        ffn_s += call_ms["expert_ffn_bwd"] * 1e-3
        ffn_bytes += 2 * R * Hp * b_el + (R * H * b_el + 3 * E * H * Hp * b_el + 2 * R * Hp * b_el + R * Hp * b_el
                                          + R * H * b_el + 2 * 2 * R * Hp * b_el + R * H * b_el + 3 * E * H * Hp * 4)
    # The burst bf16 peak applies to a kernel timed alone; when the power cap
    # engaged during the timed steps the kernel ran inside a long step, and the
    # sustained peak (measured under the same cap) is the ceiling.  Both
    # fractions are reported.
    capped = bool(clk) and "sw_power_cap" in clk.get("reasons", [])
    peak_burst = peaks.get("bf16_tflops", 1900.0)
    peak_tf = (peaks.get("bf16_tflops_sustained", 1700.0) if capped else peak_burst) \
        if shape.dtype == "bf16" else None
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    if shape.dtype != "bf16":
        # fp32 layers run on FFMA: the peak is SMs x 128 FP32 lanes x 2 FLOP x the
        # maximum SM clock (152 x 128 x 2 x 2.07 GHz = 80.5 TFLOP/s on GB300)
        import torch
        n_sm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        sm_hz = peaks.get("sm_max_mhz", 2070.0) * 1e6
        roof = {"bound": "alu", "achieved": ffn_flops / ffn_s / 1e12, "peak": n_sm * 128 * 2 * sm_hz / 1e12,
                "unit": "TFLOP/s", "peak_source": f"derived: {n_sm} SMs x 128 FP32 lanes x 2 x max SM clock"}
    elif ffn_flops / (peak_tf * 1e12) >= ffn_bytes / (hbm_peak * 1e9):
        roof = {"bound": "tensor", "achieved": ffn_flops / ffn_s / 1e12, "peak": peak_tf, "unit": "TFLOP/s",
                "peak_source": f"{peak_src} bf16_tflops" + ("_sustained (sw_power_cap seen)" if capped else
                                                            " (burst)"),
                "frac_of_burst": ffn_flops / ffn_s / 1e12 / peak_burst}
    else:  # weight streaming bounds the pair (few rows per expert)
        roof = {"bound": "hbm", "achieved": ffn_bytes / ffn_s / 1e9, "peak": hbm_peak, "unit": "GB/s",
                "peak_source": f"{peak_src} hbm_gbs"}
    roof["frac"] = roof["achieved"] / roof["peak"] if roof["peak"] else None
    if roof["bound"] == "tensor" and mode != "train" and not fused:
        # the CTA-pair GEMMs compute whole 256-row tiles per expert (gate/up:
        # 128 SwiGLU columns per tile, down: 256 columns): the share of the
        # FLOP they issue that the routed rows need
        m_pad = float(np.sum((counts + 255) // 256 * 256))
        hp128, h256, hp64 = -(-Hp // 128) * 128, -(-H // 256) * 256, -(-Hp // 64) * 64
        issued = 2.0 * m_pad * H * 2 * hp128 + 2.0 * m_pad * hp64 * h256
        roof["tile_fill"] = round(6.0 * R * H * Hp / issued, 4)
    roof["traffic"] = None if mode == "train" else FFN_DRAM_BYTES.get((shape.name, fused))
    roof["algorithmic"] = {"flops": ffn_flops, "bytes": ffn_bytes}
    hbm = {}
    for name, nbytes in algorithmic_bytes(shape, mode).items():
        if name in call_ms:
            gbs = nbytes / (call_ms[name] * 1e-3) / 1e9
            hbm[name] = {"bytes": nbytes, "GB/s": round(gbs, 1), "frac": round(gbs / hbm_peak, 4)}
            n = n_launch.get(name)
            if n in launch_floor_ms:
                best_ms = launch_floor_ms[n] + nbytes / (hbm_peak * 1e9) * 1e3
                hbm[name].update({"launches": n, "floor_us": round(launch_floor_ms[n] * 1e3, 2),
                                  "attainable_GB/s": round(nbytes / (best_ms * 1e-3) / 1e9, 1),
                                  "frac_of_attainable": round(best_ms / call_ms[name], 4)})
    result = {
        "metric": METRICS[mode],
        "value": whole_job_tokens_per_s(n_tok, world, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms,
        "eager_ms_per_step": eager_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": shape.dtype,
        "data": "synthetic",
        "config": {"workload": shape.name, "tokens_per_gpu": n_tok, "moe_tokens": T, "H": H, "E": E, "K": K,
                   "Hp": Hp, "maxvio": round(maxvio, 4), "maxvio_target": target,
                   "expert0_logit_bias": None if bias_entry is None else bias_entry["beta"],
                   "l2": "flushed between timed steps (512 MB write, then 512 MB read)", "parallelism": f"replicas{world}",
                   "route_flags": args.route_flags, "train": bool(args.train), "graph": not args.eager,
                   "fused_gather": fused, "tail_split": not args.no_tail_split},
        "calls_ms": {k: round(v, 4) for k, v in call_ms.items()},
        "roofline": {"kernel": ("moe_expert_ffn + moe_expert_ffn_bwd (grouped tcgen05 GEMMs, forward and backward)"
                                if mode == "train" else
                                "moe_expert_ffn_gather (grouped gate/up+SwiGLU GEMM gathering the rows of x, "
                                "+ down GEMM, tcgen05)" if fused else
                                "moe_expert_ffn (grouped gate/up+SwiGLU GEMM + down GEMM, tcgen05)"), **roof},
        "hbm_roofline": {"peak_GB/s": hbm_peak, "peak_source": f"{peak_src} hbm_gbs", "calls": hbm},
        "e2e": {"value": whole_job_tokens_per_s(n_tok, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "launch": ("host, call by call" if args.e2e_eager else
                           "one CUDA graph per iteration: the next step's host-to-device copies, this step's "
                           "calls and staging, the previous step's device-to-host copies")},
        "gpu_launches": launches,
        "clocks": clk,
    }
    return result, inp


# ----------------------------------------------------------------- CPU oracle arm

def oracle_sample(shape, inp, n_tok, reps=1, route_flags=0):
    """Time the CPU oracle on a bounded sample of the step: the first n_tok tokens
    (MoE workloads) or the first sequence (MoD workload).  Returns (times, tokens)."""
    import oracle as O
    from token_dispatch_gb300 import synth
    mode = inp["mode"]
    bias = None if inp["bias"] is None else inp["bias"].astype(np.float64)
    wr64 = inp["wr"].ref
    if mode == "mod":
        n_tok = shape.mod_L
    n_tok = min(n_tok, inp["x"].ref.shape[0])  # never more tokens than the batch has
    x64 = inp["x"].ref[:n_tok]

    # the experts this sample visits, copied to the host in float64
    if mode == "mod":
        s = O.mod_scores(x64, inp["wmod"].ref)
        sel, _ = O.mod_select(s, 1, shape.mod_L, shape.mod_C)
        xr = x64[sel[0]]
    else:
        xr = x64
    experts = sorted(set(O.topk_experts(O.router_logits(xr, wr64, bias), shape.K).reshape(-1).tolist()))

    class Experts:
        def __init__(self, w):
            self.shape = tuple(w.shape)
            self.a = dict(zip(experts, synth.weights_to_host(w, experts)))

        def __getitem__(self, e):
            return self.a[e]

    wg, wu, wd = Experts(inp["wg"]), Experts(inp["wu"]), Experts(inp["wd"])
    dy = None if "dy" not in inp else inp["dy"][:n_tok].float().cpu().numpy().astype(np.float64)
    dxs = None if "dxs" not in inp else inp["dxs"][:n_tok * shape.K].float().cpu().numpy().astype(np.float64)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        if mode == "mod":
            f = O.mod_forward(x64, inp["wmod"].ref, wr64, wg, wu, wd, 1, shape.mod_L, shape.mod_C, shape.K)
            inner = f["inner"]
            _, d_gate, d_score, _ = O.permute_bwd(dy, inner["h"], inner["gate"], inner["dst_row"],
                                                  row_scale=f["score"][f["flat"]], out_row=f["flat"])
            O.route_bwd_softmax_topk(d_gate, inner["logits"], inner["idx"], f["x_sel"], wr64)
            O.route_bwd_linear(d_score, f["x_sel"], inp["wmod"].ref)
        else:
            f = O.moe_forward(x64, wr64, wg, wu, wd, shape.K, bias, renorm=bool(route_flags & 1),
                              bias_select_only=bool(route_flags & 2))
            if mode == "fwd_bwd":
                O.moe_backward(f, dy, dxs, x64, wr64, renorm=bool(route_flags & 1))
            elif mode == "train":
                dh = O.permute_bwd(dy, f["h"], f["gate"], f["dst_row"])[0]
                dxs_t = np.zeros_like(f["xs"])
                for e in experts:
                    lo, hi = int(f["cu"][e]), int(f["cu"][e + 1])
                    if hi > lo:  # dxs rows and the expert's three weight gradients
                        dxs_t[lo:hi] = O.expert_swiglu_bwd(f["xs"][lo:hi], wg[e], wu[e], wd[e], dh[lo:hi])[0]
                O.moe_backward(f, dy, dxs_t, x64, wr64, renorm=bool(route_flags & 1))
        times.append(time.perf_counter() - t0)
    return times, n_tok


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def default_sample(mode):
    return {"fwd_bwd": 4096, "train": 2048, "fwd": 512, "mod": None}[mode]


def main():
    args = parse()
    rank, world, local = dist_env()
    from token_dispatch_gb300 import synth
    shape = synth.WORKLOADS[args.workload]
    mode = mode_of(shape)
    if args.train:
        if mode not in ("fwd_bwd", "fwd") or shape.dtype != "bf16":
            raise SystemExit("--train needs a bf16 MoE workload")
        mode = "train"

    if args.impl == "reference":
        if rank != 0:
            return
        import torch
        dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
        bias_np, _, target = skew_bias(shape, args.bias_target)
        inp = build_inputs(shape, dev, 0, bias_np)  # drawn exactly as the GPU arm draws them
        if mode == "train":
            inp["mode"] = "train"
            inp.pop("dxs", None)
        n_tok = args.cpu_sample_tokens or {"fwd_bwd": 32, "train": 32, "fwd": 8, "mod": None}[mode]
        oracle_sample(shape, inp, n_tok, reps=1, route_flags=args.route_flags)
        times, n_tok = oracle_sample(shape, inp, n_tok, reps=args.steps, route_flags=args.route_flags)
        ms = 1e3 * statistics.mean(times)
        val = n_tok / (ms * 1e-3)
        sample = f"first {n_tok} tokens of the batch per step" if mode != "mod" else \
            "first sequence (2048 tokens, 1024 selected) per step"
        out = {"metric": METRICS[mode], "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
               "warmup": 1, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
               "config": {"workload": shape.name, "maxvio_target": target, "route_flags": args.route_flags,
                          "train": bool(args.train)},
               "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                                "sample": sample},
               "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(out))
        return

    result, inp = run_ours(args, shape, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_tok = args.cpu_sample_tokens or default_sample(mode)
        times, n_tok = oracle_sample(shape, inp, n_tok, reps=1, route_flags=args.route_flags)
        what = "the first sequence (MoD select + MoE on 1024 tokens + route bwd)" if mode == "mod" else \
            f"first {n_tok} tokens of the batch " \
            f"({ {'fwd_bwd': 'fwd + gate/dispatch bwd', 'train': 'fwd + full bwd', 'fwd': 'fwd'}[mode] })"
        result["cpu_baseline"] = {"value": n_tok / times[0], "unit": "tokens/s", "cores": cores(),
                                  "kind": "oracle",
                                  "sample": f"{what}, float64 numpy ({times[0]:.1f} s)"}
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
