"""Benchmark of the MoE layer hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--bias-target MAXVIO]

A step is one pass of the layer on one batch of synthetic input: router GEMM +
softmax/top-K, dispatch (histogram, cu_seqlens, permutation, gather), grouped
SwiGLU expert FFN, combine, and the gate/dispatch backward (moe_permute_bwd +
moe_route_bwd).  The default workload is the Mixtral-shaped bf16 layer
(4 x 2048 tokens, H=4096, E=8, K=2, H'=14336, uniform router).

Multi-GPU runs (torchrun) are replicas: every rank processes its own batch with
no data-path collective; `value` is all ranks' tokens over the slowest rank's
time ("scaling": "weak").

`--impl reference` times the CPU oracle (float64, numpy) on the host cores on a
bounded token sample of the same workload per step; under torchrun only rank 0
runs it.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s (fwd + gate/dispatch bwd)"
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="mixtral_bf16_T8192_H4096_E8_K2_Hp14336")
    p.add_argument("--bias-target", type=float, default=None,
                   help="router skew target (maxvio) from tests/golden/skew_bias.json")
    p.add_argument("--cpu-sample-tokens", type=int, default=None)
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def skew_bias(shape, target):
    if target is None:
        return None, None
    path = os.path.join(ROOT, "tests", "golden", "skew_bias.json")
    with open(path) as fh:
        table = json.load(fh)
    entry = table[shape.name][f"{target:g}"]
    from token_dispatch_gb300 import synth
    return synth.expert_bias(shape.E, entry["beta"], expert=0), entry


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_bench_{os.getpid()}.csv")

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


def algorithmic_bytes(shape):
    """Minimum HBM bytes each HBM-bound call must move (read + write), from its
    definition: b = storage bytes, R = T*K rows; indices and gates are 4 bytes."""
    T, H, E, K = shape.T, shape.H, shape.E, shape.K
    R = T * K
    b = 2 if shape.dtype == "bf16" else 4
    return {
        # x, W_r in; logits, idx, gate out
        "route": T * H * b + H * E * b + T * E * 4 + 2 * T * K * 4,
        # idx in; x in once; xs, dst_row, src_tok, cu out
        "dispatch": T * K * 4 + T * H * b + R * H * b + 2 * R * 4 + (E + 1) * 4,
        # h, gate, dst_row in; y out
        "combine": R * H * b + T * K * 4 + R * 4 + T * H * b,
        # dy, h, dxs, gate, dst_row in; dh, dx, d_gate out
        "permute_bwd": T * H * b + 3 * R * H * b + T * H * b + T * K * 4 + R * 4 + T * K * 4,
        # d_gate, logits, idx, x, W_r in; d_logits, dW out; dx read + written
        "route_bwd": T * K * 4 + T * E * 4 + T * K * 4 + T * H * b + H * E * b + T * E * 4 + H * E * 4
                     + 2 * T * H * b,
    }


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# --------------------------------------------------------------------------- ours

def run_ours(args, shape, rank, world, local):
    import torch
    from token_dispatch_gb300 import _lib as L
    from token_dispatch_gb300 import layer, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    T, H, E, K, Hp = shape.T, shape.H, shape.E, shape.K, shape.Hp
    R = T * K
    tdt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    bias_np, bias_entry = skew_bias(shape, args.bias_target)

    # inputs: routing inputs from the host generator (each rank its own batch),
    # expert weights and the synthetic upstream gradients drawn on the device
    x, wr = synth.router_inputs(shape, seed=rank)
    x_h = x.host.pin_memory()
    wr_d = wr.host.to(dev)
    bias_d = None if bias_np is None else torch.from_numpy(bias_np).to(dev)
    wg, wu, wd = synth.expert_weights_device(shape, dev, seed=0)
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    dy_d = torch.randn((T, H), generator=g, device=dev, dtype=torch.float32).to(tdt)
    dxs_d = torch.randn((R, H), generator=g, device=dev, dtype=torch.float32).to(tdt)
    x_d = x_h.to(dev)
    b = layer.MoEBuffers(T, H, E, K, Hp, shape.dtype, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    names = ("route", "dispatch", "expert_ffn", "combine", "permute_bwd", "route_bwd")

    def step(xin, dyin, dxsin, ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        L.moe_route(xin, wr_d, bias_d, T, H, E, K, b.cdt, b.logits, b.idx, b.gate, stream=stream)
        mark(1)
        L.moe_dispatch(xin, b.idx, T, H, E, K, b.cdt, b.cu, b.dst_row, b.src_tok, b.xs, b.ws_dispatch,
                       b.ws_dispatch_bytes, stream=stream)
        mark(2)
        L.moe_expert_ffn(b.xs, b.cu, R, wg, wu, wd, E, H, Hp, b.cdt, b.act, b.h, stream=stream)
        mark(3)
        L.moe_combine(b.h, b.gate, b.dst_row, None, None, None, T, H, K, b.cdt, b.y, stream=stream)
        mark(4)
        L.moe_permute_bwd(dyin, b.h, b.gate, b.dst_row, None, None, dxsin, T, H, K, b.cdt, b.dh, b.d_gate,
                          None, b.dx, stream=stream)
        mark(5)
        L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK, b.d_gate, b.logits, b.idx, xin, wr_d, T, H, E, K, b.cdt,
                        b.d_logits, b.dw_router, b.dx, b.ws_bwd, b.ws_bwd_bytes, stream=stream)
        mark(6)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(x_d, dy_d, dxs_d)
            flush.fill_(1)
    st = L.moe_last_device_error(stream)
    if st != L.MOE_OK:
        raise RuntimeError(f"device error after warm-up: {L.moe_status_str(st)}")

    counts = np.diff(b.cu.cpu().numpy().astype(np.int64))
    maxvio = float(counts.max() / (R / E) - 1.0)

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    launches0 = L.moe_kernel_launches()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            step(x_d, dy_d, dxs_d, evs[i])
            flush.fill_(1)  # L2 flush between timed steps (outside the step's events)
    torch.cuda.synchronize(dev)
    barrier()
    launches = L.moe_kernel_launches() - launches0
    step_ms = [evs[i][0].elapsed_time(evs[i][6]) for i in range(args.steps)]
    call_ms = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
               for j, n in enumerate(names)}
    ms = statistics.mean(step_ms)

    # end to end through the public API: pinned host inputs in, results out, every step
    dy_h = dy_d.cpu().pin_memory()
    dxs_h = dxs_d.cpu().pin_memory()
    y_h = torch.empty((T, H), dtype=tdt).pin_memory()
    dx_h = torch.empty((T, H), dtype=tdt).pin_memory()
    dw_h = torch.empty((H, E), dtype=torch.float32).pin_memory()
    x_in = torch.empty_like(x_d)
    dy_in = torch.empty_like(dy_d)
    dxs_in = torch.empty_like(dxs_d)
    e2e_steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            x_in.copy_(x_h, non_blocking=True)
            dy_in.copy_(dy_h, non_blocking=True)
            dxs_in.copy_(dxs_h, non_blocking=True)
            step(x_in, dy_in, dxs_in)
            y_h.copy_(b.y, non_blocking=True)
            dx_h.copy_(b.dx, non_blocking=True)
            dw_h.copy_(b.dw_router, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    clk = clocks.stop()

    h2d = x_in.numel() * x_in.element_size() + dy_in.numel() * dy_in.element_size() + \
        dxs_in.numel() * dxs_in.element_size()
    d2h = y_h.numel() * y_h.element_size() + dx_h.numel() * dx_h.element_size() + dw_h.numel() * 4

    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms, e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, e2e_ms = float(t[0]), float(t[1])

    peaks, peak_src = measured_peaks()
    ffn_flops = 6.0 * R * H * Hp
    ffn_ms = call_ms["expert_ffn"]
    tflops = ffn_flops / (ffn_ms * 1e-3) / 1e12
    # the timed region is well under a second: the burst peak applies
    peak_tf = peaks.get("bf16_tflops", 1900.0) if shape.dtype == "bf16" else None
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    hbm = {}
    for name, nbytes in algorithmic_bytes(shape).items():
        gbs = nbytes / (call_ms[name] * 1e-3) / 1e9
        hbm[name] = {"bytes": nbytes, "GB/s": round(gbs, 1), "frac": round(gbs / hbm_peak, 4)}
    result = {
        "metric": METRIC,
        "value": world * T / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": shape.dtype,
        "data": "synthetic",
        "config": {"workload": shape.name, "tokens_per_gpu": T, "H": H, "E": E, "K": K, "Hp": Hp,
                   "maxvio": round(maxvio, 4), "bias_target": args.bias_target,
                   "l2": "flushed between timed steps (512 MB write)", "parallelism": f"replicas{world}"},
        "calls_ms": {k: round(v, 4) for k, v in call_ms.items()},
        "roofline": {"kernel": "moe_expert_ffn (grouped gate/up+SwiGLU GEMM + down GEMM)",
                     "bound": "tensor", "achieved": tflops, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": (tflops / peak_tf) if peak_tf else None, "traffic": None,
                     "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "hbm_roofline": {"peak_GB/s": hbm_peak, "peak_source": f"{peak_src} hbm_gbs", "calls": hbm},
        "e2e": {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "clocks": clk,
    }
    return result, dict(x=x, wr=wr, wg=wg, wu=wu, wd=wd, bias=bias_np, dy=dy_d, dxs=dxs_d, dev=dev)


# ----------------------------------------------------------------- CPU oracle arm

def oracle_sample(shape, inputs, n_tok, reps=1):
    """Time the CPU oracle (fwd + gate/dispatch bwd) on the first n_tok tokens."""
    import torch
    import oracle as O
    from token_dispatch_gb300 import synth

    x64 = inputs["x"].ref[:n_tok]
    wr64 = inputs["wr"].ref
    bias = None if inputs["bias"] is None else inputs["bias"].astype(np.float64)
    idx = O.topk_experts(O.router_logits(x64, wr64, bias), shape.K)
    experts = sorted(set(idx.reshape(-1).tolist()))

    class Experts:  # host float64 copies of the experts this sample visits
        def __init__(self, w):
            self.shape = tuple(w.shape)
            self.a = dict(zip(experts, synth.weights_to_host(w, experts)))

        def __getitem__(self, e):
            return self.a[e]

    wg, wu, wd = Experts(inputs["wg"]), Experts(inputs["wu"]), Experts(inputs["wd"])
    dy = inputs["dy"][:n_tok].float().cpu().numpy().astype(np.float64)
    dxs = inputs["dxs"][:n_tok * shape.K].float().cpu().numpy().astype(np.float64)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        f = O.moe_forward(x64, wr64, wg, wu, wd, shape.K, bias)
        O.moe_backward(f, dy, dxs, x64, wr64)
        times.append(time.perf_counter() - t0)
    return times


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def main():
    args = parse()
    rank, world, local = dist_env()
    from token_dispatch_gb300 import synth
    shape = synth.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        import torch
        # inputs exactly as the GPU arm draws them (expert weights on the device)
        from token_dispatch_gb300 import synth as S
        dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
        x, wr = S.router_inputs(shape, seed=0)
        wg, wu, wd = S.expert_weights_device(shape, dev, seed=0)
        g = torch.Generator(device=dev)
        g.manual_seed(1000)
        tdt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
        n_tok = args.cpu_sample_tokens or 32
        dy = torch.randn((shape.T, shape.H), generator=g, device=dev, dtype=torch.float32).to(tdt)
        dxs = torch.randn((shape.T * shape.K, shape.H), generator=g, device=dev, dtype=torch.float32).to(tdt)
        bias_np, _ = skew_bias(shape, args.bias_target)
        inputs = dict(x=x, wr=wr, wg=wg, wu=wu, wd=wd, bias=bias_np, dy=dy, dxs=dxs)
        oracle_sample(shape, inputs, n_tok, reps=max(1, args.warmup))
        times = oracle_sample(shape, inputs, n_tok, reps=args.steps)
        ms = 1e3 * statistics.mean(times)
        val = n_tok / (ms * 1e-3)
        out = {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
               "config": {"workload": shape.name, "bias_target": args.bias_target},
               "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                                "sample": f"first {n_tok} tokens of the batch per step"},
               "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(out))
        return

    result, inputs = run_ours(args, shape, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_tok = args.cpu_sample_tokens or 4096
        times = oracle_sample(shape, inputs, n_tok, reps=1)
        result["cpu_baseline"] = {"value": n_tok / times[0], "unit": "tokens/s", "cores": cores(),
                                  "kind": "oracle",
                                  "sample": f"first {n_tok} tokens of the batch, fwd + gate/dispatch bwd, "
                                            f"float64 numpy ({times[0]:.1f} s)"}
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
