"""Seeded synthetic inputs for the MoE / MoD layer workloads.

This module only draws random numbers and rounds them to the storage type; it
holds none of the layer's arithmetic.  Both the CUDA path (through the tests and
the benchmark) and the CPU oracle receive the tensors drawn here.

Generator.  Host draws use a counter-based generator: element ``i`` of stream
``(seed, stream)`` is ``splitmix64`` of a per-stream base plus ``2i`` and
``2i+1``, turned into two uniforms on (0, 1) with 53-bit resolution and mapped to
a standard normal by the Box-Muller transform (cosine branch).  The result does
not depend on how the draw is chunked, so any slice can be regenerated alone.

Very large expert-weight tensors (hundreds of millions of elements) are drawn on
the GPU with torch's seeded Philox generator instead, because host generation
and a host-to-device copy of tens of GB would dominate the run; the oracle then
receives host copies of exactly those tensors (``weights_to_host``).

Storage rounding.  bf16 values are the fp32 sample rounded to nearest-even;
the fp64 arrays handed to the oracle hold the rounded values exactly.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)


def _splitmix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser (Steele, Lea, Flood 2014) on a uint64 array."""
    z = z + _GOLDEN
    z = (z ^ (z >> np.uint64(30))) * _C1
    z = (z ^ (z >> np.uint64(27))) * _C2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed * 0x100000001B3 + stream * 0x1F3D5B79) & 0xFFFFFFFFFFFFFFFF],
                     dtype=np.uint64)
        return _splitmix64(s)[0]


def normal(seed: int, stream: int, n: int, start: int = 0, chunk: int = 1 << 22) -> np.ndarray:
    """``n`` standard normals (float64) of stream (seed, stream), from element ``start``."""
    base = _stream_base(seed, stream)
    out = np.empty(n, dtype=np.float64)
    two_pi = 2.0 * math.pi
    with np.errstate(over="ignore"):
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            i = np.arange(start + lo, start + hi, dtype=np.uint64)
            c = base + (i << np.uint64(1))
            a = _splitmix64(c)
            b = _splitmix64(c + np.uint64(1))
            u1 = ((a >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
            u2 = ((b >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
            out[lo:hi] = np.sqrt(-2.0 * np.log(u1)) * np.cos(two_pi * u2)
    return out


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` uniforms on (0, 1) (float64) of stream (seed, stream)."""
    base = _stream_base(seed, stream)
    with np.errstate(over="ignore"):
        i = np.arange(n, dtype=np.uint64)
        a = _splitmix64(base + (i << np.uint64(1)))
    return ((a >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def round_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 round-to-nearest-even of ``a``, then bf16 round-to-nearest-even; uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclasses.dataclass
class Stored:
    """A tensor in its storage type: ``ref`` holds the stored values in float64 for
    the oracle, ``host`` is the same data as a torch CPU tensor in the storage dtype."""
    ref: np.ndarray
    host: object  # torch.Tensor

    @property
    def shape(self):
        return self.ref.shape


def store(a: np.ndarray, dtype: str) -> Stored:
    """Round float64 samples to the storage dtype ("f32" or "bf16")."""
    import torch
    if dtype == "f32":
        f = np.ascontiguousarray(a, dtype=np.float32)
        return Stored(f.astype(np.float64), torch.from_numpy(f.copy()))
    if dtype == "bf16":
        bits = round_bf16_bits(a)
        t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
        return Stored(bf16_bits_to_f64(bits), t)
    raise ValueError(dtype)


def normal_stored(seed, stream, shape, std, dtype) -> Stored:
    n = int(np.prod(shape))
    return store((normal(seed, stream, n) * std).reshape(shape), dtype)


# --------------------------------------------------------------------------
# Workload descriptions (shapes and distributions of the layer configurations)
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class MoEShape:
    name: str
    T: int          # tokens entering the MoE (after MoD selection for the MoD workload)
    H: int          # hidden size
    E: int          # experts
    K: int          # experts per token
    Hp: int         # expert FFN intermediate size H'
    dtype: str      # storage type: "f32" or "bf16"
    # MoD (mixture-of-depths) front end; B*L input tokens of which C per row run the MoE
    mod_B: int = 0
    mod_L: int = 0
    mod_C: int = 0

    @property
    def R(self) -> int:
        return self.T * self.K


# Tiny fp32 layer: T=256, H=128, E=8, K=2, H'=256.
TINY_F32 = MoEShape("tiny_f32_T256_H128_E8_K2_Hp256", 256, 128, 8, 2, 256, "f32")
# Mixtral-shaped: batch 4 x seq 2048 tokens, H=4096, E=8, K=2, H'=14336.
MIXTRAL_BF16 = MoEShape("mixtral_bf16_T8192_H4096_E8_K2_Hp14336", 8192, 4096, 8, 2, 14336, "bf16")
# Fine-grained: T=16384, H=2048, E=64, K=6, H'=1408.
FINEGRAINED_BF16 = MoEShape("finegrained_bf16_T16384_H2048_E64_K6_Hp1408", 16384, 2048, 64, 6, 1408, "bf16")
# Expert-parallel benchmark shapes on one GPU: S=8192, E=384, H=7168, K=8, H'=2048.
EPBENCH_BF16 = MoEShape("epbench_bf16_T8192_H7168_E384_K8_Hp2048", 8192, 7168, 384, 8, 2048, "bf16")
# MoD + MoE: batch 4 x seq 2048, H=2048, 50% capacity -> 4096 tokens into E=16, K=2, H'=5632.
MOD_BF16 = MoEShape("mod_bf16_B4_L2048_C1024_H2048_E16_K2_Hp5632", 4096, 2048, 16, 2, 5632, "bf16",
                    mod_B=4, mod_L=2048, mod_C=1024)

# Same expert GEMM shapes as the Mixtral-shaped layer with a quarter of the
# tokens (2.8 GB of weights, 0.2 GB of activations): the case the
# hardware-counter captures run on.
PROFILE_BF16 = MoEShape("mixtral_profile_bf16_T2048_H4096_E8_K2_Hp14336", 2048, 4096, 8, 2, 14336, "bf16")

WORKLOADS = {s.name: s for s in (TINY_F32, MIXTRAL_BF16, FINEGRAINED_BF16, EPBENCH_BF16, MOD_BF16, PROFILE_BF16)}

# stream ids (seed 0 holds the forward inputs, seed 1 the upstream gradient dy,
# seed 2 the synthetic expert-input gradient dxs)
S_X, S_WR, S_WG, S_WU, S_WD, S_WMOD, S_DY, S_DXS = 1, 2, 3, 4, 5, 6, 7, 8

ROUTER_STD = 0.02


def router_inputs(shape: MoEShape, seed: int = 0, tokens: int | None = None):
    """x ~ N(0,1) [T,H] and W_r ~ N(0, 0.02) [H,E] in storage dtype.

    For the MoD workload ``tokens`` is B*L (all input tokens)."""
    T = shape.T if tokens is None else tokens
    x = normal_stored(seed, S_X, (T, shape.H), 1.0, shape.dtype)
    wr = normal_stored(seed, S_WR, (shape.H, shape.E), ROUTER_STD, shape.dtype)
    return x, wr


def mod_weight(shape: MoEShape, seed: int = 0) -> Stored:
    """MoD scalar-router weight w_mod ~ N(0, 1/sqrt(H)), so that x.w_mod ~ N(0,1)."""
    return normal_stored(seed, S_WMOD, (shape.H,), 1.0 / math.sqrt(shape.H), shape.dtype)


def expert_weights_host(shape: MoEShape, seed: int = 0):
    """Wg, Wu ~ N(0, 1/sqrt(H)) and Wd ~ N(0, 1/sqrt(H')), each one contiguous [E,H,H']."""
    E, H, Hp = shape.E, shape.H, shape.Hp
    wg = normal_stored(seed, S_WG, (E, H, Hp), 1.0 / math.sqrt(H), shape.dtype)
    wu = normal_stored(seed, S_WU, (E, H, Hp), 1.0 / math.sqrt(H), shape.dtype)
    wd = normal_stored(seed, S_WD, (E, H, Hp), 1.0 / math.sqrt(Hp), shape.dtype)
    return wg, wu, wd


def expert_weights_device(shape: MoEShape, device, seed: int = 0, experts_per_draw: int = 8):
    """Same distributions as ``expert_weights_host`` drawn on the GPU (torch Philox),
    one generator per (projection, expert) so any expert can be copied back alone."""
    import torch
    E, H, Hp = shape.E, shape.H, shape.Hp
    tdt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
    out = []
    for proj, std in ((S_WG, 1.0 / math.sqrt(H)), (S_WU, 1.0 / math.sqrt(H)), (S_WD, 1.0 / math.sqrt(Hp))):
        w = torch.empty((E, H, Hp), dtype=tdt, device=device)
        g = torch.Generator(device=device)
        for e in range(E):
            g.manual_seed((seed * 1000003 + proj) * 100003 + e)
            tmp = torch.randn((H, Hp), generator=g, device=device, dtype=torch.float32)
            w[e].copy_(tmp.mul_(std))
        out.append(w)
    return tuple(out)


def weights_to_host(w, experts=None) -> np.ndarray:
    """float64 host copy of expert weights (all experts, or the listed ones)."""
    import torch
    if experts is None:
        return w.detach().to("cpu", torch.float32).numpy().astype(np.float64)
    return np.stack([w[e].detach().to("cpu", torch.float32).numpy().astype(np.float64) for e in experts])


def upstream_grad(shape: MoEShape, rows: int, cols: int, seed: int = 1, stream: int = S_DY) -> Stored:
    """dy ~ N(0,1) (seed 1); the synthetic expert-input gradient dxs uses seed 2."""
    return normal_stored(seed, stream, (rows, cols), 1.0, shape.dtype)


def expert_bias(E: int, beta: float, expert: int = 0) -> np.ndarray:
    """Per-expert logit bias: beta on one expert, zero elsewhere (router skew)."""
    b = np.zeros(E, dtype=np.float32)
    b[expert] = beta
    return b
