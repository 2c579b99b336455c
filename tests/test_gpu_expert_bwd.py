"""GPU parity of the expert FFN backward through the C ABI: moe_expert_ffn_ex
(which also keeps the SwiGLU pre-activations g and u) and moe_expert_ffn_bwd,
against the oracle's expert_ffn / expert_ffn_bwd on the same bf16-rounded
inputs.  Row counts per expert are ragged: empty experts, a single row, exact
and inexact multiples of the 64-row K block of the weight-gradient GEMMs, H'
that is not a multiple of the 256-wide N tile."""
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
