"""A whole training step of the layer (forward, then the full backward) captured
into one CUDA graph and replayed on new inputs gives, bit for bit, what the
same calls launched one by one give.  Every launch of the library is stream
ordered, takes its workspace from the caller and reads no result back to the
host, so the capture needs no change to the path; every reduction is in a
fixed order (integer atomics only), so the two runs agree exactly."""
import pytest
import torch

from token_dispatch_gb300 import _lib as L
from token_dispatch_gb300 import layer, synth
from tests.gpu_util import DEV, dev, host_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from token_dispatch_gb300 import build
    build.build()
    assert torch.cuda.is_available()


OUTPUTS = ["logits", "idx", "gate", "cu", "dst_row", "src_tok", "xs", "act", "gu", "h", "y",
           "dh", "d_gate", "dxs", "dw_gate", "dw_up", "dw_down", "dx", "d_logits", "dw_router"]


@pytest.mark.parametrize("route_flags", [0, L.MOE_ROUTE_RENORM])
def test_graph_replay_of_a_training_step_is_bit_exact(route_flags):
    shape = synth.MoEShape("bf16_T777_H256_E8_K2_Hp192", 777, 256, 8, 2, 192, "bf16")
    T, H, E, K, Hp = shape.T, shape.H, shape.E, shape.K, shape.Hp
    x, wr, wg, wu, wd = host_layer_inputs(shape)
    weights = [dev(a) for a in (wr, wg, wu, wd)]
    wrd, wgd, wud, wdd = weights
    b = layer.MoEBuffers(T, H, E, K, Hp, "bf16", DEV, backward=True, train=True)
    x_buf = dev(x).clone()
    dy_buf = dev(synth.upstream_grad(shape, T, H)).clone()
    s = torch.cuda.Stream(device=DEV)

    def step():
        layer.moe_forward(b, x_buf, wrd, None, wgd, wud, wdd, stream=s, route_flags=route_flags)
        layer.moe_train_backward(b, x_buf, wrd, wgd, wud, wdd, dy_buf, stream=s, route_flags=route_flags)

    with torch.cuda.stream(s):  # warm the launch paths once before capturing
        step()
    torch.cuda.synchronize()
    idx_first = b.idx.clone()
    n0 = L.moe_kernel_launches()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
        step()
    assert L.moe_kernel_launches() > n0

    # new inputs of another seed into the captured buffers
    rng = torch.Generator().manual_seed(1234)
    x_new = (torch.randn((T, H), generator=rng) * 0.5).to(torch.bfloat16)
    dy_new = (torch.randn((T, H), generator=rng) * 0.1).to(torch.bfloat16)
    x_buf.copy_(x_new.to(DEV))
    dy_buf.copy_(dy_new.to(DEV))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert L.moe_last_device_error() == L.MOE_OK
    got = {n: getattr(b, n).clone() for n in OUTPUTS}

    for n in OUTPUTS:  # poison, so a stale buffer cannot pass
        getattr(b, n).fill_(7)
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    assert L.moe_last_device_error() == L.MOE_OK
    for n in OUTPUTS:
        assert torch.equal(bits(got[n]), bits(getattr(b, n))), n
    # the replay read the new inputs: its routing is not the first inputs' routing
    assert not torch.equal(got["idx"], idx_first)


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t
