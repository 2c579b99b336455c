"""moe_dispatch_noalloc: dispatch for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: their device memory belongs
to an allocator or a pre-planned arena they do not control, or they must not
call cudaMalloc on their hot path.  For them the library keeps the one scratch
table dispatch needs (per-chunk expert counts) in a static device array.  This
file checks, through the C ABI, that the variant gives exactly the results of
moe_dispatch with a caller workspace, on two calls in a row with different
sizes (the shared array keeps the previous call's contents), at the largest
table the array holds, for fp32 rows, for an empty batch and when captured in
a CUDA graph and replayed on new inputs, and that sizes past the array's
capacity are refused before anything runs.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one."""
import numpy as np
import pytest
import torch

from token_dispatch_gb300 import _lib as L

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from token_dispatch_gb300 import build
    build.build()


def idx_for(T, E, K, seed):
    rng = np.random.default_rng(seed)
    if T == 0:
        return np.zeros((0, K), np.int32)
    return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


def run_both(T, H, E, K, seed, dtype="bf16"):
    raw = L.lib()
    tdt, cdt = (torch.bfloat16, L.MOE_BF16) if dtype == "bf16" else (torch.float32, L.MOE_F32)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H), generator=g).to(tdt).to(DEV)
    idx = torch.from_numpy(idx_for(T, E, K, seed)).to(DEV)
    stream = torch.cuda.current_stream().cuda_stream

    def outputs():
        return (torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
                torch.full((T * K,), -7, dtype=torch.int32, device=DEV),
                torch.full((T * K,), -7, dtype=torch.int32, device=DEV),
                torch.zeros((T * K, H), dtype=tdt, device=DEV))

    ref = outputs()
    nbytes = raw.moe_workspace_bytes(L.MOE_OP_DISPATCH, T, H, E, K, 0)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=DEV)
    st = raw.moe_dispatch(x.data_ptr(), idx.data_ptr(), T, H, E, K, cdt, ref[0].data_ptr(),
                          ref[1].data_ptr(), ref[2].data_ptr(), ref[3].data_ptr(), ws.data_ptr(), nbytes, stream)
    assert st == L.MOE_OK, L.moe_status_str(st)

    got = outputs()
    st = raw.moe_dispatch_noalloc(x.data_ptr(), idx.data_ptr(), T, H, E, K, cdt, got[0].data_ptr(),
                                  got[1].data_ptr(), got[2].data_ptr(), got[3].data_ptr(), stream)
    assert st == L.MOE_OK, L.moe_status_str(st)
    assert raw.moe_last_device_error(stream) == L.MOE_OK
    # integer outputs and the copied rows are exact
    for a, b in zip(ref[:3], got[:3]):
        assert torch.equal(a, b)
    assert torch.equal(ref[3].view(torch.int16), got[3].view(torch.int16))  # bit patterns
    assert int(got[0][-1]) == T * K


def test_noalloc_matches_workspace_dispatch_on_two_calls_in_a_row():
    # the second call is smaller and has more experts: stale counts from the
    # first call would show up as wrong offsets
    run_both(T=4000, H=256, E=64, K=6, seed=1)
    run_both(T=1000, H=128, E=384, K=8, seed=2)


def test_noalloc_largest_table_fp32_and_empty_batch():
    # 63 chunks x 1024 experts + 1024 totals fill the array exactly (the
    # column-scan path); then fp32 rows; then no tokens at all (only
    # cu_seqlens is written, all zeros)
    run_both(T=63 * 256, H=64, E=1024, K=4, seed=3)
    run_both(T=777, H=96, E=16, K=3, seed=4, dtype="f32")
    run_both(T=0, H=64, E=8, K=2, seed=5)


def test_noalloc_refuses_sizes_past_the_static_scratch():
    raw = L.lib()
    A = 1 << 20  # never dereferenced: the size check comes first
    # ceil(T/256) * E + E = 65 * 1024 + 1024 > 65536
    st = raw.moe_dispatch_noalloc(A, A, 65 * 256, 64, 1024, 2, L.MOE_BF16, A, A, A, A, None)
    assert st == L.MOE_ERR_WORKSPACE
    # one token past the largest table that fits: 64 * 1024 + 1024 > 65536
    st = raw.moe_dispatch_noalloc(A, A, 63 * 256 + 1, 64, 1024, 2, L.MOE_BF16, A, A, A, A, None)
    assert st == L.MOE_ERR_WORKSPACE


def test_noalloc_replays_in_a_cuda_graph_on_new_inputs():
    # one eager call first (it resolves the static array's address), then the
    # call captured once on a side stream and replayed after the inputs are
    # overwritten in place: every replay must equal moe_dispatch on the same
    # inputs, bit for bit
    raw = L.lib()
    T, H, E, K = 3000, 128, 64, 6
    x = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((T, K), dtype=torch.int32, device=DEV)
    cu = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    dst = torch.empty((T * K,), dtype=torch.int32, device=DEV)
    src = torch.empty((T * K,), dtype=torch.int32, device=DEV)
    xs = torch.empty((T * K, H), dtype=torch.bfloat16, device=DEV)

    def fill(seed):
        g = torch.Generator().manual_seed(seed)
        x.copy_(torch.randn((T, H), generator=g).to(torch.bfloat16))
        idx.copy_(torch.from_numpy(idx_for(T, E, K, seed)))

    def call(stream):
        return raw.moe_dispatch_noalloc(x.data_ptr(), idx.data_ptr(), T, H, E, K, L.MOE_BF16, cu.data_ptr(),
                                        dst.data_ptr(), src.data_ptr(), xs.data_ptr(), stream)

    fill(10)
    assert call(torch.cuda.current_stream().cuda_stream) == L.MOE_OK
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        st = call(side.cuda_stream)
    assert st == L.MOE_OK
    for seed in (11, 12):
        fill(seed)
        graph.replay()
        torch.cuda.synchronize()
        assert raw.moe_last_device_error(None) == L.MOE_OK
        ref = (torch.empty_like(cu), torch.empty_like(dst), torch.empty_like(src), torch.empty_like(xs))
        nbytes = raw.moe_workspace_bytes(L.MOE_OP_DISPATCH, T, H, E, K, 0)
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=DEV)
        st = raw.moe_dispatch(x.data_ptr(), idx.data_ptr(), T, H, E, K, L.MOE_BF16, ref[0].data_ptr(),
                              ref[1].data_ptr(), ref[2].data_ptr(), ref[3].data_ptr(), ws.data_ptr(), nbytes, None)
        assert st == L.MOE_OK
        torch.cuda.synchronize()
        for a, b in zip(ref[:3], (cu, dst, src)):
            assert torch.equal(a, b)
        assert torch.equal(ref[3].view(torch.int16), xs.view(torch.int16))
