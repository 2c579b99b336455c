// Token dispatch: histogram -> cu_seqlens -> stable permutation -> row gather.
//
// Dispatch follows the MoE/MoD framework page ("What's in the box":
// a fused kernel moving tokens between experts, reading and writing the buffers
// directly) and the MoonEP page ("Step-by-step": tokens land in one contiguous
// expert-sorted buffer whose active rows are described by cu_seqlens).
//
// The histogram is atomic-free: every warp owns a private histogram in shared
// memory and groups equal expert ids of its 32 lanes with __match_any_sync, so
// one leader lane per distinct expert updates the counter.  The same pass gives
// each pair its rank among earlier pairs of the same expert (popc of lower peer
// lanes), so the permutation is stable by token and identical run to run.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int CH_TOK = 256;        // tokens per chunk (one CTA)
constexpr int CH_WARPS = 8;        // warps per chunk CTA
constexpr int TOK_PER_WARP = CH_TOK / CH_WARPS;
constexpr int MAX_E = 1024;

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }
int n_chunks(int T) { return (T + CH_TOK - 1) / CH_TOK; }

// Count the pairs of this warp's token range into its private histogram.
// Equal expert ids among the 32 lanes are grouped with __match_any_sync and the
// lowest lane of each group adds the group size: distinct groups touch distinct
// counters, so no atomics are needed.
__device__ __forceinline__ void warp_count(const int32_t* __restrict__ idx, int T, int E, int K,
                                           int t_begin, int* hist, unsigned* err) {
  const int lane = threadIdx.x & 31;
  int t_end = t_begin + TOK_PER_WARP;
  if (t_end > T) t_end = T;
  if (t_begin >= t_end) return;
  const long long j0 = (long long)t_begin * K, j1 = (long long)t_end * K;
  for (long long j = j0; j < j1; j += 32) {
    long long my = j + lane;
    int e = -1;
    if (my < j1) {
      e = __ldg(idx + my);
      if (e < 0 || e >= E) {
        set_error(err, DEV_BOUNDS);
        e = -1;
      }
    }
    unsigned active = __ballot_sync(0xffffffffu, e >= 0);
    unsigned peers = __match_any_sync(0xffffffffu, e) & active;
    if (e >= 0 && __popc(peers & ((1u << lane) - 1u)) == 0) hist[e] += __popc(peers);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(32 * CH_WARPS)
dispatch_count_kernel(const int32_t* __restrict__ idx, int T, int E, int K,
                      int* __restrict__ counts, unsigned* err) {
  __shared__ int hist[CH_WARPS][MAX_E];
  const int w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < CH_WARPS * E; i += blockDim.x) hist[i / E][i % E] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * CH_TOK + w * TOK_PER_WARP;
  warp_count(idx, T, E, K, t0, hist[w], err);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int ww = 0; ww < CH_WARPS; ++ww) c += hist[ww][e];
    counts[(long long)blockIdx.x * E + e] = c;
  }
}

// One CTA per chunk.  Besides its own per-warp counts, every CTA sums the
// chunk count table itself: the per-expert totals (an exclusive scan over
// experts gives cu_seqlens; CTA 0 writes them) and the counts of the chunks
// before its own.  Integer sums, so every CTA gets the same numbers and the
// scan needs no launch of its own.
__global__ void __launch_bounds__(32 * CH_WARPS)
dispatch_place_kernel(const int32_t* __restrict__ idx, int T, int E, int K, const int* __restrict__ counts,
                      int C, int32_t* __restrict__ cu, int32_t* __restrict__ dst_row,
                      int32_t* __restrict__ src_tok) {
  __shared__ int hist[CH_WARPS][MAX_E];
  __shared__ int tot[MAX_E], pre[MAX_E];
  __shared__ int tsum[32 * CH_WARPS];
  const int tid = threadIdx.x, w = tid >> 5, nth = blockDim.x;
  for (int i = tid; i < CH_WARPS * E; i += nth) hist[i / E][i % E] = 0;
  for (int e = tid; e < E; e += nth) tot[e] = pre[e] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * CH_TOK + w * TOK_PER_WARP;
  warp_count(idx, T, E, K, t0, hist[w], nullptr);
  // totals over all chunks and over the chunks before this one
  const long long n = (long long)C * E, before = (long long)blockIdx.x * E;
#pragma unroll 4
  for (long long i = tid; i < n; i += nth) {
    const int v = __ldg(counts + i);
    const int e = (int)(i % E);
    atomicAdd(&tot[e], v);
    if (i < before) atomicAdd(&pre[e], v);
  }
  __syncthreads();
  // exclusive scan of the totals: thread r owns a run of consecutive experts
  const int per = (E + nth - 1) / nth;
  const int e_lo = tid * per, e_hi = min(E, e_lo + per);
  int run = 0;
  for (int e = e_lo; e < e_hi; ++e) run += tot[e];
  tsum[tid] = run;
  __syncthreads();
  for (int o = 1; o < nth; o <<= 1) {
    const int v = tid >= o ? tsum[tid - o] : 0;
    __syncthreads();
    tsum[tid] += v;
    __syncthreads();
  }
  int start = tsum[tid] - run;
  for (int e = e_lo; e < e_hi; ++e) {
    const int c = tot[e];
    tot[e] = start;
    start += c;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = tid; e < E; e += nth) cu[e] = tot[e];
    if (tid == nth - 1) cu[E] = tsum[nth - 1];
  }
  // hist[w][e] <- first row of warp w for expert e
  for (int e = tid; e < E; e += nth) {
    int r = tot[e] + pre[e];
#pragma unroll
    for (int ww = 0; ww < CH_WARPS; ++ww) {
      const int c = hist[ww][e];
      hist[ww][e] = r;
      r += c;
    }
  }
  __syncthreads();
  // second pass: assign rows (the counts are not needed again, base advances in place)
  int* base = hist[w];
  const int lane = threadIdx.x & 31;
  int t_end = t0 + TOK_PER_WARP;
  if (t_end > T) t_end = T;
  if (t0 >= t_end) return;
  const long long j0 = (long long)t0 * K, j1 = (long long)t_end * K;
  for (long long j = j0; j < j1; j += 32) {
    long long my = j + lane;
    int e = -1;
    if (my < j1) {
      e = __ldg(idx + my);
      if (e < 0 || e >= E) { dst_row[my] = -1; e = -1; }
    }
    unsigned active = __ballot_sync(0xffffffffu, e >= 0);
    unsigned peers = __match_any_sync(0xffffffffu, e) & active;
    int row = 0;
    if (e >= 0) row = base[e] + __popc(peers & ((1u << lane) - 1u));
    __syncwarp();
    if (e >= 0) {
      dst_row[my] = row;
      src_tok[row] = (int)(my / K);
      if (__popc(peers & ((1u << lane) - 1u)) == 0) base[e] += __popc(peers);
    }
    __syncwarp();
  }
}

// xs[dst_row[t*K+k]] = x[t]: one warp per token, 16-byte vectors; every x row is
// read once and written to its K rows, with U vectors per lane in flight.
template <int KT>
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ dst_row, int T, int K,
                   int vec_per_row, uint4* __restrict__ xs) {
  constexpr int U = 4;
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nwarps) {
    int rows[KT];
#pragma unroll
    for (int k = 0; k < KT; ++k) rows[k] = (k < K) ? __ldg(dst_row + t * K + k) : -1;
    const uint4* src = x + t * vec_per_row;
    for (int i0 = lane; i0 < vec_per_row; i0 += 32 * U) {
      uint4 a[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + 32 * u;
        a[u] = (i < vec_per_row) ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        if (rows[k] < 0) continue;
        uint4* dst = xs + (long long)rows[k] * vec_per_row;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + 32 * u;
          if (i < vec_per_row) dst[i] = a[u];
        }
      }
    }
  }
}

int warp_grid(long long n_warps_work) {
  long long ctas = (n_warps_work + 7) / 8;
  long long cap = (long long)sm_count() * 16;
  if (ctas < 1) ctas = 1;
  return (int)(ctas < cap ? ctas : cap);
}

}  // namespace

size_t dispatch_ws_bytes(int T, int E, int K) {
  (void)K;
  return align256((size_t)n_chunks(T) * E * sizeof(int));
}

int launch_dispatch(const void* x, const int32_t* idx, int T, int H, int E, int K, int dtype,
                    int32_t* cu, int32_t* dst_row, int32_t* src_tok, void* xs, void* ws,
                    cudaStream_t s) {
  unsigned* err = device_error_word();
  const int C = n_chunks(T);
  int* counts = static_cast<int*>(ws);
  if (C > 0) {
    dispatch_count_kernel<<<C, 32 * CH_WARPS, 0, s>>>(idx, T, E, K, counts, err);
    int st = launch_status();
    if (st != MOE_OK) return st;
  }
  if (T == 0) return cudaMemsetAsync(cu, 0, (size_t)(E + 1) * sizeof(int32_t), s) == cudaSuccess ? MOE_OK
                                                                                     : MOE_ERR_CUDA;
  dispatch_place_kernel<<<C, 32 * CH_WARPS, 0, s>>>(idx, T, E, K, counts, C, cu, dst_row, src_tok);
  int st = launch_status();
  if (st != MOE_OK) return st;
  const int vec = H * (dtype == MOE_BF16 ? 2 : 4) / 16;
  const uint4* xv = static_cast<const uint4*>(x);
  uint4* xsv = static_cast<uint4*>(xs);
  const int grid = warp_grid(T);
  if (K <= 1) gather_rows_kernel<1><<<grid, 256, 0, s>>>(xv, dst_row, T, K, vec, xsv);
  else if (K <= 2) gather_rows_kernel<2><<<grid, 256, 0, s>>>(xv, dst_row, T, K, vec, xsv);
  else if (K <= 4) gather_rows_kernel<4><<<grid, 256, 0, s>>>(xv, dst_row, T, K, vec, xsv);
  else if (K <= 8) gather_rows_kernel<8><<<grid, 256, 0, s>>>(xv, dst_row, T, K, vec, xsv);
  else gather_rows_kernel<16><<<grid, 256, 0, s>>>(xv, dst_row, T, K, vec, xsv);
  return launch_status();
}

// ----------------------------------------------------------------------------
// Dispatch for callers that cannot allocate device memory.
//
// The only scratch dispatch needs is the per-chunk expert count table
// (ceil(T/256) * E ints).  Here it lives in a file-scope device array, so the
// caller passes inputs and outputs only.  The array exists once per GPU that
// loads the library and stays allocated until the process exits.  All calls
// share it: the count kernel writes every entry the later kernels read, so
// nothing has to be cleared between calls, but two calls whose kernels overlap
// on the GPU (different streams, no ordering between them) race on it.
constexpr long long kStaticScratchInts = 1 << 16;  // 256 KB
static __device__ __align__(256) int g_dispatch_static_scratch[kStaticScratchInts];

static int* g_static_scratch_dev[64];
static std::mutex g_static_scratch_mu;

long long dispatch_static_scratch_ints() { return kStaticScratchInts; }

// In host code the array's name is only a host-side stand-in; the kernels need
// its device address, resolved once per device with that device current.
static int* static_scratch_address(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (!g_static_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_static_scratch) != cudaSuccess || !p) {
      *status = MOE_ERR_CUDA;
      return nullptr;
    }
    g_static_scratch_dev[dev] = static_cast<int*>(p);
  }
  *status = MOE_OK;
  return g_static_scratch_dev[dev];
}

int launch_dispatch_static(const void* x, const int32_t* idx, int T, int H, int E, int K, int dtype,
                           int32_t* cu, int32_t* dst_row, int32_t* src_tok, void* xs, cudaStream_t s) {
  if ((long long)n_chunks(T) * E > kStaticScratchInts) return MOE_ERR_WORKSPACE;
  int st = MOE_OK;
  int* scratch = static_scratch_address(&st);
  if (!scratch) return st;
  return launch_dispatch(x, idx, T, H, E, K, dtype, cu, dst_row, src_tok, xs, scratch, s);
}

}  // namespace moe
