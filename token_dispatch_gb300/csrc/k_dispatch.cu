// Token dispatch: histogram -> cu_seqlens -> stable permutation -> row gather.
//
// Dispatch follows the MoE/MoD framework page ("What's in the box":
// a fused kernel moving tokens between experts, reading and writing the buffers
// directly) and the MoonEP page ("Step-by-step": tokens land in one contiguous
// expert-sorted buffer whose active rows are described by cu_seqlens).
//
// Tokens are cut into chunks of 256 (one CTA each).  Per chunk the expert
// histogram is built without atomics: every warp owns a private histogram in
// shared memory and groups equal expert ids of its 32 lanes with
// __match_any_sync, so one leader lane per distinct expert updates the
// counter.  The same grouping gives each pair its rank among earlier pairs of
// the same expert (popc of lower peer lanes), so the permutation is stable by
// token and identical run to run.  Every warp loads all its expert ids at once
// before the first match, so a chunk costs one memory round trip, not one per
// 32 pairs.
//
// The row of pair (t, k) of chunk c with expert e is
//   cu[e] + (pairs of e in chunks before c) + (pairs of e earlier in chunk c),
// so the chunk counts need two scans: over chunks per expert, and over the
// expert totals.  Small count tables (chunks x experts <= 8192) are summed by
// every place CTA itself with per-thread strided sums (no atomics; integer
// sums, so all CTAs agree).  Larger tables get one column-scan launch (a thread
// per expert, warps over chunk ranges) that overwrites the table with the
// exclusive per-expert prefixes and writes the totals, so the work stays
// linear in chunks x experts.  The scan over experts (cu_seqlens) is a block
// scan in every place CTA; CTA 0 writes cu_seqlens.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int CH_TOK = 256;        // tokens per chunk (one CTA)
constexpr int CH_WARPS = 8;        // warps per chunk CTA
constexpr int CH_THREADS = 32 * CH_WARPS;
constexpr int TOK_PER_WARP = CH_TOK / CH_WARPS;
constexpr int MAX_E = 1024;
constexpr int PF = 8;                    // expert ids per lane loaded at once
constexpr long long SMALL_TABLE = 8192;  // count tables summed by every place CTA

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }
int n_chunks(int T) { return (T + CH_TOK - 1) / CH_TOK; }
bool small_table(int T, int E) { return (long long)n_chunks(T) * E <= SMALL_TABLE; }
// ints of scratch: the chunk x expert count table and the expert totals
long long scratch_ints(int T, int E) { return (long long)n_chunks(T) * E + E; }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Pairs (t*K + k order) of warp w of chunk c: [j0, j1).
__device__ __forceinline__ void warp_pairs(int T, int K, int c, int w, int& j0, int& j1) {
  int t0 = c * CH_TOK + w * TOK_PER_WARP;
  int t1 = min(t0 + TOK_PER_WARP, T);
  if (t0 > t1) t0 = t1;
  j0 = t0 * K;
  j1 = t1 * K;
}

// PF expert ids per lane: pair jb + 32u + lane.  All loads are issued before
// any is checked.  -1: no pair there; -2: an id outside [0, E).
__device__ __forceinline__ void load_ids(const int32_t* __restrict__ idx, int jb, int j1, int E, int (&e)[PF]) {
  const int lane = threadIdx.x & 31;
  int raw[PF];
#pragma unroll
  for (int u = 0; u < PF; ++u) {
    const int j = jb + 32 * u + lane;
    raw[u] = j < j1 ? __ldg(idx + j) : -1;
  }
#pragma unroll
  for (int u = 0; u < PF; ++u) {
    const int j = jb + 32 * u + lane;
    e[u] = j >= j1 ? -1 : (raw[u] < 0 || raw[u] >= E) ? -2 : raw[u];
  }
}

// One group of 32 pairs into the warp's histogram: the lowest lane of each
// group of equal ids adds the group's size (distinct groups, distinct counters).
__device__ __forceinline__ void count32(int e, int* hist) {
  const unsigned active = __ballot_sync(0xffffffffu, e >= 0);
  const unsigned peers = __match_any_sync(0xffffffffu, e) & active;
  if (e >= 0 && (peers & lanemask_lt()) == 0) hist[e] += __popc(peers);
  __syncwarp();
}

// One group of 32 pairs: row = the warp's next row of the expert + rank among
// lower lanes with the same id; the group's leader advances the next row.
__device__ __forceinline__ int assign32(int e, int* next) {
  const unsigned active = __ballot_sync(0xffffffffu, e >= 0);
  const unsigned peers = __match_any_sync(0xffffffffu, e) & active;
  const int rank = __popc(peers & lanemask_lt());
  const int row = e >= 0 ? next[e] + rank : -1;
  __syncwarp();
  if (e >= 0 && rank == 0) next[e] += __popc(peers);
  __syncwarp();
  return row;
}

// Count the chunk's pairs per warp into hist[w][.]; true if an id was bad.
// The first batch of ids stays in e0 for the assign pass.
__device__ __forceinline__ bool warp_count(const int32_t* __restrict__ idx, int E, int j0, int j1, int* hist,
                                           int (&e0)[PF]) {
  bool bad = false;
  for (int jb = j0; jb < j1; jb += 32 * PF) {
    int e[PF];
    load_ids(idx, jb, j1, E, e);
#pragma unroll
    for (int u = 0; u < PF; ++u) {
      if (jb + 32 * u >= j1) break;  // uniform over the warp
      bad |= e[u] == -2;
      count32(e[u], hist);
    }
    if (jb == j0) {
#pragma unroll
      for (int u = 0; u < PF; ++u) e0[u] = e[u];
    }
  }
  return bad;
}

__global__ void __launch_bounds__(CH_THREADS)
dispatch_count_kernel(const int32_t* __restrict__ idx, int T, int E, int K, int* __restrict__ counts,
                      unsigned* err) {
  __shared__ int hist[CH_WARPS][MAX_E];
  const int w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < CH_WARPS * E; i += CH_THREADS) hist[i / E][i % E] = 0;
  __syncthreads();
  int j0, j1;
  warp_pairs(T, K, blockIdx.x, w, j0, j1);
  int e0[PF];
  const bool bad = warp_count(idx, E, j0, j1, hist[w], e0);
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) set_error(err, DEV_BOUNDS);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += CH_THREADS) {
    int c = 0;
#pragma unroll
    for (int ww = 0; ww < CH_WARPS; ++ww) c += hist[ww][e];
    counts[(long long)blockIdx.x * E + e] = c;
  }
}

// Large count tables: per expert, the exclusive prefix over chunks replaces
// the counts in place and the total goes to tot[e].  CTA = 32 consecutive
// experts (one per lane, 128-byte rows); its 8 warps own consecutive chunk
// ranges, whose sums meet in shared memory in warp order.
__global__ void __launch_bounds__(CH_THREADS)
dispatch_scan_kernel(int* __restrict__ counts, int C, int E, int* __restrict__ tot) {
  __shared__ int wsum[CH_WARPS][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const bool live = e < E;
  const int cb = (int)((long long)w * C / CH_WARPS), ce = (int)((long long)(w + 1) * C / CH_WARPS);
  int s = 0;
  for (int c0 = cb; c0 < ce; c0 += 8) {
    int v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = (live && c0 + u < ce) ? counts[(long long)(c0 + u) * E + e] : 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) s += v[u];
  }
  wsum[w][lane] = s;
  __syncthreads();
  int run = 0;
  for (int ww = 0; ww < w; ++ww) run += wsum[ww][lane];
  if (w == CH_WARPS - 1 && live) tot[e] = run + s;
  for (int c0 = cb; c0 < ce; c0 += 8) {
    int v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = (live && c0 + u < ce) ? counts[(long long)(c0 + u) * E + e] : 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (live && c0 + u < ce) counts[(long long)(c0 + u) * E + e] = run;
      run += v[u];
    }
  }
}

// One CTA per chunk: its per-warp counts, the chunk's offsets (summed here for
// small tables, read from the column scan otherwise), the scan over experts,
// then stable rows for every pair.
__global__ void __launch_bounds__(CH_THREADS)
dispatch_place_kernel(const int32_t* __restrict__ idx, int T, int E, int K, const int* __restrict__ counts,
                      int C, const int* __restrict__ tot_scanned, int32_t* __restrict__ cu,
                      int32_t* __restrict__ dst_row, int32_t* __restrict__ src_tok) {
  __shared__ int hist[CH_WARPS][MAX_E];
  __shared__ int tot[MAX_E], pre[MAX_E];
  __shared__ int part_t[CH_THREADS], part_p[CH_THREADS];
  __shared__ int wsum[CH_WARPS];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.x;
  for (int i = tid; i < CH_WARPS * E; i += CH_THREADS) hist[i / E][i % E] = 0;
  __syncthreads();
  int j0, j1;
  warp_pairs(T, K, blk, w, j0, j1);
  int e0[PF];
  (void)warp_count(idx, E, j0, j1, hist[w], e0);

  // totals per expert and the pairs of each expert in earlier chunks
  if (tot_scanned) {
    for (int e = tid; e < E; e += CH_THREADS) {
      tot[e] = __ldg(tot_scanned + e);
      pre[e] = __ldg(counts + (long long)blk * E + e);
    }
  } else if (E <= CH_THREADS) {
    const int ng = CH_THREADS / E;  // chunk groups: thread (g, e) sums chunks g, g + ng, ...
    int st = 0, sp = 0;
    if (tid < ng * E) {
      const int g = tid / E, e = tid - g * E;
#pragma unroll 4
      for (int c = g; c < C; c += ng) {
        const int v = __ldg(counts + (long long)c * E + e);
        st += v;
        sp += c < blk ? v : 0;
      }
    }
    part_t[tid] = st;
    part_p[tid] = sp;
    __syncthreads();
    for (int e = tid; e < E; e += CH_THREADS) {
      int a = 0, b = 0;
      for (int g = 0; g < ng; ++g) {
        a += part_t[g * E + e];
        b += part_p[g * E + e];
      }
      tot[e] = a;
      pre[e] = b;
    }
  } else {
    for (int e = tid; e < E; e += CH_THREADS) {
      int a = 0, b = 0;
#pragma unroll 4
      for (int c = 0; c < C; ++c) {
        const int v = __ldg(counts + (long long)c * E + e);
        a += v;
        b += c < blk ? v : 0;
      }
      tot[e] = a;
      pre[e] = b;
    }
  }
  __syncthreads();

  // exclusive scan of the totals over experts: thread r owns a run of
  // consecutive experts; runs are scanned with warp shuffles, then warp sums
  const int per = (E + CH_THREADS - 1) / CH_THREADS;
  const int e_lo = min(E, tid * per), e_hi = min(E, e_lo + per);
  int run = 0;
  for (int e = e_lo; e < e_hi; ++e) run += tot[e];
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  int start = incl - run, total = 0;
#pragma unroll
  for (int ww = 0; ww < CH_WARPS; ++ww) {
    start += ww < w ? wsum[ww] : 0;
    total += wsum[ww];
  }
  for (int e = e_lo; e < e_hi; ++e) {
    const int c = tot[e];
    tot[e] = start;
    start += c;
  }
  __syncthreads();
  if (blk == 0) {
    for (int e = tid; e < E; e += CH_THREADS) cu[e] = tot[e];
    if (tid == 0) cu[E] = total;
  }
  // hist[w][e] <- first row of warp w for expert e
  for (int e = tid; e < E; e += CH_THREADS) {
    int r = tot[e] + pre[e];
#pragma unroll
    for (int ww = 0; ww < CH_WARPS; ++ww) {
      const int c = hist[ww][e];
      hist[ww][e] = r;
      r += c;
    }
  }
  __syncthreads();

  // assign rows in pair order (the first batch of ids is still in registers)
  int* next = hist[w];
  for (int jb = j0; jb < j1; jb += 32 * PF) {
    int e[PF];
    if (jb == j0) {
#pragma unroll
      for (int u = 0; u < PF; ++u) e[u] = e0[u];
    } else {
      load_ids(idx, jb, j1, E, e);
    }
#pragma unroll
    for (int u = 0; u < PF; ++u) {
      if (jb + 32 * u >= j1) break;
      const int j = jb + 32 * u + lane;
      const int row = assign32(e[u], next);
      if (e[u] >= 0) {
        dst_row[j] = row;
        src_tok[row] = j / K;
      } else if (e[u] == -2) {
        dst_row[j] = -1;
      }
    }
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
  return align256((size_t)scratch_ints(T, E) * sizeof(int));
}

int launch_dispatch(const void* x, const int32_t* idx, int T, int H, int E, int K, int dtype,
                    int32_t* cu, int32_t* dst_row, int32_t* src_tok, void* xs, void* ws,
                    cudaStream_t s) {
  unsigned* err = device_error_word();
  const int C = n_chunks(T);
  if (T == 0) return cudaMemsetAsync(cu, 0, (size_t)(E + 1) * sizeof(int32_t), s) == cudaSuccess ? MOE_OK
                                                                                     : MOE_ERR_CUDA;
  int* counts = static_cast<int*>(ws);
  int* tot = counts + (long long)C * E;
  dispatch_count_kernel<<<C, CH_THREADS, 0, s>>>(idx, T, E, K, counts, err);
  int st = launch_status();
  if (st != MOE_OK) return st;
  const bool scanned = !small_table(T, E);
  if (scanned) {
    dispatch_scan_kernel<<<(E + 31) / 32, CH_THREADS, 0, s>>>(counts, C, E, tot);
    if ((st = launch_status()) != MOE_OK) return st;
  }
  dispatch_place_kernel<<<C, CH_THREADS, 0, s>>>(idx, T, E, K, counts, C, scanned ? tot : nullptr, cu, dst_row,
                                                  src_tok);
  if ((st = launch_status()) != MOE_OK) return st;
  if (!xs) return MOE_OK;  // index maps only: the rows are gathered by the expert FFN's operand load
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
// The only scratch dispatch needs is the per-chunk expert count table and the
// expert totals (ceil(T/256) * E + E ints).  Here it lives in a file-scope
// device array, so the caller passes inputs and outputs only.  The array
// exists once per GPU that loads the library and stays allocated until the
// process exits.  All calls share it: every entry a later kernel reads is
// written earlier in the same call, so nothing has to be cleared between calls,
// but two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on it.
constexpr long long kStaticScratchInts = 1 << 16;  // 256 KB
static __device__ __align__(256) int g_dispatch_static_scratch[kStaticScratchInts];

static int* g_static_scratch_dev[64];
static std::mutex g_static_scratch_mu;

long long dispatch_static_scratch_ints() { return kStaticScratchInts; }
long long dispatch_scratch_ints(int T, int E) { return scratch_ints(T, E); }

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
  if (scratch_ints(T, E) > kStaticScratchInts) return MOE_ERR_WORKSPACE;
  int st = MOE_OK;
  int* scratch = static_scratch_address(&st);
  if (!scratch) return st;
  return launch_dispatch(x, idx, T, H, E, K, dtype, cu, dst_row, src_tok, xs, scratch, s);
}

}  // namespace moe
