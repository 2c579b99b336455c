// Token dispatch (histogram -> cu_seqlens -> stable permutation -> row gather),
// combine (gate-weighted gather-sum back to token order) and their backward.
//
// Dispatch/combine follow the MoE/MoD framework page ("What's in the box":
// a fused kernel moving tokens between experts, reading and writing the buffers
// directly) and the MoonEP page ("Step-by-step": tokens land in one contiguous
// expert-sorted buffer whose active rows are described by cu_seqlens).
//
// The histogram is atomic-free: every warp owns a private histogram in shared
// memory and groups equal expert ids of its 32 lanes with __match_any_sync, so
// one leader lane per distinct expert updates the counter.  The same pass gives
// each pair its rank among earlier pairs of the same expert (popc of lower peer
// lanes), so the permutation is stable by token and identical run to run.
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

// One CTA: per-expert totals over chunks, exclusive scan over experts -> cu,
// then per-chunk starting rows (written over the counts).
__global__ void __launch_bounds__(1024)
dispatch_scan_kernel(int* __restrict__ counts, int C, int E, int32_t* __restrict__ cu) {
  __shared__ int sc[MAX_E];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E)
    for (int c = 0; c < C; ++c) total += counts[(long long)c * E + e];
  sc[e] = total;
  __syncthreads();
  // inclusive Hillis-Steele scan over 1024 entries
  for (int o = 1; o < 1024; o <<= 1) {
    int v = e >= o ? sc[e - o] : 0;
    __syncthreads();
    sc[e] += v;
    __syncthreads();
  }
  int excl = sc[e] - total;
  if (e < E) {
    cu[e] = excl;
    if (e == E - 1) cu[E] = sc[e];
    int run = excl;
    for (int c = 0; c < C; ++c) {
      int n = counts[(long long)c * E + e];
      counts[(long long)c * E + e] = run;
      run += n;
    }
  }
}

__global__ void __launch_bounds__(32 * CH_WARPS)
dispatch_place_kernel(const int32_t* __restrict__ idx, int T, int E, int K,
                      const int* __restrict__ chunk_off, int32_t* __restrict__ dst_row,
                      int32_t* __restrict__ src_tok) {
  __shared__ int hist[CH_WARPS][MAX_E];
  const int w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < CH_WARPS * E; i += blockDim.x) hist[i / E][i % E] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * CH_TOK + w * TOK_PER_WARP;
  warp_count(idx, T, E, K, t0, hist[w], nullptr);
  __syncthreads();
  // hist[w][e] <- first row of warp w for expert e
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_off[(long long)blockIdx.x * E + e];
#pragma unroll
    for (int ww = 0; ww < CH_WARPS; ++ww) {
      int n = hist[ww][e];
      hist[ww][e] = run;
      run += n;
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

// xs[dst_row[t*K+k]] = x[t]: one warp per token, 16-byte vectors, x read once.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ dst_row, int T, int K,
                   int vec_per_row, uint4* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nwarps) {
    int rows[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) rows[k] = (k < K) ? __ldg(dst_row + t * K + k) : -1;
    const uint4* src = x + t * vec_per_row;
    for (int i = lane; i < vec_per_row; i += 64) {
      uint4 a = __ldg(src + i);
      bool two = i + 32 < vec_per_row;
      uint4 b = two ? __ldg(src + i + 32) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k < K && rows[k] >= 0) {
          uint4* dst = xs + (long long)rows[k] * vec_per_row;
          dst[i] = a;
          if (two) dst[i + 32] = b;
        }
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ h, const float* __restrict__ gate,
               const int32_t* __restrict__ dst_row, const float* __restrict__ scale,
               const T* __restrict__ residual, const int32_t* __restrict__ out_row,
               int Tn, int H, int K, T* __restrict__ y) {
  constexpr int V = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = H / V;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < Tn; t += nwarps) {
    int rows[16];
    float g[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      rows[k] = (k < K) ? (dst_row ? __ldg(dst_row + t * K + k) : (int)(t * K + k)) : -1;
      g[k] = (k < K) ? __ldg(gate + t * K + k) : 0.f;
    }
    const float s = scale ? __ldg(scale + t) : 1.0f;
    const long long o = out_row ? (long long)__ldg(out_row + t) : t;
    for (int i = lane; i < nvec; i += 32) {
      float acc[V];
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k < K && rows[k] >= 0) {
          float hv[V];
          Vec16<T>::load(h + (long long)rows[k] * H + (long long)i * V, hv);
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] = fmaf(g[k], hv[v], acc[v]);
        }
      }
      float out[V];
      if (residual) {
        float rv[V];
        Vec16<T>::load(residual + o * H + (long long)i * V, rv);
#pragma unroll
        for (int v = 0; v < V; ++v) out[v] = fmaf(s, acc[v], rv[v]);
      } else {
#pragma unroll
        for (int v = 0; v < V; ++v) out[v] = s * acc[v];
      }
      Vec16<T>::store(y + o * H + (long long)i * V, out);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
permute_bwd_kernel(const T* __restrict__ dy, const T* __restrict__ h, const float* __restrict__ gate,
                   const int32_t* __restrict__ dst_row, const float* __restrict__ scale,
                   const int32_t* __restrict__ out_row, const T* __restrict__ dxs,
                   int Tn, int H, int K, T* __restrict__ dh, float* __restrict__ d_gate,
                   float* __restrict__ d_scale, T* __restrict__ dx) {
  constexpr int V = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = H / V;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < Tn; t += nwarps) {
    int rows[16];
    float g[16], dot[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      rows[k] = (k < K) ? (dst_row ? __ldg(dst_row + t * K + k) : (int)(t * K + k)) : -1;
      g[k] = (k < K) ? __ldg(gate + t * K + k) : 0.f;
      dot[k] = 0.f;
    }
    const float s = scale ? __ldg(scale + t) : 1.0f;
    const long long o = out_row ? (long long)__ldg(out_row + t) : t;
    for (int i = lane; i < nvec; i += 32) {
      float gy[V], ax[V];
      Vec16<T>::load(dy + o * H + (long long)i * V, gy);
#pragma unroll
      for (int v = 0; v < V; ++v) ax[v] = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k < K && rows[k] >= 0) {
          const long long off = (long long)rows[k] * H + (long long)i * V;
          if (d_gate || d_scale) {
            float hv[V];
            Vec16<T>::load(h + off, hv);
#pragma unroll
            for (int v = 0; v < V; ++v) dot[k] = fmaf(gy[v], hv[v], dot[k]);
          }
          if (dh) {
            float d[V];
            const float c = s * g[k];
#pragma unroll
            for (int v = 0; v < V; ++v) d[v] = c * gy[v];
            Vec16<T>::store(dh + off, d);
          }
          if (dx) {
            float xv[V];
            Vec16<T>::load(dxs + off, xv);
#pragma unroll
            for (int v = 0; v < V; ++v) ax[v] += xv[v];
          }
        }
      }
      if (dx) Vec16<T>::store(dx + t * H + (long long)i * V, ax);
    }
    if (d_gate || d_scale) {
      float ds = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k < K) {
          float d = warp_sum(dot[k]);
          if (lane == 0 && d_gate) d_gate[t * K + k] = s * d;
          ds = fmaf(g[k], d, ds);
        }
      }
      if (lane == 0 && d_scale) d_scale[t] = ds;
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
  dispatch_scan_kernel<<<1, 1024, 0, s>>>(counts, C, E, cu);
  int st = launch_status();
  if (st != MOE_OK || T == 0) return st;
  dispatch_place_kernel<<<C, 32 * CH_WARPS, 0, s>>>(idx, T, E, K, counts, dst_row, src_tok);
  st = launch_status();
  if (st != MOE_OK) return st;
  const int row_bytes = H * (dtype == MOE_BF16 ? 2 : 4);
  gather_rows_kernel<<<warp_grid(T), 256, 0, s>>>(static_cast<const uint4*>(x), dst_row, T, K,
                                                  row_bytes / 16, static_cast<uint4*>(xs));
  return launch_status();
}

int launch_combine(const void* h, const float* gate, const int32_t* dst_row, const float* scale,
                   const void* residual, const int32_t* out_row, int T, int H, int K, int dtype,
                   void* y, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  int grid = warp_grid(T);
  if (dtype == MOE_BF16)
    combine_kernel<bf16><<<grid, 256, 0, s>>>(static_cast<const bf16*>(h), gate, dst_row, scale,
                                              static_cast<const bf16*>(residual), out_row, T, H, K,
                                              static_cast<bf16*>(y));
  else
    combine_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(h), gate, dst_row, scale,
                                               static_cast<const float*>(residual), out_row, T, H, K,
                                               static_cast<float*>(y));
  return launch_status();
}

int launch_permute_bwd(const void* dy, const void* h, const float* gate, const int32_t* dst_row,
                       const float* scale, const int32_t* out_row, const void* dxs, int T, int H,
                       int K, int dtype, void* dh, float* d_gate, float* d_scale, void* dx,
                       cudaStream_t s) {
  if (T == 0) return MOE_OK;
  int grid = warp_grid(T);
  if (dtype == MOE_BF16)
    permute_bwd_kernel<bf16><<<grid, 256, 0, s>>>(
        static_cast<const bf16*>(dy), static_cast<const bf16*>(h), gate, dst_row, scale, out_row,
        static_cast<const bf16*>(dxs), T, H, K, static_cast<bf16*>(dh), d_gate, d_scale,
        static_cast<bf16*>(dx));
  else
    permute_bwd_kernel<float><<<grid, 256, 0, s>>>(
        static_cast<const float*>(dy), static_cast<const float*>(h), gate, dst_row, scale, out_row,
        static_cast<const float*>(dxs), T, H, K, static_cast<float*>(dh), d_gate, d_scale,
        static_cast<float*>(dx));
  return launch_status();
}

}  // namespace moe
