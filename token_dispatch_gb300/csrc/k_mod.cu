// Mixture-of-Depths capacity router (MoE/MoD framework page, MoD paragraph:
// part of the tokens skips the layer entirely; 50% capacity).
//
//   score[t] = x[t] . w_mod                         (one warp per token)
//   per sequence: the C highest scores are selected, equal scores -> lower
//   position.  One CTA per sequence sorts (score desc, position asc) keys with a
//   shared-memory bitonic network, flags the first C positions and compacts
//   them in position order with a block scan.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int SEL_THREADS = 1024;

template <typename T>
__global__ void __launch_bounds__(256)
mod_score_kernel(const T* __restrict__ x, const T* __restrict__ w, long long n_tok, int H,
                 float* __restrict__ score) {
  constexpr int V = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = H / V;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_tok; t += nwarps) {
    float acc = 0.f;
    for (int i = lane; i < nvec; i += 32) {
      float xv[V], wv[V];
      Vec16<T>::load(x + t * H + (long long)i * V, xv);
      Vec16<T>::load(w + (long long)i * V, wv);
#pragma unroll
      for (int v = 0; v < V; ++v) acc = fmaf(xv[v], wv[v], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) score[t] = acc;
  }
}

// Order-preserving map of a float to uint32 (ascending), -0 folded onto +0.
__device__ __forceinline__ unsigned ordered_bits(float f) {
  if (f == 0.f) f = 0.f;
  unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(SEL_THREADS)
mod_select_kernel(const float* __restrict__ score, int L, int C, int P, int32_t* __restrict__ sel,
                  float* __restrict__ sel_score, uint8_t* __restrict__ mask) {
  extern __shared__ unsigned long long smem_keys[];
  unsigned long long* key = smem_keys;                       // P keys
  int* flag = reinterpret_cast<int*>(smem_keys + P);         // P flags
  __shared__ int part[SEL_THREADS];
  const int b = blockIdx.x;
  const float* s = score + (long long)b * L;
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    // ascending sort of (~ordered(score), position) == score desc, position asc
    key[i] = (i < L) ? ((unsigned long long)(~ordered_bits(s[i])) << 32) | (unsigned)i : ~0ull;
    flag[i] = 0;
  }
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        int l = i ^ j;
        if (l > i) {
          unsigned long long a = key[i], c = key[l];
          bool up = (i & k) == 0;
          if ((a > c) == up) { key[i] = c; key[l] = a; }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < C; i += blockDim.x) flag[key[i] & 0xffffffffu] = 1;
  __syncthreads();
  // compact flagged positions in increasing order: each thread owns a run of positions
  const int per = (P + SEL_THREADS - 1) / SEL_THREADS;
  const int lo = threadIdx.x * per;
  int cnt = 0;
  for (int i = lo; i < lo + per && i < L; ++i) cnt += flag[i];
  part[threadIdx.x] = cnt;
  __syncthreads();
  for (int o = 1; o < SEL_THREADS; o <<= 1) {
    int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int r = part[threadIdx.x] - cnt;
  for (int i = lo; i < lo + per && i < L; ++i) {
    mask[(long long)b * L + i] = (uint8_t)flag[i];
    if (flag[i]) {
      sel[(long long)b * C + r] = b * L + i;
      if (sel_score) sel_score[(long long)b * C + r] = s[i];
      ++r;
    }
  }
}

// x_sel[j] = x[sel[j]]  (sel holds flat token indices)
__global__ void __launch_bounds__(256)
gather_selected_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sel, long long n_sel,
                       int vec_per_row, uint4* __restrict__ x_sel) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long j = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < n_sel; j += nwarps) {
    long long src = __ldg(sel + j);
    for (int i = lane; i < vec_per_row; i += 32)
      x_sel[j * vec_per_row + i] = __ldg(x + src * vec_per_row + i);
  }
}

// y[t] = x[t] for tokens that skip the layer
__global__ void __launch_bounds__(256)
skip_copy_kernel(const uint4* __restrict__ x, const uint8_t* __restrict__ mask, long long n_tok,
                 int vec_per_row, uint4* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_tok; t += nwarps) {
    if (mask[t]) continue;
    for (int i = lane; i < vec_per_row; i += 32) y[t * vec_per_row + i] = __ldg(x + t * vec_per_row + i);
  }
}

int warp_grid(long long n) {
  long long ctas = (n + 7) / 8;
  long long cap = (long long)sm_count() * 16;
  if (ctas < 1) ctas = 1;
  return (int)(ctas < cap ? ctas : cap);
}

}  // namespace

int launch_mod_select(const void* x, const void* w, int B, int L, int H, int C, int dtype,
                      float* score, int32_t* sel, float* sel_score, uint8_t* mask, void* x_sel,
                      void* y_skip, cudaStream_t s) {
  const long long n_tok = (long long)B * L;
  if (n_tok == 0) return MOE_OK;
  if (dtype == MOE_BF16)
    mod_score_kernel<bf16><<<warp_grid(n_tok), 256, 0, s>>>(static_cast<const bf16*>(x),
                                                            static_cast<const bf16*>(w), n_tok, H, score);
  else
    mod_score_kernel<float><<<warp_grid(n_tok), 256, 0, s>>>(static_cast<const float*>(x),
                                                             static_cast<const float*>(w), n_tok, H, score);
  int st = launch_status();
  if (st != MOE_OK) return st;
  int P = 1;
  while (P < L) P <<= 1;
  size_t smem = (size_t)P * (sizeof(unsigned long long) + sizeof(int));
  if (cudaFuncSetAttribute(mod_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  mod_select_kernel<<<B, SEL_THREADS, smem, s>>>(score, L, C, P, sel, sel_score, mask);
  st = launch_status();
  if (st != MOE_OK) return st;
  const int vec = H * (dtype == MOE_BF16 ? 2 : 4) / 16;
  if (x_sel && C > 0) {
    gather_selected_kernel<<<warp_grid((long long)B * C), 256, 0, s>>>(
        static_cast<const uint4*>(x), sel, (long long)B * C, vec, static_cast<uint4*>(x_sel));
    st = launch_status();
    if (st != MOE_OK) return st;
  }
  if (y_skip) {
    skip_copy_kernel<<<warp_grid(n_tok), 256, 0, s>>>(static_cast<const uint4*>(x), mask, n_tok, vec,
                                                      static_cast<uint4*>(y_skip));
    st = launch_status();
  }
  return st;
}

}  // namespace moe
