// Router for few experts (E <= 16) in one launch: logits = x W_r + bias,
// softmax over experts, top-K with the lowest-index tie-break, gates.
//
// MoE/MoD framework page, "What's in the box": softmax over experts and top-k
// selection "in one launch", with warp-level primitives.  With E <= 16 the
// router does at most 16 FLOP per byte of x, far below the tensor-core ridge:
// it is an HBM stream, so it runs on the FFMA pipes and reads x exactly once.
//
// W_r is staged once per CTA in shared memory as fp32, in chunks of the V rows
// that one 16-byte vector of x covers (chunk stride padded by 16 bytes so the
// 32 lanes of a warp hit 32 different banks).  A warp takes TPW tokens at a
// time; lane l accumulates chunks l, l+32, ... of all TPW tokens (each W value
// read from shared memory serves TPW tokens), the partial logits are summed
// across the warp with shuffles, and lane j < TPW finishes token j: bias,
// logits store, softmax, top-K.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int RF_WARPS = 16;  // 512 threads, one CTA per SM (W_r fills shared memory)
constexpr int RF_TPW = 4;     // tokens per warp pass

template <typename T> constexpr int chunk_rows() { return 16 / (int)sizeof(T); }
template <int EP, typename T> constexpr int chunk_stride() { return chunk_rows<T>() * EP + 4; }

template <int EP>
__device__ __forceinline__ void finish_token(const float (&acc)[EP], long long t, int E, int K, const float* bias,
                                             float* logits, int32_t* idx, float* gate) {
  float l[EP];
#pragma unroll
  for (int e = 0; e < EP; ++e) l[e] = e < E ? acc[e] + (bias ? __ldg(bias + e) : 0.f) : -INFINITY;
#pragma unroll
  for (int e = 0; e < EP; ++e)
    if (e < E) logits[t * E + e] = l[e];
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < EP; ++e) m = fmaxf(m, l[e]);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < EP; ++e) s += e < E ? expf(l[e] - m) : 0.f;
  unsigned taken = 0;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int be = 0;
    bool found = false;
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      // strict '>' keeps the lowest index among equal logits
      if (e < E && !((taken >> e) & 1u) && (!found || l[e] > bv)) { bv = l[e]; be = e; found = true; }
    }
    taken |= 1u << be;
    idx[t * K + k] = be;
    gate[t * K + k] = expf(bv - m) / s;
  }
}

template <typename T, int EP>
__global__ void __launch_bounds__(32 * RF_WARPS, 1)
router_fused_kernel(const T* __restrict__ x, const T* __restrict__ w, const float* __restrict__ bias, int Tn,
                    int H, int E, int K, float* __restrict__ logits, int32_t* __restrict__ idx,
                    float* __restrict__ gate) {
  constexpr int V = chunk_rows<T>();
  constexpr int CF = V * EP;                 // W values of one chunk
  constexpr int CS = chunk_stride<EP, T>();  // padded chunk stride (floats)
  extern __shared__ __align__(16) float wsm[];
  const int nchunk = H / V;
  for (int i = threadIdx.x; i < nchunk * CF; i += blockDim.x) {
    const int c = i / CF, r = i % CF;
    const int h = c * V + r / EP, e = r % EP;
    wsm[c * CS + r] = e < E ? to_f32(w[(long long)h * E + e]) : 0.f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long nw = (long long)gridDim.x * RF_WARPS;
  for (long long t0 = ((long long)blockIdx.x * RF_WARPS + (threadIdx.x >> 5)) * RF_TPW; t0 < Tn;
       t0 += nw * RF_TPW) {
    float acc[RF_TPW][EP];
#pragma unroll
    for (int j = 0; j < RF_TPW; ++j)
#pragma unroll
      for (int e = 0; e < EP; ++e) acc[j][e] = 0.f;
    for (int c = lane; c < nchunk; c += 32) {
      float xv[RF_TPW][V];
#pragma unroll
      for (int j = 0; j < RF_TPW; ++j) {
        if (t0 + j < Tn) {
          Vec16<T>::load(x + (t0 + j) * H + (long long)c * V, xv[j]);
        } else {
#pragma unroll
          for (int v = 0; v < V; ++v) xv[j][v] = 0.f;
        }
      }
      const float* wc = wsm + c * CS;
#pragma unroll
      for (int hv = 0; hv < V; ++hv) {
        float wr[EP];
#pragma unroll
        for (int q = 0; q < EP / 4; ++q) {
          const float4 f = *reinterpret_cast<const float4*>(wc + hv * EP + 4 * q);
          wr[4 * q] = f.x; wr[4 * q + 1] = f.y; wr[4 * q + 2] = f.z; wr[4 * q + 3] = f.w;
        }
#pragma unroll
        for (int j = 0; j < RF_TPW; ++j)
#pragma unroll
          for (int e = 0; e < EP; ++e) acc[j][e] = fmaf(xv[j][hv], wr[e], acc[j][e]);
      }
    }
#pragma unroll
    for (int j = 0; j < RF_TPW; ++j)
#pragma unroll
      for (int e = 0; e < EP; ++e) acc[j][e] = warp_sum(acc[j][e]);
#pragma unroll
    for (int j = 0; j < RF_TPW; ++j)
      if (lane == j && t0 + j < Tn) finish_token<EP>(acc[j], t0 + j, E, K, bias, logits, idx, gate);
  }
}

template <typename T, int EP>
size_t fused_smem(int H) {
  return (size_t)(H / chunk_rows<T>()) * chunk_stride<EP, T>() * sizeof(float);
}

template <typename T, int EP>
int launch_fused(const void* x, const void* w, const float* bias, int T_, int H, int E, int K, float* logits,
                 int32_t* idx, float* gate, cudaStream_t s) {
  const size_t smem = fused_smem<T, EP>(H);
  auto k = router_fused_kernel<T, EP>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  long long warps = ((long long)T_ + RF_TPW - 1) / RF_TPW;
  long long ctas = (warps + RF_WARPS - 1) / RF_WARPS;
  const long long cap = sm_count();
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  k<<<(unsigned)ctas, 32 * RF_WARPS, smem, s>>>(static_cast<const T*>(x), static_cast<const T*>(w), bias, T_, H, E,
                                                  K, logits, idx, gate);
  return launch_status();
}

constexpr size_t RF_SMEM_LIMIT = 200 * 1024;

}  // namespace

// The one-launch router serves E <= 16 whenever W_r (fp32) fits in shared memory.
bool router_fused_ok(int H, int E, int dtype) {
  if (E > 16 || E < 1) return false;
  const int V = dtype == MOE_BF16 ? 8 : 4;
  if (H % V != 0) return false;
  const size_t smem = dtype == MOE_BF16 ? (E <= 8 ? fused_smem<bf16, 8>(H) : fused_smem<bf16, 16>(H))
                                        : (E <= 8 ? fused_smem<float, 8>(H) : fused_smem<float, 16>(H));
  return smem <= RF_SMEM_LIMIT;
}

int launch_router_fused(const void* x, const void* w, const float* bias, int T, int H, int E, int K, int dtype,
                        float* logits, int32_t* idx, float* gate, cudaStream_t s) {
  if (dtype == MOE_BF16)
    return E <= 8 ? launch_fused<bf16, 8>(x, w, bias, T, H, E, K, logits, idx, gate, s)
                  : launch_fused<bf16, 16>(x, w, bias, T, H, E, K, logits, idx, gate, s);
  return E <= 8 ? launch_fused<float, 8>(x, w, bias, T, H, E, K, logits, idx, gate, s)
                : launch_fused<float, 16>(x, w, bias, T, H, E, K, logits, idx, gate, s);
}

}  // namespace moe
