// Router: logits GEMM, fused softmax + top-K gate, and the router backward.
//
// Softmax/top-K follows the routing/gating kernel of the MoE/MoD framework page
// ("What's in the box": softmax over experts and top-k in one launch, warp-level
// primitives for top-k).  One warp per token row: the row is read with 128-bit
// loads, max / sum / arg-max are warp-shuffle reductions, and the K winners are
// taken by K rounds of a (value desc, expert asc) arg-max, which gives the
// lowest-index tie-break exactly.  Selection is on the fp32 logits themselves.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int ROWS_PER_CTA = 8;  // warps per CTA

// Values per lane: VPL (multiple of 4); element e of the row lives in lane
// (e/4) % 32, slot 4*(e/128) + e%4.
template <int VPL>
__device__ __forceinline__ void load_row(const float* row, int E, int lane, float (&v)[VPL]) {
#pragma unroll
  for (int q = 0; q < VPL / 4; ++q) {
    int e4 = (q * 32 + lane) * 4;
    if (e4 < E) {
      float4 f = __ldg(reinterpret_cast<const float4*>(row + e4));
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    } else {
      v[4 * q] = v[4 * q + 1] = v[4 * q + 2] = v[4 * q + 3] = -INFINITY;
    }
  }
}
__device__ __forceinline__ int slot_expert(int slot, int lane) {
  return ((slot >> 2) * 32 + lane) * 4 + (slot & 3);
}

template <int VPL>
__global__ void __launch_bounds__(32 * ROWS_PER_CTA)
softmax_topk_kernel(const float* __restrict__ logits, int T, int E, int K,
                    int32_t* __restrict__ idx, float* __restrict__ gate) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * ROWS_PER_CTA;
  for (long long t = (long long)blockIdx.x * ROWS_PER_CTA + (threadIdx.x >> 5); t < T; t += nwarps) {
    float v[VPL];
    load_row<VPL>(logits + t * E, E, lane, v);
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPL; ++j) m = fmaxf(m, v[j]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) s += (slot_expert(j, lane) < E) ? expf(v[j] - m) : 0.f;
    s = warp_sum(s);
    unsigned taken = 0;
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        int e = slot_expert(j, lane);
        bool ok = e < E && !((taken >> j) & 1u);
        if (ok && (v[j] > bv || (v[j] == bv && e < be))) { bv = v[j]; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      if (((be >> 2) & 31) == lane) taken |= 1u << ((be >> 7) * 4 + (be & 3));
      if (lane == 0) {
        idx[t * K + k] = be;
        gate[t * K + k] = expf(bv - m) / s;
      }
    }
  }
}

// d_logits[t,j] = p_j (G_j - sum_k d_gate[t,k] p[idx[t,k]])
template <int VPL>
__global__ void __launch_bounds__(32 * ROWS_PER_CTA)
softmax_topk_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                        const float* __restrict__ d_gate, int T, int E, int K,
                        float* __restrict__ d_logits) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * ROWS_PER_CTA;
  for (long long t = (long long)blockIdx.x * ROWS_PER_CTA + (threadIdx.x >> 5); t < T; t += nwarps) {
    float v[VPL];
    load_row<VPL>(logits + t * E, E, lane, v);
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPL; ++j) m = fmaxf(m, v[j]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) s += (slot_expert(j, lane) < E) ? expf(v[j] - m) : 0.f;
    s = warp_sum(s);
    float p[VPL], G[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      p[j] = (slot_expert(j, lane) < E) ? expf(v[j] - m) / s : 0.f;
      G[j] = 0.f;
    }
    float inner = 0.f;
    for (int k = 0; k < K; ++k) {
      int e = __ldg(idx + t * K + k);
      float dg = __ldg(d_gate + t * K + k);
      if (((e >> 2) & 31) == lane) {
        int slot = (e >> 7) * 4 + (e & 3);
#pragma unroll
        for (int j = 0; j < VPL; ++j)
          if (j == slot) { G[j] = dg; inner += dg * p[j]; }
      }
    }
    inner = warp_sum(inner);
    float* out = d_logits + t * E;
#pragma unroll
    for (int q = 0; q < VPL / 4; ++q) {
      int e4 = (q * 32 + lane) * 4;
      if (e4 < E) {
        float4 r;
        r.x = p[4 * q] * (G[4 * q] - inner);
        r.y = p[4 * q + 1] * (G[4 * q + 1] - inner);
        r.z = p[4 * q + 2] * (G[4 * q + 2] - inner);
        r.w = p[4 * q + 3] * (G[4 * q + 3] - inner);
        *reinterpret_cast<float4*>(out + e4) = r;
      }
    }
  }
}

__global__ void copy_f32_kernel(const float* __restrict__ a, float* __restrict__ b, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    b[i] = a[i];
}

// dw[i] = sum_s part[s][i], in split order (deterministic).
__global__ void reduce_splits_kernel(const float* __restrict__ part, int S, long long n, float* __restrict__ out) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) acc += part[(long long)s * n + i];
    out[i] = acc;
  }
}

int rows_grid(long long T) {
  long long ctas = (T + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
  long long cap = (long long)sm_count() * 16;
  return (int)(ctas < cap ? (ctas > 0 ? ctas : 1) : cap);
}

int splits_for(int T, int H, int E) {
  long long by_t = T / 512;
  long long by_mem = (64ll << 20) / ((long long)H * E * 4);
  long long s = by_t < by_mem ? by_t : by_mem;
  if (s > 16) s = 16;
  return s < 1 ? 1 : (int)s;
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

int launch_router_tc(const void* x, const void* w, const float* bias, int T, int H, int E, float* logits,
                     cudaStream_t s);

// bf16: tcgen05 GEMM with the bias added in the epilogue.  fp32: FFMA GEMM.
int launch_router_logits(const void* x, const void* w, const float* bias, int T, int H, int E,
                         int dtype, float* logits, cudaStream_t s) {
  if (dtype == MOE_BF16) return launch_router_tc(x, w, bias, T, H, E, logits, s);
  SimtGemmArgs a{};
  a.A = x; a.a_sm = H; a.a_sk = 1;
  a.B = w; a.b_sg = 0; a.b_sk = E; a.b_sn = 1;
  a.C = logits; a.c_sm = E;
  a.bias = bias; a.cu = nullptr;
  a.M = T; a.N = E; a.K = H; a.groups = 1;
  a.epilogue = 2; a.swiglu = false;
  return launch_simt_gemm(a, dtype, dtype, MOE_F32, s);
}

int launch_softmax_topk(const float* logits, int T, int E, int K, int32_t* idx, float* gate,
                        cudaStream_t s) {
  if (T == 0) return MOE_OK;
  int grid = rows_grid(T);
  int vpl = (E + 127) / 128 * 4;
  if (vpl <= 4) softmax_topk_kernel<4><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, T, E, K, idx, gate);
  else if (vpl <= 8) softmax_topk_kernel<8><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, T, E, K, idx, gate);
  else if (vpl <= 16) softmax_topk_kernel<16><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, T, E, K, idx, gate);
  else softmax_topk_kernel<32><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, T, E, K, idx, gate);
  return launch_status();
}

size_t route_bwd_ws_bytes(int T, int H, int E) {
  int S = splits_for(T, H, E);
  return align256((size_t)S * H * E * 4) + align256((size_t)T * E * 4);
}

int launch_route_bwd(int mode, const float* d_gate, const float* logits, const int32_t* idx,
                     const void* x, const void* w, int T, int H, int E, int K, int dtype,
                     float* d_logits, float* dw, void* dx, bool dx_write, void* ws, cudaStream_t s) {
  if (T == 0) {
    if (dw) {
      cudaMemsetAsync(dw, 0, (size_t)H * E * 4, s);
    }
    return launch_status();
  }
  const int S = splits_for(T, H, E);
  float* part = static_cast<float*>(ws);
  float* dl = d_logits;
  if (!dl) dl = reinterpret_cast<float*>(static_cast<char*>(ws) + align256((size_t)S * H * E * 4));

  if (mode == MOE_ROUTE_SOFTMAX_TOPK) {
    int grid = rows_grid(T);
    int vpl = (E + 127) / 128 * 4;
    if (vpl <= 4) softmax_topk_bwd_kernel<4><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, idx, d_gate, T, E, K, dl);
    else if (vpl <= 8) softmax_topk_bwd_kernel<8><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, idx, d_gate, T, E, K, dl);
    else if (vpl <= 16) softmax_topk_bwd_kernel<16><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, idx, d_gate, T, E, K, dl);
    else softmax_topk_bwd_kernel<32><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, idx, d_gate, T, E, K, dl);
  } else {
    // linear score: the score gradient is the logit gradient (E = K = 1)
    copy_f32_kernel<<<rows_grid(T), 256, 0, s>>>(d_gate, dl, (long long)T);
  }
  int st = launch_status();
  if (st != MOE_OK) return st;

  if (dw) {
    // dw[h,e] = sum_t x[t,h] dl[t,e], split over T for parallelism, reduced in order
    int chunk = (T + S - 1) / S;
    for (int sp = 0; sp < S; ++sp) {
      int t0 = sp * chunk;
      int len = T - t0 < chunk ? T - t0 : chunk;
      float* out = part + (size_t)sp * H * E;
      SimtGemmArgs a{};
      a.A = static_cast<const char*>(x) + (size_t)t0 * H * (dtype == MOE_BF16 ? 2 : 4);
      a.a_sm = 1; a.a_sk = H;
      a.B = dl + (size_t)t0 * E; a.b_sg = 0; a.b_sk = E; a.b_sn = 1;
      a.C = out; a.c_sm = E;
      a.M = H; a.N = E; a.K = len > 0 ? len : 0; a.groups = 1; a.epilogue = 0;
      if (len <= 0) {
        cudaMemsetAsync(out, 0, (size_t)H * E * 4, s);
        continue;
      }
      st = launch_simt_gemm(a, dtype, MOE_F32, MOE_F32, s);
      if (st != MOE_OK) return st;
    }
    long long n = (long long)H * E;
    int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    reduce_splits_kernel<<<grid, 256, 0, s>>>(part, S, n, dw);
    st = launch_status();
    if (st != MOE_OK) return st;
  }
  if (dx) {
    // dx[t,h] += sum_e dl[t,e] w[h,e]
    SimtGemmArgs a{};
    a.A = dl; a.a_sm = E; a.a_sk = 1;
    a.B = w; a.b_sg = 0; a.b_sk = 1; a.b_sn = E;
    a.C = dx; a.c_sm = H;
    a.M = T; a.N = H; a.K = E; a.groups = 1; a.epilogue = dx_write ? 0 : 1;
    st = launch_simt_gemm(a, MOE_F32, dtype, dtype, s);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

}  // namespace moe
