// Combine (gate-weighted gather-sum back to token order) and the backward of
// combine and of the dispatch gather.
//
// MoE/MoD framework page, "What's in the box": dispatch and combine move tokens
// between experts with a kernel that reads and writes the buffers directly, and
// the gating/dispatch gradients come from one sparse backward kernel.  The
// scatter-add of the combine is written as a gather over each token's K rows
// (dst_row), which gives the same sum in a fixed k order without atomics.
//
// Both kernels are HBM-bound row streams: one warp per token, 16-byte vectors,
// and the loads of U vector columns of all K rows are issued before the
// arithmetic so enough bytes are in flight per SM to cover DRAM latency.
#include "moe_internal.cuh"

namespace moe {
namespace {

template <typename T> struct Raw;
template <> struct Raw<bf16> {
  static constexpr int V = 8;
  __device__ __forceinline__ static void unpack(const uint4& q, float* v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  __device__ __forceinline__ static uint4 pack(const float* v) {
    uint4 q;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return q;
  }
};
template <> struct Raw<float> {
  static constexpr int V = 4;
  __device__ __forceinline__ static void unpack(const uint4& q, float* v) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
  __device__ __forceinline__ static uint4 pack(const float* v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
  }
};

__device__ __forceinline__ uint4 zero16() { return make_uint4(0, 0, 0, 0); }

constexpr int WARPS = 8;

// y[o(t)] = residual[o(t)] + s_t * sum_k gate[t,k] h[dst_row[t*K+k]]   (k order)
template <typename T, int KT>
__global__ void __launch_bounds__(32 * WARPS)
combine_kernel(const uint4* __restrict__ h, const float* __restrict__ gate, const int32_t* __restrict__ dst_row,
               const float* __restrict__ scale, const uint4* __restrict__ residual,
               const int32_t* __restrict__ out_row, int Tn, int nvec, int K, uint4* __restrict__ y) {
  constexpr int V = Raw<T>::V;
  constexpr int U = KT <= 2 ? 4 : KT <= 8 ? 2 : 1;  // U*KT h rows of 16 bytes per lane in flight
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * WARPS;
  for (long long t = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5); t < Tn; t += nwarps) {
    int rows[KT];
    float g[KT];
#pragma unroll
    for (int k = 0; k < KT; ++k) {
      rows[k] = (k < K) ? (dst_row ? __ldg(dst_row + t * K + k) : (int)(t * K + k)) : -1;
      g[k] = (k < K) ? __ldg(gate + t * K + k) : 0.f;
    }
    const float s = scale ? __ldg(scale + t) : 1.0f;
    const long long o = out_row ? (long long)__ldg(out_row + t) : t;
    for (int i0 = lane; i0 < nvec; i0 += 32 * U) {
      uint4 raw[U][KT], rr[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + 32 * u;
#pragma unroll
        for (int k = 0; k < KT; ++k)
          raw[u][k] = (i < nvec && rows[k] >= 0) ? __ldg(h + (long long)rows[k] * nvec + i) : zero16();
        rr[u] = (residual && i < nvec) ? __ldg(residual + o * nvec + i) : zero16();
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + 32 * u;
        if (i >= nvec) break;
        float acc[V], hv[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
#pragma unroll
        for (int k = 0; k < KT; ++k) {
          if (rows[k] < 0) continue;
          Raw<T>::unpack(raw[u][k], hv);
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] = fmaf(g[k], hv[v], acc[v]);
        }
        float out[V];
        if (residual) {
          float rv[V];
          Raw<T>::unpack(rr[u], rv);
#pragma unroll
          for (int v = 0; v < V; ++v) out[v] = fmaf(s, acc[v], rv[v]);
        } else {
#pragma unroll
          for (int v = 0; v < V; ++v) out[v] = s * acc[v];
        }
        y[o * nvec + i] = Raw<T>::pack(out);
      }
    }
  }
}

// With g(t) = dy[o(t)]:  dh[row] = s_t gate[t,k] g(t);  d_gate = s_t <g(t), h[row]>;
// d_scale[t] = sum_k gate[t,k] <g(t), h[row]>;  dx[t] = sum_k dxs[row].
// The K rows are taken in groups of KT (a single group unless K > 8); dx is
// written by the first group and accumulated by later ones.
// Small CTAs and a register cap of 128 (four CTAs of four warps per SM): with
// K rows of h and dxs plus dy requested at once per lane, the loads in flight
// per SM grow with the resident warps.
constexpr int PB_WARPS = 4;

template <typename T, int KT>
__global__ void __launch_bounds__(32 * PB_WARPS, 4)
permute_bwd_kernel(const uint4* __restrict__ dy, const uint4* __restrict__ h, const float* __restrict__ gate,
                   const int32_t* __restrict__ dst_row, const float* __restrict__ scale,
                   const int32_t* __restrict__ out_row, const uint4* __restrict__ dxs, int Tn, int nvec, int K,
                   uint4* __restrict__ dh, float* __restrict__ d_gate, float* __restrict__ d_scale,
                   uint4* __restrict__ dx) {
  constexpr int V = Raw<T>::V;
  constexpr int U = KT <= 2 ? 2 : 1;
  const int lane = threadIdx.x & 31;
  const bool want_dot = d_gate || d_scale;
  const int n_groups = (K + KT - 1) / KT;
  const long long nwarps = (long long)gridDim.x * PB_WARPS;
  for (long long t = (long long)blockIdx.x * PB_WARPS + (threadIdx.x >> 5); t < Tn; t += nwarps) {
    const float s = scale ? __ldg(scale + t) : 1.0f;
    const long long o = out_row ? (long long)__ldg(out_row + t) : t;
    float ds = 0.f;
#pragma unroll 1
    for (int grp = 0; grp < n_groups; ++grp) {
      int rows[KT];
      float g[KT], dot[KT];
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        const int kk = grp * KT + k;
        rows[k] = (kk < K) ? (dst_row ? __ldg(dst_row + t * K + kk) : (int)(t * K + kk)) : -1;
        g[k] = (kk < K) ? __ldg(gate + t * K + kk) : 0.f;
        dot[k] = 0.f;
      }
      for (int i0 = lane; i0 < nvec; i0 += 32 * U) {
        uint4 gr[U], hr[U][KT], xr[U][KT], pr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + 32 * u;
          gr[u] = (i < nvec && (dh || want_dot)) ? __ldg(dy + o * nvec + i) : zero16();
          pr[u] = (dx && grp > 0 && i < nvec) ? dx[t * nvec + i] : zero16();
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            const bool ok = i < nvec && rows[k] >= 0;
            hr[u][k] = (ok && want_dot) ? __ldg(h + (long long)rows[k] * nvec + i) : zero16();
            xr[u][k] = (ok && dx) ? __ldg(dxs + (long long)rows[k] * nvec + i) : zero16();
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + 32 * u;
          if (i >= nvec) break;
          float gy[V], ax[V];
          Raw<T>::unpack(gr[u], gy);
          Raw<T>::unpack(pr[u], ax);
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            if (rows[k] < 0) continue;
            if (want_dot) {
              float hv[V];
              Raw<T>::unpack(hr[u][k], hv);
#pragma unroll
              for (int v = 0; v < V; ++v) dot[k] = fmaf(gy[v], hv[v], dot[k]);
            }
            if (dh) {
              float d[V];
              const float c = s * g[k];
#pragma unroll
              for (int v = 0; v < V; ++v) d[v] = c * gy[v];
              dh[(long long)rows[k] * nvec + i] = Raw<T>::pack(d);
            }
            if (dx) {
              float xv[V];
              Raw<T>::unpack(xr[u][k], xv);
#pragma unroll
              for (int v = 0; v < V; ++v) ax[v] += xv[v];
            }
          }
          if (dx) dx[t * nvec + i] = Raw<T>::pack(ax);
        }
      }
      if (want_dot) {
#pragma unroll
        for (int k = 0; k < KT; ++k) {
          const int kk = grp * KT + k;
          const float d = warp_sum(dot[k]);
          if (kk < K) {
            if (lane == 0 && d_gate) d_gate[t * K + kk] = s * d;
            ds = fmaf(g[k], d, ds);
          }
        }
      }
    }
    if (lane == 0 && d_scale) d_scale[t] = ds;
  }
}

int warp_grid(long long n_warps_work) {
  long long ctas = (n_warps_work + WARPS - 1) / WARPS;
  long long cap = (long long)sm_count() * 16;
  if (ctas < 1) ctas = 1;
  return (int)(ctas < cap ? ctas : cap);
}

template <typename T, int KT>
void combine_t(const void* h, const float* gate, const int32_t* dst_row, const float* scale, const void* residual,
               const int32_t* out_row, int Tn, int nvec, int K, void* y, cudaStream_t s) {
  combine_kernel<T, KT><<<warp_grid(Tn), 32 * WARPS, 0, s>>>(
      static_cast<const uint4*>(h), gate, dst_row, scale, static_cast<const uint4*>(residual), out_row, Tn, nvec, K,
      static_cast<uint4*>(y));
}

template <typename T, int KT>
void permute_bwd_t(const void* dy, const void* h, const float* gate, const int32_t* dst_row, const float* scale,
                   const int32_t* out_row, const void* dxs, int Tn, int nvec, int K, void* dh, float* d_gate,
                   float* d_scale, void* dx, cudaStream_t s) {
  long long ctas = (Tn + PB_WARPS - 1) / PB_WARPS;
  const long long cap = (long long)sm_count() * 32;
  if (ctas > cap) ctas = cap;
  permute_bwd_kernel<T, KT><<<(unsigned)(ctas > 0 ? ctas : 1), 32 * PB_WARPS, 0, s>>>(
      static_cast<const uint4*>(dy), static_cast<const uint4*>(h), gate, dst_row, scale, out_row,
      static_cast<const uint4*>(dxs), Tn, nvec, K, static_cast<uint4*>(dh), d_gate, d_scale, static_cast<uint4*>(dx));
}

}  // namespace

int launch_combine(const void* h, const float* gate, const int32_t* dst_row, const float* scale,
                   const void* residual, const int32_t* out_row, int T, int H, int K, int dtype,
                   void* y, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int nvec = H * (dtype == MOE_BF16 ? 2 : 4) / 16;
#define MOE_COMBINE(TT)                                                                         \
  if (K <= 1) combine_t<TT, 1>(h, gate, dst_row, scale, residual, out_row, T, nvec, K, y, s);   \
  else if (K <= 2) combine_t<TT, 2>(h, gate, dst_row, scale, residual, out_row, T, nvec, K, y, s); \
  else if (K <= 4) combine_t<TT, 4>(h, gate, dst_row, scale, residual, out_row, T, nvec, K, y, s); \
  else if (K <= 8) combine_t<TT, 8>(h, gate, dst_row, scale, residual, out_row, T, nvec, K, y, s); \
  else combine_t<TT, 16>(h, gate, dst_row, scale, residual, out_row, T, nvec, K, y, s);
  if (dtype == MOE_BF16) { MOE_COMBINE(bf16) } else { MOE_COMBINE(float) }
#undef MOE_COMBINE
  return launch_status();
}

int launch_permute_bwd(const void* dy, const void* h, const float* gate, const int32_t* dst_row,
                       const float* scale, const int32_t* out_row, const void* dxs, int T, int H,
                       int K, int dtype, void* dh, float* d_gate, float* d_scale, void* dx,
                       cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int nvec = H * (dtype == MOE_BF16 ? 2 : 4) / 16;
#define MOE_PBWD(TT)                                                                                          \
  if (K <= 1) permute_bwd_t<TT, 1>(dy, h, gate, dst_row, scale, out_row, dxs, T, nvec, K, dh, d_gate, d_scale, dx, s); \
  else if (K <= 2) permute_bwd_t<TT, 2>(dy, h, gate, dst_row, scale, out_row, dxs, T, nvec, K, dh, d_gate, d_scale, dx, s); \
  else if (K <= 4) permute_bwd_t<TT, 4>(dy, h, gate, dst_row, scale, out_row, dxs, T, nvec, K, dh, d_gate, d_scale, dx, s); \
  else permute_bwd_t<TT, 8>(dy, h, gate, dst_row, scale, out_row, dxs, T, nvec, K, dh, d_gate, d_scale, dx, s);
  if (dtype == MOE_BF16) { MOE_PBWD(bf16) } else { MOE_PBWD(float) }
#undef MOE_PBWD
  return launch_status();
}

}  // namespace moe
