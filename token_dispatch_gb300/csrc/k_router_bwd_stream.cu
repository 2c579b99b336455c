// Router backward for few experts (E = 8 or 16 with the softmax/top-K gate, or
// the MoD linear score with E = 1), bf16, as one streaming pass.
//
// The sparse backward of the MoE/MoD framework page ("What's in the box": the
// gating gradients computed in one kernel without saved intermediates) needs,
// per token t, the logit gradient dl[t, :] (from the saved logits, the chosen
// experts and d_gate), then
//     dx[t, h]  (+)= sum_e dl[t, e] W_r[h, e]
//     dW_r[h, e]  += x[t, h] dl[t, e]          (summed over all tokens).
// With E <= 16 both products are 2E flops per element of x / dx, far below what
// the FMA pipes sustain per byte of HBM, so the pass is a stream of x and dx:
//   * a CTA owns a contiguous range of tokens and one slice of H; each of its
//     512 threads owns CPT consecutive columns (CPT * E = 32 products per
//     token), so the thread's W_r values and its dW_r sums stay in registers
//     for the whole range, and W_r is read once per CTA;
//   * dl for a chunk of the range is computed first, one thread per token,
//     into shared memory, where every thread of a row reads it as a broadcast;
//   * loads of x and dx for U tokens are issued before any of them is used
//     (addresses clamped into the range, so no load is predicated), x and dx
//     go from global memory straight into registers and dx back;
//   * both products run on the paired fp32 FMA (two columns per instruction):
//     column pairs of x, dx and W_r against (dl, dl);
//   * the dW_r partial of each (token range, row lane) goes to the workspace
//     and a fixed-order reduction adds the partials: the same bits every run.
// (Staging x and dx through shared memory with bulk asynchronous copies, with
// a CTA barrier per stage or per-warp rings, measured slower at 8192 tokens:
// the pass is bound by instruction issue as much as by HBM.)
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int RB_THREADS = 512;
constexpr int RB_CHUNK = 256;  // tokens whose dl sits in shared memory at a time

// CPT columns per thread (CPT * E = 32 products per token, or 8 with E = 1)
// and U tokens whose loads are in flight per thread: the thread's W_r values,
// its dW_r sums and the loads take the 128 registers a 512-thread CTA allows
// (a few bytes spill at E = 8 and 16; one token more in flight measured faster
// than no spill)
template <int E> struct RbCols {
  static constexpr int CPT = E == 1 ? 8 : E == 8 ? 4 : 2;
  static constexpr int U = E == 8 ? 5 : E == 16 ? 6 : 8;
};

// CPT bf16 values of one row: one 16-, 8- or 4-byte load
template <int CPT> struct RowVec;
template <> struct RowVec<8> {
  uint4 v;
  __device__ __forceinline__ void load(const bf16* p) { v = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ unsigned word(int i) const { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
  __device__ __forceinline__ void set(int i, unsigned w) {
    if (i == 0) v.x = w; else if (i == 1) v.y = w; else if (i == 2) v.z = w; else v.w = w;
  }
  __device__ __forceinline__ void store(bf16* p) const { *reinterpret_cast<uint4*>(p) = v; }
};
template <> struct RowVec<4> {
  uint2 v;
  __device__ __forceinline__ void load(const bf16* p) { v = __ldg(reinterpret_cast<const uint2*>(p)); }
  __device__ __forceinline__ unsigned word(int i) const { return i == 0 ? v.x : v.y; }
  __device__ __forceinline__ void set(int i, unsigned w) { if (i == 0) v.x = w; else v.y = w; }
  __device__ __forceinline__ void store(bf16* p) const { *reinterpret_cast<uint2*>(p) = v; }
};
template <> struct RowVec<2> {
  unsigned v;
  __device__ __forceinline__ void load(const bf16* p) { v = __ldg(reinterpret_cast<const unsigned*>(p)); }
  __device__ __forceinline__ unsigned word(int) const { return v; }
  __device__ __forceinline__ void set(int, unsigned w) { v = w; }
  __device__ __forceinline__ void store(bf16* p) const { *reinterpret_cast<unsigned*>(p) = v; }
};

// the two bf16 of a 32-bit word as (low, high) fp32
__device__ __forceinline__ float2 bf_pair(unsigned w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ unsigned pack_bf2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<unsigned*>(&h);
}

// dl[e] for token t: softmax over the E logits, then the gradient of the K
// chosen gates (renormalised to sum 1 when renorm):
//   plain:  dl_j = p_j (G_j - sum_k d_gate_k p_{idx_k})
//   renorm: q_j = p_j / sum_k p_{idx_k} on the chosen experts, 0 elsewhere;
//           dl_j = q_j (G_j - sum_k d_gate_k q_{idx_k})
// G_j = d_gate_k where idx_k = j, else 0.  Linear score (E = 1): dl = d_gate.
template <int E>
__device__ __forceinline__ void token_dl(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                                         const float* __restrict__ d_gate, int K, int renorm, int linear,
                                         long long t, float (&dl)[E]) {
  if (linear) {
#pragma unroll
    for (int j = 0; j < E; ++j) dl[j] = j == 0 ? __ldg(d_gate + t) : 0.f;
    return;
  }
  float v[E];
  if constexpr (E % 4 == 0) {
#pragma unroll
    for (int q = 0; q < E / 4; ++q) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(logits + t * E) + q);
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) v[j] = __ldg(logits + t * E + j);
  }
  float m = v[0];
#pragma unroll
  for (int j = 1; j < E; ++j) m = fmaxf(m, v[j]);
  float s = 0.f, p[E], G[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    p[j] = expf(v[j] - m);
    s += p[j];
    G[j] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < E; ++j) p[j] = p[j] / s;
  float inner = 0.f, csum = 0.f;
  unsigned chosen = 0;
  for (int k = 0; k < K; ++k) {
    const int e = __ldg(idx + t * K + k);
    const float dg = __ldg(d_gate + t * K + k);
#pragma unroll
    for (int j = 0; j < E; ++j)
      if (j == e) { G[j] = dg; inner += dg * p[j]; csum += p[j]; chosen |= 1u << j; }
  }
  if (renorm) {
    inner = inner / csum;
#pragma unroll
    for (int j = 0; j < E; ++j) p[j] = ((chosen >> j) & 1u) ? p[j] / csum : 0.f;
  }
#pragma unroll
  for (int j = 0; j < E; ++j) dl[j] = p[j] * (G[j] - inner);
}

// grid = G token ranges x NS slices of H (blockIdx.x = range * NS + slice).
// A slice holds HS = H / NS columns; TPR = HS / CPT threads cover one row and
// RPI = floor(512 / TPR) rows are processed side by side.  part (nullable)
// receives [G * RPI][H][E] partial sums of dW_r; dx (nullable) is accumulated
// into, or written when dx_write; d_logits (nullable) is written by slice 0.
template <int E>
__global__ void __launch_bounds__(RB_THREADS, 1)
router_bwd_stream_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                         const float* __restrict__ d_gate, int K, int renorm, int linear,
                         const bf16* __restrict__ x, const bf16* __restrict__ w, int T, int H, int NS, int G,
                         float* __restrict__ d_logits, float* __restrict__ part, bf16* __restrict__ dx,
                         int dx_write) {
  constexpr int CPT = RbCols<E>::CPT, U = RbCols<E>::U, CP = CPT / 2;
  // dl of the chunk, each value twice: (dl, dl) is the broadcast operand of
  // the paired FMAs
  __shared__ __align__(16) float2 sdl[RB_CHUNK * E];
  const int tid = threadIdx.x;
  const int slice = blockIdx.x % NS, range = blockIdx.x / NS;
  const int HS = H / NS, TPR = HS / CPT, RPI = RB_THREADS / TPR;
  const int r = tid / TPR;  // threads with r >= RPI (when TPR does not divide 512) only compute dl
  const bool active = r < RPI;
  const int c0 = slice * HS + (tid % TPR) * CPT;
  const long long t0 = (long long)T * range / G, t1 = (long long)T * (range + 1) / G;

  // this thread's columns of W_r in column pairs: wp[c2][e] = (W[c0+2c2][e], W[c0+2c2+1][e])
  float2 wp[CP][E];
  if constexpr (E == 1) {
    RowVec<CPT> q;
    q.load(w + c0);
#pragma unroll
    for (int c2 = 0; c2 < CP; ++c2) wp[c2][0] = bf_pair(q.word(c2));
  } else {
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
      for (int q = 0; q < E / 8; ++q) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(w + (long long)(c0 + c) * E) + q);
        const unsigned ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = bf_pair(ws[i]);
          if (c & 1) { wp[c / 2][8 * q + 2 * i].y = f.x; wp[c / 2][8 * q + 2 * i + 1].y = f.y; }
          else { wp[c / 2][8 * q + 2 * i].x = f.x; wp[c / 2][8 * q + 2 * i + 1].x = f.y; }
        }
      }
  }
  // dW_r sums in column pairs: acc[c2][e] = (sum for column c0+2c2, for c0+2c2+1)
  float2 acc[CP][E];
#pragma unroll
  for (int c2 = 0; c2 < CP; ++c2)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[c2][e] = make_float2(0.f, 0.f);

  const bool do_dx = active && dx != nullptr, do_dw = active && part != nullptr;
  const bool load_dx = do_dx && !dx_write;
  for (long long cs = t0; cs < t1; cs += RB_CHUNK) {
    const int n = (int)(t1 - cs < RB_CHUNK ? t1 - cs : RB_CHUNK);
    if (tid < n) {
      float dl[E];
      token_dl<E>(logits, idx, d_gate, K, renorm, linear, cs + tid, dl);
#pragma unroll
      for (int e = 0; e < E; ++e) sdl[tid * E + e] = make_float2(dl[e], dl[e]);
      if (d_logits && slice == 0) {
        if constexpr (E % 4 == 0) {
#pragma unroll
          for (int q = 0; q < E / 4; ++q)
            reinterpret_cast<float4*>(d_logits + (cs + tid) * E)[q] =
                make_float4(dl[4 * q], dl[4 * q + 1], dl[4 * q + 2], dl[4 * q + 3]);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) d_logits[(cs + tid) * E + e] = dl[e];
        }
      }
    }
    __syncthreads();
    if (do_dx || do_dw) {
      for (int i0 = r; i0 < n; i0 += RPI * U) {
        RowVec<CPT> xv[U], dv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          int i = i0 + u * RPI;
          i = i < n ? i : n - 1;  // clamped: a valid row, its result unused
          const long long off = (cs + i) * H + c0;
          if (do_dw) xv[u].load(x + off);
          if (load_dx) dv[u].load(dx + off);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + u * RPI;
          if (i >= n) break;
          // x and dx of the token in column pairs; the dx sums start from the
          // old dx and run in two halves (even / odd experts) to halve the
          // dependent chain
          float2 xp[CP], v[CP], v2[CP];
#pragma unroll
          for (int c2 = 0; c2 < CP; ++c2) {
            xp[c2] = do_dw ? bf_pair(xv[u].word(c2)) : make_float2(0.f, 0.f);
            v[c2] = load_dx ? bf_pair(dv[u].word(c2)) : make_float2(0.f, 0.f);
            v2[c2] = make_float2(0.f, 0.f);
          }
          // dl pairs two experts at a time (one 16-byte shared load), used at
          // once; both products always (one that is not wanted is not stored)
#pragma unroll
          for (int e0 = 0; e0 < E; e0 += 2) {
            float2 d2[2];
            if constexpr (E % 2 == 0) {
              const float4 f = reinterpret_cast<const float4*>(sdl + i * E + e0)[0];
              d2[0] = make_float2(f.x, f.y);
              d2[1] = make_float2(f.z, f.w);
            } else {
              d2[0] = sdl[i * E + e0];
              d2[1] = d2[0];
            }
#pragma unroll
            for (int c2 = 0; c2 < CP; ++c2) {
              acc[c2][e0] = __ffma2_rn(xp[c2], d2[0], acc[c2][e0]);
              v[c2] = __ffma2_rn(d2[0], wp[c2][e0], v[c2]);
              if (e0 + 1 < E) {
                acc[c2][e0 + 1] = __ffma2_rn(xp[c2], d2[1], acc[c2][e0 + 1]);
                v2[c2] = __ffma2_rn(d2[1], wp[c2][e0 + 1], v2[c2]);
              }
            }
          }
          if (do_dx) {
            RowVec<CPT> o;
#pragma unroll
            for (int c2 = 0; c2 < CP; ++c2) o.set(c2, pack_bf2(v[c2].x + v2[c2].x, v[c2].y + v2[c2].y));
            o.store(dx + (cs + i) * H + c0);
          }
        }
      }
    }
    __syncthreads();  // sdl is rewritten by the next chunk
  }
  if (do_dw) {
    // CPT * E consecutive floats of [H][E]: 16-byte stores
    float* dst = part + ((long long)(range * RPI + r) * H + c0) * E;
    float flat[CPT * E];
#pragma unroll
    for (int c2 = 0; c2 < CP; ++c2)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        flat[(2 * c2) * E + e] = acc[c2][e].x;
        flat[(2 * c2 + 1) * E + e] = acc[c2][e].y;
      }
#pragma unroll
    for (int j = 0; j < CPT * E; j += 4)
      *reinterpret_cast<float4*>(dst + j) = make_float4(flat[j], flat[j + 1], flat[j + 2], flat[j + 3]);
  }
}

int rb_cpt(int E) { return E == 1 ? 8 : E == 8 ? 4 : 2; }

struct RbGeom {
  int ns, hs, rpi, g;
};

// NS = the fewest slices of at most 512 * CPT columns
RbGeom rb_geom(int T, int H, int E) {
  const int cpt = rb_cpt(E);
  const int cw = RB_THREADS * cpt;
  RbGeom q;
  q.ns = (H + cw - 1) / cw;
  q.hs = H / q.ns;
  q.rpi = RB_THREADS / (q.hs / cpt);
  long long g = sm_count() / q.ns;
  if (g < 1) g = 1;
  if (g > T) g = T > 0 ? T : 1;
  q.g = (int)g;
  return q;
}

}  // namespace

// The streaming router backward serves bf16 layers with the softmax/top-K gate
// over 8 or 16 experts, or the linear MoD score (E = 1), whose H splits into
// NS equal slices of whole warps (each slice a multiple of 32 * CPT columns).
bool router_bwd_stream_applies(int mode, int dtype, int H, int E, int K) {
  if (dtype != MOE_BF16) return false;
  const bool topk = mode == MOE_ROUTE_SOFTMAX_TOPK && (E == 8 || E == 16) && K >= 1 && K <= E;
  const bool lin = mode == MOE_ROUTE_MOD_LINEAR && E == 1;
  if (!topk && !lin) return false;
  const int cpt = rb_cpt(E);
  const int cw = RB_THREADS * cpt;
  if (H <= 0) return false;
  const int ns = (H + cw - 1) / cw;
  return H % ns == 0 && (H / ns) % (32 * cpt) == 0;
}

// partial sums of dW_r the kernel leaves in the workspace (one per token range
// and row lane)
int router_bwd_stream_splits(int T, int H, int E) {
  if (router_bwd_mma_applies(MOE_ROUTE_SOFTMAX_TOPK, MOE_BF16, H, E, 1)) return router_bwd_mma_splits(T, H);
  const RbGeom q = rb_geom(T, H, E);
  return q.g * q.rpi;
}

int launch_router_bwd_stream(int mode, const float* d_gate, const float* logits, const int32_t* idx, const void* x,
                             const void* w, int T, int H, int E, int K, bool renorm, float* d_logits, float* part,
                             void* dx, bool dx_write, cudaStream_t s) {
  // 8 or 16 experts with whole 512-column slices: both products on the warp MMA
  if (router_bwd_mma_applies(mode, MOE_BF16, H, E, K))
    return launch_router_bwd_mma(d_gate, logits, idx, x, w, T, H, E, K, renorm, d_logits, part, dx, dx_write, s);
  const RbGeom q = rb_geom(T, H, E);
  const int grid = q.g * q.ns;
  const int lin = mode == MOE_ROUTE_MOD_LINEAR ? 1 : 0;
  const int rn = renorm ? 1 : 0;
  const bf16* xb = static_cast<const bf16*>(x);
  const bf16* wb = static_cast<const bf16*>(w);
  bf16* dxb = static_cast<bf16*>(dx);
  const int dxw = dx_write ? 1 : 0;
  if (E == 1)
    router_bwd_stream_kernel<1><<<grid, RB_THREADS, 0, s>>>(logits, idx, d_gate, K, rn, lin, xb, wb, T, H, q.ns, q.g,
                                                            d_logits, part, dxb, dxw);
  else if (E == 8)
    router_bwd_stream_kernel<8><<<grid, RB_THREADS, 0, s>>>(logits, idx, d_gate, K, rn, lin, xb, wb, T, H, q.ns, q.g,
                                                            d_logits, part, dxb, dxw);
  else
    router_bwd_stream_kernel<16><<<grid, RB_THREADS, 0, s>>>(logits, idx, d_gate, K, rn, lin, xb, wb, T, H, q.ns,
                                                             q.g, d_logits, part, dxb, dxw);
  return launch_status();
}

}  // namespace moe
