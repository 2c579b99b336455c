// Router: logits GEMM, fused softmax + top-K gate, and the router backward.
//
// Softmax/top-K follows the routing/gating kernel of the MoE/MoD framework page
// ("What's in the box": softmax over experts and top-k in one launch, warp-level
// primitives for top-k).  One warp per token row: the row is read with 128-bit
// loads, max / sum / arg-max are warp-shuffle reductions, and the K winners are
// taken by K rounds of a (value desc, expert asc) arg-max, which gives the
// lowest-index tie-break exactly.  Selection is on the fp32 logits themselves.
#include <climits>
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

// With S > 1 the router GEMM left S partial sums over slices of H in `part`
// ([S][T][E]); they are added in slice order, the bias added last, and the
// logits written before the softmax (a fixed order: the same bits every run).
template <int VPL>
__global__ void __launch_bounds__(32 * ROWS_PER_CTA)
softmax_topk_kernel(float* __restrict__ logits, const float* __restrict__ part, int S,
                    const float* __restrict__ bias, const float* __restrict__ sel_bias, int renorm, int T, int E,
                    int K, int32_t* __restrict__ idx, float* __restrict__ gate) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * ROWS_PER_CTA;
  for (long long t = (long long)blockIdx.x * ROWS_PER_CTA + (threadIdx.x >> 5); t < T; t += nwarps) {
    float v[VPL];
    if (S > 1) {
      load_row<VPL>(part + t * E, E, lane, v);
      for (int s = 1; s < S; ++s) {
        float w[VPL];
        load_row<VPL>(part + (long long)s * T * E + t * E, E, lane, w);
#pragma unroll
        for (int j = 0; j < VPL; ++j) v[j] += w[j];
      }
#pragma unroll
      for (int q = 0; q < VPL / 4; ++q) {
        const int e4 = (q * 32 + lane) * 4;
        if (e4 < E) {
          if (bias) {
            const float4 bb = __ldg(reinterpret_cast<const float4*>(bias + e4));
            v[4 * q] += bb.x; v[4 * q + 1] += bb.y; v[4 * q + 2] += bb.z; v[4 * q + 3] += bb.w;
          }
          *reinterpret_cast<float4*>(logits + t * E + e4) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2],
                                                                        v[4 * q + 3]);
        }
      }
    } else {
      load_row<VPL>(logits + t * E, E, lane, v);
    }
    // selection values: the logits, or the logits plus a selection-only bias
    float sv[VPL];
    if (sel_bias) {
      load_row<VPL>(sel_bias, E, lane, sv);
#pragma unroll
      for (int j = 0; j < VPL; ++j) sv[j] += v[j];
    } else {
#pragma unroll
      for (int j = 0; j < VPL; ++j) sv[j] = v[j];
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < VPL; ++j) m = fmaxf(m, v[j]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) s += (slot_expert(j, lane) < E) ? expf(v[j] - m) : 0.f;
    s = warp_sum(s);
    // Top-K by selection value, descending, lowest expert first on ties.
    // A lane's slots hold increasing experts, so scanning them in slot order
    // with a strict comparison already breaks ties by expert.  Slots past E
    // and taken slots hold NaN, which no comparison accepts.  Each lane caches
    // its best two untaken slots (an empty cache still accepts -inf); a round
    // takes the warp's best cached candidate with two warp reductions (the
    // largest order-preserving integer key, then the smallest expert among
    // the lanes holding it); the winning lane promotes its second and scans
    // again only when its cache ran empty.
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (slot_expert(j, lane) >= E) sv[j] = __int_as_float(0x7fffffff);
    float c1v, c2v, c1r, c2r;
    int c1j, c2j;
    auto rescan = [&]() {
      c1v = c2v = -INFINITY;
      c1j = c2j = -1;
      c1r = c2r = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const float x = sv[j];
        if (x > c1v || (c1j < 0 && x == x)) {
          c2v = c1v; c2j = c1j; c2r = c1r;
          c1v = x; c1j = j; c1r = v[j];
        } else if (x > c2v || (c2j < 0 && x == x)) {
          c2v = x; c2j = j; c2r = v[j];
        }
      }
    };
    rescan();
    float chosen_sum = 0.f;
    for (int k = 0; k < K; ++k) {
      // order-preserving integer key of the cached value (finite or +-inf);
      // a lane with nothing left offers the smallest key
      int key = __float_as_int(c1v);
      key = key >= 0 ? key : key ^ 0x7fffffff;
      if (c1v == 0.f) key = 0;  // -0 and +0 are equal values
      if (c1j < 0) key = INT_MIN;
      const int kmax = __reduce_max_sync(0xffffffffu, key);
      const int my_e = (c1j >= 0 && key == kmax) ? slot_expert(c1j, lane) : 0x7fffffff;
      const int be = __reduce_min_sync(0xffffffffu, (unsigned)my_e);
      const bool mine = my_e == be && c1j >= 0;
      // the winner's own logit (not its selection value) gives its probability
      const int owner = (be >> 2) & 31;
      const float vw = __shfl_sync(0xffffffffu, mine ? c1r : 0.f, owner);
      if (mine) {
#pragma unroll
        for (int j = 0; j < VPL; ++j)
          if (j == c1j) sv[j] = __int_as_float(0x7fffffff);
        c1v = c2v; c1j = c2j; c1r = c2r;
        c2v = -INFINITY; c2j = -1;
        if (c1j < 0) rescan();
      }
      const float pk = expf(vw - m) / s;
      chosen_sum += pk;
      if (lane == 0) {
        idx[t * K + k] = be;
        gate[t * K + k] = pk;
      }
    }
    // Mixtral-style renormalisation: the K gates rescaled to sum to 1
    if (renorm && lane == 0)
      for (int k = 0; k < K; ++k) gate[t * K + k] = gate[t * K + k] / chosen_sum;
  }
}

// d_logits[t,j] = p_j (G_j - sum_k d_gate[t,k] p[idx[t,k]])
// Exact split of an fp32 value into three bf16 parts, v = hi + mid + lo: each
// subtraction is exact in fp32 and each rounding keeps the next 8+ significant
// bits, so three parts hold the full 24-bit significand.
__device__ __forceinline__ void split3(float v, bf16& hi, bf16& mid, bf16& lo) {
  hi = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(hi);
  mid = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(mid);
  lo = __float2bfloat16_rn(r2);
}

template <int VPL>
__global__ void __launch_bounds__(32 * ROWS_PER_CTA)
softmax_topk_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                        const float* __restrict__ d_gate, int renorm, int T, int E, int K,
                        float* __restrict__ d_logits, bf16* __restrict__ dl3) {
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
    float inner = 0.f, csum = 0.f;
    unsigned chosen = 0;
    // the K (expert, d_gate) pairs of the row: lane k loads pair k (K <= 32), all
    // loads in flight at once, then each is broadcast
    const int my_e = lane < K ? __ldg(idx + t * K + lane) : 0;
    const float my_dg = lane < K ? __ldg(d_gate + t * K + lane) : 0.f;
    for (int k = 0; k < K; ++k) {
      const int e = __shfl_sync(0xffffffffu, my_e, k);
      const float dg = __shfl_sync(0xffffffffu, my_dg, k);
      if (((e >> 2) & 31) == lane) {
        int slot = (e >> 7) * 4 + (e & 3);
#pragma unroll
        for (int j = 0; j < VPL; ++j)
          if (j == slot) { G[j] = dg; inner += dg * p[j]; csum += p[j]; chosen |= 1u << j; }
      }
    }
    inner = warp_sum(inner);
    if (renorm) {
      // renormalised gates q = p / (sum of the chosen p): only the chosen
      // logits get a gradient, q_j (G_j - sum_k d_gate_k q_k)
      csum = warp_sum(csum);
      inner = inner / csum;
#pragma unroll
      for (int j = 0; j < VPL; ++j) p[j] = ((chosen >> j) & 1u) ? p[j] / csum : 0.f;
    }
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
        if (dl3) {
          const float vv[4] = {r.x, r.y, r.z, r.w};
          __align__(8) bf16 part[3][4];
#pragma unroll
          for (int j = 0; j < 4; ++j) split3(vv[j], part[0][j], part[1][j], part[2][j]);
          const long long plane = (long long)T * E;
#pragma unroll
          for (int s = 0; s < 3; ++s)
            *reinterpret_cast<uint2*>(dl3 + s * plane + t * E + e4) = *reinterpret_cast<const uint2*>(part[s]);
        }
      }
    }
  }
}

__global__ void copy_f32_kernel(const float* __restrict__ a, float* __restrict__ b, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    b[i] = a[i];
}

// dw[i] = sum_s part[s][i] in a fixed order (the same result every run).  A
// block covers 32 consecutive outputs with 8 warps: warp q adds splits q, q+8,
// q+16, ... in increasing order for output base + lane, so every load
// instruction reads 128 contiguous bytes and a thread's loads are independent
// of one another; the 8 warp sums then meet in shared memory, added in warp
// order.
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float* __restrict__ part, int S, long long n,
                                                            float* __restrict__ out) {
  __shared__ float red[8][33];
  const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
  for (long long base = blockIdx.x * 32LL; base < n; base += gridDim.x * 32LL) {
    const long long i = base + lane;
    float acc = 0.f;
    if (i < n) {
#pragma unroll 8
      for (int s = q; s < S; s += 8) acc += __ldg(part + (long long)s * n + i);
    }
    red[q][lane] = acc;
    __syncthreads();
    if (q == 0 && i < n) {
      float t = red[0][lane];
#pragma unroll
      for (int j = 1; j < 8; ++j) t += red[j][lane];
      out[i] = t;
    }
    __syncthreads();
  }
}

int rows_grid(long long T) {
  long long ctas = (T + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
  long long cap = (long long)sm_count() * 16;
  return (int)(ctas < cap ? (ctas > 0 ? ctas : 1) : cap);
}

// ---------------------------------------------------------------------------
// Router weight gradient  dw[h,e] = sum_t x[t,h] dl[t,e].
// Split over tokens; a thread owns CPT consecutive columns h and EB experts
// (CPT*EB = 64 fp32 accumulators), reads its x columns with one 16/32-byte load
// per token and the token's dl values from a shared-memory tile (broadcast).
// Each split writes its partial [H, E]; a second kernel adds the splits in
// order, so the result does not depend on scheduling.
constexpr int DW_THREADS = 256;
constexpr int DW_TB = 32;  // tokens per shared-memory dl tile

struct DwPlan {
  int cpt, eb, col_blocks, exp_blocks, splits, rows_per_split;
};

DwPlan dw_plan(int T, int H, int E) {
  DwPlan p;
  p.eb = E <= 8 ? 8 : E <= 16 ? 16 : E <= 32 ? 32 : 64;
  p.cpt = 64 / p.eb;
  p.col_blocks = (H + DW_THREADS * p.cpt - 1) / (DW_THREADS * p.cpt);
  p.exp_blocks = (E + p.eb - 1) / p.eb;
  // about two CTAs per SM (the workspace size then depends on the current
  // device's SM count, which moe_workspace_bytes reads the same way)
  const long long target = 2LL * sm_count();
  long long want = (target + p.col_blocks * p.exp_blocks - 1) / (p.col_blocks * p.exp_blocks);
  long long by_t = (T + 7) / 8;
  long long s = want < by_t ? want : by_t;
  if (s > 256) s = 256;
  if (s < 1) s = 1;
  p.splits = (int)s;
  p.rows_per_split = (T + p.splits - 1) / p.splits;
  return p;
}

template <typename T> __device__ __forceinline__ void load_cols(const T* p, int n, float* v);
template <> __device__ __forceinline__ void load_cols<bf16>(const bf16* p, int n, float* v) {
  if (n == 8) {
    Vec16<bf16>::load(p, v);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) if (j < n) v[j] = __bfloat162float(p[j]);
  }
}
template <> __device__ __forceinline__ void load_cols<float>(const float* p, int n, float* v) {
  if (n == 8) {
    Vec16<float>::load(p, v);
    Vec16<float>::load(p + 4, v + 4);
  } else if (n == 4) {
    Vec16<float>::load(p, v);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) if (j < n) v[j] = p[j];
  }
}

// E <= 8: a thread owns 8 columns x 8 experts and streams its own x columns
// through a private slot of a DW8_NS-stage shared-memory ring with cp.async
// (16-byte copies, zero-filled past the tensor), so DW8_NS * DW8_RB tokens per
// thread are in flight without holding registers.  The slot layout
// [stage][row][chunk][thread] keeps every access conflict-free, and since no
// thread reads another's slot no block barrier is needed.
constexpr int DW8_NS = 3;
template <typename T> struct Dw8 {
  static constexpr int CH = sizeof(T) == 2 ? 1 : 2;  // 16-byte chunks per row (8 columns)
  static constexpr int RB = sizeof(T) == 2 ? 8 : 4;  // rows per stage
  static constexpr int STAGE = RB * CH * DW_THREADS;  // uint4 per stage
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const int src_size = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(gmem), "r"(src_size) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(DW_THREADS, 2)
router_dw8_kernel(const T* __restrict__ x, const float* __restrict__ dl, int Tn, int H, int E,
                  int rows_per_split, float* __restrict__ part) {
  using P = Dw8<T>;
  extern __shared__ uint4 ring[];  // [DW8_NS][RB][CH][DW_THREADS]
  const int tid = threadIdx.x;
  const int h0 = (blockIdx.x * DW_THREADS + tid) * 8;
  const bool col_ok = h0 < H;
  const int split = blockIdx.z;
  const int t_begin = split * rows_per_split;
  const int t_end = min(Tn, t_begin + rows_per_split);
  const int nb = t_end > t_begin ? (t_end - t_begin + P::RB - 1) / P::RB : 0;
  auto issue = [&](int blk) {
    const int stage = blk % DW8_NS;
#pragma unroll
    for (int r = 0; r < P::RB; ++r) {
      const int t = t_begin + blk * P::RB + r;
      const bool ok = col_ok && blk < nb && t < t_end;
      const T* src = x + (ok ? (long long)t * H + h0 : 0);
#pragma unroll
      for (int c = 0; c < P::CH; ++c) {
        // chunk c holds columns h0 + c*V .. h0 + (c+1)*V - 1 (V = 16 / sizeof(T))
        const bool okc = ok && h0 + (c + 1) * (16 / (int)sizeof(T)) <= H;
        cp_async16(&ring[((stage * P::RB + r) * P::CH + c) * DW_THREADS + tid],
                   reinterpret_cast<const uint4*>(src) + (okc ? c : 0), okc);
      }
    }
  };
  float acc[8][8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
#pragma unroll
  for (int s = 0; s < DW8_NS - 1; ++s) {
    issue(s);
    cp_async_commit();
  }
  for (int b = 0; b < nb; ++b) {
    issue(b + DW8_NS - 1);
    cp_async_commit();
    cp_async_wait<DW8_NS - 1>();
    const int stage = b % DW8_NS;
#pragma unroll
    for (int r = 0; r < P::RB; ++r) {
      const int t = t_begin + b * P::RB + r;
      if (t >= t_end) break;
      float xv[8];
      if (sizeof(T) == 2) {
        Vec16<bf16>::load_raw_unpack(ring[((stage * P::RB + r) * P::CH) * DW_THREADS + tid], xv);
      } else {
#pragma unroll
        for (int c = 0; c < P::CH; ++c) {
          const uint4 q = ring[((stage * P::RB + r) * P::CH + c) * DW_THREADS + tid];
          xv[4 * c] = __uint_as_float(q.x); xv[4 * c + 1] = __uint_as_float(q.y);
          xv[4 * c + 2] = __uint_as_float(q.z); xv[4 * c + 3] = __uint_as_float(q.w);
        }
      }
      float dv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) dv[e] = e < E ? __ldg(dl + (long long)t * E + e) : 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(xv[j], dv[e], acc[j][e]);
    }
  }
  cp_async_wait<0>();
  if (!col_ok) return;
  float* out = part + (long long)split * H * E + (long long)h0 * E;
  const int ncol = min(8, H - h0);
  if (E == 8 && ncol == 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      reinterpret_cast<float4*>(out)[2 * j] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
      reinterpret_cast<float4*>(out)[2 * j + 1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (j < ncol && e < E) out[j * E + e] = acc[j][e];
  }
}

template <typename T, int CPT, int EB>
__global__ void __launch_bounds__(DW_THREADS)
router_dw_partial_kernel(const T* __restrict__ x, const float* __restrict__ dl, int Tn, int H, int E,
                         int rows_per_split, float* __restrict__ part) {
  __shared__ float dls[DW_TB][EB];
  const int h0 = (blockIdx.x * DW_THREADS + threadIdx.x) * CPT;
  const int e0 = blockIdx.y * EB;
  const int split = blockIdx.z;
  const int t_begin = split * rows_per_split;
  const int t_end = min(Tn, t_begin + rows_per_split);
  float acc[CPT][EB];
#pragma unroll
  for (int j = 0; j < CPT; ++j)
#pragma unroll
    for (int e = 0; e < EB; ++e) acc[j][e] = 0.f;
  const bool col_ok = h0 < H;
  const int ncol = col_ok ? min(CPT, H - h0) : 0;
  for (int t0 = t_begin; t0 < t_end; t0 += DW_TB) {
    __syncthreads();
    for (int i = threadIdx.x; i < DW_TB * EB; i += DW_THREADS) {
      const int tt = i / EB, e = i % EB;
      const int t = t0 + tt, ge = e0 + e;
      dls[tt][e] = (t < t_end && ge < E) ? __ldg(dl + (long long)t * E + ge) : 0.f;
    }
    __syncthreads();
    const int n_rows = min(DW_TB, t_end - t0);
    if (col_ok) {
      int tt = 0;
      // four tokens' x columns are loaded before their FMAs (loads in flight)
      for (; tt + 4 <= n_rows; tt += 4) {
        float xv[4][8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int j = 0; j < 8; ++j) xv[q][j] = 0.f;
          load_cols<T>(x + (long long)(t0 + tt + q) * H + h0, ncol, xv[q]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int j = 0; j < CPT; ++j)
#pragma unroll
            for (int e = 0; e < EB; ++e) acc[j][e] = fmaf(xv[q][j], dls[tt + q][e], acc[j][e]);
      }
      for (; tt < n_rows; ++tt) {
        float xv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        load_cols<T>(x + (long long)(t0 + tt) * H + h0, ncol, xv);
#pragma unroll
        for (int j = 0; j < CPT; ++j)
#pragma unroll
          for (int e = 0; e < EB; ++e) acc[j][e] = fmaf(xv[j], dls[tt][e], acc[j][e]);
      }
    }
  }
  if (!col_ok) return;
  float* out = part + (long long)split * H * E;
#pragma unroll
  for (int j = 0; j < CPT; ++j)
#pragma unroll
    for (int e = 0; e < EB; ++e)
      if (j < ncol && e0 + e < E) out[(long long)(h0 + j) * E + e0 + e] = acc[j][e];
}

// ---------------------------------------------------------------------------
// Router input gradient  dx[t,h] (+)= sum_e dl[t,e] w[h,e].
// A CTA covers DX_TR tokens x DX_HB columns; w[h, e-chunk] is staged in shared
// memory transposed ([e][h], so a warp's 8-column reads are contiguous) together
// with the tokens' dl chunk; a thread owns 8 consecutive columns of one token.
constexpr int DX_TR = 32, DX_HB = 256, DX_EC = 32, DX_THREADS = 256;
// thread (r, c): r = tid / 32 (+ 8 * i), c = tid % 32 -> columns 8c .. 8c+7

constexpr int DX_RT = 4;  // row tiles per CTA

// four consecutive values of the storage type (8 bytes of bf16, 16 of fp32);
// an invalid load yields zeros
template <typename T> __device__ __forceinline__ void load4(const T* p, bool ok, float* v);
template <> __device__ __forceinline__ void load4<bf16>(const bf16* p, bool ok, float* v) {
  uint2 q = ok ? __ldg(reinterpret_cast<const uint2*>(p)) : make_uint2(0, 0);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
  float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
template <> __device__ __forceinline__ void load4<float>(const float* p, bool ok, float* v) {
  float4 q = ok ? __ldg(reinterpret_cast<const float4*>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
template <typename T> __device__ __forceinline__ void store4(T* p, const float* v);
template <> __device__ __forceinline__ void store4<bf16>(bf16* p, const float* v) {
  uint2 q;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
  h[0] = __floats2bfloat162_rn(v[0], v[1]);
  h[1] = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = q;
}
template <> __device__ __forceinline__ void store4<float>(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

template <typename T>
__global__ void __launch_bounds__(DX_THREADS)
router_dx_kernel(const float* __restrict__ dl, const T* __restrict__ w, int Tn, int H, int E, bool write,
                 T* __restrict__ dx) {
  __shared__ __align__(16) float ws[DX_EC][DX_HB];
  __shared__ float ds[DX_TR][DX_EC];
  const int hb = blockIdx.x * DX_HB;
  const int c = threadIdx.x & 31;
  const int r0 = threadIdx.x >> 5;  // 0..7; rows r0, r0+8, r0+16, r0+24 of a tile
  // a thread owns columns hb+4c..+3 and hb+128+4c..+3: consecutive lanes read
  // consecutive 16-byte words of ws (no bank conflicts) and a warp's stores of
  // each 4-column group are contiguous; H % 4 == 0 makes each group all-in or all-out
  const int ha = hb + 4 * c, hbb = hb + 128 + 4 * c;
  const bool oka = ha < H, okb = hbb < H;
  const bool one_chunk = E <= DX_EC;
  auto stage_w = [&](int e0) {
    const int ne = min(DX_EC, E - e0);
    for (int i = threadIdx.x; i < ne * DX_HB; i += DX_THREADS) {
      const int hh = i % DX_HB, e = i / DX_HB;  // consecutive threads write consecutive h
      const int gh = hb + hh;
      ws[e][hh] = gh < H ? to_f32(w[(long long)gh * E + e0 + e]) : 0.f;
    }
  };
  if (one_chunk) stage_w(0);
  for (int rt = 0; rt < DX_RT; ++rt) {
    const int tb = (blockIdx.y * DX_RT + rt) * DX_TR;
    if (tb >= Tn) break;
    float acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int e0 = 0; e0 < E; e0 += DX_EC) {
      const int ne = min(DX_EC, E - e0);
      __syncthreads();
      if (!one_chunk) stage_w(e0);
      for (int i = threadIdx.x; i < DX_TR * ne; i += DX_THREADS) {
        const int r = i / ne, e = i % ne;
        const int t = tb + r;
        ds[r][e] = t < Tn ? __ldg(dl + (long long)t * E + e0 + e) : 0.f;
      }
      __syncthreads();
      for (int e = 0; e < ne; ++e) {
        float wv[8];
        const float4 a = *reinterpret_cast<const float4*>(&ws[e][4 * c]);
        const float4 b = *reinterpret_cast<const float4*>(&ws[e][128 + 4 * c]);
        wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w; wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float d = ds[r0 + 8 * i][e];
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(d, wv[j], acc[i][j]);
        }
      }
    }
    float old[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // all read-modify-write loads first
      const int t = tb + r0 + 8 * i;
      const bool rok = t < Tn && !write;
      const T* p = dx + (long long)t * H;
      load4<T>(p + ha, rok && oka, old[i]);
      load4<T>(p + hbb, rok && okb, old[i] + 4);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = tb + r0 + 8 * i;
      if (t >= Tn) continue;
      T* p = dx + (long long)t * H;
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = old[i][j] + acc[i][j];
      if (oka) store4<T>(p + ha, v);
      if (okb) store4<T>(p + hbb, v + 4);
    }
  }
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

int launch_router_tc(const void* x, const void* w, const float* bias, const float* sel_bias, bool renorm, int T,
                     int H, int E, float* out, int S, int K, int32_t* idx, float* gate, cudaStream_t s);
int router_tc_splits(int T, int H, int E);

size_t route_ws_bytes(int T, int H, int E) {
  if (router_stream_applies(MOE_BF16, H, E)) return 0;
  const int S = router_tc_splits(T, H, E);
  return S > 1 ? align256((size_t)S * T * E * 4) : 0;
}

// Router forward.  bf16 with 8 or 16 experts: one streaming launch (logits,
// softmax and top-K); other bf16 shapes: tcgen05 GEMM, split over H into S
// partial sums when the token tiles alone would leave SMs idle (the partials,
// the bias and the softmax/top-k meet in one pass); fp32: FFMA GEMM with the
// bias in its epilogue.
int launch_route(const void* x, const void* w, const float* bias, int T, int H, int E, int K, int dtype, int flags,
                 float* logits, int32_t* idx, float* gate, void* ws, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const bool renorm = flags & MOE_ROUTE_RENORM;
  // a selection-only bias never reaches the GEMM: it is added to copies of the
  // logits where the experts are chosen
  const float* sel_bias = (flags & MOE_ROUTE_BIAS_SELECT) ? bias : nullptr;
  const float* gemm_bias = sel_bias ? nullptr : bias;
  if (router_stream_applies(dtype, H, E))
    return launch_router_stream(x, w, gemm_bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
  int S = 1;
  float* part = nullptr;
  int st;
  if (dtype == MOE_BF16) {
    S = router_tc_splits(T, H, E);
    part = S > 1 ? static_cast<float*>(ws) : nullptr;
    if (S == 1 && E <= 64) {  // the whole expert row is one tile: one launch
      return launch_router_tc(x, w, gemm_bias, sel_bias, renorm, T, H, E, logits, 1, K, idx, gate, s);
    }
    st = launch_router_tc(x, w, gemm_bias, nullptr, false, T, H, E, S > 1 ? part : logits, S, 0, nullptr, nullptr,
                          s);
  } else {
    SimtGemmArgs a{};
    a.A = x; a.a_sm = H; a.a_sk = 1;
    a.B = w; a.b_sg = 0; a.b_sk = E; a.b_sn = 1;
    a.C = logits; a.c_sm = E;
    a.bias = gemm_bias; a.cu = nullptr;
    a.M = T; a.N = E; a.K = H; a.groups = 1;
    a.epilogue = 2; a.swiglu = false;
    st = launch_simt_gemm(a, dtype, dtype, MOE_F32, s);
  }
  if (st != MOE_OK) return st;
  const int grid = rows_grid(T);
  const int vpl = (E + 127) / 128 * 4;
  const float* pb = S > 1 ? gemm_bias : nullptr;
  const int rn = renorm ? 1 : 0;
  if (vpl <= 4)
    softmax_topk_kernel<4><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, part, S, pb, sel_bias, rn, T, E, K, idx, gate);
  else if (vpl <= 8)
    softmax_topk_kernel<8><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, part, S, pb, sel_bias, rn, T, E, K, idx, gate);
  else if (vpl <= 12)
    softmax_topk_kernel<12><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, part, S, pb, sel_bias, rn, T, E, K, idx, gate);
  else if (vpl <= 16)
    softmax_topk_kernel<16><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, part, S, pb, sel_bias, rn, T, E, K, idx, gate);
  else
    softmax_topk_kernel<32><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, part, S, pb, sel_bias, rn, T, E, K, idx, gate);
  return launch_status();
}

int router_dw_tc_splits(int T, int H, int E);
int launch_router_dw_tc(const void* x, const void* dl3, int T, int H, int E, float* part, cudaStream_t s);
bool router_bwd_tc_applies(int H, int E);
int router_bwd_tc_splits(int T, int H, int E);
int launch_router_bwd_tc(const void* x, const void* dl3, const void* w, int T, int H, int E, float* part, bool write,
                         void* dx, cudaStream_t s);
int launch_router_dx_tc(const void* dl3, const void* w, int T, int H, int E, bool write, void* dx, cudaStream_t s);

// The tensor-core router backward serves bf16 layers whose W_r rows are
// 16-byte multiples (E % 8 == 0) and whose dx rows tile by 64 columns.
static bool route_bwd_on_tensor_cores(int mode, int dtype, int H, int E) {
  return mode == MOE_ROUTE_SOFTMAX_TOPK && dtype == MOE_BF16 && E % 8 == 0 && H % 64 == 0;
}

// workspace: [fp32 partials of dW][fp32 dl (when d_logits is not given)][bf16 dl in three parts]
struct BwdWs {
  size_t part, dl, dl3;
};
static BwdWs bwd_ws(int T, int H, int E) {
  const DwPlan pl = dw_plan(T, H, E);
  long long splits = pl.splits;
  const long long tcs = router_dw_tc_splits(T, H, E);
  if (tcs > splits) splits = tcs;
  const long long fused = router_bwd_tc_applies(H, E) ? router_bwd_tc_splits(T, H, E) : 0;
  if (fused > splits) splits = fused;
  const long long sts = (E == 1 || E == 8 || E == 16) ? router_bwd_stream_splits(T, H, E) : 0;
  if (sts > splits) splits = sts;
  return BwdWs{align256((size_t)splits * H * E * 4), align256((size_t)T * E * 4), align256((size_t)3 * T * E * 2)};
}

size_t route_bwd_ws_bytes(int T, int H, int E) {
  const BwdWs w = bwd_ws(T, H, E);
  return w.part + w.dl + w.dl3;
}

template <typename T>
int launch_dw(const T* x, const float* dl, int Tn, int H, int E, float* part, float* dw, cudaStream_t s) {
  const DwPlan pl = dw_plan(Tn, H, E);
  dim3 grid(pl.col_blocks, pl.exp_blocks, pl.splits);
  if (pl.eb == 8) {
    const int smem = DW8_NS * Dw8<T>::STAGE * (int)sizeof(uint4);
    if (cudaFuncSetAttribute(router_dw8_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    router_dw8_kernel<T><<<grid, DW_THREADS, smem, s>>>(x, dl, Tn, H, E, pl.rows_per_split, part);
  } else if (pl.eb == 16) router_dw_partial_kernel<T, 4, 16><<<grid, DW_THREADS, 0, s>>>(x, dl, Tn, H, E, pl.rows_per_split, part);
  else if (pl.eb == 32) router_dw_partial_kernel<T, 2, 32><<<grid, DW_THREADS, 0, s>>>(x, dl, Tn, H, E, pl.rows_per_split, part);
  else router_dw_partial_kernel<T, 1, 64><<<grid, DW_THREADS, 0, s>>>(x, dl, Tn, H, E, pl.rows_per_split, part);
  return launch_status();
}

int launch_reduce(const float* part, int S, int H, int E, float* dw, cudaStream_t s) {
  const long long n = (long long)H * E;
  const long long blocks = (n + 31) / 32;
  reduce_splits_kernel<<<(int)(blocks < 16384 ? blocks : 16384), 256, 0, s>>>(part, S, n, dw);
  return launch_status();
}

template <typename T>
int launch_dx(const float* dl, const T* w, int Tn, int H, int E, bool write, T* dx, cudaStream_t s) {
  dim3 grid((H + DX_HB - 1) / DX_HB, (Tn + DX_TR * DX_RT - 1) / (DX_TR * DX_RT));
  router_dx_kernel<T><<<grid, DX_THREADS, 0, s>>>(dl, w, Tn, H, E, write, dx);
  return launch_status();
}

int launch_route_bwd(int mode, const float* d_gate, const float* logits, const int32_t* idx,
                     const void* x, const void* w, int T, int H, int E, int K, int dtype,
                     float* d_logits, float* dw, void* dx, bool dx_write, bool renorm, void* ws, cudaStream_t s) {
  if (T == 0) {
    if (dw && cudaMemsetAsync(dw, 0, (size_t)H * E * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const BwdWs lay = bwd_ws(T, H, E);
  char* wsb = static_cast<char*>(ws);
  float* part = reinterpret_cast<float*>(wsb);
  if (router_bwd_stream_applies(mode, dtype, H, E, K)) {  // one streaming pass, then the dW_r reduction
    int st = launch_router_bwd_stream(mode, d_gate, logits, idx, x, w, T, H, E, K, renorm, d_logits,
                                      dw ? part : nullptr, dx, dx_write, s);
    if (st == MOE_OK && dw) st = launch_reduce(part, router_bwd_stream_splits(T, H, E), H, E, dw, s);
    return st;
  }
  // linear score (E = K = 1): the score gradient is the logit gradient, used as is
  float* dl = mode == MOE_ROUTE_MOD_LINEAR ? const_cast<float*>(d_gate)
              : d_logits ? d_logits : reinterpret_cast<float*>(wsb + lay.part);
  const bool tc = route_bwd_on_tensor_cores(mode, dtype, H, E);
  bf16* dl3 = tc ? reinterpret_cast<bf16*>(wsb + lay.part + lay.dl) : nullptr;

  if (mode == MOE_ROUTE_SOFTMAX_TOPK) {
    int grid = rows_grid(T);
    int vpl = (E + 127) / 128 * 4;
    const int rn = renorm ? 1 : 0;
    if (vpl <= 4)
      softmax_topk_bwd_kernel<4><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, idx, d_gate, rn, T, E, K, dl, dl3);
    else if (vpl <= 8)
      softmax_topk_bwd_kernel<8><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, idx, d_gate, rn, T, E, K, dl, dl3);
    else if (vpl <= 16)
      softmax_topk_bwd_kernel<16><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, idx, d_gate, rn, T, E, K, dl, dl3);
    else
      softmax_topk_bwd_kernel<32><<<grid, 32 * ROWS_PER_CTA, 0, s>>>(logits, idx, d_gate, rn, T, E, K, dl, dl3);
  } else if (d_logits) {
    // the logit gradient output of the linear score is d_score itself
    copy_f32_kernel<<<rows_grid(T), 256, 0, s>>>(d_gate, d_logits, (long long)T);
  }
  int st = (mode == MOE_ROUTE_SOFTMAX_TOPK || d_logits) ? launch_status() : MOE_OK;
  if (st != MOE_OK) return st;

  if (tc && router_bwd_tc_applies(H, E) && (dw || dx)) {
    // dW partials and dx in one pass over x and dx, then the partials' reduction
    st = launch_router_bwd_tc(x, dl3, w, T, H, E, dw ? part : nullptr, dx_write, dx, s);
    if (st == MOE_OK && dw) st = launch_reduce(part, router_bwd_tc_splits(T, H, E), H, E, dw, s);
    return st;
  }
  if (dw) {
    if (tc) {
      st = launch_router_dw_tc(x, dl3, T, H, E, part, s);
      if (st == MOE_OK) st = launch_reduce(part, router_dw_tc_splits(T, H, E), H, E, dw, s);
    } else {
      st = dtype == MOE_BF16 ? launch_dw<bf16>(static_cast<const bf16*>(x), dl, T, H, E, part, dw, s)
                             : launch_dw<float>(static_cast<const float*>(x), dl, T, H, E, part, dw, s);
      if (st == MOE_OK) st = launch_reduce(part, dw_plan(T, H, E).splits, H, E, dw, s);
    }
    if (st != MOE_OK) return st;
  }
  if (dx) {
    if (tc) st = launch_router_dx_tc(dl3, w, T, H, E, dx_write, dx, s);
    else
      st = dtype == MOE_BF16
               ? launch_dx<bf16>(dl, static_cast<const bf16*>(w), T, H, E, dx_write, static_cast<bf16*>(dx), s)
               : launch_dx<float>(dl, static_cast<const float*>(w), T, H, E, dx_write, static_cast<float*>(dx), s);
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

}  // namespace moe
