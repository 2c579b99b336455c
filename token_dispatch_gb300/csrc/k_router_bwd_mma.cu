// Router backward for 8 or 16 experts (bf16, softmax/top-K gate) as one
// streaming pass with both products on the warp-level tensor-core MMA.
//
// The sparse backward of the MoE/MoD framework page ("What's in the box": the
// gating gradients in one kernel without saved intermediates) needs, per token
// t, the logit gradient dl[t, :] (from the saved logits, the chosen experts
// and d_gate), then
//     dx[t, h]    (+)= sum_e dl[t, e] W_r[h, e]
//     dW_r[h, e]   += sum_t x[t, h] dl[t, e].
// At 2E flops per element of x and dx the pass is a stream of x and dx; what
// it must not be is bound by instruction issue, which is where per-thread FMAs
// left it.  Here both products are bf16 m16n8k16 / m16n8k8 MMAs with fp32
// accumulation, with dl carried exactly: dl = hi + mid + lo, three bf16 parts
// (each part keeps the next 8 significant bits; the subtractions are exact),
// so every product of a bf16 x or W_r value with a part is exact in fp32 and
// the three products land in the same fp32 sums.
//
//   * A CTA owns a contiguous token range and a 512-column slice of H; each of
//     its 8 warps owns 64 columns, and lane group g (lanes 4g..4g+3) owns 8
//     consecutive columns of them.  Tokens go in groups of 16; lane (g, c)
//     touches the rows of tokens 2c, 2c+1, 2c+8, 2c+9 of the group at its 8
//     columns: it copies them from x and dx (16 bytes each: whole 128-byte
//     lines per 8 lanes) into its own slots of a shared-memory ring with
//     cp.async, six groups ahead for 8 experts and four for 16, reads them
//     back when the group comes up, and writes dx back to the same places.
//   * dx: D[h, t] = W_r[h, :] . dl[t, :]^T per 8 tokens.  Row m of M tile i is
//     column 8g + 2i (m = g) or 8g + 2i + 1 (m = g + 8), so after the four
//     tiles each lane holds whole 8-column row pieces of its two tokens; the
//     accumulators start from the old dx (or zero when dx is overwritten).
//     K runs over (part, expert): with 8 experts hi|mid in one k16 MMA and lo
//     in a k8 one; with 16 experts one k16 MMA per part.  W_r sits in
//     registers as A fragments for the whole range.
//   * dW: D[e-part, h] += dl^T[e-part, t] . x[t, h] per 16 tokens, N tile j
//     column n = h 8n + j, so the B fragments (pairs of tokens at one column)
//     come from the lane's own x loads by byte permutes.  The accumulators
//     stay in registers over the range and are written once as this range's
//     fp32 partial [H][E]; a fixed-order reduction adds the ranges.
//   * dl of a chunk of 256 tokens is computed one thread per token into shared
//     memory in two layouts: expert pairs per token (dx B fragments) and token
//     pairs per expert (dW A fragments), rows padded against bank conflicts.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int RM_WARPS = 8;
constexpr int RM_THREADS = 32 * RM_WARPS;
constexpr int RM_VW = 8;                     // columns per lane group: one 16-byte piece of a row
constexpr int RM_CS = RM_WARPS * 8 * RM_VW;  // columns per CTA slice: 512
constexpr int RM_MT = RM_VW / 2;             // dx M tiles per warp
constexpr int RM_CHUNK = 256;             // tokens whose dl sits in shared memory
constexpr int RM_GROUPS = RM_CHUNK / 16;  // 16-token groups per chunk

template <int E> struct RmCfg {
  static constexpr int NPART = 3;
  static constexpr int EP = E / 2;                      // expert pairs per token
  static constexpr int EPS = E == 16 ? EP + 4 : EP;     // padded row (words)
  static constexpr int TPS = RM_CHUNK / 2 + 4;          // token pairs per expert row, padded
  static constexpr int DLP_WORDS = NPART * RM_CHUNK * EPS;
  static constexpr int DLT_WORDS = NPART * E * TPS;
  static constexpr int DWM = E == 8 ? 2 : 3;           // dW MMAs per N tile
  // groups whose x and dx pieces are in flight ahead, each thread's in its own
  // slots of a shared-memory ring (filled by cp.async, read back by the same
  // thread): 8 pieces of 16 bytes per thread and group
  static constexpr int D = E == 8 ? 6 : 4;
  static constexpr int RING_OFF = ((DLP_WORDS + DLT_WORDS) * 4 + 15) / 16 * 16;  // bytes
  static constexpr int SMEM = RING_OFF + D * 8 * RM_THREADS * 16;
};

__device__ __forceinline__ void mma_k16(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                        unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_k8(float (&d)[4], unsigned a0, unsigned a1, unsigned b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ float bf_lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(unsigned w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ unsigned pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<unsigned*>(&h);
}

// 16 bytes of a row into shared memory, through L2 only (zeros when !ok)
__device__ __forceinline__ void cp16(void* smem, const bf16* p, bool ok) {
  const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(p), "r"(ok ? 16 : 0) : "memory");
}
__device__ __forceinline__ unsigned word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// dl[e] of token t: softmax of the E logits, then the gradient of the K chosen
// gates (renormalised to sum 1 when renorm):
//   plain:  dl_j = p_j (G_j - sum_k d_gate_k p_{idx_k})
//   renorm: q_j = p_j / sum_k p_{idx_k} on the chosen experts, 0 elsewhere;
//           dl_j = q_j (G_j - sum_k d_gate_k q_{idx_k})
// G_j = d_gate_k where idx_k = j, else 0.
template <int E>
__device__ __forceinline__ void logit_grad(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                                           const float* __restrict__ d_gate, int K, int renorm, long long t,
                                           float (&dl)[E]) {
  float v[E];
#pragma unroll
  for (int q = 0; q < E / 4; ++q) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(logits + t * E) + q);
    v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
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

// grid = G token ranges x NS slices of 512 columns (blockIdx.x = range * NS +
// slice).  part (nullable): [G][H][E] fp32 partials of dW_r; dx (nullable):
// accumulated into, or written when dx_write; d_logits (nullable): written by
// slice 0.
template <int E>
__global__ void __launch_bounds__(RM_THREADS, 1)
router_bwd_mma_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                      const float* __restrict__ d_gate, int K, int renorm, const bf16* __restrict__ x,
                      const bf16* __restrict__ w, int T, int H, int NS, int G, float* __restrict__ d_logits,
                      float* __restrict__ part, bf16* __restrict__ dx, int dx_write) {
  using C = RmCfg<E>;
  extern __shared__ unsigned rm_smem[];
  unsigned* dlp = rm_smem;                  // [part][token][expert pair]
  unsigned* dlt = rm_smem + C::DLP_WORDS;   // [part][expert][token pair]
  uint16_t* dlt16 = reinterpret_cast<uint16_t*>(dlt);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int slice = blockIdx.x % NS, range = blockIdx.x / NS;
  const int col = slice * RM_CS + warp * (8 * RM_VW) + RM_VW * g;  // this lane group's 8 columns
  const int t0 = (int)((long long)T * range / G), t1 = (int)((long long)T * (range + 1) / G);
  const int n_groups = (t1 - t0 + 15) / 16;
  const bool do_dw = part != nullptr, do_dx = dx != nullptr, load_dx = do_dx && !dx_write;

  // W_r A fragments of the dx MMAs: tile i, rows m = g (column col + 2i) and
  // m = g + 8 (column col + 2i + 1); experts 2c, 2c+1 (and 2c+8, 2c+9)
  unsigned wa[RM_MT][E == 16 ? 4 : 2];
#pragma unroll
  for (int i = 0; i < RM_MT; ++i) {
    const bf16* r0 = w + (long long)(col + 2 * i) * E;
    const bf16* r1 = r0 + E;
    wa[i][0] = __ldg(reinterpret_cast<const unsigned*>(r0) + c);
    wa[i][1] = __ldg(reinterpret_cast<const unsigned*>(r1) + c);
    if constexpr (E == 16) {
      wa[i][2] = __ldg(reinterpret_cast<const unsigned*>(r0) + c + 4);
      wa[i][3] = __ldg(reinterpret_cast<const unsigned*>(r1) + c + 4);
    }
  }
  // dW accumulators: [MMA][N tile j][4]
  float acc[C::DWM][RM_VW][4];
#pragma unroll
  for (int m = 0; m < C::DWM; ++m)
#pragma unroll
    for (int j = 0; j < RM_VW; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[m][j][q] = 0.f;

  // rows of a group this lane touches: tokens 2c, 2c+1, 2c+8, 2c+9
  auto row_tok = [&](int grp, int r) { return t0 + grp * 16 + 2 * c + (r & 1) + (r >> 1) * 8; };
  // ring slot of group grp: piece j (x rows 0-3, then dx rows 0-3) of thread
  // tid at [slot][j][tid] (consecutive lanes 16 bytes apart: no bank conflicts)
  uint4* ring = reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(rm_smem) + C::RING_OFF);
  auto piece = [&](int grp, int j) { return ring + ((grp % C::D) * 8 + j) * RM_THREADS + tid; };
  // every thread commits one copy group per ring group, copies or not, so the
  // per-thread wait counts stay aligned
  auto load_group = [&](int grp) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = row_tok(grp, r);
      const bool ok = grp < n_groups && t < t1;
      const long long off = (long long)(ok ? t : 0) * H + col;
      if (do_dw) cp16(piece(grp, r), x + off, ok);
      // dx is written by this kernel (a piece is read groups before it is
      // written back, by the same thread): the copies read through L2
      if (load_dx) cp16(piece(grp, 4 + r), dx + off, ok);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
#pragma unroll
  for (int d = 0; d < C::D; ++d) load_group(d);

  auto process = [&](uint4 (&xr)[4], uint4 (&dr)[4], int grp) {
    const int lg = grp % RM_GROUPS;  // group inside the chunk
    if (lg == 0) {
      // logit gradients of the chunk into shared memory (tokens past the range: 0)
      __syncthreads();
      const int cs = t0 + grp * 16;
      if (tid < RM_CHUNK) {
        float dl[E];
        const long long t = cs + tid;
        if (t < t1) {
          logit_grad<E>(logits, idx, d_gate, K, renorm, t, dl);
          if (d_logits && slice == 0) {
#pragma unroll
            for (int q = 0; q < E / 4; ++q)
              reinterpret_cast<float4*>(d_logits + t * E)[q] =
                  make_float4(dl[4 * q], dl[4 * q + 1], dl[4 * q + 2], dl[4 * q + 3]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) dl[e] = 0.f;
        }
        // exact split dl = hi + mid + lo
        float pt[3][E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float hi = __bfloat162float(__float2bfloat16_rn(dl[e]));
          const float r1 = dl[e] - hi;
          const float mid = __bfloat162float(__float2bfloat16_rn(r1));
          const float lo = __bfloat162float(__float2bfloat16_rn(r1 - mid));
          pt[0][e] = hi; pt[1][e] = mid; pt[2][e] = lo;
        }
#pragma unroll
        for (int p = 0; p < 3; ++p) {
#pragma unroll
          for (int e2 = 0; e2 < C::EP; ++e2)
            dlp[(p * RM_CHUNK + tid) * C::EPS + e2] = pack2(pt[p][2 * e2], pt[p][2 * e2 + 1]);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const __nv_bfloat16 b = __float2bfloat16_rn(pt[p][e]);
            dlt16[(p * E + e) * (2 * C::TPS) + tid] = *reinterpret_cast<const uint16_t*>(&b);
          }
        }
      }
      __syncthreads();
    }

    // ---- dW: B fragments from the lane's x rows (tokens 2c,2c+1 | 2c+8,2c+9)
    if (do_dw) {
      const int tp = lg * 8 + c;  // token pair (2c, 2c+1) of the group
      // A fragments of the group (the same for every N tile): rows e = g
      // (and g + 8) of each part, token pairs c and c + 4
      unsigned af[3][4];
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        af[p][0] = dlt[(p * E + g) * C::TPS + tp];
        af[p][2] = dlt[(p * E + g) * C::TPS + tp + 4];
        if constexpr (E == 16) {
          af[p][1] = dlt[(p * E + g + 8) * C::TPS + tp];
          af[p][3] = dlt[(p * E + g + 8) * C::TPS + tp + 4];
        } else {
          af[p][1] = af[p][3] = 0u;
        }
      }
#pragma unroll
      for (int j = 0; j < RM_VW; ++j) {
        const unsigned sel = (j & 1) ? 0x7632u : 0x5410u;
        const unsigned w0a = word(xr[0], j >> 1), w0b = word(xr[1], j >> 1);
        const unsigned w1a = word(xr[2], j >> 1), w1b = word(xr[3], j >> 1);
        const unsigned b0 = __byte_perm(w0a, w0b, sel), b1 = __byte_perm(w1a, w1b, sel);
        if constexpr (E == 8) {
          // rows 0-7 hi, 8-15 mid; then rows 0-7 lo
          mma_k16(acc[0][j], af[0][0], af[1][0], af[0][2], af[1][2], b0, b1);
          mma_k16(acc[1][j], af[2][0], 0u, af[2][2], 0u, b0, b1);
        } else {
#pragma unroll
          for (int p = 0; p < 3; ++p) mma_k16(acc[p][j], af[p][0], af[p][1], af[p][2], af[p][3], b0, b1);
        }
      }
    }

    // ---- dx: per 8 tokens (s = 0: rows 0, 1; s = 1: rows 2, 3 of the lane)
    if (do_dx) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const uint4 o0 = dr[2 * s], o1 = dr[2 * s + 1];  // tokens 2c, 2c+1 of the 8
        float d[RM_MT][4];
#pragma unroll
        for (int i = 0; i < RM_MT; ++i) {
          const unsigned u0 = word(o0, i), u1 = word(o1, i);
          d[i][0] = load_dx ? bf_lo(u0) : 0.f;  // column 2i, token 2c
          d[i][1] = load_dx ? bf_lo(u1) : 0.f;  // column 2i, token 2c+1
          d[i][2] = load_dx ? bf_hi(u0) : 0.f;  // column 2i+1, token 2c
          d[i][3] = load_dx ? bf_hi(u1) : 0.f;  // column 2i+1, token 2c+1
        }
        const int tk = lg * 16 + s * 8 + g;  // token of this lane's B column
        if constexpr (E == 8) {
          const unsigned bh = dlp[(0 * RM_CHUNK + tk) * C::EPS + c];
          const unsigned bm = dlp[(1 * RM_CHUNK + tk) * C::EPS + c];
          const unsigned bl = dlp[(2 * RM_CHUNK + tk) * C::EPS + c];
#pragma unroll
          for (int i = 0; i < RM_MT; ++i) {
            mma_k16(d[i], wa[i][0], wa[i][1], wa[i][0], wa[i][1], bh, bm);
            mma_k8(d[i], wa[i][0], wa[i][1], bl);
          }
        } else {
#pragma unroll
          for (int p = 0; p < 3; ++p) {
            const unsigned b0 = dlp[(p * RM_CHUNK + tk) * C::EPS + c];
            const unsigned b1 = dlp[(p * RM_CHUNK + tk) * C::EPS + c + 4];
#pragma unroll
            for (int i = 0; i < RM_MT; ++i) mma_k16(d[i], wa[i][0], wa[i][1], wa[i][2], wa[i][3], b0, b1);
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int t = row_tok(grp, 2 * s + r);
          if (t < t1) {
            uint4 o;
            o.x = pack2(d[0][r], d[0][r + 2]);
            o.y = pack2(d[1][r], d[1][r + 2]);
            o.z = pack2(d[2][r], d[2][r + 2]);
            o.w = pack2(d[3][r], d[3][r + 2]);
            *reinterpret_cast<uint4*>(dx + (long long)t * H + col) = o;
          }
        }
      }
    }
  };

  // every thread takes part in the chunk barriers: the group loop is uniform
  for (int grp = 0; grp < n_groups; ++grp) {
    // this thread's copies of group grp have landed (the D - 1 newer groups may
    // still be in flight)
    asm volatile("cp.async.wait_group %0;" ::"n"(C::D - 1) : "memory");
    uint4 xr[4], dr[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      xr[r] = do_dw ? *piece(grp, r) : make_uint4(0, 0, 0, 0);
      dr[r] = load_dx ? *piece(grp, 4 + r) : make_uint4(0, 0, 0, 0);
    }
    process(xr, dr, grp);
    load_group(grp + C::D);  // into the slot just read
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  if (do_dw) {
    // dW[h][e] of column h = col + j (N tile j, n = g of the lane group that
    // owns it): lane (g, c) holds columns n = 2c, 2c+1 of every tile, i.e.
    // h = (warp columns) + 8 * (2c) + j and + 8 * (2c + 1) + j
    float* dst = part + (long long)range * H * E;
    const int wcol = slice * RM_CS + warp * (8 * RM_VW);
#pragma unroll
    for (int j = 0; j < RM_VW; ++j)
#pragma unroll
      for (int nn = 0; nn < 2; ++nn) {
        const int h = wcol + RM_VW * (2 * c + nn) + j;
        if constexpr (E == 8) {
          dst[(long long)h * E + g] = (acc[0][j][nn] + acc[0][j][nn + 2]) + acc[1][j][nn];
        } else {
          dst[(long long)h * E + g] = (acc[0][j][nn] + acc[1][j][nn]) + acc[2][j][nn];
          dst[(long long)h * E + g + 8] = (acc[0][j][nn + 2] + acc[1][j][nn + 2]) + acc[2][j][nn + 2];
        }
      }
  }
}

struct RmGeom {
  int ns, g;
};

RmGeom rm_geom(int T, int H) {
  RmGeom q;
  q.ns = H / RM_CS;
  long long g = sm_count() / (q.ns > 0 ? q.ns : 1);
  if (g < 1) g = 1;
  if (g > (T + 15) / 16) g = (T + 15) / 16;
  if (g < 1) g = 1;
  q.g = (int)g;
  return q;
}

}  // namespace

// bf16 softmax/top-K gate over 8 or 16 experts with H a multiple of 512
bool router_bwd_mma_applies(int mode, int dtype, int H, int E, int K) {
  return dtype == MOE_BF16 && mode == MOE_ROUTE_SOFTMAX_TOPK && (E == 8 || E == 16) && K >= 1 && K <= E &&
         H >= RM_CS && H % RM_CS == 0;
}

int router_bwd_mma_splits(int T, int H) { return rm_geom(T, H).g; }

int launch_router_bwd_mma(const float* d_gate, const float* logits, const int32_t* idx, const void* x,
                          const void* w, int T, int H, int E, int K, bool renorm, float* d_logits, float* part,
                          void* dx, bool dx_write, cudaStream_t s) {
  const RmGeom q = rm_geom(T, H);
  const int grid = q.g * q.ns;
  const bf16* xb = static_cast<const bf16*>(x);
  const bf16* wb = static_cast<const bf16*>(w);
  bf16* dxb = static_cast<bf16*>(dx);
  const int rn = renorm ? 1 : 0, dxw = dx_write ? 1 : 0;
  if (E == 8) {
    auto k = router_bwd_mma_kernel<8>;
    const int smem = RmCfg<8>::SMEM;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    k<<<grid, RM_THREADS, smem, s>>>(logits, idx, d_gate, K, rn, xb, wb, T, H, q.ns, q.g, d_logits, part, dxb,
                                     dxw);
  } else {
    auto k = router_bwd_mma_kernel<16>;
    const int smem = RmCfg<16>::SMEM;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    k<<<grid, RM_THREADS, smem, s>>>(logits, idx, d_gate, K, rn, xb, wb, T, H, q.ns, q.g, d_logits, part, dxb,
                                     dxw);
  }
  return launch_status();
}

}  // namespace moe
