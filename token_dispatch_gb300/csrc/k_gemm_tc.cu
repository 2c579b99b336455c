// Grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Two persistent, warp-specialised kernels: a one-CTA kernel (described below;
// the router GEMMs of up to 128 experts and the router backward's dW and dx
// GEMMs), and a CTA-pair kernel (two-CTA MMA, 256 x 256 tiles, each CTA staging
// half of B; its own section further down) for the expert FFN forward (with
// the dispatch gather optionally fused into its gate/up operand load) and
// backward and the router logits of more than 128 experts.  The backward of the expert FFN adds
//   da = dh Wd[e] with the SwiGLU backward in the epilogue, dxs = [dg | du]
//   [Wg[e] ; Wu[e]]^T, and the grouped-K weight gradients dW[e] = A_e^T B_e.
//
// The contractions of the layer:
//   * gate/up projection of every expert with SwiGLU fused in the epilogue
//       act[r, n] = silu(sum_k xs[r,k] Wg[e][k,n]) * (sum_k xs[r,k] Wu[e][k,n])
//   * down projection  h[r, n] = sum_k act[r,k] Wd[e][n,k]
//   * router GEMM      logits[t, e] = sum_h x[t,h] W_r[h,e] + bias[e]   (fp32 out)
//   * router backward  dW_r[h, e] = sum_t x[t,h] dl[t,e]  (A = x^T read MN-major,
//                      split over t into fp32 partials) and
//                      dx[t, h] (+)= sum_e dl[t,e] W_r[h,e]
//     with the fp32 logit gradient dl carried exactly as three bf16 parts
//     (dl = hi + mid + lo covers fp32's 24-bit significand): the three products
//     accumulate into the same fp32 TMEM accumulator.
// The weights are one contiguous [E, H, H'] tensor per projection and experts are
// addressed by their index (MoonEP page, "Step-by-step"); the rows of expert e
// are [cu[e], cu[e+1]) of the expert-sorted activation buffer, read on the device
// (no host synchronisation).
//
// Design of the one-CTA kernel (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer: A tile 128x64 (K-major x, or x^T read MN-major)
//               and B tile (MN-major [64 K x BN] chunks for W_r [H, E] or the
//               logit gradient; K-major [BN x 64 K] for W_r read as [E, H])
//               into a STAGES-deep shared-memory ring, 128-byte swizzled.
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16) from one
//               thread into one of two fp32 TMEM accumulators, committing each
//               stage back to the producer and each finished tile to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31 = tile rows), apply the bias / softmax and top-K,
//               convert, store;
//               the next tile's mainloop runs meanwhile in the other accumulator.
// Tiles are (expert, m-tile, n-tile) with m fastest inside an expert so the CTAs
// running at the same time share weight columns in L2.  Rows past an expert's
// end are computed (they belong to the next expert or are zero-filled by TMA past
// the buffer) and masked at the store.
//
// Every mbarrier wait is bounded: past the limit the kernel records
// MOE_ERR_TIMEOUT in the device error word, raises an abort flag that the other
// roles poll, waits (bounded) for its own copies and MMAs in flight, frees TMEM
// and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;            // 64 bf16 = 128 bytes: one swizzle row
constexpr int NUM_THREADS = 192;  // 6 warps
constexpr int GATHER_WARPS = 8;   // extra warps per CTA copying gathered A rows (the gate/up GEMM)
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int STG_LD = 33;  // row stride (floats) of an epilogue staging tile

// EPI_SWIGLU_BWD: the accumulator is da; with g, u read back from p.aux it
// writes dg and du (bf16) side by side.  EPI_F32_GK: fp32 tile of a grouped-K
// product (one output slab per group), zeros for a group without rows.
enum Epi { EPI_SWIGLU = 0, EPI_BF16 = 1, EPI_F32_BIAS = 2, EPI_ROUTER = 3, EPI_SWIGLU_BWD = 4, EPI_F32_GK = 5 };

struct Params {
  const int32_t* cu;  // nullptr: one group of M rows
  int G, M, N, K;     // N = output columns, K = reduction length
  void* out;
  long long ldo;
  const float* bias;
  unsigned* err;
  unsigned long long wait_limit;  // clock64 cycles
  int ksplit;                     // K split into this many ranges (fp32 partial outputs)
  long long part_stride;          // elements between the partial outputs of two splits
  int accumulate;                 // bf16 output: add the existing values
  // EPI_ROUTER: the whole expert row sits in one tile; the epilogue also takes
  // the softmax and the top-k of it
  int topk = 0;
  int32_t* topk_idx = nullptr;
  float* topk_gate = nullptr;
  const float* sel_bias = nullptr;  // added only where experts are chosen
  int renorm = 0;                   // the K gates rescaled to sum to 1
  // EPI_SWIGLU: when set, g and u are also stored (bf16, [g | u] per row of
  // ld_aux elements); EPI_SWIGLU_BWD: where g and u are read from
  void* aux = nullptr;
  long long ld_aux = 0;
  // K-major B from two tensors along K: k < kcat from tmB, k >= kcat from tmB2
  int kcat = 0;
  int b_col_off = 0;  // grouped K (CTA pairs): added to the N coordinate of the B loads
  // CTA pairs, bf16 output: when the last round holds at most half as many
  // tiles as there are pairs, its tiles run as two K halves on two pairs,
  // whose fp32 partials meet in split_ws; split_cnt holds one arrival counter
  // per (tile slot, CTA, epilogue warp), zeroed by the previous kernel on the
  // stream (zero_cnt / zero_n: the counters this kernel zeroes for the next)
  float* split_ws = nullptr;
  int* split_cnt = nullptr;
  int* zero_cnt = nullptr;
  int zero_n = 0;
  // K-major A rows gathered from another matrix (the gate/up GEMM on CTA
  // pairs): row r of A is row gather[r] of gather_src [gather_n, K] (bf16),
  // copied into the swizzled stages by GATHER_WARPS extra warps per CTA with
  // 16-byte asynchronous copies (the dispatch gather fused into the operand
  // load)
  const int32_t* gather = nullptr;
  const bf16* gather_src = nullptr;
  int gather_n = 0;
  // EPI_SWIGLU / EPI_SWIGLU_BWD: p.out and p.aux (when set) are 32-byte
  // aligned (their row strides are multiples of 128 bytes), so the epilogue
  // moves 64-byte row pieces as two 32-byte vectors
  int vec32 = 0;
};

// Waits for copies and MMAs already in flight when a role stops always use
// this bound, so a kernel that gave up early still leaves nothing running.
constexpr unsigned long long DRAIN_LIMIT = 4000000000ull;

// ------------------------------------------------------------------ PTX ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait.  Returns false (and raises the abort flag) on timeout, or if
// another role already aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             const Params& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if ((unsigned long long)(clock64() - t0) > p.wait_limit) {
        *abort_flag = 1;
        set_error(p.err, DEV_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns
// Order-preserving integer key of a float: a > b iff key(a) > key(b); -0 and
// +0 give the same key.  Keys of real values are >= 0x007fffff (that of -inf).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format): start, leading/stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // version
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A = B = bf16; bit 15 / 16 select
// MN-major A / B.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// NA A tiles and NB B tiles per stage; MMA pair p uses A tile min(p, NA-1) and
// B tile min(p, NB-1), all into one accumulator.
template <int BN, int EPI, int NA, int NB>
struct Cfg {
  static constexpr int B_TILE_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = NA * A_STAGE_BYTES + NB * B_TILE_BYTES;
  static constexpr int NP = NA > NB ? NA : NB;
  static constexpr int OUT_BN = (EPI == EPI_SWIGLU) ? BN / 2 : BN;  // output columns per tile
  static constexpr int TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
  // bf16 epilogue: per warp a [32 rows][33] fp32 staging tile, so the global
  // stores (and the reads of the old values) go out row-contiguous
  static constexpr int STG_LD = tc::STG_LD;
  static constexpr int EPI_BYTES = (EPI == EPI_BF16 || EPI == EPI_ROUTER) ? 4 * 32 * STG_LD * 4 : 0;
};

struct TileInfo {
  int g, row0, rows, n0;
};

// Tile t -> (group, rows, first output column).  mt_pre[g] = m-tiles before g.
__device__ __forceinline__ TileInfo decode(int t, const int* mt_pre, const int* cu, int G, int n_tiles,
                                           const Params& p, int out_bn) {
  // largest g with mt_pre[g] * n_tiles <= t
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (mt_pre[mid] * n_tiles <= t) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo;
  const int mt_g = mt_pre[g + 1] - mt_pre[g];
  const int local = t - mt_pre[g] * n_tiles;
  const int m = local % mt_g, n = local / mt_g;
  const int beg = cu ? cu[g] : 0;
  const int end = cu ? cu[g + 1] : p.M;
  TileInfo ti;
  ti.g = g;
  ti.row0 = beg + m * BM;
  ti.rows = min(BM, end - ti.row0);
  ti.n0 = n * out_bn;
  return ti;
}

// ------------------------------------------------------------ epilogues ---
// The thread owns TMEM lane (row) q*32 + lane of the tile's accumulator at
// tbase; grow is that row's index in the output, row_ok whether it exists.

// 32 bytes (two uint4) from or to a 32-byte aligned global address
__device__ __forceinline__ void ld_v8(uint4& a, uint4& b, const void* p) {
  asm volatile("ld.global.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "l"(p));
}
__device__ __forceinline__ void st_v8(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

// 64 bytes of one row: two 32-byte vector stores when p.vec32, else four 16-byte
__device__ __forceinline__ void st_row64(const Params& p, bf16* dst, const uint4 (&v)[4]) {
  if (p.vec32) {
    st_v8(dst, v[0], v[1]);
    st_v8(dst + 16, v[2], v[3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) reinterpret_cast<uint4*>(dst)[j] = v[j];
  }
}

// EPI_SWIGLU: columns [0, OUT_BN) hold g, [OUT_BN, 2 OUT_BN) hold u; act =
// silu(g) * u goes out as bf16 (and g, u to p.aux when set).
template <int OUT_BN>
__device__ __forceinline__ void epi_swiglu(const Params& p, uint32_t tbase, const TileInfo& ti, bool row_ok,
                                           long long grow, int c_begin = 0, int c_end = OUT_BN / 32) {
  bf16* out = static_cast<bf16*>(p.out);
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    float gv[32], uv[32];
    tmem_ld32(tbase + c * 32, gv);
    tmem_ld32(tbase + OUT_BN + c * 32, uv);
    const int col = ti.n0 + c * 32;
    if (row_ok && col < p.N) {
      uint4 pk[4];
      __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(pk);
      if (p.aux) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float a0 = gv[2 * j] / (1.0f + __expf(-gv[2 * j])) * uv[2 * j];
          float a1 = gv[2 * j + 1] / (1.0f + __expf(-gv[2 * j + 1])) * uv[2 * j + 1];
          h2[j] = __floats2bfloat162_rn(a0, a1);
        }
      } else {
        // without g and u to store: the approximate divide (2 ulp; silu of
        // g < -87 comes out 0), measured 1.5-1.8% faster at the short-K shapes;
        // with the stores it measured slower, so that path keeps the IEEE one
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float a0 = __fdividef(gv[2 * j], 1.0f + __expf(-gv[2 * j])) * uv[2 * j];
          float a1 = __fdividef(gv[2 * j + 1], 1.0f + __expf(-gv[2 * j + 1])) * uv[2 * j + 1];
          h2[j] = __floats2bfloat162_rn(a0, a1);
        }
      }
      st_row64(p, out + grow * p.ldo + col, pk);
      if (p.aux) {  // keep g and u for the backward
        uint4 gp[4], up[4];
        __nv_bfloat162* g2 = reinterpret_cast<__nv_bfloat162*>(gp);
        __nv_bfloat162* u2 = reinterpret_cast<__nv_bfloat162*>(up);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          g2[j] = __floats2bfloat162_rn(gv[2 * j], gv[2 * j + 1]);
          u2[j] = __floats2bfloat162_rn(uv[2 * j], uv[2 * j + 1]);
        }
        bf16* ax = static_cast<bf16*>(p.aux) + grow * p.ld_aux;
        st_row64(p, ax + col, gp);
        st_row64(p, ax + p.N + col, up);
      }
    }
  }
}

// EPI_SWIGLU_BWD: the accumulator is da; with g, u read back from p.aux it
// writes dg and du (bf16) side by side.
template <int OUT_BN>
__device__ __forceinline__ void epi_swiglu_bwd(const Params& p, uint32_t tbase, const TileInfo& ti, bool row_ok,
                                               long long grow, int c_begin = 0, int c_end = OUT_BN / 32) {
  // da for 32 columns at a time; g and u of the same columns come from
  // p.aux ([g | u] per row); dg and du go to p.out ([dg | du] per row)
  //   dg = da * u * s(g) * (1 + g * (1 - s(g))),  du = da * g * s(g)
  // The g, u loads of chunk c + 1 are issued before chunk c is computed (the
  // loop stays rolled: the next chunk's registers move into the current's).
  bf16* out = static_cast<bf16*>(p.out);
  const bf16* ax = static_cast<const bf16*>(p.aux);
  uint4 gq[4], uq[4], gn[4], un[4];
  auto load = [&](int c, uint4 (&g)[4], uint4 (&u)[4]) {
    const int col = ti.n0 + c * 32;
    if (row_ok && col < p.N) {
      const bf16* gs = ax + grow * p.ld_aux + col;
      const bf16* us = gs + p.N;
      if (p.vec32) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          ld_v8(g[2 * j], g[2 * j + 1], gs + 16 * j);
          ld_v8(u[2 * j], u[2 * j + 1], us + 16 * j);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          g[j] = reinterpret_cast<const uint4*>(gs)[j];
          u[j] = reinterpret_cast<const uint4*>(us)[j];
        }
      }
    }
  };
  load(c_begin, gq, uq);
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    if (c + 1 < c_end) load(c + 1, gn, un);
    float da[32];
    tmem_ld32(tbase + c * 32, da);
    const int col = ti.n0 + c * 32;
    if (row_ok && col < p.N) {
      uint4 dgp[4], dup[4];
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(gq);
      const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(uq);
      __nv_bfloat162* dg2 = reinterpret_cast<__nv_bfloat162*>(dgp);
      __nv_bfloat162* du2 = reinterpret_cast<__nv_bfloat162*>(dup);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float2 g = __bfloat1622float2(g2[j]);
        const float2 u = __bfloat1622float2(u2[j]);
        const float s0 = 1.0f / (1.0f + __expf(-g.x)), s1 = 1.0f / (1.0f + __expf(-g.y));
        const float a0 = da[2 * j], a1 = da[2 * j + 1];
        dg2[j] = __floats2bfloat162_rn(a0 * u.x * s0 * (1.0f + g.x * (1.0f - s0)),
                                       a1 * u.y * s1 * (1.0f + g.y * (1.0f - s1)));
        du2[j] = __floats2bfloat162_rn(a0 * g.x * s0, a1 * g.y * s1);
      }
      bf16* dgd = out + grow * p.ldo + col;
      bf16* dud = dgd + p.N;
      if (p.vec32) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          st_v8(dgd + 16 * j, dgp[2 * j], dgp[2 * j + 1]);
          st_v8(dud + 16 * j, dup[2 * j], dup[2 * j + 1]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          reinterpret_cast<uint4*>(dgd)[j] = dgp[j];
          reinterpret_cast<uint4*>(dud)[j] = dup[j];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      gq[j] = gn[j];
      uq[j] = un[j];
    }
  }
}

// EPI_F32_BIAS (CTA pairs): the fp32 tile plus the bias of its columns,
// 32 columns at a time through the warp's staging tile: 4 rows x 128 bytes per
// store instruction; columns at or past N are not stored.
template <int OUT_BN>
__device__ __forceinline__ void epi_f32_bias(const Params& p, uint32_t tbase, const TileInfo& ti, float* epi_stage,
                                             int q, int lane) {
  float* out = static_cast<float*>(p.out);
  float* stg = epi_stage + q * 32 * STG_LD;
  const int seg = (lane & 7) * 4;
#pragma unroll 1
  for (int c = 0; c < OUT_BN / 32; ++c) {
    float v[32];
    tmem_ld32(tbase + c * 32, v);
#pragma unroll
    for (int j = 0; j < 32; ++j) stg[lane * STG_LD + j] = v[j];
    __syncwarp();
    const int col = ti.n0 + c * 32 + seg;
    float4 bb = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.bias && col < p.N) bb = __ldg(reinterpret_cast<const float4*>(p.bias + col));
#pragma unroll
    for (int ps = 0; ps < 8; ++ps) {
      const int rw = ps * 4 + (lane >> 3);
      const int rr = q * 32 + rw;
      const long long gr = (long long)ti.row0 + rr;
      if (rr < ti.rows && gr < p.M && col < p.N) {
        const float* sp = stg + rw * STG_LD + seg;
        *reinterpret_cast<float4*>(out + gr * p.ldo + col) =
            make_float4(sp[0] + bb.x, sp[1] + bb.y, sp[2] + bb.z, sp[3] + bb.w);
      }
    }
    __syncwarp();
  }
}

// EPI_F32_GK through tensor stores: each 32-column chunk of the warp's 32
// TMEM lanes goes to one of the warp's GK_OUT_BUFS 4 KB staging tiles in the
// 128-byte swizzled layout (16-byte piece j of row r at j ^ (r & 7): the
// lanes' writes fall in distinct banks) and leaves as one [32 x 32] fp32 store
// into slab `slab` of the map's [G][M][N] output, which clips rows and columns
// past the output.  Lane 0 issues one bulk group per chunk; `chunk` counts the
// warp's chunks across tiles, and a staging tile is refilled GK_OUT_BUFS
// chunks later, once the store from it has read it (two tiles per warp: deeper
// rotations measured the same).
constexpr int GK_OUT_BUFS = 2;
template <int OUT_BN>
__device__ __forceinline__ void epi_f32_gk_tma(const CUtensorMap* tmO, const Params& p, uint32_t tbase,
                                               const TileInfo& ti, int slab, bool empty, float* stage_w, int q,
                                               int lane, int& chunk) {
  if (ti.rows <= q * 32) return;  // none of this warp's rows is an output row
  const uint32_t buf = smem_u32(stage_w);
#pragma unroll 1
  for (int c = 0; c < OUT_BN / 32; ++c) {
    const int col = ti.n0 + c * 32;
    if (col >= p.N) break;
    float v[32];
    if (!empty) {
      tmem_ld32(tbase + c * 32, v);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    }
    const uint32_t dst = buf + (chunk % GK_OUT_BUFS) * 4096;
    ++chunk;
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(GK_OUT_BUFS - 1) : "memory");
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t a = dst + lane * 128 + ((j ^ (lane & 7)) << 4);
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v[4 * j]), "f"(v[4 * j + 1]),
                   "f"(v[4 * j + 2]), "f"(v[4 * j + 3])
                   : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(tmO),
                   "r"(col), "r"(ti.row0 + q * 32), "r"(slab), "r"(dst)
                   : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
  }
}

// EPI_BF16: the fp32 tile rounded to bf16 (plus the old values with
// p.accumulate), through the warp's [32][STG_LD] staging tile.
template <int OUT_BN>
__device__ __forceinline__ void epi_bf16(const Params& p, uint32_t tbase, const TileInfo& ti, float* epi_stage,
                                         int q, int lane, const float* addp = nullptr) {
  // TMEM row per thread -> this warp's staging tile -> 8 rows x 64 bytes
  // per store instruction (4 lanes per row segment of 32 columns).  With
  // accumulate, every old value the warp will add is requested first.
  bf16* out = static_cast<bf16*>(p.out);
  constexpr int NCH = OUT_BN / 32;
  float* stg = epi_stage + q * 32 * STG_LD;
  const int seg = (lane & 3) * 8;
  uint4 old[NCH][4];
  if (p.accumulate) {
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
#pragma unroll
      for (int ps = 0; ps < 4; ++ps) {
        const int rr = q * 32 + ps * 8 + (lane >> 2);
        const long long gr = (long long)ti.row0 + rr;
        const int col = ti.n0 + c * 32 + seg;
        const bool ok = rr < ti.rows && gr < p.M && col < p.N;
        old[c][ps] = ok ? *reinterpret_cast<const uint4*>(out + gr * p.ldo + col) : make_uint4(0, 0, 0, 0);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    float v[32];
    tmem_ld32(tbase + c * 32, v);
    if (addp) {
      // the other K half's partial of this thread's row (split tiles)
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 o = __ldcg(reinterpret_cast<const float4*>(addp) + (c * 8 + j4) * 32 + lane);
        v[4 * j4] += o.x;
        v[4 * j4 + 1] += o.y;
        v[4 * j4 + 2] += o.z;
        v[4 * j4 + 3] += o.w;
      }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) stg[lane * STG_LD + j] = v[j];
    __syncwarp();
#pragma unroll
    for (int ps = 0; ps < 4; ++ps) {
      const int rw = ps * 8 + (lane >> 2);
      const int rr = q * 32 + rw;
      const long long gr = (long long)ti.row0 + rr;
      const int col = ti.n0 + c * 32 + seg;
      if (rr < ti.rows && gr < p.M && col < p.N) {
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = stg[rw * STG_LD + seg + j];
        if (p.accumulate) {
          const __nv_bfloat162* oh = reinterpret_cast<const __nv_bfloat162*>(&old[c][ps]);
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {
            const float2 f = __bfloat1622float2(oh[q2]);
            a[2 * q2] += f.x;
            a[2 * q2 + 1] += f.y;
          }
        }
        uint4 pk;
        __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
        for (int j = 0; j < 4; ++j) h2[j] = __floats2bfloat162_rn(a[2 * j], a[2 * j + 1]);
        *reinterpret_cast<uint4*>(out + gr * p.ldo + col) = pk;
      }
    }
    __syncwarp();
  }
}

// Tail split (CTA pairs): tile slots, and the fp32 partial of one K half of one
// epilogue warp's 32 rows x 256 columns, stored so that every store and load
// instruction covers 512 contiguous bytes (float4 j of chunk c of lane l at
// (c * 8 + j) * 32 + l).
constexpr int SPLIT_SLOTS = 64;
constexpr long long SPLIT_WARP_ELEMS = 32LL * 256;
constexpr size_t SPLIT_PART_BYTES = (size_t)SPLIT_SLOTS * 2 * 4 * 2 * SPLIT_WARP_ELEMS * 4;
constexpr int SPLIT_COUNTERS = SPLIT_SLOTS * 2 * 4;

// EPI_BF16 of a split tile, first part: each epilogue warp stores its partial,
// then counts itself in with a device-scope fence before the atomic.  Returns
// the other half's partial when this warp arrived second (it then adds that
// partial, in epi_bf16, and writes the bf16 rows; fp32 addition commutes, so
// the result does not depend on which half finishes first), else nullptr: the
// warp is done once its partial is out.  Nothing waits.
template <int OUT_BN>
__device__ __forceinline__ const float* split_partial(const Params& p, uint32_t tbase, int slot, int half,
                                                      uint32_t rank, int q, int lane) {
  static_assert(32LL * OUT_BN == SPLIT_WARP_ELEMS, "one warp's partial is 32 rows x 256 columns");
  float* base = p.split_ws + (((long long)slot * 2 + rank) * 4 + q) * 2 * SPLIT_WARP_ELEMS;
  float4* mine = reinterpret_cast<float4*>(base + half * SPLIT_WARP_ELEMS);
#pragma unroll 1
  for (int c = 0; c < OUT_BN / 32; ++c) {
    float v[32];
    tmem_ld32(tbase + c * 32, v);
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4)
      __stcg(mine + (c * 8 + j4) * 32 + lane, make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]));
  }
  __threadfence();
  __syncwarp();
  int first = 0;
  if (lane == 0) first = atomicAdd(p.split_cnt + ((slot * 2 + (int)rank) * 4 + q), 1) == 0;
  if (__shfl_sync(0xffffffffu, first, 0)) return nullptr;
  __threadfence();
  return base + (half ^ 1) * SPLIT_WARP_ELEMS;
}

// KSUB > 1: the NA = NB = KSUB tile pairs of a stage are consecutive 64-wide
// slices of K (a stage covers 64*KSUB of K), so each row of a streamed operand
// is requested as 128*KSUB contiguous bytes at once.
template <int EPI, bool A_MN, bool B_MN, int BN, int STAGES, int NA, int NB, int KSUB = 1>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmB2, const Params p) {
  using C = Cfg<BN, EPI, NA, NB>;
  static_assert(KSUB == 1 || (NA == KSUB && NB == KSUB && !A_MN), "k sub-blocks pair A and B slices");
  constexpr int KSTAGE = BK * KSUB;  // K covered by one stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  float* epi_stage = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + C::EPI_BYTES);
  // bars: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;
  __shared__ int mt_pre[1025];
  __shared__ int cu_s[1025];  // the group boundaries, read once from global memory
  __shared__ int total_tiles_s;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int n_tiles = (p.N + C::OUT_BN - 1) / C::OUT_BN;

  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto accf_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + a]); };
  auto acce_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 4]);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 128);
    }
    mbar_init(drain_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (p.kcat) prefetch_tmap(&tmB2);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_slot)),
                 "r"((uint32_t)C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == 2 && p.cu) {
    // eight loads per lane in flight at a time
    for (int base = 0; base <= G; base += 32 * 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * 32 + lane;
        v[u] = i <= G ? p.cu[i] : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * 32 + lane;
        if (i <= G) cu_s[i] = v[u];
      }
    }
    __syncwarp();
  }
  const int* cu = p.cu ? cu_s : nullptr;
  if (warp == 2) {
    // m-tile prefix over groups: each lane owns a contiguous run of groups
    const int per = (G + 31) / 32;
    int sum = 0;
    for (int g = lane * per; g < min(G, lane * per + per); ++g) {
      int rows = cu ? max(0, cu[g + 1] - cu[g]) : p.M;
      sum += (rows + BM - 1) / BM;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int g = lane * per; g < min(G, lane * per + per); ++g) {
      mt_pre[g] = run;
      int rows = cu ? max(0, cu[g + 1] - cu[g]) : p.M;
      run += (rows + BM - 1) / BM;
    }
    if (lane == 0 && cu && (cu[0] != 0 || cu[G] != p.M)) set_error(p.err, DEV_BOUNDS);
    if (lane == 31) {
      mt_pre[G] = incl;
      total_tiles_s = incl * n_tiles * p.ksplit;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  const int total_tiles = total_tiles_s;
  const int base_tiles = total_tiles / p.ksplit;  // tiles of one K range
  const int KB_ALL = (p.K + KSTAGE - 1) / KSTAGE;
  // k-blocks [kb_lo, kb_hi) of split s (every split non-empty: ksplit <= KB_ALL)
  auto kb_lo = [&](int s) { return (int)((long long)s * KB_ALL / p.ksplit); };
  // One work item: its output tile, its k-blocks and its K split.
  struct Work {
    TileInfo ti;
    int kb_begin, kb_end, split;
  };
  auto work = [&](int t) {
    Work w;
    w.split = t / base_tiles;
    w.ti = decode(t - w.split * base_tiles, mt_pre, cu, G, n_tiles, p, C::OUT_BN);
    w.kb_begin = kb_lo(w.split);
    w.kb_end = kb_lo(w.split + 1);
    return w;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int filled_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) filled_parity[s] = -1;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        const Work wk = work(t);
        const TileInfo& ti = wk.ti;
        for (int kb = wk.kb_begin; kb < wk.kb_end; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, &abort_flag, p)) { ok = false; break; }
          const uint32_t a_dst = smem_u32(stage_base + stage * C::STAGE_BYTES);
          const uint32_t b_dst = a_dst + NA * A_STAGE_BYTES;
          const int k0 = kb * KSTAGE;
          mbar_expect_tx(full_bar(stage), C::STAGE_BYTES);
          filled_parity[stage] = (int)phase;
#pragma unroll
          for (int ia = 0; ia < NA; ++ia) {
            const uint32_t dst = a_dst + ia * A_STAGE_BYTES;
            if (A_MN) {  // [64 K rows x 64 M] boxes, the two M halves LBO apart
              tma_load_3d(dst, &tmA, full_bar(stage), ti.row0, k0, ia);
              tma_load_3d(dst + 64 * BK * 2, &tmA, full_bar(stage), ti.row0 + 64, k0, ia);
            } else {
              if (KSUB > 1) tma_load_3d(dst, &tmA, full_bar(stage), k0 + ia * BK, ti.row0, 0);
              else tma_load_3d(dst, &tmA, full_bar(stage), k0, ti.row0, ia);
            }
          }
#pragma unroll
          for (int ib = 0; ib < NB; ++ib) {
            const uint32_t dst = b_dst + ib * C::B_TILE_BYTES;
            const int z = (NB > 1 && KSUB == 1) ? ib : ti.g;
            const int kb0 = KSUB > 1 ? k0 + ib * BK : k0;
            if (B_MN) {
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                tma_load_3d(dst + c * (64 * BK * 2), &tmB, full_bar(stage), ti.n0 + c * 64, kb0, z);
            } else if (p.kcat && kb0 >= p.kcat) {
              tma_load_3d(dst, &tmB2, full_bar(stage), kb0 - p.kcat, ti.n0, z);
            } else {
              tma_load_3d(dst, &tmB, full_bar(stage), kb0, ti.n0, z);
            }
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // drain: every stage this thread filled must have landed before exit
      for (int s = 0; s < STAGES; ++s) {
        if (filled_parity[s] < 0) continue;
        const long long t0 = clock64();
        while (!mbar_try_wait(full_bar(s), (uint32_t)filled_parity[s])) {
          if ((unsigned long long)(clock64() - t0) > DRAIN_LIMIT) { set_error(p.err, DEV_TIMEOUT); break; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = instr_desc(BM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued = false;
      int i = 0;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, ++i) {
        const int acc = i & 1;
        if (!wait_bounded(acce_bar(acc), (((uint32_t)i >> 1) & 1u) ^ 1u, &abort_flag, p)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const Work wk = work(t);
        const int kb_begin = wk.kb_begin, kb_end = wk.kb_end;
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, &abort_flag, p)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stage_base + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + NA * A_STAGE_BYTES;
#pragma unroll
          for (int pp = 0; pp < C::NP; ++pp) {
            const uint32_t a_t = a_addr + (pp < NA ? pp : NA - 1) * A_STAGE_BYTES;
            const uint32_t b_t = b_addr + (pp < NB ? pp : NB - 1) * C::B_TILE_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              // K-major: +32 bytes per 16-element K step inside the 128-byte
              // swizzle row; MN-major: +16 rows of 128 bytes, 64-wide M/N atoms
              // 8 KB apart (leading byte offset), 8-row groups 1 KB apart
              const uint64_t adesc = A_MN ? smem_desc(a_t + k * 16 * 128, 64 * BK * 2, 1024)
                                          : smem_desc(a_t + k * 32, 16, 1024);
              const uint64_t bdesc = B_MN ? smem_desc(b_t + k * 16 * 128, 64 * BK * 2, 1024)
                                          : smem_desc(b_t + k * 32, 16, 1024);
              tc_mma(d_tmem, adesc, bdesc, IDESC, (kb > kb_begin || pp > 0 || k > 0) ? 1u : 0u);
            }
          }
          issued = true;
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(accf_bar(acc));
      }
      // drain: all issued MMAs complete before TMEM is released
      if (issued) {
        tc_commit(drain_bar);
        const long long t0 = clock64();
        while (!mbar_try_wait(drain_bar, 0)) {
          if ((unsigned long long)(clock64() - t0) > DRAIN_LIMIT) { set_error(p.err, DEV_TIMEOUT); break; }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_local = q * 32 + lane;
    int i = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++i) {
      const int acc = i & 1;
      if (!wait_bounded(accf_bar(acc), ((uint32_t)i >> 1) & 1u, &abort_flag, p)) break;
      tc_fence_after();
      const Work wk = work(t);
      const TileInfo& ti = wk.ti;
      const int split = wk.split;
      const long long grow = (long long)ti.row0 + r_local;
      const bool row_ok = r_local < ti.rows && grow >= 0 && grow < p.M;
      const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
      if (EPI == EPI_BF16) {
        epi_bf16<C::OUT_BN>(p, tbase, ti, epi_stage, q, lane);
      } else if (EPI == EPI_ROUTER) {
        // one thread = one token: its BN logits (E valid) come out of TMEM, get
        // the bias and are stored; the softmax and the top-k (value descending,
        // lowest expert first on ties) run in registers as balanced trees, so
        // every level is BN/2^l independent operations instead of one chain
        // of BN dependent ones
        float v[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(tbase + c * 32, *reinterpret_cast<float(*)[32]>(v + c * 32));
        if (p.bias) {
#pragma unroll
          for (int j = 0; j < BN; j += 4) {
            if (j < p.N) {
              const float4 bb = __ldg(reinterpret_cast<const float4*>(p.bias + j));
              v[j] += bb.x; v[j + 1] += bb.y; v[j + 2] += bb.z; v[j + 3] += bb.w;
            }
          }
        }
        {
          // logits through this warp's staging tile, 32 columns at a time: each
          // store instruction writes 4 rows x 128 contiguous bytes (a row per
          // thread would touch 32 lines per instruction)
          float* out = static_cast<float*>(p.out);
          float* stg = epi_stage + q * 32 * C::STG_LD;
          const int seg = (lane & 7) * 4;
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
#pragma unroll
            for (int j = 0; j < 32; ++j) stg[lane * C::STG_LD + j] = v[c * 32 + j];
            __syncwarp();
#pragma unroll
            for (int ps = 0; ps < 8; ++ps) {
              const int rw = ps * 4 + (lane >> 3);
              const int rr = q * 32 + rw;
              const long long gr = (long long)ti.row0 + rr;
              const int col = c * 32 + seg;
              if (rr < ti.rows && gr < p.M && col < p.N) {
                const float* sp = stg + rw * C::STG_LD + seg;
                *reinterpret_cast<float4*>(out + gr * p.ldo + col) = make_float4(sp[0], sp[1], sp[2], sp[3]);
              }
            }
            __syncwarp();
          }
        }
        if (row_ok) {
          // selection keys: the logits (plus the selection-only bias when
          // given) as order-preserving integers, -0 folded onto +0 (equal
          // values are equal keys); 0 marks a column past E or an expert
          // already chosen (every real value has a larger key)
          uint32_t key[BN];
#pragma unroll
          for (int j = 0; j < BN; j += 4) {
            float4 sb = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p.sel_bias && j < p.N) sb = __ldg(reinterpret_cast<const float4*>(p.sel_bias + j));
            const float sv[4] = {v[j] + sb.x, v[j + 1] + sb.y, v[j + 2] + sb.z, v[j + 3] + sb.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) key[j + u] = j < p.N ? order_key(sv[u]) : 0u;
          }
          float m[BN / 2];
#pragma unroll
          for (int j = 0; j < BN / 2; ++j) {
            const float a = j < p.N ? v[j] : -INFINITY, b = j + BN / 2 < p.N ? v[j + BN / 2] : -INFINITY;
            m[j] = fmaxf(a, b);
          }
#pragma unroll
          for (int w = BN / 4; w >= 1; w >>= 1)
#pragma unroll
            for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
          // exp(v - max) = 2^(v log2(e) - max log2(e)): one fused multiply-add
          // and the base-2 exponential per expert
          const float mx = m[0];
          const float mxl = mx * 1.4426950408889634f;
          float e[BN], sm[BN / 2];
#pragma unroll
          for (int j = 0; j < BN; ++j) e[j] = j < p.N ? exp2f(fmaf(v[j], 1.4426950408889634f, -mxl)) : 0.f;
#pragma unroll
          for (int j = 0; j < BN / 2; ++j) sm[j] = e[j] + e[j + BN / 2];
#pragma unroll
          for (int w = BN / 4; w >= 1; w >>= 1)
#pragma unroll
            for (int j = 0; j < w; ++j) sm[j] += sm[j + w];
          const float sum = sm[0];
          float chosen = 0.f;
          for (int k = 0; k < p.topk; ++k) {
            // arg-max tree over adjacent pairs: the left operand always holds
            // the lower expert ids, so a tie keeps the left one; the winner's
            // exp value rides along
            uint32_t tk[BN / 2];
            int ti_[BN / 2];
            float te[BN / 2];
#pragma unroll
            for (int j = 0; j < BN / 2; ++j) {
              const bool r = key[2 * j + 1] > key[2 * j];
              tk[j] = r ? key[2 * j + 1] : key[2 * j];
              ti_[j] = r ? 2 * j + 1 : 2 * j;
              te[j] = r ? e[2 * j + 1] : e[2 * j];
            }
#pragma unroll
            for (int w = BN / 4; w >= 1; w >>= 1)
#pragma unroll
              for (int j = 0; j < w; ++j) {
                const bool r = tk[2 * j + 1] > tk[2 * j];
                tk[j] = r ? tk[2 * j + 1] : tk[2 * j];
                ti_[j] = r ? ti_[2 * j + 1] : ti_[2 * j];
                te[j] = r ? te[2 * j + 1] : te[2 * j];
              }
            const int be = ti_[0];
#pragma unroll
            for (int j = 0; j < BN; ++j) key[j] = j == be ? 0u : key[j];
            const float pk = te[0] / sum;
            chosen += pk;
            p.topk_idx[grow * p.topk + k] = be;
            p.topk_gate[grow * p.topk + k] = pk;
          }
          if (p.renorm)
            for (int k = 0; k < p.topk; ++k) p.topk_gate[grow * p.topk + k] = p.topk_gate[grow * p.topk + k] / chosen;
        }
      } else {
        float* out = static_cast<float*>(p.out) + (long long)split * p.part_stride;
#pragma unroll 1
        for (int c = 0; c < C::OUT_BN / 32; ++c) {
          float v[32];
          tmem_ld32(tbase + c * 32, v);
          if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = ti.n0 + c * 32 + j;
              if (col < p.N) out[grow * p.ldo + col] = v[j] + (p.bias ? __ldg(p.bias + col) : 0.f);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acce_bar(acc));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"((uint32_t)C::TMEM_COLS));
  }
}

// ------------------------------------------------------ CTA-pair GEMM ---
// The expert FFN's gate/up (SwiGLU epilogue) and down (bf16 epilogue) GEMMs
// on pairs of SMs with the 5th-generation tensor core's two-CTA MMA
// (tcgen05 cta_group::2): one 256 x 256 tile per pair, each CTA holding 128
// rows of A and half of the B columns in its own shared memory, each CTA's
// tensor memory holding the accumulator rows of its A rows.  Per SM a stage is
// 32 KB instead of 48 KB (B is not duplicated), so shared-memory traffic per
// MMA falls by a third and six stages fit where four did.
//
// Protocol (barriers at the same offsets in both CTAs):
//   full[s]   leader's only: its producer expects both CTAs' bytes; the two
//             producers' loads (cta_group::2 form) complete on it;
//   empty[s]  each CTA's own: the leader's MMA commit arrives on both;
//   accf[a]   each CTA's own: the leader's accumulator commit arrives on both;
//   acce[a]   leader's only: 128 epilogue threads of each CTA arrive (the
//             peer's remotely) before the leader reuses accumulator a.
// Tensor memory is allocated and freed by both CTAs together (the same
// columns in each); cluster barriers after set-up and before the release.
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_BN = 256;

template <int EPI>
struct PairCfg {
  // grouped K keeps GK_OUT_BUFS 4 KB staging tiles per epilogue warp for its
  // tensor stores, in place of pipeline stages
  static constexpr int STAGES = EPI == EPI_F32_GK ? (GK_OUT_BUFS <= 3 ? PAIR_STAGES - 1 : PAIR_STAGES - 2)
                                                 : PAIR_STAGES;
  static constexpr int B_HALF_BYTES = (PAIR_BN / 2) * BK * 2;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_HALF_BYTES;
  static constexpr int OUT_BN = EPI == EPI_SWIGLU ? PAIR_BN / 2 : PAIR_BN;
  // B N-contiguous (MN-major: Wg / Wu / Wd read as [K = H][N = H'], W_r as
  // [K = H][N = E]) or K-contiguous (Wd, or Wg / Wu in the backward, read as
  // [N = H][K = H'])
  static constexpr bool B_MN = EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD || EPI == EPI_F32_BIAS || EPI == EPI_F32_GK;
  // grouped K (weight gradients): A read transposed from a row-major [rows, M]
  // matrix, M-contiguous
  static constexpr bool A_MN = EPI == EPI_F32_GK;
  static constexpr int TMEM_COLS = 2 * PAIR_BN;
  static constexpr int EPI_BYTES =
      EPI == EPI_F32_GK ? 4 * GK_OUT_BUFS * 32 * 32 * 4 : (EPI == EPI_BF16 || EPI == EPI_F32_BIAS) ? 4 * 32 * STG_LD * 4 : 0;
  // barriers: full, empty, gathered [STAGES] each; accf, acce [2] each; drain
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + EPI_BYTES + (3 * STAGES + 5) * 8 + 1024;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// the shared::cluster address of the same offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// the pipeline stage n K blocks after stage s
template <int STAGES>
__device__ __forceinline__ int pair_stage(int s, int n) { return (s + n) % STAGES; }
// Zero K rows [from, BK) of both 64-column halves of a grouped-K A stage in
// both CTAs of the pair.  In the MN-major boxes each K row is one 128-byte
// line, so the swizzle does not matter; the 32 lanes of a warp take one K row
// (8 chunks x 2 halves x 2 CTAs) per step, then fence their generic writes
// against the MMAs' async-proxy reads.
__device__ __forceinline__ void clear_rows_pair(uint32_t a_stage, int from, int lane) {
  const int n = (BK - from) * 32;
  for (int idx = lane; idx < n; idx += 32) {
    const int j = idx & 7, half = (idx >> 3) & 1, cta = (idx >> 4) & 1, r = from + (idx >> 5);
    const uint32_t a = cluster_addr(a_stage + half * (64 * BK * 2) + r * 128 + j * 16, cta);
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
  }
  asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA load into this CTA's shared memory, completing on an mbarrier of
// either CTA of the pair (a shared::cluster address)
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                                 int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, %4, "
      "%5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// arrive (once the MMAs issued so far complete) on the mbarrier at this
// offset in every CTA of ctaMask
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(mask)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait with cluster-scope acquire (for arrivals from the peer CTA)
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                     const Params& p) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if ((unsigned long long)(clock64() - t0) > p.wait_limit) {
        *abort_flag = 1;
        set_error(p.err, DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Pair tile t -> (group, this CTA's 128 rows, first output column): m-tiles of
// 256 rows per group (mt_pre counts them), CTA `rank` takes rows 128 rank ..
template <int OUT_BN>
__device__ __forceinline__ TileInfo decode_pair(int t, const int* mt_pre, const int* cu, int G, int n_tiles,
                                                uint32_t rank) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (mt_pre[mid] * n_tiles <= t) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo;
  const int mt_g = mt_pre[g + 1] - mt_pre[g];
  const int local = t - mt_pre[g] * n_tiles;
  const int m = local % mt_g, n = local / mt_g;
  TileInfo ti;
  ti.g = g;
  ti.row0 = cu[g] + m * 2 * BM + (int)rank * BM;
  ti.rows = max(0, min(BM, cu[g + 1] - ti.row0));
  ti.n0 = n * OUT_BN;
  return ti;
}

// GATHER (gate/up only): the A rows are gathered from p.gather_src by
// GATHER_WARPS extra warps per CTA instead of loaded by TMA, each CTA copying
// its own 128 rows (rows past the group's end are not copied: their outputs
// are masked, and an accumulator row depends on its own A row only).  Every
// gather lane's copies complete on its CTA's `gathered` barrier; one more warp
// per CTA relays each completed stage to the leader's full barrier: it fences
// the copies (generic proxy) against the MMA's reads (async proxy) and sends
// 16 bytes to the leader by a bulk copy that completes on that barrier, like
// the TMA loads (a plain remote arrival at cluster scope, measured, made the
// MMA's waits about twice as long).
constexpr int PAIR_GATHER_THREADS = NUM_THREADS + 32 * (GATHER_WARPS + 1);
// Epilogue warps of the pair kernel: the SwiGLU backward keeps two warps per
// TMEM lane quadrant, each taking half of the tile's columns.  Its epilogue
// (g and u read, dg and du written, a row per lane) takes about twice as long
// as a tile's MMAs at K = 2048; the second warp per quadrant took the
// fine-grained layer's expert backward from 2.90 to 2.80 ms (measured), while
// the forward SwiGLU epilogue with g and u stored ran slower with it.
template <int EPI, bool GATHER>
__host__ __device__ constexpr int pair_epi_warps() {
  return EPI == EPI_SWIGLU_BWD && !GATHER ? 8 : 4;
}
template <int EPI, bool GATHER>
__host__ __device__ constexpr int pair_threads() {
  return GATHER ? PAIR_GATHER_THREADS : 64 + 32 * pair_epi_warps<EPI, GATHER>();
}
template <int EPI, bool GATHER = false>
__global__ void __launch_bounds__(pair_threads<EPI, GATHER>(), 1) __cluster_dims__(2, 1, 1)
tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB2, const Params p) {
  static_assert(EPI == EPI_SWIGLU || EPI == EPI_BF16 || EPI == EPI_SWIGLU_BWD || EPI == EPI_F32_BIAS ||
                    EPI == EPI_F32_GK,
                "pair kernel: GEMMs with a row-major output");
  static_assert(!GATHER || EPI == EPI_SWIGLU, "gathered A rows: the gate/up GEMM only");
  using C = PairCfg<EPI>;
  constexpr bool B_MN = C::B_MN;
  constexpr bool A_MN = C::A_MN;
  constexpr bool GK = EPI == EPI_F32_GK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  float* epi_stage = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES);
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;
  __shared__ int mt_pre[1025];
  __shared__ int cu_s[1025];
  __shared__ int total_tiles_s, full_tiles_s;
  __shared__ alignas(16) uint32_t relay_buf[8 * PAIR_STAGES];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int n_tiles = (p.N + C::OUT_BN - 1) / C::OUT_BN;

  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[C::STAGES + s]); };
  auto accf_bar = [&](int a) { return smem_u32(&bars[2 * C::STAGES + a]); };
  auto acce_bar = [&](int a) { return smem_u32(&bars[2 * C::STAGES + 2 + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * C::STAGES + 4]);
  auto gath_bar = [&](int s) { return smem_u32(&bars[2 * C::STAGES + 5 + s]); };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      if (GATHER) mbar_init(gath_bar(s), 32 * GATHER_WARPS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 2 * 32 * pair_epi_warps<EPI, GATHER>());  // the epilogue threads of both CTAs
    }
    mbar_init(drain_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (EPI == EPI_SWIGLU || p.kcat) prefetch_tmap(&tmB2);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_slot)),
                 "r"((uint32_t)C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  if (warp == 2) {
    // group boundaries (no cu: one group of M rows)
    for (int base = 0; base <= G; base += 32 * 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * 32 + lane;
        v[u] = i <= G ? (p.cu ? p.cu[i] : (i == 0 ? 0 : p.M)) : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * 32 + lane;
        if (i <= G) cu_s[i] = v[u];
      }
    }
    __syncwarp();
    // pair m-tiles (256 rows) per group, prefix over groups
    const int per = (G + 31) / 32;
    int sum = 0;
    for (int g = lane * per; g < min(G, lane * per + per); ++g) sum += (max(0, cu_s[g + 1] - cu_s[g]) + 2 * BM - 1) / (2 * BM);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int g = lane * per; g < min(G, lane * per + per); ++g) {
      mt_pre[g] = run;
      run += (max(0, cu_s[g + 1] - cu_s[g]) + 2 * BM - 1) / (2 * BM);
    }
    if (lane == 0 && (cu_s[0] != 0 || cu_s[G] != (GK ? p.K : p.M))) set_error(p.err, DEV_BOUNDS);
    if (lane == 31) {
      mt_pre[G] = incl;
      // grouped K: every group has all (M / 256) x (N / 256) output tiles
      int total = GK ? G * ((p.M + 2 * BM - 1) / (2 * BM)) * n_tiles : incl * n_tiles;
      int full = total;
      if (EPI == EPI_BF16 && p.split_ws && (p.K + BK - 1) / BK >= 2) {
        // tail split: the last round's tiles become two K halves each
        const int P = gridDim.x >> 1, rem = total % P;
        if (rem > 0 && 2 * rem <= P && rem <= SPLIT_SLOTS) {
          full = total - rem;
          total = full + 2 * rem;
        }
      }
      total_tiles_s = total;
      full_tiles_s = full;
    }
  }
  // counters of the next kernel on the stream (its split tiles' arrivals)
  if (p.zero_cnt && blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.zero_n; i += blockDim.x) p.zero_cnt[i] = 0;
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before anything arrives on them
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  const int total_tiles = total_tiles_s, full_tiles = full_tiles_s;
  const int KB_ALL = (p.K + BK - 1) / BK;
  // One pair tile: this CTA's output rows, its K blocks, the first K row of
  // block 0, the output slab (group) and the valid K rows of its last block.
  struct PairWork {
    TileInfo ti;
    int kb_end, k_base, slab, last_valid;
    int slot, half;  // split tiles: the tile's slot and K half (slot -1: a whole tile)
  };
  const int gk_mt = (p.M + 2 * BM - 1) / (2 * BM);
  auto pair_work = [&](int t) {
    PairWork w;
    if constexpr (GK) {
      const int per_g = gk_mt * n_tiles;
      const int g = t / per_g, rem = t - g * per_g;
      const int m = rem % gk_mt, n = rem / gk_mt;
      w.ti.g = g;
      w.ti.row0 = m * 2 * BM + (int)rank * BM;
      w.ti.rows = max(0, min(BM, p.M - w.ti.row0));
      w.ti.n0 = n * C::OUT_BN;
      const int beg = cu_s[g], rows = max(0, cu_s[g + 1] - beg);
      w.kb_end = (rows + BK - 1) / BK;
      w.k_base = beg;
      w.slab = g;
      w.last_valid = rows - (w.kb_end - 1) * BK;
      w.slot = -1;
      w.half = 0;
    } else {
      w.slab = 0;
      w.last_valid = BK;
      if (t < full_tiles) {
        w.ti = decode_pair<C::OUT_BN>(t, mt_pre, cu_s, G, n_tiles, rank);
        w.kb_end = KB_ALL;
        w.k_base = 0;
        w.slot = -1;
        w.half = 0;
      } else {
        // units full, full + 1 are the two K halves of tile full, and so on
        const int v = t - full_tiles, kb_mid = KB_ALL / 2;
        w.ti = decode_pair<C::OUT_BN>(full_tiles + (v >> 1), mt_pre, cu_s, G, n_tiles, rank);
        w.slot = v >> 1;
        w.half = v & 1;
        w.k_base = w.half ? kb_mid * BK : 0;
        w.kb_end = w.half ? KB_ALL - kb_mid : kb_mid;
      }
    }
    return w;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int filled_parity[C::STAGES];
      for (int s = 0; s < C::STAGES; ++s) filled_parity[s] = -1;
      bool ok = true;
      for (int t = pair; ok && t < total_tiles; t += n_pairs) {
        const PairWork wk = pair_work(t);
        const TileInfo& ti = wk.ti;
        for (int kb = 0; kb < wk.kb_end; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, &abort_flag, p)) { ok = false; break; }
          const uint32_t a_dst = smem_u32(stage_base + stage * C::STAGE_BYTES);
          const uint32_t b_dst = a_dst + A_STAGE_BYTES;
          const int k0 = wk.k_base + kb * BK;
          if (leader) {
            // this CTA's bytes and the peer's (gathered A: B and the two
            // relays' 16 bytes)
            mbar_expect_tx(full_bar(stage), GATHER ? 2 * C::B_HALF_BYTES + 32 : 2 * C::STAGE_BYTES);
            filled_parity[stage] = (int)phase;
          }
          const uint32_t fb = cluster_addr(full_bar(stage), 0);
          if constexpr (GATHER) {
            // A rows: the gather warps
          } else if constexpr (A_MN) {
            // [64 K rows x 64 M] boxes, the two M halves 8 KB apart (a
            // group's last block is cleared past the group before its MMAs)
            tma_load_3d_pair(a_dst, &tmA, fb, ti.row0, k0, 0);
            tma_load_3d_pair(a_dst + 64 * BK * 2, &tmA, fb, ti.row0 + 64, k0, 0);
          } else {
            tma_load_3d_pair(a_dst, &tmA, fb, k0, ti.row0, 0);
          }
          if constexpr (EPI == EPI_SWIGLU) {
            // the leader stages the gate columns, the peer the up columns
            const CUtensorMap* m = leader ? &tmB : &tmB2;
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_3d_pair(b_dst + c * (64 * BK * 2), m, fb, ti.n0 + c * 64, k0, ti.g);
          } else if constexpr (B_MN) {
            // each CTA stages its half of the 256 output columns (grouped K:
            // rows k0.. of one [rows, .] matrix, columns from b_col_off)
#pragma unroll
            for (int c = 0; c < 2; ++c)
              tma_load_3d_pair(b_dst + c * (64 * BK * 2), &tmB, fb,
                               ti.n0 + (int)rank * (PAIR_BN / 2) + c * 64 + p.b_col_off, k0, GK ? 0 : ti.g);
          } else if (p.kcat && k0 >= p.kcat) {
            // K concatenated from two tensors: k >= kcat reads the second
            tma_load_3d_pair(b_dst, &tmB2, fb, k0 - p.kcat, ti.n0 + (int)rank * (PAIR_BN / 2), ti.g);
          } else {
            tma_load_3d_pair(b_dst, &tmB, fb, k0, ti.n0 + (int)rank * (PAIR_BN / 2), ti.g);
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // drain (leader): every stage filled must have landed, both CTAs' bytes
      if (leader) {
        for (int s = 0; s < C::STAGES; ++s) {
          if (filled_parity[s] < 0) continue;
          const long long t0 = clock64();
          while (!mbar_try_wait(full_bar(s), (uint32_t)filled_parity[s])) {
            if ((unsigned long long)(clock64() - t0) > DRAIN_LIMIT) { set_error(p.err, DEV_TIMEOUT); break; }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer (leader only)
    // Lane 0 waits and issues.  Grouped K: the other lanes follow the same
    // tile sequence and meet lane 0 only in a group's last, partial K block,
    // whose rows past the group (the next group's) they clear to zeros in
    // both CTAs' A stages before its MMAs.  After a failed wait lane 0 keeps
    // walking the tiles without issuing, so the meetings still happen.
    if (leader && (lane == 0 || GK)) {
      constexpr uint32_t IDESC = instr_desc(2 * BM, PAIR_BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued = false;
      int i = 0;
      for (int t = pair; t < total_tiles; t += n_pairs, ++i) {
        const int acc = i & 1;
        const PairWork wk_m = pair_work(t);
        const int kb_end = wk_m.kb_end, last_valid = wk_m.last_valid;
        const bool clear = GK && kb_end > 0 && last_valid < BK;
        if (lane != 0) {
          // follower: the clearing of this tile's last block
          if (clear) {
            __syncwarp();
            const uint32_t a_t = smem_u32(stage_base + pair_stage<C::STAGES>(stage, kb_end - 1) * C::STAGE_BYTES);
            clear_rows_pair(a_t, last_valid, lane);
            __syncwarp();
          }
          stage = pair_stage<C::STAGES>(stage, kb_end);
          continue;
        }
        if (ok && !wait_bounded_cluster(acce_bar(acc), (((uint32_t)i >> 1) & 1u) ^ 1u, &abort_flag, p)) ok = false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * PAIR_BN;
        for (int kb = 0; kb < kb_end; ++kb) {
          const bool last_clear = clear && kb == kb_end - 1;
          if (ok && !(last_clear ? wait_bounded_cluster(full_bar(stage), phase, &abort_flag, p)
                                 : wait_bounded(full_bar(stage), phase, &abort_flag, p)))
            ok = false;
          tc_fence_after();
          const uint32_t a_t = smem_u32(stage_base + stage * C::STAGE_BYTES);
          const uint32_t b_t = a_t + A_STAGE_BYTES;
          if (last_clear) {
            __syncwarp();
            clear_rows_pair(a_t, last_valid, lane);
            __syncwarp();
          }
          if (ok) {
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              // K-major: +32 bytes per 16-element K step in the 128-byte row;
              // MN-major: +16 rows of 128 bytes, 64-wide atoms 8 KB apart
              const uint64_t adesc =
                  A_MN ? smem_desc(a_t + k * 16 * 128, 64 * BK * 2, 1024) : smem_desc(a_t + k * 32, 16, 1024);
              const uint64_t bdesc =
                  B_MN ? smem_desc(b_t + k * 16 * 128, 64 * BK * 2, 1024) : smem_desc(b_t + k * 32, 16, 1024);
              tc_mma_pair(d_tmem, adesc, bdesc, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
            }
            issued = true;
            tc_commit_pair(empty_bar(stage), 3);
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (ok) tc_commit_pair(accf_bar(acc), 3);
        else if (!GK) break;
      }
      if (lane == 0 && issued) {
        tc_commit_pair(drain_bar, 1);
        const long long t0 = clock64();
        while (!mbar_try_wait(drain_bar, 0)) {
          if ((unsigned long long)(clock64() - t0) > DRAIN_LIMIT) { set_error(p.err, DEV_TIMEOUT); break; }
        }
      }
    }
  } else if (GATHER && warp == NUM_THREADS / 32 + GATHER_WARPS) {
    // ------------------------------------- relay of the gathered A rows
    // Per stage, once every gather lane's copies have landed: fence them
    // against the async proxy, then 16 bytes from this CTA's relay slot to the
    // leader's by a bulk copy completing on the leader's full barrier.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = pair; ok && t < total_tiles; t += n_pairs) {
        const int kb_end = pair_work(t).kb_end;
        for (int kb = 0; kb < kb_end; ++kb) {
          if (!wait_bounded(gath_bar(stage), phase, &abort_flag, p)) { ok = false; break; }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          const uint32_t slot = smem_u32(&relay_buf[8 * stage + 4 * rank]);
          asm volatile(
              "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], 16, [%2];" ::"r"(
                  cluster_addr(slot, 0)),
              "r"(slot), "r"(cluster_addr(full_bar(stage), 0))
              : "memory");
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (GATHER && warp >= NUM_THREADS / 32) {
    // ------------------------------------------------ gathered A rows
    // Warp 6 + w copies rows RW*w .. RW*w + RW-1 of this CTA's 128 A rows
    // (RW = 128 / GATHER_WARPS): instruction j takes 4 rows, 8 lanes per row,
    // one 16-byte chunk each (whole 128-byte row segments), to the chunk's
    // 128-byte-swizzled place.  Rows past the group's end are skipped.
    constexpr int RW = BM / GATHER_WARPS;
    const int gw = warp - NUM_THREADS / 32;
    const int crow = lane >> 3, chunk = lane & 7;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = pair; ok && t < total_tiles; t += n_pairs) {
      const PairWork wk = pair_work(t);
      const int r_own = wk.ti.row0 + RW * gw + (lane % RW);
      int src = r_own < p.M ? __ldg(p.gather + r_own) : 0;
      if (src < 0 || src >= p.gather_n) {
        set_error(p.err, DEV_BOUNDS);
        src = 0;
      }
      for (int kb = 0; kb < wk.kb_end; ++kb) {
        if (lane == 0) ok = wait_bounded(empty_bar(stage), phase ^ 1u, &abort_flag, p);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const uint32_t a_dst = smem_u32(stage_base + stage * C::STAGE_BYTES);
        const int k0 = wk.k_base + kb * BK;
#pragma unroll
        for (int j = 0; j < RW / 4; ++j) {
          const int rr = 4 * j + crow;  // row inside this warp's RW
          const int r = RW * gw + rr;   // row inside the CTA's 128
          const int srow = __shfl_sync(0xffffffffu, src, rr);
          const bf16* g = p.gather_src + (long long)srow * p.K + k0 + chunk * 8;
          if (r < wk.ti.rows)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(a_dst + r * 128 + ((chunk ^ (r & 7)) << 4)),
                         "l"(g)
                         : "memory");
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(gath_bar(stage)) : "memory");
        if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_local = q * 32 + lane;
    // with two warps per quadrant, each takes half of the 32-column chunks
    constexpr int EPI_H = pair_epi_warps<EPI, GATHER>() / 4;
    constexpr int NCH = C::OUT_BN / 32;
    const int c_begin = ((warp - 2) >> 2) * (NCH / EPI_H), c_end = c_begin + NCH / EPI_H;
    int i = 0;
    int out_chunk = 0;  // grouped K: this warp's output chunks so far (staging tile rotation)
    for (int t = pair; t < total_tiles; t += n_pairs, ++i) {
      const int acc = i & 1;
      if (!wait_bounded(accf_bar(acc), ((uint32_t)i >> 1) & 1u, &abort_flag, p)) break;
      tc_fence_after();
      const PairWork wk = pair_work(t);
      const TileInfo& ti = wk.ti;
      const long long grow = (long long)ti.row0 + r_local;
      const bool row_ok = r_local < ti.rows && grow < p.M;
      const uint32_t tbase = tmem_base + acc * PAIR_BN + ((uint32_t)(q * 32) << 16);
      if constexpr (EPI == EPI_SWIGLU) epi_swiglu<C::OUT_BN>(p, tbase, ti, row_ok, grow, c_begin, c_end);
      else if constexpr (EPI == EPI_SWIGLU_BWD) epi_swiglu_bwd<C::OUT_BN>(p, tbase, ti, row_ok, grow, c_begin, c_end);
      else if constexpr (EPI == EPI_F32_BIAS) epi_f32_bias<C::OUT_BN>(p, tbase, ti, epi_stage, q, lane);
      else if constexpr (GK) {
        // the fp32 output's tensor map comes in place of the second B map
        epi_f32_gk_tma<C::OUT_BN>(&tmB2, p, tbase, ti, wk.slab, wk.kb_end == 0,
                                  epi_stage + q * GK_OUT_BUFS * 32 * 32, q, lane, out_chunk);
      } else {
        const float* addp = nullptr;
        if (wk.slot >= 0) addp = split_partial<C::OUT_BN>(p, tbase, wk.slot, wk.half, rank, q, lane);
        if (wk.slot < 0 || addp) epi_bf16<C::OUT_BN>(p, tbase, ti, epi_stage, q, lane, addp);
      }
      tc_fence_before();
      if (leader) mbar_arrive(acce_bar(acc));
      else mbar_arrive_remote(cluster_addr(acce_bar(acc), 0));
    }
    // the tensor stores are complete (and done reading shared memory) before
    // the CTA exits
    if constexpr (GK)
      if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs are done with tensor memory and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"((uint32_t)C::TMEM_COLS));
  }
}

// Failure-detection probe: one thread waits on an mbarrier that nothing ever
// arrives at, with the bounded wait of the pipelined kernels above; it gives up
// after p.wait_limit cycles and records DEV_TIMEOUT, as a stalled pipeline would.
__global__ void wait_probe_kernel(const Params p) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  (void)wait_bounded(smem_u32(&bar), 0, &abort_flag, p);
}

// ------------------------------------------------------------------ host ----

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle; dims/strides innermost first (strides in
// bytes for dims 1..rank-1).
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dt, rank, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

unsigned long long g_wait_limit = 4000000000ull;  // ~2 s at 2 GHz

template <int EPI, bool A_MN, bool B_MN, int BN, int STAGES, int NA, int NB, int KSUB = 1>
int launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const Params& p,
           long long tiles_upper, cudaStream_t s) {
  using C = Cfg<BN, EPI, NA, NB>;
  const size_t smem = (size_t)STAGES * C::STAGE_BYTES + C::EPI_BYTES + (2 * STAGES + 5) * 8 + 1024;
  static_assert((size_t)STAGES * C::STAGE_BYTES + C::EPI_BYTES + (2 * STAGES + 5) * 8 + 1024 + 8500 <= 227 * 1024,
                "smem (dynamic + static)");
  auto k = tc_gemm_kernel<EPI, A_MN, B_MN, BN, STAGES, NA, NB, KSUB>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  long long grid = sm_count();
  if (tiles_upper < grid) grid = tiles_upper;
  if (grid < 1) return MOE_OK;
  k<<<(unsigned)grid, NUM_THREADS, smem, s>>>(a, b, b2, p);
  return launch_status();
}

// Pairs resident at once for the pair kernel (cached per device and kernel):
// clusters of two SMs with one CTA each.
template <int EPI, bool GATHER = false>
int pair_slots() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return sm_count() / 2;
  }
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(pair_threads<EPI, GATHER>());
  cfg.dynamicSmemBytes = PairCfg<EPI>::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_pair_kernel<EPI, GATHER>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sm_count() / 2;
  }
  cached[dev] = n;
  return n;
}

template <int EPI, bool GATHER = false>
int launch_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const Params& p,
                long long pair_tiles_upper, cudaStream_t s) {
  using C = PairCfg<EPI>;
  static_assert(C::SMEM + 8500 <= 227 * 1024, "smem (dynamic + static)");
  auto k = tc_gemm_pair_kernel<EPI, GATHER>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) != cudaSuccess)
    return MOE_ERR_CUDA;
  long long pairs = pair_slots<EPI, GATHER>();
  if (pair_tiles_upper < pairs) pairs = pair_tiles_upper;
  if (pairs < 1) return MOE_OK;
  k<<<(unsigned)(2 * pairs), pair_threads<EPI, GATHER>(), C::SMEM, s>>>(a, b, b2, p);
  return launch_status();
}

// [rows, inner] bf16 matrix as a 3D map {inner, rows, 1}
bool map_2d_as_3d(CUtensorMap* m, const void* base, long long inner, long long rows, int box_inner, int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, 1};
  cuuint64_t str[2] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * rows * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  return make_map(m, base, 3, dims, str, box);
}

// [depth, rows, inner] bf16 tensor as a 3D map {inner, rows, depth}
bool map_3d(CUtensorMap* m, const void* base, long long inner, long long rows, long long depth, int box_inner,
            int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)depth};
  cuuint64_t str[2] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * rows * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
  return make_map(m, base, 3, dims, str, box);
}

Params params(const int32_t* cu, int G, int M, int N, int K, void* out, long long ldo, const float* bias) {
  return Params{cu, G, M, N, K, out, ldo, bias, device_error_word(), g_wait_limit, 1, 0, 0};
}

// ---------------------------------------------- router backward, one pass ---
// Router backward for bf16 routers with 32..64 experts (E % 8 == 0, padded to
// 64 by TMA zero fill) in one launch after the softmax backward: with the
// logit gradient split exactly into three bf16 parts dl = hi + mid + lo,
//   dW_r[h, e] = sum_t x[t, h] dl[t, e]        (fp32 partials per token range)
//   dx[t, h]  (+)= sum_e dl[t, e] W_r[h, e]    (bf16, read-modify-write)
// A CTA owns a 128-column slice of H and a range of 128-token blocks.  Per
// block one TMA stage brings the x tile (128 tokens x 128 columns, two
// M-contiguous boxes) and the three dl parts (128 tokens x 64 experts each);
// the same dl boxes are the N-contiguous B operand of dW (N = 192: the three
// parts side by side) and the K-major A operand of dx (M = 128 tokens, K = 3 x
// 64), so dl is read once for both products and x once.  dW accumulates in
// tensor memory over the CTA's whole token range (columns [0, 192)); dx uses two
// accumulators (columns [256, 384) and [384, 512)) so the epilogue of one block
// overlaps the next block's MMAs.  W_r's slice (128 x 64) is loaded once.
constexpr int RB_STAGES = 2;
constexpr int RB_TB = 128;                               // tokens per block
constexpr int RB_HS = 128;                               // H columns per CTA
constexpr int RB_X_BYTES = RB_TB * RB_HS * 2;            // 32 KB: two 64-column boxes
constexpr int RB_DL_BYTES = 3 * RB_TB * 64 * 2;          // 48 KB: three parts
constexpr int RB_STAGE_BYTES = RB_X_BYTES + RB_DL_BYTES;
constexpr int RB_W_BYTES = RB_HS * 64 * 2;               // 16 KB
// two epilogue warp groups, one per dx accumulator: consecutive blocks'
// read-modify-write round trips overlap
constexpr int RB_THREADS = 64 + 2 * 128;
constexpr int RB_STG_BYTES = 8 * 32 * STG_LD * 4;
constexpr size_t RB_SMEM = (size_t)RB_STAGES * RB_STAGE_BYTES + RB_W_BYTES + RB_STG_BYTES + 16 * 8 + 1024;

__global__ void __launch_bounds__(RB_THREADS, 1)
router_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmDL,
                     const __grid_constant__ CUtensorMap tmW, const Params p, int n_slices, int splits,
                     int n_blocks, float* part, int E) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* w_tile = smem + RB_STAGES * RB_STAGE_BYTES;
  float* epi_stage = reinterpret_cast<float*>(w_tile + RB_W_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(epi_stage) + RB_STG_BYTES);
  // bars: full[2], empty[2], accf[2], acce[2], w_full, dw_full, drain
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[RB_STAGES + s]); };
  auto accf_bar = [&](int a) { return smem_u32(&bars[2 * RB_STAGES + a]); };
  auto acce_bar = [&](int a) { return smem_u32(&bars[2 * RB_STAGES + 2 + a]); };
  const uint32_t w_bar = smem_u32(&bars[2 * RB_STAGES + 4]);
  const uint32_t dw_bar = smem_u32(&bars[2 * RB_STAGES + 5]);
  const uint32_t drain_bar = smem_u32(&bars[2 * RB_STAGES + 6]);
  // this CTA's slice of H and range of token blocks
  const int slice = blockIdx.x % n_slices, split = blockIdx.x / n_slices;
  const int h0 = slice * RB_HS;
  const int b_lo = (int)((long long)split * n_blocks / splits), b_hi = (int)((long long)(split + 1) * n_blocks / splits);
  const bool do_dw = part != nullptr, do_dx = p.out != nullptr;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < RB_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 128);
    }
    mbar_init(w_bar, 1);
    mbar_init(dw_bar, 1);
    mbar_init(drain_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmDL);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_slot)),
                 "r"(512u));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int filled_parity[RB_STAGES];
      for (int s = 0; s < RB_STAGES; ++s) filled_parity[s] = -1;
      if (do_dx) {
        mbar_expect_tx(w_bar, RB_W_BYTES);
        tma_load_3d(smem_u32(w_tile), &tmW, w_bar, 0, h0, 0);
      }
      for (int b = b_lo; b < b_hi; ++b) {
        if (!wait_bounded(empty_bar(stage), phase ^ 1u, &abort_flag, p)) break;
        const uint32_t xs = smem_u32(stage_base + stage * RB_STAGE_BYTES), ds = xs + RB_X_BYTES;
        const int t0 = b * RB_TB;
        mbar_expect_tx(full_bar(stage), (do_dw ? RB_X_BYTES : 0) + RB_DL_BYTES);
        filled_parity[stage] = (int)phase;
        if (do_dw) {  // x tile: columns h0.. and h0 + 64.. of 128 token rows
          tma_load_3d(xs, &tmX, full_bar(stage), h0, t0, 0);
          tma_load_3d(xs + RB_TB * 128, &tmX, full_bar(stage), h0 + 64, t0, 0);
        }
#pragma unroll
        for (int q = 0; q < 3; ++q) tma_load_3d(ds + q * (RB_TB * 128), &tmDL, full_bar(stage), 0, t0, q);
        if (++stage == RB_STAGES) { stage = 0; phase ^= 1u; }
      }
      // drain: every copy this thread started has landed before exit
      for (int s = 0; s < RB_STAGES; ++s) {
        if (filled_parity[s] < 0) continue;
        const long long t0 = clock64();
        while (!mbar_try_wait(full_bar(s), (uint32_t)filled_parity[s])) {
          if ((unsigned long long)(clock64() - t0) > DRAIN_LIMIT) { set_error(p.err, DEV_TIMEOUT); break; }
        }
      }
      if (do_dx) {
        const long long t0 = clock64();
        while (!mbar_try_wait(w_bar, 0)) {
          if ((unsigned long long)(clock64() - t0) > DRAIN_LIMIT) { set_error(p.err, DEV_TIMEOUT); break; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // dW: M = 128 columns of H (x^T, M-contiguous), N = 192 (the three dl
      // parts, N-contiguous), K = 128 tokens per block
      constexpr uint32_t IDW = instr_desc(128, 192, true, true);
      // dx: M = 128 tokens (dl part, K-major), N = 128 columns of H (W_r slice,
      // K-major), K = 64 experts per part
      constexpr uint32_t IDX = instr_desc(128, 128, false, false);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = !do_dx || wait_bounded(w_bar, 0, &abort_flag, p);
      bool issued = false;
      tc_fence_after();
      const uint32_t wt = smem_u32(w_tile);
      int i = 0;
      for (int b = b_lo; ok && b < b_hi; ++b, ++i) {
        const int acc = i & 1;
        if (do_dx && !wait_bounded(acce_bar(acc), (((uint32_t)i >> 1) & 1u) ^ 1u, &abort_flag, p)) { ok = false; break; }
        if (!wait_bounded(full_bar(stage), phase, &abort_flag, p)) { ok = false; break; }
        tc_fence_after();
        const uint32_t xs = smem_u32(stage_base + stage * RB_STAGE_BYTES), ds = xs + RB_X_BYTES;
        if (do_dw) {
#pragma unroll
          for (int k = 0; k < RB_TB / 16; ++k) {
            // 16 token rows per step; 64-wide atoms one 16 KB box apart
            const uint64_t adesc = smem_desc(xs + k * 16 * 128, RB_TB * 128, 1024);
            const uint64_t bdesc = smem_desc(ds + k * 16 * 128, RB_TB * 128, 1024);
            tc_mma(tmem_base, adesc, bdesc, IDW, (b > b_lo || k > 0) ? 1u : 0u);
          }
        }
        if (do_dx) {
          const uint32_t d = tmem_base + 256 + acc * 128;
#pragma unroll
          for (int q = 0; q < 3; ++q)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t adesc = smem_desc(ds + q * (RB_TB * 128) + k * 32, 16, 1024);
              const uint64_t bdesc = smem_desc(wt + k * 32, 16, 1024);
              tc_mma(d, adesc, bdesc, IDX, (q > 0 || k > 0) ? 1u : 0u);
            }
        }
        issued = true;
        tc_commit(empty_bar(stage));
        if (do_dx) tc_commit(accf_bar(acc));
        if (++stage == RB_STAGES) { stage = 0; phase ^= 1u; }
      }
      if (ok && do_dw) tc_commit(dw_bar);
      if (issued) {
        tc_commit(drain_bar);
        const long long t0 = clock64();
        while (!mbar_try_wait(drain_bar, 0)) {
          if ((unsigned long long)(clock64() - t0) > DRAIN_LIMIT) { set_error(p.err, DEV_TIMEOUT); break; }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // group eg (warps 2-5 or 6-9) takes the blocks of accumulator eg
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int eg = (warp - 2) >> 2;
    float* stg_g = epi_stage + eg * 4 * 32 * STG_LD;
    if (do_dx) {
      for (int b = b_lo + eg, i = eg; b < b_hi; b += 2, i += 2) {
        const int acc = eg;
        if (!wait_bounded(accf_bar(acc), ((uint32_t)i >> 1) & 1u, &abort_flag, p)) break;
        tc_fence_after();
        TileInfo ti;
        ti.g = 0;
        ti.row0 = b * RB_TB;
        ti.rows = min(RB_TB, p.M - ti.row0);
        ti.n0 = h0;
        const uint32_t tbase = tmem_base + 256 + acc * 128 + ((uint32_t)(q * 32) << 16);
        epi_bf16<RB_HS>(p, tbase, ti, stg_g, q, lane);
        tc_fence_before();
        mbar_arrive(acce_bar(acc));
      }
    }
    if (do_dw && wait_bounded(dw_bar, 0, &abort_flag, p)) {
      // TMEM lane = column h of W_r; dW[h, e] = hi + mid + lo (fixed order);
      // group eg writes experts 32 eg .. 32 eg + 31; a CTA without tokens
      // writes zeros
      tc_fence_after();
      const bool empty = b_hi <= b_lo;
      const int h = h0 + q * 32 + lane;
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
      float* out = part + ((long long)split * p.N + h) * E;
      {
        const int c = eg;
        float hi[32], mid[32], lo[32];
        if (!empty) {
          tmem_ld32(tb + c * 32, hi);
          tmem_ld32(tb + 64 + c * 32, mid);
          tmem_ld32(tb + 128 + c * 32, lo);
        }
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          if (c * 32 + j < E) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!empty)
              v = make_float4(hi[j] + mid[j] + lo[j], hi[j + 1] + mid[j + 1] + lo[j + 1],
                              hi[j + 2] + mid[j + 2] + lo[j + 2], hi[j + 3] + mid[j + 3] + lo[j + 3]);
            *reinterpret_cast<float4*>(out + c * 32 + j) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512u));
  }
}

}  // namespace tc

// act = silu(xs Wg[e]) * (xs Wu[e]);  h = act Wd[e]^T   (bf16, grouped by cu)
size_t expert_ffn_ws_bytes() { return tc::SPLIT_PART_BYTES + (size_t)tc::SPLIT_COUNTERS * sizeof(int); }

int launch_expert_ffn_tc(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                         const void* wd, int E, int H, int Hp, void* act, void* gu, void* h, cudaStream_t s,
                         const int32_t* gather, int gather_n, void* ws, size_t ws_bytes) {
  using namespace tc;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  CUtensorMap mA, mG, mU, mA2, mD;
  // gathered rows: the A map is not read (the gather warps copy rows themselves)
  if (!map_2d_as_3d(&mA, xs, H, gather ? gather_n : rows, BK, BM)) return MOE_ERR_CUDA;
  if (!map_3d(&mG, wg, Hp, H, E, 64, BK)) return MOE_ERR_CUDA;
  if (!map_3d(&mU, wu, Hp, H, E, 64, BK)) return MOE_ERR_CUDA;
  if (!map_2d_as_3d(&mA2, act, Hp, rows, BK, BM)) return MOE_ERR_CUDA;
  // down-projection B: 128-row halves, one per CTA of a pair
  if (!map_3d(&mD, wd, Hp, H, E, BK, PAIR_BN / 2)) return MOE_ERR_CUDA;
  Params p1 = params(cu, E, rows, Hp, H, act, Hp, nullptr);
  p1.aux = gu;  // nullable: g and u kept for the backward
  p1.ld_aux = 2LL * Hp;
  p1.vec32 = (reinterpret_cast<uintptr_t>(act) | reinterpret_cast<uintptr_t>(gu)) % 32 == 0;
  Params p2 = params(cu, E, rows, H, Hp, h, H, nullptr);
  // CTA pairs: 256-row tiles, each CTA staging half of the B columns.  With
  // the workspace, the gate/up kernel zeroes the counters with which the
  // down projection's split tiles (if its last round has any) meet.
  if (ws && ws_bytes >= expert_ffn_ws_bytes()) {
    p2.split_ws = static_cast<float*>(ws);
    p2.split_cnt = reinterpret_cast<int*>(static_cast<char*>(ws) + SPLIT_PART_BYTES);
    p1.zero_cnt = p2.split_cnt;
    p1.zero_n = SPLIT_COUNTERS;
  }
  const long long ptiles = (rows + 2 * BM - 1) / (2 * BM) + E;
  int st;
  if (gather) {
    p1.gather = gather;
    p1.gather_src = static_cast<const bf16*>(xs);
    p1.gather_n = gather_n;
    st = launch_pair<EPI_SWIGLU, true>(mA, mG, mU, p1, ptiles * ((Hp + 127) / 128), s);
  } else {
    st = launch_pair<EPI_SWIGLU>(mA, mG, mU, p1, ptiles * ((Hp + 127) / 128), s);
  }
  if (st != MOE_OK) return st;
  return launch_pair<EPI_BF16>(mA2, mD, mD, p2, ptiles * ((H + 255) / 256), s);
}

// Backward of the grouped SwiGLU FFN (bf16, tcgen05), given dh [rows, H]:
//   dgu = [dg | du] from da = dh Wd[e] and the saved [g | u]      (per row group)
//   dxs = dg Wg[e]^T + du Wu[e]^T                                  (K = 2 H', B switches at H')
//   dWd[e] = dh_e^T act_e,  dWg[e] = xs_e^T dg_e,  dWu[e] = xs_e^T du_e   (grouped K, fp32)
int launch_expert_ffn_bwd_tc(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                             const void* wd, int E, int H, int Hp, const void* gu, const void* act, const void* dh,
                             void* dgu, void* dxs, float* dwg, float* dwu, float* dwd, cudaStream_t s) {
  using namespace tc;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  // da and dxs on CTA pairs (256-row tiles)
  const long long ptiles = (rows + 2 * BM - 1) / (2 * BM) + E;
  int st;
  {  // dgu: A = dh (K-major, K = H), B = Wd[e] read as [K = H, N = H'] (MN-major)
    CUtensorMap mA, mB;
    if (!map_2d_as_3d(&mA, dh, H, rows, BK, BM)) return MOE_ERR_CUDA;
    if (!map_3d(&mB, wd, Hp, H, E, 64, BK)) return MOE_ERR_CUDA;
    Params p = params(cu, E, rows, Hp, H, dgu, 2LL * Hp, nullptr);
    p.aux = const_cast<void*>(gu);
    p.ld_aux = 2LL * Hp;
    // rows of [g | u] and [dg | du] are 4 H' bytes apart (H' % 64 == 0)
    p.vec32 = (reinterpret_cast<uintptr_t>(gu) | reinterpret_cast<uintptr_t>(dgu)) % 32 == 0;
    st = launch_pair<EPI_SWIGLU_BWD>(mA, mB, mB, p, ptiles * ((Hp + 255) / 256), s);
    if (st != MOE_OK) return st;
  }
  if (dxs) {  // A = dgu (K-major, K = 2H'), B = Wg[e] then Wu[e], each [N = H rows, K = H'] (K-major)
    CUtensorMap mA, mG, mU;
    if (!map_2d_as_3d(&mA, dgu, 2LL * Hp, rows, BK, BM)) return MOE_ERR_CUDA;
    if (!map_3d(&mG, wg, Hp, H, E, BK, PAIR_BN / 2)) return MOE_ERR_CUDA;
    if (!map_3d(&mU, wu, Hp, H, E, BK, PAIR_BN / 2)) return MOE_ERR_CUDA;
    Params p = params(cu, E, rows, H, 2 * Hp, dxs, H, nullptr);
    p.kcat = Hp;
    st = launch_pair<EPI_BF16>(mA, mG, mU, p, ptiles * ((H + 255) / 256), s);
    if (st != MOE_OK) return st;
  }
  // weight gradients: M = H (A = an [rows, H] matrix read transposed, MN-major),
  // N = H' (B = an [rows, .] matrix, MN-major), K = the rows of each expert
  // (CTA pairs: 256 x 256 output tiles)
  const long long gk_tiles = (long long)E * ((H + 2 * BM - 1) / (2 * BM)) * ((Hp + 255) / 256);
  auto wgrad = [&](const void* a_rows, const void* b_rows, long long b_ld, int b_off, float* out) {
    CUtensorMap mA, mB;
    if (!map_2d_as_3d(&mA, a_rows, H, rows, 64, BK)) return (int)MOE_ERR_CUDA;
    if (!map_2d_as_3d(&mB, b_rows, b_ld, rows, 64, BK)) return (int)MOE_ERR_CUDA;
    Params p = params(cu, E, H, Hp, rows, out, Hp, nullptr);
    p.b_col_off = b_off;
    // fp32 [E][H][H'] output as a map of [32 x 32] store boxes (the C ABI
    // guarantees a 16-byte aligned base; H' % 64 == 0 makes every row a
    // 16-byte multiple)
    CUtensorMap mO;
    cuuint64_t dims[3] = {(cuuint64_t)Hp, (cuuint64_t)H, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)Hp * 4, (cuuint64_t)H * Hp * 4};
    cuuint32_t box[3] = {32, 32, 1};
    if (!make_map(&mO, out, 3, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32)) return (int)MOE_ERR_CUDA;
    return launch_pair<EPI_F32_GK>(mA, mB, mO, p, gk_tiles, s);
  };
  if (dwd && (st = wgrad(dh, act, Hp, 0, dwd)) != MOE_OK) return st;
  if (dwg && (st = wgrad(xs, dgu, 2LL * Hp, 0, dwg)) != MOE_OK) return st;
  if (dwu && (st = wgrad(xs, dgu, 2LL * Hp, Hp, dwu)) != MOE_OK) return st;
  return MOE_OK;
}

int launch_wait_probe(unsigned long long wait_cycles, cudaStream_t s) {
  tc::Params p = tc::params(nullptr, 1, 0, 0, 0, nullptr, 0, nullptr);
  p.wait_limit = wait_cycles;
  tc::wait_probe_kernel<<<1, 32, 0, s>>>(p);
  return launch_status();
}

// N tile of the router GEMM: the whole expert row up to 128 experts; beyond,
// 192-wide tiles when they cover E exactly (E = 384: two tiles, no padded
// columns), else 256
static int router_bn(int E) { return E <= 64 ? 64 : E <= 128 ? 128 : E % 192 == 0 ? 192 : 256; }

// Splits of H for the router GEMM: a CTA streams x from DRAM at a limited rate,
// so when the token tiles alone would occupy fewer than about two thirds of the
// SMs the reduction over H is split (fp32 partials summed by the softmax pass).
int router_tc_splits(int T, int H, int E) {
  const long long tiles = ((T + tc::BM - 1) / tc::BM) * (long long)((E + router_bn(E) - 1) / router_bn(E));
  const long long sms = sm_count();
  if (3 * tiles >= 2 * sms) return 1;
  long long s = sms / (tiles > 0 ? tiles : 1);
  // every split needs at least one stage of K (64 * k sub-blocks per stage)
  const int ksub = E <= 64 ? 4 : E <= 128 ? 2 : 1;
  const long long kb = (H + tc::BK * ksub - 1) / (tc::BK * ksub);
  if (s > kb) s = kb;
  if (s > 8) s = 8;
  return s < 1 ? 1 : (int)s;
}

// out = x W_r (+ bias when S == 1): bf16 inputs, fp32 [T,E]; with S > 1, out
// holds S partial sums [S][T][E] over consecutive slices of H (no bias).
// E % 8 == 0, H % 8 == 0.  With idx given (S == 1 and E <= 64 only) the
// epilogue also writes the top-K experts and gates.
int launch_router_tc(const void* x, const void* w, const float* bias, const float* sel_bias, bool renorm, int T,
                     int H, int E, float* out, int S, int K, int32_t* idx, float* gate, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB;
  if (!map_2d_as_3d(&mA, x, H, T, BK, BM)) return MOE_ERR_CUDA;
  if (!map_3d(&mB, w, E, H, 1, 64, BK)) return MOE_ERR_CUDA;
  Params p = params(nullptr, 1, T, E, H, out, E, S > 1 ? nullptr : bias);
  p.ksplit = S;
  p.part_stride = (long long)T * E;
  const long long tiles = (T + BM - 1) / BM * (long long)S;
  if (idx) {  // S == 1, E <= 64: logits, softmax and top-k in the GEMM's epilogue
    p.topk = K;
    p.topk_idx = idx;
    p.topk_gate = gate;
    p.sel_bias = sel_bias;
    p.renorm = renorm ? 1 : 0;
    return launch<EPI_ROUTER, false, true, 64, 2, 4, 4, 4>(mA, mB, mB, p, tiles, s);
  }
  // x is streamed from DRAM once: stages of 4 (2) consecutive 64-wide K slices
  // request 512 (256) contiguous bytes of every row at a time
  if (E <= 64) return launch<EPI_F32_BIAS, false, true, 64, 2, 4, 4, 4>(mA, mB, mB, p, tiles, s);
  if (E <= 128) return launch<EPI_F32_BIAS, false, true, 128, 3, 2, 2, 2>(mA, mB, mB, p, tiles, s);
  if (S == 1) {
    // CTA pairs: 256 tokens x 256 experts per tile (columns past E read as
    // zeros and are not stored)
    const long long ptiles = (T + 2 * BM - 1) / (2 * BM) * ((E + PAIR_BN - 1) / PAIR_BN);
    return launch_pair<EPI_F32_BIAS>(mA, mB, mB, p, ptiles, s);
  }
  if (E % 192 == 0) return launch<EPI_F32_BIAS, false, true, 192, 5, 1, 1>(mA, mB, mB, p, tiles * (E / 192), s);
  return launch<EPI_F32_BIAS, false, true, 256, 4, 1, 1>(mA, mB, mB, p, tiles * ((E + 255) / 256), s);
}

// Split count for the router weight gradient on tensor cores: the (h tile x
// token split) work items run in ceil(items / SMs) rounds, and a round costs a
// fixed part (the first stage's latency, the fp32 partial tile's epilogue:
// about 12 K blocks' worth) plus its K blocks; the split count (up to 64, each
// split at least one 64-token block) with the smallest estimate wins, the
// smaller count on ties.
int router_dw_tc_splits(int T, int H, int E) {
  const long long tiles = ((H + tc::BM - 1) / tc::BM) * (long long)(E <= 64 ? 1 : (E + 127) / 128);
  const long long kb = (T + tc::BK - 1) / tc::BK;
  const long long sms = sm_count();
  constexpr long long FIXED = 12;
  long long best = 1, best_cost = -1;
  for (long long s = 1; s <= 64 && s <= kb; ++s) {
    const long long rounds = (tiles * s + sms - 1) / sms;
    const long long cost = rounds * (FIXED + (kb + s - 1) / s);
    if (best_cost < 0 || cost < best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  return (int)best;
}

// part[s][h][e] = sum over the tokens of split s of x[t,h] (hi+mid+lo)[t,e]
// x [T,H] bf16; dl3 [3,T,E] bf16 (the exact three-part split of the fp32 dl)
int launch_router_dw_tc(const void* x, const void* dl3, int T, int H, int E, float* part, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB;
  if (!map_2d_as_3d(&mA, x, H, T, 64, BK)) return MOE_ERR_CUDA;  // A = x^T, MN-major boxes [64 t x 64 h]
  if (!map_3d(&mB, dl3, E, T, 3, 64, BK)) return MOE_ERR_CUDA;
  const int S = router_dw_tc_splits(T, H, E);
  Params p = params(nullptr, 1, H, E, T, part, E, nullptr);
  p.ksplit = S;
  p.part_stride = (long long)H * E;
  const long long mtiles = (H + BM - 1) / BM;
  if (E <= 64) return launch<EPI_F32_BIAS, true, true, 64, 5, 1, 3>(mA, mB, mB, p, mtiles * S, s);
  return launch<EPI_F32_BIAS, true, true, 128, 3, 1, 3>(mA, mB, mB, p, mtiles * ((E + 127) / 128) * S, s);
}

// dx[t,h] (+)= sum_e (hi+mid+lo)[t,e] W_r[h,e]; dx bf16 [T,H], H % 64 == 0
// One-pass router backward (dW partials and dx) for 32..64 experts: one CTA per
// (128-column slice of H, range of token blocks), the token ranges sized so
// that all CTAs run in one wave.
bool router_bwd_tc_applies(int H, int E) { return E % 8 == 0 && E > 16 && E <= 64 && H % tc::RB_HS == 0; }

int router_bwd_tc_splits(int T, int H, int E) {
  const long long n_slices = H / tc::RB_HS, n_blocks = (T + tc::RB_TB - 1) / tc::RB_TB;
  long long sp = sm_count() / (n_slices > 0 ? n_slices : 1);
  if (sp > n_blocks) sp = n_blocks;
  if (sp > 64) sp = 64;
  return sp < 1 ? 1 : (int)sp;
}

int launch_router_bwd_tc(const void* x, const void* dl3, const void* w, int T, int H, int E, float* part, bool write,
                         void* dx, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mX, mDL, mW;
  if (!map_3d(&mDL, dl3, E, T, 3, 64, RB_TB)) return MOE_ERR_CUDA;
  if (part) {
    if (!map_2d_as_3d(&mX, x, H, T, 64, RB_TB)) return MOE_ERR_CUDA;
  } else {
    mX = mDL;  // not read
  }
  if (dx) {
    if (!map_2d_as_3d(&mW, w, E, H, 64, RB_HS)) return MOE_ERR_CUDA;
  } else {
    mW = mDL;  // not read
  }
  Params p = params(nullptr, 1, T, H, E, dx, H, nullptr);
  p.accumulate = write ? 0 : 1;
  const int n_slices = H / RB_HS, n_blocks = (T + RB_TB - 1) / RB_TB, splits = router_bwd_tc_splits(T, H, E);
  if (cudaFuncSetAttribute(router_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RB_SMEM) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  router_bwd_tc_kernel<<<n_slices * splits, RB_THREADS, RB_SMEM, s>>>(mX, mDL, mW, p, n_slices, splits, n_blocks,
                                                                      part, E);
  return launch_status();
}

int launch_router_dx_tc(const void* dl3, const void* w, int T, int H, int E, bool write, void* dx, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB;
  if (!map_3d(&mA, dl3, E, T, 3, BK, BM)) return MOE_ERR_CUDA;
  if (!map_2d_as_3d(&mB, w, E, H, BK, 256)) return MOE_ERR_CUDA;
  Params p = params(nullptr, 1, T, H, E, dx, H, nullptr);
  p.accumulate = write ? 0 : 1;
  const long long tiles = ((T + BM - 1) / BM) * (long long)((H + 255) / 256);
  return launch<EPI_BF16, false, false, 256, 2, 3, 1>(mA, mB, mB, p, tiles, s);
}

}  // namespace moe
