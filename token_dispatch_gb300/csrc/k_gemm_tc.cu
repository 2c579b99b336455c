// Grouped bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Serves the three dense contractions of the layer:
//   * gate/up projection of every expert with SwiGLU fused in the epilogue
//       act[r, n] = silu(sum_k xs[r,k] Wg[e][k,n]) * (sum_k xs[r,k] Wu[e][k,n])
//   * down projection  h[r, n] = sum_k act[r,k] Wd[e][n,k]
//   * router GEMM      logits[t, e] = sum_h x[t,h] W_r[h,e] + bias[e]   (fp32 out)
// The weights are one contiguous [E, H, H'] tensor per projection and experts are
// addressed by their index (MoonEP page, "Step-by-step"); the rows of expert e
// are [cu[e], cu[e+1]) of the expert-sorted activation buffer, read on the device
// (no host synchronisation).
//
// Design (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer: A tile 128x64 (K-major) and B tile (MN-major
//               [64 K x BN] chunks for W[e] stored [H, H'] or W_r [H, E];
//               K-major [BN x 64 K] for Wd[e] stored [H, H']) into a STAGES-deep
//               shared-memory ring, 128-byte swizzled.
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16) from one
//               thread into one of two fp32 TMEM accumulators, committing each
//               stage back to the producer and each finished tile to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31 = tile rows), apply SwiGLU / bias, convert, store;
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
constexpr int A_STAGE_BYTES = BM * BK * 2;

enum Epi { EPI_SWIGLU = 0, EPI_BF16 = 1, EPI_F32_BIAS = 2 };

struct Params {
  const int32_t* cu;  // nullptr: one group of M rows
  int G, M, N, K;     // N = output columns, K = reduction length
  void* out;
  long long ldo;
  const float* bias;
  unsigned* err;
  unsigned long long wait_limit;  // clock64 cycles
};

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

// Instruction descriptor, kind::f16: D fp32, A = B = bf16, A K-major.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

template <int BN, int EPI>
struct Cfg {
  static constexpr int B_STAGE_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
  static constexpr int OUT_BN = (EPI == EPI_SWIGLU) ? BN / 2 : BN;  // output columns per tile
  static constexpr int TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                   : (2 * BN <= 256) ? 256 : 512;
};

struct TileInfo {
  int g, row0, rows, n0;
};

// Tile t -> (group, rows, first output column).  mt_pre[g] = m-tiles before g.
__device__ __forceinline__ TileInfo decode(int t, const int* mt_pre, int G, int n_tiles, const Params& p,
                                           int out_bn) {
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
  const int beg = p.cu ? p.cu[g] : 0;
  const int end = p.cu ? p.cu[g + 1] : p.M;
  TileInfo ti;
  ti.g = g;
  ti.row0 = beg + m * BM;
  ti.rows = min(BM, end - ti.row0);
  ti.n0 = n * out_bn;
  return ti;
}

template <int EPI, bool B_MN, int BN, int STAGES>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmB2, const Params p) {
  using C = Cfg<BN, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;
  __shared__ int mt_pre[1025];
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
    if (EPI == EPI_SWIGLU) prefetch_tmap(&tmB2);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_slot)),
                 "r"((uint32_t)C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == 2) {
    // m-tile prefix over groups: each lane owns a contiguous run of groups
    const int per = (G + 31) / 32;
    int sum = 0;
    for (int g = lane * per; g < min(G, lane * per + per); ++g) {
      int rows = p.cu ? max(0, p.cu[g + 1] - p.cu[g]) : p.M;
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
      int rows = p.cu ? max(0, p.cu[g + 1] - p.cu[g]) : p.M;
      run += (rows + BM - 1) / BM;
    }
    if (lane == 0 && p.cu && (p.cu[0] != 0 || p.cu[G] != p.M)) set_error(p.err, DEV_BOUNDS);
    if (lane == 31) {
      mt_pre[G] = incl;
      total_tiles_s = incl * n_tiles;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_slot;
  const int total_tiles = total_tiles_s;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int filled_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) filled_parity[s] = -1;
      const int KB = (p.K + BK - 1) / BK;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        const TileInfo ti = decode(t, mt_pre, G, n_tiles, p, C::OUT_BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_bounded(empty_bar(stage), phase ^ 1u, &abort_flag, p)) { ok = false; break; }
          const uint32_t a_dst = smem_u32(stage_base + stage * C::STAGE_BYTES);
          const uint32_t b_dst = a_dst + A_STAGE_BYTES;
          mbar_expect_tx(full_bar(stage), C::STAGE_BYTES);
          filled_parity[stage] = (int)phase;
          tma_load_2d(a_dst, &tmA, full_bar(stage), kb * BK, ti.row0);
          if (EPI == EPI_SWIGLU) {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c) {
              const CUtensorMap* m = (c < BN / 128) ? &tmB : &tmB2;
              const int col = ti.n0 + (c % (BN / 128)) * 64;
              tma_load_3d(b_dst + c * (64 * BK * 2), m, full_bar(stage), col, kb * BK, ti.g);
            }
          } else if (B_MN) {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_3d(b_dst + c * (64 * BK * 2), &tmB, full_bar(stage), ti.n0 + c * 64, kb * BK, ti.g);
          } else {
            tma_load_3d(b_dst, &tmB, full_bar(stage), kb * BK, ti.n0, ti.g);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // drain: every stage this thread filled must have landed before exit
      for (int s = 0; s < STAGES; ++s) {
        if (filled_parity[s] < 0) continue;
        const long long t0 = clock64();
        while (!mbar_try_wait(full_bar(s), (uint32_t)filled_parity[s])) {
          if ((unsigned long long)(clock64() - t0) > p.wait_limit) { set_error(p.err, DEV_TIMEOUT); break; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = instr_desc(BM, BN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      const int KB = (p.K + BK - 1) / BK;
      bool ok = true;
      bool issued = false;
      int i = 0;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, ++i) {
        const int acc = i & 1;
        if (!wait_bounded(acce_bar(acc), (((uint32_t)i >> 1) & 1u) ^ 1u, &abort_flag, p)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_bounded(full_bar(stage), phase, &abort_flag, p)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stage_base + stage * C::STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t adesc = smem_desc(a_addr + k * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? smem_desc(b_addr + k * 16 * 128, 64 * BK * 2, 1024)
                                        : smem_desc(b_addr + k * 32, 16, 1024);
            tc_mma(d_tmem, adesc, bdesc, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
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
          if ((unsigned long long)(clock64() - t0) > p.wait_limit) { set_error(p.err, DEV_TIMEOUT); break; }
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
      const TileInfo ti = decode(t, mt_pre, G, n_tiles, p, C::OUT_BN);
      const long long grow = (long long)ti.row0 + r_local;
      const bool row_ok = r_local < ti.rows && grow >= 0 && grow < p.M;
      const uint32_t tbase = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
      if (EPI == EPI_SWIGLU) {
        bf16* out = static_cast<bf16*>(p.out);
#pragma unroll 1
        for (int c = 0; c < C::OUT_BN / 32; ++c) {
          float gv[32], uv[32];
          tmem_ld32(tbase + c * 32, gv);
          tmem_ld32(tbase + C::OUT_BN + c * 32, uv);
          const int col = ti.n0 + c * 32;
          if (row_ok && col < p.N) {
            uint4 pk[4];
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float a0 = gv[2 * j] / (1.0f + __expf(-gv[2 * j])) * uv[2 * j];
              float a1 = gv[2 * j + 1] / (1.0f + __expf(-gv[2 * j + 1])) * uv[2 * j + 1];
              h2[j] = __floats2bfloat162_rn(a0, a1);
            }
            uint4* dst = reinterpret_cast<uint4*>(out + grow * p.ldo + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = pk[j];
          }
        }
      } else if (EPI == EPI_BF16) {
        bf16* out = static_cast<bf16*>(p.out);
#pragma unroll 1
        for (int c = 0; c < C::OUT_BN / 32; ++c) {
          float v[32];
          tmem_ld32(tbase + c * 32, v);
          const int col = ti.n0 + c * 32;
          if (row_ok && col < p.N) {
            uint4 pk[4];
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
            for (int j = 0; j < 16; ++j) h2[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
            uint4* dst = reinterpret_cast<uint4*>(out + grow * p.ldo + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = pk[j];
          }
        }
      } else {
        float* out = static_cast<float*>(p.out);
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
              const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

unsigned long long g_wait_limit = 4000000000ull;  // ~2 s at 2 GHz

template <int EPI, bool B_MN, int BN, int STAGES>
int launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2, const Params& p,
           long long tiles_upper, cudaStream_t s) {
  using C = Cfg<BN, EPI>;
  const size_t smem = (size_t)STAGES * C::STAGE_BYTES + (2 * STAGES + 5) * 8 + 1024;
  auto k = tc_gemm_kernel<EPI, B_MN, BN, STAGES>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  long long grid = sm_count();
  if (tiles_upper < grid) grid = tiles_upper;
  if (grid < 1) return MOE_OK;
  k<<<(unsigned)grid, NUM_THREADS, smem, s>>>(a, b, b2, p);
  return launch_status();
}

}  // namespace tc

// act = silu(xs Wg[e]) * (xs Wu[e]);  h = act Wd[e]^T   (bf16, grouped by cu)
int launch_expert_ffn_tc(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                         const void* wd, int E, int H, int Hp, void* act, void* h, cudaStream_t s) {
  using namespace tc;
  if (E > 1024) return MOE_ERR_UNSUPPORTED;
  CUtensorMap mA, mG, mU, mA2, mD;
  {
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t str[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {BK, BM};
    if (!make_map(&mA, xs, 2, dims, str, box)) return MOE_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)Hp, (cuuint64_t)H, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)Hp * 2, (cuuint64_t)H * Hp * 2};
    cuuint32_t box[3] = {64, BK, 1};
    if (!make_map(&mG, wg, 3, dims, str, box)) return MOE_ERR_CUDA;
    if (!make_map(&mU, wu, 3, dims, str, box)) return MOE_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)Hp, (cuuint64_t)rows};
    cuuint64_t str[1] = {(cuuint64_t)Hp * 2};
    cuuint32_t box[2] = {BK, BM};
    if (!make_map(&mA2, act, 2, dims, str, box)) return MOE_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)Hp, (cuuint64_t)H, (cuuint64_t)E};
    cuuint64_t str[2] = {(cuuint64_t)Hp * 2, (cuuint64_t)H * Hp * 2};
    cuuint32_t box[3] = {BK, 256, 1};
    if (!make_map(&mD, wd, 3, dims, str, box)) return MOE_ERR_CUDA;
  }
  const long long mtiles = (rows + BM - 1) / BM + E;
  Params p1{cu, E, rows, Hp, H, act, Hp, nullptr, device_error_word(), g_wait_limit};
  int st = launch<EPI_SWIGLU, true, 256, 4>(mA, mG, mU, p1, mtiles * ((Hp + 127) / 128), s);
  if (st != MOE_OK) return st;
  Params p2{cu, E, rows, H, Hp, h, H, nullptr, device_error_word(), g_wait_limit};
  return launch<EPI_BF16, false, 256, 4>(mA2, mD, mD, p2, mtiles * ((H + 255) / 256), s);
}

// logits = x W_r + bias  (bf16 inputs, fp32 out); E % 8 == 0, H % 8 == 0
int launch_router_tc(const void* x, const void* w, const float* bias, int T, int H, int E, float* logits,
                     cudaStream_t s) {
  using namespace tc;
  CUtensorMap mA, mB;
  {
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t str[1] = {(cuuint64_t)H * 2};
    cuuint32_t box[2] = {BK, BM};
    if (!make_map(&mA, x, 2, dims, str, box)) return MOE_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)E, (cuuint64_t)H, 1};
    cuuint64_t str[2] = {(cuuint64_t)E * 2, (cuuint64_t)H * E * 2};
    cuuint32_t box[3] = {64, BK, 1};
    if (!make_map(&mB, w, 3, dims, str, box)) return MOE_ERR_CUDA;
  }
  Params p{nullptr, 1, T, E, H, logits, E, bias, device_error_word(), g_wait_limit};
  const long long mtiles = (T + BM - 1) / BM;
  if (E <= 64) return launch<EPI_F32_BIAS, true, 64, 8>(mA, mB, mB, p, mtiles, s);
  if (E <= 128) return launch<EPI_F32_BIAS, true, 128, 6>(mA, mB, mB, p, mtiles, s);
  return launch<EPI_F32_BIAS, true, 256, 4>(mA, mB, mB, p, mtiles * ((E + 255) / 256), s);
}

}  // namespace moe
