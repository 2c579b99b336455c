// Router forward for few experts (E = 8 or 16, bf16) in one launch: logits,
// softmax and top-K gate.
//
// The routing/gating kernel of the MoE/MoD framework page ("What's in the box":
// softmax over experts and top-k selection in one launch) runs here on top of
// the logits GEMM itself.  With E <= 16 the GEMM is a pure stream of x from
// HBM (16 or 32 flops per byte), so the design is about bytes in flight, not
// about tensor-core rate:
//   * x goes from global memory straight into registers (128-bit loads, 16
//     per lane in flight: 2 to 16 token blocks ahead depending on the width
//     of the warp's slice of H; each register is refilled as soon as it is
//     consumed); nothing of x passes through shared memory;
//   * the products run on the warp-level bf16 MMA (m16n8k16, fp32
//     accumulate) with W_r^T as the 16-row A operand (experts) and x^T as B
//     (8 tokens), so one 128-bit load of x feeds two MMAs;
//   * W_r sits in shared memory once per persistent CTA, pre-arranged in the
//     MMA's A-fragment order (one conflict-free 128-bit load per lane per 32
//     values of H); each thread loads 8 whole rows of W_r and writes their
//     fragments with an in-register 8 x 8 transpose (byte permutes), so the
//     staging costs a few instructions per 16 bytes instead of one store per
//     element;
//   * the 16 warps of a CTA own 16 consecutive slices of H; their partial
//     logits meet in shared memory in warp order (fixed: the same bits every
//     run) and get the bias; the E threads of a token then take the softmax
//     and the K winners (value descending, lowest expert first on ties) with
//     butterfly shuffles.  The partial
//     tile is double-buffered, so one CTA barrier per block of 8 tokens
//     suffices, and the loads already in flight keep HBM busy across it.
//
// The k index inside each 32-wide chunk of H is permuted: lane (g, c) of the
// MMA holds k = 2c, 2c+1, 2c+8, 2c+9 of A and B alike, and MMA j of a chunk
// maps them to h = 8c + 4j + {0, 1, 2, 3}.  A and B use the same map, so the
// sum over k is unchanged and each lane's x values are 8 contiguous bf16.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int RS_WARPS = 16;   // warps per CTA = slices of H
constexpr int RS_THREADS = RS_WARPS * 32;
constexpr int RS_TOK = 8;      // tokens per n-tile (the MMA's N)
constexpr int RS_RED_LD = 20;  // row stride of the partial-logit tile (banks)

// 16 bytes of x into v when ok; otherwise v keeps what it held.  The load is
// predicated (no select on its result), so nothing waits for it until the
// MMA that consumes v.
__device__ __forceinline__ void ldg_stream(uint4& v, const bf16* p, bool ok) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.b32 q, %4, 0;\n"
      " @q ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%5];\n}"
      : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
      : "r"((int)ok), "l"(p));
}

__device__ __forceinline__ unsigned word4(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// D += A B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Token blocks of 8 * NT tokens (NT n-tiles of the MMA) and D blocks of loads
// in flight per warp, NT * CH * D <= 16 loads per lane: narrow slices of H
// take bigger blocks, so the per-block barrier and softmax stay small next to
// the bytes a block streams.
template <int CH, bool E16>
struct StreamCfg {
  static constexpr int NT = CH >= 6 ? 2 : CH >= 5 ? 1 : (8 / CH < (E16 ? 4 : 8) ? 8 / CH : (E16 ? 4 : 8));
  static constexpr int D = NT * CH > 8 ? 1 : (16 / (NT * CH) < 2 ? 2 : 16 / (NT * CH));
  static constexpr int TOK = RS_TOK * NT;                       // tokens per block
  static constexpr int RED_FLOATS = 2 * RS_WARPS * TOK * RS_RED_LD;  // double-buffered partials
};

// CH: 32-wide chunks of H per warp (H = 512 * CH).  E16: experts 8..15 exist
// (A rows g + 8); otherwise those rows are zero.
template <int CH, bool E16>
__global__ void __launch_bounds__(RS_THREADS, 1)
router_stream_kernel(const bf16* __restrict__ x, const bf16* __restrict__ w, const float* __restrict__ bias,
                     const float* __restrict__ sel_bias, int renorm, int T, int H, int E, int K,
                     float* __restrict__ logits, int32_t* __restrict__ idx, float* __restrict__ gate) {
  using C = StreamCfg<CH, E16>;
  constexpr int NF = E16 ? 2 : 1;  // 16-byte fragments per lane per chunk
  constexpr int NT = C::NT, D = C::D, TOK = C::TOK;
  extern __shared__ uint4 smem_dyn[];
  float* red = reinterpret_cast<float*>(smem_dyn);  // [2][RS_WARPS][TOK][RS_RED_LD]
  uint4* wfrag = smem_dyn + C::RED_FLOATS / 4;       // [H/32][32 lanes][NF]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  // CTA b streams the contiguous tokens [tb0, tb1), an even share of T (the
  // last block of a range may be partial), so every SM moves the same bytes
  const int G = gridDim.x;
  const int tb0 = (int)((long long)blockIdx.x * T / G), tb1 = (int)((long long)(blockIdx.x + 1) * T / G);
  const int my_blocks = (tb1 - tb0 + TOK - 1) / TOK;
  const bf16* xw = x + warp * (CH * 32) + 8 * c;  // this lane's columns of every chunk

  // loads of block i of the range into r; rows past the range are not loaded (their
  // MMA columns hold stale values and are never written out)
  auto load_block = [&](uint4 (&r)[NT][CH], int i) {
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      const int tok = tb0 + i * TOK + q * RS_TOK + g;
      const bool ok = i < my_blocks && tok < tb1;
      const bf16* p = xw + (long long)(ok ? tok : 0) * H;
#pragma unroll
      for (int j = 0; j < CH; ++j) ldg_stream(r[q][j], p + j * 32, ok);
    }
  };

  // W_r [H, E] row-major -> A fragments: chunk ch, lane (g', c'), row half q,
  // element j = W_r[ch*32 + 8c' + j][g' + 8q].  Thread u owns the 8
  // consecutive rows 8u .. 8u+7 (128 or 256 contiguous bytes, loaded at once)
  // and transposes each 8 x 8 block of bf16 in registers with byte permutes:
  // word a of the fragment of column g' is (row 2a, row 2a+1) of that column.
  uint4 xr[D][NT][CH] = {};
  {
    const bool has_unit = tid < H / 8;  // H <= 4096: at most one unit per thread
    uint4 wv[NF][8];
    if (has_unit) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int q = 0; q < NF; ++q) wv[q][j] = __ldg(reinterpret_cast<const uint4*>(w + (size_t)(8 * tid + j) * E) + q);
    }
    if (has_unit) {
      const int ch = tid >> 2, cc = tid & 3;
      // two halves (rows 0-3, rows 4-7): 8-byte stores, fewer live registers
#pragma unroll
      for (int q = 0; q < NF; ++q)
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int gg = 0; gg < 8; ++gg) {
            const unsigned sel = (gg & 1) ? 0x7632u : 0x5410u;
            uint2 o;
            o.x = __byte_perm(word4(wv[q][4 * half], gg >> 1), word4(wv[q][4 * half + 1], gg >> 1), sel);
            o.y = __byte_perm(word4(wv[q][4 * half + 2], gg >> 1), word4(wv[q][4 * half + 3], gg >> 1), sel);
            reinterpret_cast<uint2*>(wfrag + (ch * 32 + 4 * gg + cc) * NF + q)[half] = o;
          }
    }
    // the first D blocks of x go out once the fragments are written: issued
    // earlier, the x loads (16 per thread) fill the load queues and the W_r
    // loads wait behind them (measured: 4.5 us of staging instead of 6 us)
    asm volatile("" ::: "memory");
#pragma unroll
    for (int d = 0; d < D; ++d) load_block(xr[d], d);
  }
  __syncthreads();

  const uint4* wl = wfrag + (warp * CH * 32 + lane) * NF;
  // block i of this CTA: multiply the loads in r, refill r with block i + D,
  // then sum the 16 slices (warp order), add the bias and take the softmax /
  // top-K
  auto process = [&](uint4 (&r)[NT][CH], int i) {
    const int buf = i & 1;
    const int nxt = i + D;
    float d[NT][4] = {};
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const uint4 a = wl[j * 32 * NF];
      const uint4 a8 = E16 ? wl[j * 32 * NF + 1] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < NT; ++q) {
        mma_16816(d[q], a.x, a8.x, a.y, a8.y, r[q][j].x, r[q][j].y);
        mma_16816(d[q], a.z, a8.z, a.w, a8.w, r[q][j].z, r[q][j].w);
        const int tok = tb0 + nxt * TOK + q * RS_TOK + g;
        const bool ok = nxt < my_blocks && tok < tb1;
        ldg_stream(r[q][j], xw + (long long)(ok ? tok : 0) * H + j * 32, ok);
      }
    }
    // d0, d1: expert g, tokens 2c, 2c+1 of n-tile q; d2, d3: expert g + 8
    float* rw = red + (buf * RS_WARPS + warp) * TOK * RS_RED_LD;
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      float* rq = rw + q * RS_TOK * RS_RED_LD;
      rq[(2 * c) * RS_RED_LD + g] = d[q][0];
      rq[(2 * c + 1) * RS_RED_LD + g] = d[q][1];
      if (E16) {
        rq[(2 * c) * RS_RED_LD + g + 8] = d[q][2];
        rq[(2 * c + 1) * RS_RED_LD + g + 8] = d[q][3];
      }
    }
    __syncthreads();
    // thread (t, e): the logit of token t, expert e; the E threads of a token
    // are E consecutive lanes, so max, sum and the K arg-max rounds are
    // butterfly shuffles inside the group
    if (tid < TOK * E) {
      const int t = tid / E, e = tid - t * E;
      const float* rt = red + buf * RS_WARPS * TOK * RS_RED_LD + t * RS_RED_LD + e;
      float v = 0.f;
#pragma unroll
      for (int ww = 0; ww < RS_WARPS; ++ww) v += rt[ww * TOK * RS_RED_LD];
      if (bias) v += __ldg(bias + e);
      const int tk = tb0 + i * TOK + t;
      const bool live = tk < tb1;
      if (live) logits[(long long)tk * E + e] = v;
      float m = v;
#pragma unroll
      for (int o = E16 ? 8 : 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float sum = expf(v - m);
#pragma unroll
      for (int o = E16 ? 8 : 4; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      // selection value: the logit, plus the selection-only bias when given
      const float sel = sel_bias ? v + __ldg(sel_bias + e) : v;
      int my_k = -1;
      for (int k = 0; k < K; ++k) {
        float bv = my_k >= 0 ? -INFINITY : sel;
        int be = my_k >= 0 ? 0x7fffffff : e;
#pragma unroll
        for (int o = E16 ? 8 : 4; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
        if (e == be) {
          my_k = k;
          if (live) idx[(long long)tk * K + k] = be;
        }
      }
      // each chosen expert's thread writes its gate: its own probability, over
      // the sum of the chosen probabilities when renormalising
      const float pe = expf(v - m) / sum;
      float norm = 1.f;
      if (renorm) {
        norm = my_k >= 0 ? pe : 0.f;
#pragma unroll
        for (int o = E16 ? 8 : 4; o > 0; o >>= 1) norm += __shfl_xor_sync(0xffffffffu, norm, o);
      }
      if (my_k >= 0 && live) gate[(long long)tk * K + my_k] = pe / norm;
    }
  };

  for (int i = 0; i < my_blocks; i += D) {
#pragma unroll
    for (int d = 0; d < D; ++d)
      if (i + d < my_blocks) process(xr[d], i + d);
  }
}

template <int CH>
int launch_ch(const void* x, const void* w, const float* bias, const float* sel_bias, bool renorm, int T, int H,
              int E, int K, float* logits, int32_t* idx, float* gate, cudaStream_t s) {
  const int tok = E > 8 ? StreamCfg<CH, true>::TOK : StreamCfg<CH, false>::TOK;
  const int red = E > 8 ? StreamCfg<CH, true>::RED_FLOATS : StreamCfg<CH, false>::RED_FLOATS;
  const int nblk = (T + tok - 1) / tok;
  int grid = sm_count();
  if (grid > nblk) grid = nblk;
  const size_t smem = (size_t)red * 4 + (size_t)H * (E > 8 ? 2 : 1) * 16;
  if (E > 8) {
    auto k = router_stream_kernel<CH, true>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    k<<<grid, RS_THREADS, smem, s>>>(static_cast<const bf16*>(x), static_cast<const bf16*>(w), bias, sel_bias,
                                     renorm ? 1 : 0, T, H, E, K, logits, idx, gate);
  } else {
    auto k = router_stream_kernel<CH, false>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    k<<<grid, RS_THREADS, smem, s>>>(static_cast<const bf16*>(x), static_cast<const bf16*>(w), bias, sel_bias,
                                     renorm ? 1 : 0, T, H, E, K, logits, idx, gate);
  }
  return launch_status();
}

}  // namespace

bool router_stream_applies(int dtype, int H, int E) {
  return dtype == MOE_BF16 && (E == 8 || E == 16) && H % 512 == 0 && H >= 512 && H <= 4096;
}

int launch_router_stream(const void* x, const void* w, const float* bias, const float* sel_bias, bool renorm,
                         int T, int H, int E, int K, float* logits, int32_t* idx, float* gate, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  switch (H / 512) {
    case 1: return launch_ch<1>(x, w, bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
    case 2: return launch_ch<2>(x, w, bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
    case 3: return launch_ch<3>(x, w, bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
    case 4: return launch_ch<4>(x, w, bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
    case 5: return launch_ch<5>(x, w, bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
    case 6: return launch_ch<6>(x, w, bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
    case 7: return launch_ch<7>(x, w, bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
    case 8: return launch_ch<8>(x, w, bias, sel_bias, renorm, T, H, E, K, logits, idx, gate, s);
    default: return MOE_ERR_UNSUPPORTED;
  }
}

}  // namespace moe
