// Mixture-of-Depths capacity router (MoE/MoD framework page, MoD paragraph:
// part of the tokens skips the layer entirely; 50% capacity).
//
//   score[t] = x[t] . w_mod                         (one warp per token)
//   per sequence: the C highest scores are selected, equal scores -> lower
//   position, i.e. token i is selected iff its rank
//     #{j : s_j > s_i  or  (s_j == s_i and j < i)}
//   is below C.
// The selection runs as a radix select on order-preserving integer keys of
// the scores (-0 folded onto +0, so equal scores are equal keys): four 8-bit
// passes from the top find the C-th largest key k*; keys above k* are
// selected, and of the keys equal to k* the first (C - #{key > k*}) by
// position.  One launch does the select and the row copies: every CTA of a
// sequence runs the same select on the sequence's scores (identical integer
// work, identical result), the first CTA writes mask, sel and sel_score, and
// each CTA copies its share of the rows: the selected ones to the MoE input
// x_sel in position order, the others to y (y = x for tokens that skip).
#include "moe_internal.cuh"

namespace moe {
namespace {

template <typename T>
__global__ void __launch_bounds__(256)
mod_score_kernel(const T* __restrict__ x, const T* __restrict__ w, long long n_tok, int H,
                 float* __restrict__ score) {
  constexpr int V = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = H / V;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long t = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_tok; t += nwarps) {
    // all U vectors of a lane's share of the row are requested before any is used
    constexpr int U = 8;
    float acc = 0.f;
    for (int base = 0; base < nvec; base += 32 * U) {
      uint4 xr[U], wr[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + 32 * u + lane;
        if (i < nvec) {
          xr[u] = __ldg(reinterpret_cast<const uint4*>(x + t * H) + i);
          wr[u] = __ldg(reinterpret_cast<const uint4*>(w) + i);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (base + 32 * u + lane < nvec) {
          float xv[V], wv[V];
          Vec16<T>::load_raw_unpack(xr[u], xv);
          Vec16<T>::load_raw_unpack(wr[u], wv);
#pragma unroll
          for (int v = 0; v < V; ++v) acc = fmaf(xv[v], wv[v], acc);
        }
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) score[t] = acc;
  }
}

constexpr int MS_THREADS = 512;
constexpr int MS_WARPS = MS_THREADS / 32;
constexpr int MS_MAX_RUN = 16;  // positions per thread: L <= 8192

// Order-preserving key: a > b as floats iff key(a) > key(b); -0 and +0 map to
// the same key (they are equal scores).
__device__ __forceinline__ unsigned score_key(float s) {
  const unsigned u = __float_as_uint(s == 0.f ? 0.f : s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive prefix of v over the CTA's threads in thread order (warp shuffles,
// then the warp totals); total gets the sum over all threads.
__device__ __forceinline__ int block_excl_scan(int v, int* wtot, int& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();  // wtot may still be read by a previous scan
  if (lane == 31) wtot[w] = incl;
  __syncthreads();
  int before = incl - v;
  total = 0;
#pragma unroll
  for (int ww = 0; ww < MS_WARPS; ++ww) {
    before += ww < w ? wtot[ww] : 0;
    total += wtot[ww];
  }
  return before;
}

// grid (R, B): CTA r of sequence b.  Dynamic shared memory: L ints (the keys,
// then the row map: selected position -> rank among the selected, else -1).
__global__ void __launch_bounds__(MS_THREADS)
mod_select_rows_kernel(const float* __restrict__ score, int L, int C, const uint4* __restrict__ x,
                       int vec_per_row, int32_t* __restrict__ sel, float* __restrict__ sel_score,
                       uint8_t* __restrict__ mask, uint4* __restrict__ x_sel, uint4* __restrict__ y_skip) {
  extern __shared__ unsigned keys[];
  __shared__ int hist[256];
  __shared__ int wtot[MS_WARPS];
  __shared__ int s_bin, s_need;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int b = blockIdx.y, R = gridDim.x, r = blockIdx.x;
  const float* s = score + (long long)b * L;
  for (int i = tid; i < L; i += MS_THREADS) keys[i] = score_key(__ldg(s + i));
  __syncthreads();

  // radix select of the C-th largest key: after the pass at `shift`, the bits
  // of `prefix` under `pmask` are fixed and `need` keys are still to be taken
  // among the keys that match them
  unsigned prefix = 0, pmask = 0;
  int need = C;
  const bool partial = C > 0 && C < L;
  if (partial) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      for (int i0 = 0; i0 < L; i0 += MS_THREADS) {
        const int i = i0 + tid;
        const unsigned k = i < L ? keys[i] : 0u;
        const int d = (i < L && (k & pmask) == prefix) ? (int)((k >> shift) & 255u) : -1;
        // lanes with the same digit add once (the lowest of them)
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (d >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&hist[d], __popc(peers));
      }
      __syncthreads();
      if (w == 0) {
        // lane l owns digits 255 - 8l - j, j = 0..7 (descending); the digit
        // where the count from the top reaches `need` holds the C-th key
        int c[8], local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[255 - 8 * lane - j];
          local += c[j];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        const int before = incl - local;
        if (before < need && need <= incl) {
          int run = before;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (run + c[j] >= need) {
              s_bin = 255 - 8 * lane - j;
              s_need = need - run;
              break;
            }
            run += c[j];
          }
        }
      }
      __syncthreads();
      prefix |= (unsigned)s_bin << shift;
      pmask |= 255u << shift;
      need = s_need;
    }
  }
  const unsigned kth = prefix;  // the C-th largest key (when 0 < C < L)

  // each thread owns a run of consecutive positions: selection flags with the
  // tie rule (equal keys taken by position), then ranks among the selected
  const int per = (L + MS_THREADS - 1) / MS_THREADS;
  const int lo = min(L, tid * per), hi = min(L, lo + per);
  int n_eq = 0;
  for (int i = lo; i < hi; ++i) n_eq += (partial && keys[i] == kth) ? 1 : 0;
  int tot;
  int eq_before = block_excl_scan(n_eq, wtot, tot);
  unsigned flags = 0;
  int n_sel = 0;
  for (int i = lo; i < hi; ++i) {
    const unsigned k = keys[i];
    bool take;
    if (!partial) {
      take = C >= L;
    } else if (k > kth) {
      take = true;
    } else if (k == kth) {
      take = eq_before < need;
      ++eq_before;
    } else {
      take = false;
    }
    if (take) {
      flags |= 1u << (i - lo);
      ++n_sel;
    }
  }
  int pos = block_excl_scan(n_sel, wtot, tot);
  // the row map replaces the keys (each thread rewrites only its own run)
  for (int i = lo; i < hi; ++i) {
    const bool take = (flags >> (i - lo)) & 1u;
    const long long t = (long long)b * L + i;
    if (r == 0) {
      mask[t] = take ? 1 : 0;
      if (take) {
        sel[(long long)b * C + pos] = (int32_t)t;
        if (sel_score) sel_score[(long long)b * C + pos] = __ldg(s + i);
      }
    }
    keys[i] = take ? (unsigned)pos : 0xffffffffu;
    pos += take ? 1 : 0;
  }
  __syncthreads();

  // this CTA's rows: one warp per row, 16-byte vectors, all of a lane's
  // vectors of the row in flight before the first store
  const int r_lo = (int)((long long)L * r / R), r_hi = (int)((long long)L * (r + 1) / R);
  for (int i = r_lo + w; i < r_hi; i += MS_WARPS) {
    const int m = (int)keys[i];
    uint4* dst;
    if (m >= 0) {
      if (!x_sel) continue;
      dst = x_sel + ((long long)b * C + m) * vec_per_row;
    } else {
      if (!y_skip) continue;
      dst = y_skip + ((long long)b * L + i) * vec_per_row;
    }
    const uint4* src = x + ((long long)b * L + i) * vec_per_row;
    constexpr int U = 8;
    for (int i0 = lane; i0 < vec_per_row; i0 += 32 * U) {
      uint4 a[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + 32 * u < vec_per_row) a[u] = __ldg(src + i0 + 32 * u);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + 32 * u < vec_per_row) dst[i0 + 32 * u] = a[u];
    }
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
  if (L > MS_THREADS * MS_MAX_RUN) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_BF16)
    mod_score_kernel<bf16><<<warp_grid(n_tok), 256, 0, s>>>(static_cast<const bf16*>(x),
                                                            static_cast<const bf16*>(w), n_tok, H, score);
  else
    mod_score_kernel<float><<<warp_grid(n_tok), 256, 0, s>>>(static_cast<const float*>(x),
                                                             static_cast<const float*>(w), n_tok, H, score);
  int st = launch_status();
  if (st != MOE_OK) return st;
  const int vec = H * (dtype == MOE_BF16 ? 2 : 4) / 16;
  // about two CTAs per SM over all sequences, at least 8 rows each
  long long R = (2LL * sm_count() + B - 1) / B;
  if (R > (L + 7) / 8) R = (L + 7) / 8;
  if (R < 1) R = 1;
  const size_t smem = (size_t)L * sizeof(unsigned);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(mod_select_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  mod_select_rows_kernel<<<dim3((unsigned)R, B), MS_THREADS, smem, s>>>(
      score, L, C, static_cast<const uint4*>(x), vec, sel, sel_score, mask, static_cast<uint4*>(x_sel),
      static_cast<uint4*>(y_skip));
  return launch_status();
}

}  // namespace moe
