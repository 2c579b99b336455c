// Mixture-of-Depths capacity router (MoE/MoD framework page, MoD paragraph:
// part of the tokens skips the layer entirely; 50% capacity).
//
//   score[t] = x[t] . w_mod
//   per sequence: the C highest scores are selected, equal scores -> lower
//   position, i.e. token i is selected iff its rank
//     #{j : s_j > s_i  or  (s_j == s_i and j < i)}
//   is below C.
// The selection runs on order-preserving integer keys of the scores (-0
// folded onto +0, so equal scores are equal keys): the C-th largest key k* is
// found bit by bit from the top (a radix select with one-bit digits); keys
// above k* are selected, and of the keys equal to k* the first
// (C - #{key > k*}) by position.
//
// One launch when the rows fit in shared memory (every CTA holds at most
// ~54 rows of 4 KB, as at 4 x 2048 tokens of H = 2048 on 152 SMs): each CTA
// brings its contiguous rows in with bulk copies (groups of 16 rows on their
// own mbarriers, each row scored as soon as its group lands), then
// waits until every score of its sequence(s) is written (the score buffer is
// first filled with a bit pattern no dot product produces, so the wait needs
// no counter and two calls never share state), runs the select and stores
// its rows from shared memory to x_sel or y: x is read from HBM once.  The
// CTAs wait on one another, so the launch is cooperative (all CTAs resident).
// Otherwise two launches: a score kernel (one warp per token), then the
// select and the row copies, every CTA of a sequence running the same select
// on the sequence's scores and copying its share of the rows.
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

// Select of one sequence: keys[i] (i < L) holds score_key of position i on
// entry and, on return, the rank of position i among the selected positions,
// or 0xffffffff when it is not selected.  All threads of the CTA call it;
// hist ([2][256]) and wcnt ([2][MS_WARPS]) are the CTA's shared scratch.
//
// Radix select: up to four 8-bit passes from the top find the C-th largest key
// k*.  Each thread keeps its run of consecutive positions in registers; in the
// first pass lanes with the same digit add to the histogram once (the lowest
// of them), in later passes (only the keys under the chosen prefix) each key
// adds itself; the two histograms alternate so a pass clears the next one's
// while it counts.
// When the digit bucket holding the C-th key is taken whole (every key with
// that prefix is among the C largest), the remaining passes are skipped: the
// selection is then every key whose prefix is at least that bucket's, the
// same set the full passes give (ties between equal keys can only fall inside
// the bucket, all of which is taken).
__device__ void seq_row_map(unsigned* keys, int L, int C, int (*hist)[256], int (*wcnt)[MS_WARPS], int* s_sel) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const bool partial = C > 0 && C < L;
  const int per = (L + MS_THREADS - 1) / MS_THREADS;
  const int lo = min(L, tid * per), hi = min(L, lo + per);
  unsigned kr[MS_MAX_RUN];
#pragma unroll
  for (int j = 0; j < MS_MAX_RUN; ++j) kr[j] = lo + j < hi ? keys[lo + j] : 0u;
  unsigned lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
  // after the pass at `shift`, the bits of `prefix` under `pmask` are fixed
  // and `need` keys are still to be taken among the keys that match them
  unsigned prefix = 0, pmask = 0;
  int need = C;
  if (partial) {
    if (tid < 256) hist[0][tid] = 0;
    __syncthreads();
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      int* h = hist[pass & 1];
      if (tid < 256) hist[(pass + 1) & 1][tid] = 0;  // the next pass's histogram
      int d[MS_MAX_RUN];
#pragma unroll
      for (int j = 0; j < MS_MAX_RUN; ++j)
        d[j] = (lo + j < hi && (kr[j] & pmask) == prefix) ? (int)((kr[j] >> shift) & 255u) : -1;
      if (pass == 0) {
        // all keys count, and scores crowd into few top digits: lanes with
        // equal digits add once
#pragma unroll
        for (int j = 0; j < MS_MAX_RUN; ++j) {
          if (j >= per) break;  // uniform: per is the same for every thread
          const unsigned peers = __match_any_sync(0xffffffffu, d[j]);
          if (d[j] >= 0 && (peers & lt) == 0) atomicAdd(&h[d[j]], __popc(peers));
        }
      } else {
        // only the keys under the chosen prefix count, spread over the digits
#pragma unroll
        for (int j = 0; j < MS_MAX_RUN; ++j)
          if (d[j] >= 0) atomicAdd(&h[d[j]], 1);
      }
      __syncthreads();
      if (w == 0) {
        // lane l owns digits 255 - 8l - j, j = 0..7 (descending); the digit
        // where the count from the top reaches `need` holds the C-th key
        int c[8], local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = h[255 - 8 * lane - j];
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
              // digit, and a flag (bit 8) when the bucket is taken whole
              s_sel[2 * (pass & 1)] = (255 - 8 * lane - j) | (run + c[j] == need ? 256 : 0);
              s_sel[2 * (pass & 1) + 1] = need - run;
              break;
            }
            run += c[j];
          }
        }
      }
      __syncthreads();
      const int dsel = s_sel[2 * (pass & 1)];
      prefix |= (unsigned)(dsel & 255) << shift;
      pmask |= 255u << shift;
      need = s_sel[2 * (pass & 1) + 1];
      if (dsel & 256) break;  // uniform: every thread read the same flag
    }
  }
  // the C-th largest key's prefix under pmask (the whole key after four passes)
  const unsigned kth = prefix;

  // selection flags with the tie rule (equal keys taken by position), then
  // ranks among the selected
  int n_eq = 0;
#pragma unroll
  for (int j = 0; j < MS_MAX_RUN; ++j) n_eq += (lo + j < hi && partial && (kr[j] & pmask) == kth) ? 1 : 0;
  int tot;
  int eq_before = block_excl_scan(n_eq, wcnt[1], tot);
  unsigned flags = 0;
  int n_sel = 0;
#pragma unroll
  for (int j = 0; j < MS_MAX_RUN; ++j) {
    if (lo + j >= hi) break;
    const unsigned k = kr[j] & pmask;
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
      flags |= 1u << j;
      ++n_sel;
    }
  }
  int pos = block_excl_scan(n_sel, wcnt[0], tot);
  // the row map replaces the keys (each thread rewrites only its own run)
#pragma unroll
  for (int j = 0; j < MS_MAX_RUN; ++j) {
    if (lo + j >= hi) break;
    const bool take = (flags >> j) & 1u;
    keys[lo + j] = take ? (unsigned)pos : 0xffffffffu;
    pos += take ? 1 : 0;
  }
  __syncthreads();
}

// grid (R, B): CTA r of sequence b.  Dynamic shared memory: L ints (the keys,
// then the row map: selected position -> rank among the selected, else -1).
__global__ void __launch_bounds__(MS_THREADS)
mod_select_rows_kernel(const float* __restrict__ score, int L, int C, const uint4* __restrict__ x,
                       int vec_per_row, int32_t* __restrict__ sel, float* __restrict__ sel_score,
                       uint8_t* __restrict__ mask, uint4* __restrict__ x_sel, uint4* __restrict__ y_skip) {
  extern __shared__ unsigned keys[];
  __shared__ int hist[2][256];
  __shared__ int wcnt[2][MS_WARPS];
  __shared__ int s_sel[4];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int b = blockIdx.y, R = gridDim.x, r = blockIdx.x;
  const float* s = score + (long long)b * L;
  for (int i = tid; i < L; i += MS_THREADS) keys[i] = score_key(__ldg(s + i));
  __syncthreads();
  seq_row_map(keys, L, C, hist, wcnt, s_sel);
  if (r == 0) {
    for (int i = tid; i < L; i += MS_THREADS) {
      const unsigned m = keys[i];
      const long long t = (long long)b * L + i;
      mask[t] = m != 0xffffffffu ? 1 : 0;
      if (m != 0xffffffffu) {
        sel[(long long)b * C + m] = (int32_t)t;
        if (sel_score) sel_score[(long long)b * C + m] = __ldg(s + i);
      }
    }
  }

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

// ---------------------------------------------------------- one launch ---
constexpr unsigned SCORE_UNSET = 0xffffffffu;  // a NaN bit pattern no dot product yields
constexpr unsigned long long MF_WAIT_LIMIT = 4000000000ull;  // clock64 cycles, ~2 s
constexpr int MF_GROUPS = 8;  // row groups (mbarriers) per CTA

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool mbar_try_wait0(uint32_t bar) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar)
      : "memory");
  return ok != 0;
}
// waits (bounded) for the mbarrier's first phase; false on timeout
__device__ __forceinline__ bool mbar_wait0_bounded(uint32_t bar) {
  const long long t0 = clock64();
  while (!mbar_try_wait0(bar))
    if ((unsigned long long)(clock64() - t0) > MF_WAIT_LIMIT) return false;
  return true;
}

// grid: G CTAs, all resident (cooperative launch); CTA g owns the tokens
// [g n / G, (g+1) n / G) of the n = B L.  Dynamic shared memory: rows_cap
// rows of H elements, then L keys.
template <typename T>
__global__ void __launch_bounds__(MS_THREADS, 1)
mod_fused_kernel(const T* __restrict__ x, const T* __restrict__ w, int B, int L, int H, int C, int rows_cap,
                 float* score, int32_t* __restrict__ sel, float* __restrict__ sel_score,
                 uint8_t* __restrict__ mask, T* __restrict__ x_sel, T* __restrict__ y_skip, unsigned* err) {
  extern __shared__ __align__(128) unsigned char smem_rows[];
  __shared__ __align__(8) unsigned long long bar[MF_GROUPS];
  __shared__ int rows_bad;
  __shared__ int hist[2][256];
  __shared__ int wcnt[2][MS_WARPS];
  __shared__ int s_sel[4];
  constexpr int V = Vec16<T>::N;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long n_tok = (long long)B * L;
  const int G = gridDim.x;
  const long long r0 = n_tok * blockIdx.x / G, r1 = n_tok * (blockIdx.x + 1) / G;
  const int nr = (int)(r1 - r0);
  const uint32_t rb = (uint32_t)H * (uint32_t)sizeof(T);
  const int nvec = H / V;
  unsigned* keys = reinterpret_cast<unsigned*>(smem_rows + (size_t)rows_cap * rb);
  // rows [MS_WARPS g, MS_WARPS (g + 1)) arrive on barrier g (the last one takes
  // the rest): the warps score the first rows while the later ones land
  const int n_groups = min(MF_GROUPS, (nr + MS_WARPS - 1) / MS_WARPS);
  auto group_of = [&](int r) { return min(r / MS_WARPS, MF_GROUPS - 1); };

  // 1. the CTA's rows into shared memory (bulk copies, one mbarrier per group)
  if (tid == 0) {
    rows_bad = 0;
    for (int g = 0; g < n_groups; ++g)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bar[g])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) {
    for (int g = 0; g < n_groups; ++g) {
      const int ra = g * MS_WARPS, rz = g == MF_GROUPS - 1 ? nr : min(nr, ra + MS_WARPS);
      const uint32_t bg = smem_addr(&bar[g]);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bg), "r"((uint32_t)(rz - ra) * rb)
                   : "memory");
      for (int r = ra; r < rz; ++r)
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_addr(smem_rows + (size_t)r * rb)),
            "l"(x + (r0 + r) * H), "r"(rb), "r"(bg)
            : "memory");
    }
  }
  // a lane's share of w_mod (WV vectors of 16 bytes) is requested while the
  // rows arrive and stays in registers for all the warp's rows
  constexpr int WV = 8;  // H * sizeof(T) <= 32 * WV * 16 bytes: one pass over a row
  const uint4* wv = reinterpret_cast<const uint4*>(w);
  uint4 wr[WV];
#pragma unroll
  for (int u = 0; u < WV; ++u) wr[u] = lane + 32 * u < nvec ? __ldg(wv + lane + 32 * u) : make_uint4(0, 0, 0, 0);

  // 2. scores of the CTA's rows: one warp per row, as its group lands (a row
  //    whose copy timed out is still scored, so no CTA waits on it forever)
  {
    for (int r = warp; r < nr; r += MS_WARPS) {
      if (!mbar_wait0_bounded(smem_addr(&bar[group_of(r)])) && lane == 0) rows_bad = 1;
      const uint4* rv = reinterpret_cast<const uint4*>(smem_rows + (size_t)r * rb);
      float acc = 0.f;
      if (nvec <= 32 * WV) {
        // WV independent partial sums (short dependency chains), added in a
        // fixed order
        uint4 xr[WV];
        float part[WV];
#pragma unroll
        for (int u = 0; u < WV; ++u) xr[u] = lane + 32 * u < nvec ? rv[lane + 32 * u] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < WV; ++u) {
          float xv[V], ww[V];
          Vec16<T>::load_raw_unpack(xr[u], xv);
          Vec16<T>::load_raw_unpack(wr[u], ww);
          part[u] = 0.f;
#pragma unroll
          for (int v = 0; v < V; ++v) part[u] = fmaf(xv[v], ww[v], part[u]);
        }
#pragma unroll
        for (int u = 0; u < WV; ++u) acc += part[u];
      } else {
        for (int i = lane; i < nvec; i += 32) {
          float xv[V], ww[V];
          Vec16<T>::load_raw_unpack(rv[i], xv);
          Vec16<T>::load_raw_unpack(__ldg(wv + i), ww);
#pragma unroll
          for (int v = 0; v < V; ++v) acc = fmaf(xv[v], ww[v], acc);
        }
      }
      acc = warp_sum(acc);
      if (__float_as_uint(acc) == SCORE_UNSET) acc = __uint_as_float(0x7fffffffu);
      if (lane == 0) score[r0 + r] = acc;
    }
  }
  const bool rows_ok = !__syncthreads_or(rows_bad);
  if (!rows_ok && tid == 0) set_error(err, DEV_TIMEOUT);

  // 3. per sequence the CTA's tokens belong to: wait for all its scores, select,
  //    then write the CTA's share of mask / sel / sel_score and of the rows
  if (nr > 0) {
    const long long b_lo = r0 / L, b_hi = (r1 - 1) / L;
    for (long long b = b_lo; b <= b_hi; ++b) {
      const unsigned* s = reinterpret_cast<const unsigned*>(score + b * L);
      const long long t0 = clock64();
      for (;;) {
        int missing = 0;
        for (int i = tid; i < L; i += MS_THREADS) {
          const unsigned u = __ldcg(s + i);
          missing |= u == SCORE_UNSET;
          keys[i] = score_key(__uint_as_float(u));
        }
        if (!__syncthreads_or(missing)) break;
        // one clock decides for the whole CTA (the loop exit stays uniform)
        if (__syncthreads_or(tid == 0 && (unsigned long long)(clock64() - t0) > MF_WAIT_LIMIT)) {
          if (tid == 0) set_error(err, DEV_TIMEOUT);
          break;
        }
        __nanosleep(256);
      }
      seq_row_map(keys, L, C, hist, wcnt, s_sel);
      const long long t_lo = r0 > b * L ? r0 : b * L;
      const long long t_hi = r1 < (b + 1) * L ? r1 : (b + 1) * L;
      for (long long t = t_lo + tid; t < t_hi; t += MS_THREADS) {
        const int i = (int)(t - b * L);
        const unsigned m = keys[i];
        mask[t] = m != 0xffffffffu ? 1 : 0;
        T* dst = nullptr;
        if (m != 0xffffffffu) {
          sel[b * C + m] = (int32_t)t;
          if (sel_score) sel_score[b * C + m] = __uint_as_float(__ldcg(s + i));
          if (x_sel) dst = x_sel + (b * C + m) * H;
        } else if (y_skip) {
          dst = y_skip + t * H;
        }
        if (dst && rows_ok)
          asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                       "r"(smem_addr(smem_rows + (size_t)(t - r0) * rb)), "r"(rb)
                       : "memory");
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      __syncthreads();  // the keys are rewritten for the next sequence
    }
    // shared memory stays until the bulk stores have read it
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
  if (!rows_ok && tid == 0)  // copies still in flight land before exit
    for (int g = 0; g < n_groups; ++g) mbar_wait0_bounded(smem_addr(&bar[g]));
}

int warp_grid(long long n) {
  long long ctas = (n + 7) / 8;
  long long cap = (long long)sm_count() * 16;
  if (ctas < 1) ctas = 1;
  return (int)(ctas < cap ? ctas : cap);
}

}  // namespace

template <typename T>
int launch_mod_fused(const void* x, const void* w, int B, int L, int H, int C, float* score, int32_t* sel,
                     float* sel_score, uint8_t* mask, void* x_sel, void* y_skip, int rows_cap, int G, size_t smem,
                     cudaStream_t s) {
  auto k = mod_fused_kernel<T>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  // every score starts as the unset pattern (0xff bytes)
  if (cudaMemsetAsync(score, 0xff, (size_t)B * L * sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(MS_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, k, static_cast<const T*>(x), static_cast<const T*>(w), B, L, H, C, rows_cap, score, sel,
                     sel_score, mask, static_cast<T*>(x_sel), static_cast<T*>(y_skip), device_error_word());
  return launch_status();
}

// The one-launch form applies when every CTA's rows and the keys of a
// sequence fit in shared memory with all CTAs resident (one per SM).
bool mod_fused_plan(int B, int L, int H, int dtype, int* rows_cap, int* G, size_t* smem) {
  const long long n_tok = (long long)B * L;
  const int esz = dtype == MOE_BF16 ? 2 : 4;
  int dev = 0, max_optin = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (!coop || n_tok < 1) return false;
  cudaFuncAttributes fa;
  if ((dtype == MOE_BF16 ? cudaFuncGetAttributes(&fa, mod_fused_kernel<bf16>)
                         : cudaFuncGetAttributes(&fa, mod_fused_kernel<float>)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const long long g = n_tok < sm_count() ? n_tok : sm_count();
  const long long cap = (n_tok + g - 1) / g;
  const size_t need = (size_t)cap * H * esz + (size_t)L * 4;
  if (need + fa.sharedSizeBytes > (size_t)max_optin) return false;  // + the static shared memory
  *rows_cap = (int)cap;
  *G = (int)g;
  *smem = need;
  return true;
}

int launch_mod_select(const void* x, const void* w, int B, int L, int H, int C, int dtype,
                      float* score, int32_t* sel, float* sel_score, uint8_t* mask, void* x_sel,
                      void* y_skip, cudaStream_t s) {
  const long long n_tok = (long long)B * L;
  if (n_tok == 0) return MOE_OK;
  if (L > MS_THREADS * MS_MAX_RUN) return MOE_ERR_UNSUPPORTED;
  int rows_cap = 0, G = 0;
  size_t fsmem = 0;
  if (mod_fused_plan(B, L, H, dtype, &rows_cap, &G, &fsmem)) {
    return dtype == MOE_BF16
               ? launch_mod_fused<bf16>(x, w, B, L, H, C, score, sel, sel_score, mask, x_sel, y_skip, rows_cap, G,
                                        fsmem, s)
               : launch_mod_fused<float>(x, w, B, L, H, C, score, sel, sel_score, mask, x_sel, y_skip, rows_cap, G,
                                         fsmem, s);
  }
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
