// Mixture-of-Depths capacity router (MoE/MoD framework page, MoD paragraph:
// part of the tokens skips the layer entirely; 50% capacity).
//
//   score[t] = x[t] . w_mod                         (one warp per token)
//   per sequence: the C highest scores are selected, equal scores -> lower
//   position.  Token i of a sequence is selected iff its rank
//     #{j : s_j > s_i  or  (s_j == s_i and j < i)}
//   is below C; every token's rank is counted directly against the whole
//   sequence held in shared memory (L compares per token, all tokens in
//   parallel across many CTAs).  One CTA per sequence then compacts the
//   selected positions in order with a block scan, and one launch copies both
//   the selected rows (the MoE input) and the skipped rows (y = x).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int SEL_THREADS = 1024;

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

constexpr int RANK_TOK = 32;    // tokens per rank CTA
constexpr int RANK_SPLIT = 8;   // threads per token, each counting 1/8 of the sequence

// mask[b, i] = (rank of token i in sequence b) < C.  grid (ceil(L / RANK_TOK), B).
// The RANK_SPLIT threads of a token are consecutive lanes; they read
// consecutive 16-byte words of the shared scores (other tokens of the warp read
// the same words: broadcasts) and add their counts with shuffles.
__global__ void __launch_bounds__(RANK_TOK * RANK_SPLIT)
mod_rank_kernel(const float* __restrict__ score, int L, int C, uint8_t* __restrict__ mask) {
  extern __shared__ float4 s4[];  // the sequence's scores, padded to a multiple of 4 with -inf
  float* sv = reinterpret_cast<float*>(s4);
  const int b = blockIdx.y;
  const float* s = score + (long long)b * L;
  const int L4 = (L + 3) / 4;
  for (int j = threadIdx.x; j < 4 * L4; j += blockDim.x) sv[j] = j < L ? s[j] : -INFINITY;
  __syncthreads();
  const int part = threadIdx.x % RANK_SPLIT;
  const int i = blockIdx.x * RANK_TOK + threadIdx.x / RANK_SPLIT;
  const int ii = i < L ? i : L - 1;  // rows past L count too (uniform shuffles), nothing is written
  const float si = sv[ii];
  int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
#pragma unroll 4
  for (int q = part; q < L4; q += RANK_SPLIT) {
    const float4 v = s4[q];
    const int j = 4 * q;
    r0 += (v.x > si) | ((v.x == si) & (j < ii));
    r1 += (v.y > si) | ((v.y == si) & (j + 1 < ii));
    r2 += (v.z > si) | ((v.z == si) & (j + 2 < ii));
    r3 += (v.w > si) | ((v.w == si) & (j + 3 < ii));
  }
  int rank = (r0 + r1) + (r2 + r3);
#pragma unroll
  for (int o = RANK_SPLIT / 2; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
  if (part == 0 && i < L) mask[(long long)b * L + i] = (uint8_t)(rank < C);
}

// sel[b, r] = b*L + i for the r-th selected position i of sequence b (and its score)
__global__ void __launch_bounds__(SEL_THREADS)
mod_compact_kernel(const float* __restrict__ score, const uint8_t* __restrict__ mask, int L, int C,
                   int32_t* __restrict__ sel, float* __restrict__ sel_score) {
  __shared__ int part[SEL_THREADS];
  const int b = blockIdx.x;
  const uint8_t* m = mask + (long long)b * L;
  // each thread owns a run of positions
  const int per = (L + SEL_THREADS - 1) / SEL_THREADS;
  const int lo = threadIdx.x * per, hi = min(L, lo + per);
  int cnt = 0;
  for (int i = lo; i < hi; ++i) cnt += m[i];
  part[threadIdx.x] = cnt;
  __syncthreads();
  for (int o = 1; o < SEL_THREADS; o <<= 1) {
    const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int r = part[threadIdx.x] - cnt;
  for (int i = lo; i < hi; ++i) {
    if (m[i] && r < C) {
      sel[(long long)b * C + r] = b * L + i;
      if (sel_score) sel_score[(long long)b * C + r] = score[(long long)b * L + i];
      ++r;
    }
  }
}

// Row copies in one launch, one warp per item, U 16-byte vectors per lane in
// flight: items [0, n_sel) gather x_sel[j] = x[sel[j]] (sel holds flat token
// indices); items [n_sel, n_sel + n_tok) copy y[t] = x[t] for the tokens that
// skip the layer.
__global__ void __launch_bounds__(256)
mod_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sel, long long n_sel,
                const uint8_t* __restrict__ mask, long long n_tok, int vec_per_row, uint4* __restrict__ x_sel,
                uint4* __restrict__ y_skip) {
  constexpr int U = 4;
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < n_sel + n_tok;
       it += nwarps) {
    long long src, dst;
    uint4* out;
    if (it < n_sel) {
      src = __ldg(sel + it);
      dst = it;
      out = x_sel;
    } else {
      src = dst = it - n_sel;
      if (mask[src]) continue;
      out = y_skip;
    }
    const uint4* in = x + src * vec_per_row;
    uint4* o = out + dst * vec_per_row;
    for (int i0 = lane; i0 < vec_per_row; i0 += 32 * U) {
      uint4 a[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + 32 * u < vec_per_row) a[u] = __ldg(in + i0 + 32 * u);
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + 32 * u < vec_per_row) o[i0 + 32 * u] = a[u];
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
  if (dtype == MOE_BF16)
    mod_score_kernel<bf16><<<warp_grid(n_tok), 256, 0, s>>>(static_cast<const bf16*>(x),
                                                            static_cast<const bf16*>(w), n_tok, H, score);
  else
    mod_score_kernel<float><<<warp_grid(n_tok), 256, 0, s>>>(static_cast<const float*>(x),
                                                             static_cast<const float*>(w), n_tok, H, score);
  int st = launch_status();
  if (st != MOE_OK) return st;
  const int vec = H * (dtype == MOE_BF16 ? 2 : 4) / 16;
  const size_t smem = (size_t)((L + 3) / 4) * 16;
  mod_rank_kernel<<<dim3((L + RANK_TOK - 1) / RANK_TOK, B), RANK_TOK * RANK_SPLIT, smem, s>>>(score, L, C,
                                                                                            mask);
  st = launch_status();
  if (st != MOE_OK) return st;
  if (C > 0) {
    mod_compact_kernel<<<B, SEL_THREADS, 0, s>>>(score, mask, L, C, sel, sel_score);
    st = launch_status();
    if (st != MOE_OK) return st;
  }
  const long long n_sel = x_sel ? (long long)B * C : 0;
  const long long n_skip = y_skip ? n_tok : 0;
  if (n_sel + n_skip > 0) {
    mod_rows_kernel<<<warp_grid(n_sel + n_skip), 256, 0, s>>>(static_cast<const uint4*>(x), sel, n_sel, mask,
                                                              n_skip, vec, static_cast<uint4*>(x_sel),
                                                              static_cast<uint4*>(y_skip));
    st = launch_status();
  }
  return st;
}

}  // namespace moe
