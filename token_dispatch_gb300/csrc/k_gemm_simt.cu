// SIMT (FFMA) tiled GEMM with fp32 accumulation.
//
// Used where the contraction is fp32 end to end (the fp32 layer: tf32 tensor
// cores cannot hold a 1e-5 relative error) and for the small router-gradient
// contractions.  A 64x64 output tile per 256-thread CTA, 4x4 outputs per thread,
// K staged through shared memory 16 at a time.  Operands are addressed through
// element strides so one kernel serves x.W, x^T.dlogits and dlogits.W^T, and
// optionally per expert group (rows [cu[g], cu[g+1]) with weights g*b_sg).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <typename TA, typename TB, typename TC, bool SWIGLU>
__global__ void __launch_bounds__(NT) simt_gemm_kernel(SimtGemmArgs a) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float Bs2[SWIGLU ? BK : 1][SWIGLU ? BN + 4 : 1];

  const int g = blockIdx.z;
  long long row_lo = 0, row_hi = a.M;
  if (a.cu) { row_lo = a.cu[g]; row_hi = a.cu[g + 1]; }
  const long long m0 = row_lo + (long long)blockIdx.y * BM;
  if (m0 >= row_hi) return;
  const int n0 = blockIdx.x * BN;

  const TA* A = static_cast<const TA*>(a.A);
  const TB* B = static_cast<const TB*>(a.B) + (long long)g * a.b_sg;
  const TB* B2 = SWIGLU ? static_cast<const TB*>(a.B2) + (long long)g * a.b_sg : nullptr;

  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  float acc[4][4] = {}, acc2[4][4] = {};

  const bool a_krow = (a.a_sk == 1);
  const bool b_nrow = (a.b_sn == 1);

  for (int k0 = 0; k0 < a.K; k0 += BK) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = tid + j * NT;
      int m = a_krow ? e / BK : e % BM;
      int k = a_krow ? e % BK : e / BM;
      long long gm = m0 + m;
      int gk = k0 + k;
      float v = 0.f;
      if (gm < row_hi && gk < a.K) {
        const long long am = a.a_rows ? (long long)__ldg(a.a_rows + gm) : gm;
        v = to_f32(A[am * a.a_sm + (long long)gk * a.a_sk]);
      }
      As[k][m] = v;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = tid + j * NT;
      int k = b_nrow ? e / BN : e % BK;
      int n = b_nrow ? e % BN : e / BK;
      int gk = k0 + k, gn = n0 + n;
      float v = 0.f, v2 = 0.f;
      if (gk < a.K && gn < a.N) {
        long long off = (long long)gk * a.b_sk + (long long)gn * a.b_sn;
        v = to_f32(B[off]);
        if (SWIGLU) v2 = to_f32(B2[off]);
      }
      Bs[k][n] = v;
      if (SWIGLU) Bs2[k][n] = v2;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float av[4], bv[4], bv2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[k][ty * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i) bv[i] = Bs[k][tx * 4 + i];
      if (SWIGLU) {
#pragma unroll
        for (int i = 0; i < 4; ++i) bv2[i] = Bs2[k][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
          if (SWIGLU) acc2[i][j] = fmaf(av[i], bv2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }

  TC* C = static_cast<TC*>(a.C);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    long long gm = m0 + ty * 4 + i;
    if (gm >= row_hi) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int gn = n0 + tx * 4 + j;
      if (gn >= a.N) continue;
      float v = acc[i][j];
      if (SWIGLU) v = v / (1.0f + expf(-v)) * acc2[i][j];
      TC* p = C + gm * a.c_sm + gn;
      if (a.epilogue == 1) v += to_f32(*p);
      else if (a.epilogue == 2 && a.bias) v += a.bias[gn];
      *p = from_f32<TC>(v);
    }
  }
}

template <typename TA, typename TB, typename TC>
int launch_typed(const SimtGemmArgs& a, cudaStream_t s) {
  long long rows = a.M;
  dim3 grid((a.N + BN - 1) / BN, (unsigned)((rows + BM - 1) / BM), a.cu ? a.groups : 1);
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return MOE_OK;
  if (a.swiglu) simt_gemm_kernel<TA, TB, TC, true><<<grid, NT, 0, s>>>(a);
  else simt_gemm_kernel<TA, TB, TC, false><<<grid, NT, 0, s>>>(a);
  return launch_status();
}

}  // namespace

int launch_simt_gemm(const SimtGemmArgs& a, int ta, int tb, int tc, cudaStream_t s) {
  if (ta == MOE_F32 && tb == MOE_F32 && tc == MOE_F32) return launch_typed<float, float, float>(a, s);
  if (ta == MOE_BF16 && tb == MOE_BF16 && tc == MOE_BF16) return launch_typed<bf16, bf16, bf16>(a, s);
  if (ta == MOE_BF16 && tb == MOE_F32 && tc == MOE_F32) return launch_typed<bf16, float, float>(a, s);
  if (ta == MOE_F32 && tb == MOE_BF16 && tc == MOE_BF16) return launch_typed<float, bf16, bf16>(a, s);
  if (ta == MOE_BF16 && tb == MOE_BF16 && tc == MOE_F32) return launch_typed<bf16, bf16, float>(a, s);
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
