// Grouped SwiGLU expert FFN over contiguous [E, H, H'] weights (MoonEP page,
// "Step-by-step": one contiguous tensor per projection, experts addressed by row
// index; T4 bottleneck page, SwiGLU table: three matrix products).
//
// The row split per expert is read on the device from cu_seqlens, so no host
// synchronisation happens between dispatch and the expert GEMMs.
#include "moe_internal.cuh"

namespace moe {

int launch_expert_ffn_tc(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                         const void* wd, int E, int H, int Hp, void* act, void* gu, void* h, cudaStream_t s,
                         const int32_t* gather, int gather_n, void* ws, size_t ws_bytes);
int launch_expert_ffn_bwd_tc(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                             const void* wd, int E, int H, int Hp, const void* gu, const void* act, const void* dh,
                             void* dgu, void* dxs, float* dwg, float* dwu, float* dwd, cudaStream_t s);

// bf16: tcgen05 grouped GEMMs.  fp32: FFMA grouped GEMMs (a 1e-5 relative error
// is out of reach of the tf32 tensor-core path).
int launch_expert_ffn(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                      const void* wd, int E, int H, int Hp, int dtype, void* act, void* gu, void* h,
                      cudaStream_t s, const int32_t* gather, int gather_n, void* ws, size_t ws_bytes) {
  if (rows == 0) return MOE_OK;
  if (dtype == MOE_BF16)
    return launch_expert_ffn_tc(xs, cu, rows, wg, wu, wd, E, H, Hp, act, gu, h, s, gather, gather_n, ws, ws_bytes);
  // act = silu(xs . Wg[e]) * (xs . Wu[e])
  SimtGemmArgs a{};
  a.A = xs; a.a_sm = H; a.a_sk = 1;
  a.a_rows = gather;
  a.B = wg; a.B2 = wu; a.b_sg = (long long)H * Hp; a.b_sk = Hp; a.b_sn = 1;
  a.C = act; a.c_sm = Hp;
  a.cu = cu; a.M = rows; a.N = Hp; a.K = H; a.groups = E;
  a.epilogue = 0; a.swiglu = true;
  int st = launch_simt_gemm(a, dtype, dtype, dtype, s);
  if (st != MOE_OK) return st;
  // h = act . Wd[e]^T   (Wd[e] stored [H, H'])
  SimtGemmArgs d{};
  d.A = act; d.a_sm = Hp; d.a_sk = 1;
  d.B = wd; d.b_sg = (long long)H * Hp; d.b_sk = 1; d.b_sn = Hp;
  d.C = h; d.c_sm = H;
  d.cu = cu; d.M = rows; d.N = H; d.K = Hp; d.groups = E;
  d.epilogue = 0; d.swiglu = false;
  return launch_simt_gemm(d, dtype, dtype, dtype, s);
}

// Backward (bf16 only): dgu is workspace [rows, 2H'] bf16.
int launch_expert_ffn_bwd(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                          const void* wd, int E, int H, int Hp, const void* gu, const void* act, const void* dh,
                          void* dxs, float* dwg, float* dwu, float* dwd, void* ws, cudaStream_t s) {
  if (rows == 0) {  // no rows: the weight gradients are zero
    const size_t n = (size_t)E * H * Hp * sizeof(float);
    for (float* d : {dwg, dwu, dwd})
      if (d && cudaMemsetAsync(d, 0, n, s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  return launch_expert_ffn_bwd_tc(xs, cu, rows, wg, wu, wd, E, H, Hp, gu, act, dh, ws, dxs, dwg, dwu, dwd, s);
}

size_t expert_ffn_bwd_ws_bytes(int rows, int Hp) { return (((size_t)rows * 2 * Hp * 2) + 255) & ~(size_t)255; }

}  // namespace moe
