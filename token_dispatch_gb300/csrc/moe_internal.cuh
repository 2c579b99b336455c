// Internal declarations shared by the libmoe translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- errors ---
// Device error codes written into the per-device error word (first error wins).
enum : unsigned { DEV_OK = 0, DEV_TIMEOUT = MOE_ERR_TIMEOUT, DEV_BOUNDS = MOE_ERR_DEVICE_BOUNDS };

__device__ __forceinline__ void set_error(unsigned* err, unsigned code) {
  if (err) atomicCAS(err, 0u, code);
}

// Address of the current device's error word (resolved once per device).
unsigned* device_error_word();

// ------------------------------------------------------------ conversions ---
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// A 16-byte vector of the storage type: 4 floats or 8 bf16.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const float* p, float* v) {
    float4 q = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ __forceinline__ static void load_raw_unpack(const uint4& q, float* v) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
  __device__ __forceinline__ static void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <> struct Vec16<bf16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const bf16* p, float* v) {
    uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
  }
  __device__ __forceinline__ static void load_raw_unpack(const uint4& q, float* v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
  }
  __device__ __forceinline__ static void store(bf16* p, const float* v) {
    uint4 q;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = q;
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// SMs of the current device.  Without a device to ask (workspace sizes queried
// on a host with no GPU) the answer is that of GB300, the part this library is
// built for: 152.
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  return n;
}

// Kernels this library has launched in this process (every launch site is
// followed by exactly one launch_status()).
extern unsigned long long g_kernel_launches;

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  __atomic_fetch_add(&g_kernel_launches, 1ull, __ATOMIC_RELAXED);
  return MOE_OK;
}

// ------------------------------------------------------- kernel launchers ---
// Each returns a moe_status.  Arguments have been validated by the C ABI layer.

// route
size_t route_ws_bytes(int T, int H, int E);
bool router_stream_applies(int dtype, int H, int E);
// bias: added to the stored logits; sel_bias: added only where experts are
// chosen (nullable both); renorm: the K gates rescaled to sum to 1
int launch_router_stream(const void* x, const void* w, const float* bias, const float* sel_bias, bool renorm,
                         int T, int H, int E, int K, float* logits, int32_t* idx, float* gate, cudaStream_t s);
int launch_route(const void* x, const void* w, const float* bias, int T, int H, int E, int K, int dtype, int flags,
                 float* logits, int32_t* idx, float* gate, void* ws, cudaStream_t s);
int launch_route_bwd(int mode, const float* d_gate, const float* logits, const int32_t* idx,
                     const void* x, const void* w, int T, int H, int E, int K, int dtype,
                     float* d_logits, float* dw, void* dx, bool dx_write, bool renorm, void* ws, cudaStream_t s);
size_t route_bwd_ws_bytes(int T, int H, int E);
// streaming router backward (bf16; E = 8 or 16 softmax/top-K, E = 1 linear)
bool router_bwd_stream_applies(int mode, int dtype, int H, int E, int K);
int router_bwd_stream_splits(int T, int H, int E);
// the same pass with both products on the warp-level MMA (8 or 16 experts, H % 512 == 0)
bool router_bwd_mma_applies(int mode, int dtype, int H, int E, int K);
int router_bwd_mma_splits(int T, int H);
int launch_router_bwd_mma(const float* d_gate, const float* logits, const int32_t* idx, const void* x,
                          const void* w, int T, int H, int E, int K, bool renorm, float* d_logits, float* part,
                          void* dx, bool dx_write, cudaStream_t s);
int launch_router_bwd_stream(int mode, const float* d_gate, const float* logits, const int32_t* idx, const void* x,
                             const void* w, int T, int H, int E, int K, bool renorm, float* d_logits, float* part,
                             void* dx, bool dx_write, cudaStream_t s);

// dispatch / combine / permute backward
size_t dispatch_ws_bytes(int T, int E, int K);
int launch_dispatch(const void* x, const int32_t* idx, int T, int H, int E, int K, int dtype,
                    int32_t* cu, int32_t* dst_row, int32_t* src_tok, void* xs, void* ws,
                    cudaStream_t s);
int launch_dispatch_static(const void* x, const int32_t* idx, int T, int H, int E, int K, int dtype,
                           int32_t* cu, int32_t* dst_row, int32_t* src_tok, void* xs, cudaStream_t s);
long long dispatch_static_scratch_ints();
long long dispatch_scratch_ints(int T, int E);  // ints of scratch one dispatch call uses
int launch_combine(const void* h, const float* gate, const int32_t* dst_row, const float* scale,
                   const void* residual, const int32_t* out_row, int T, int H, int K, int dtype,
                   void* y, cudaStream_t s);
int launch_permute_bwd(const void* dy, const void* h, const float* gate, const int32_t* dst_row,
                       const float* scale, const int32_t* out_row, const void* dxs, int T, int H,
                       int K, int dtype, void* dh, float* d_gate, float* d_scale, void* dx,
                       cudaStream_t s);

// expert FFN
// gather (nullable): row r of the FFN input is row gather[r] of xs [gather_n, H]
// (the dispatch gather fused into the gate/up operand load).  ws (nullable):
// with expert_ffn_ws_bytes() bytes, the bf16 down projection may split its
// last round of tiles along K (fp32 partials and arrival counters in ws)
int launch_expert_ffn(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                      const void* wd, int E, int H, int Hp, int dtype, void* act, void* gu, void* h,
                      cudaStream_t s, const int32_t* gather = nullptr, int gather_n = 0, void* ws = nullptr,
                      size_t ws_bytes = 0);
size_t expert_ffn_ws_bytes();
int launch_expert_ffn_bwd(const void* xs, const int32_t* cu, int rows, const void* wg, const void* wu,
                          const void* wd, int E, int H, int Hp, const void* gu, const void* act, const void* dh,
                          void* dxs, float* dwg, float* dwu, float* dwd, void* ws, cudaStream_t s);
size_t expert_ffn_bwd_ws_bytes(int rows, int Hp);

// failure-detection probe (a bounded wait that times out)
int launch_wait_probe(unsigned long long wait_cycles, cudaStream_t s);

// MoD
int launch_mod_select(const void* x, const void* w, int B, int L, int H, int C, int dtype,
                      float* score, int32_t* sel, float* sel_score, uint8_t* mask, void* x_sel,
                      void* y_skip, cudaStream_t s);

// Generic SIMT GEMM (fp32 accumulate):  C[m, n] (+)= sum_k A(m, k) * B(k, n)
//   A(m,k) = A[m*a_sm + k*a_sk], B(k,n) = B[g*b_sg + k*b_sk + n*b_sn]
//   Grouped when `cu` != nullptr: group g = blockIdx.z covers rows [cu[g], cu[g+1]).
//   epilogue: 0 store, 1 accumulate into C, 2 store + bias[n] (fp32 only).
//   swiglu: B2 (same strides) is the up projection; C = silu(A.B) * (A.B2).
struct SimtGemmArgs {
  const void* A; long long a_sm, a_sk;
  const void* B; const void* B2; long long b_sg, b_sk, b_sn;
  void* C; long long c_sm;
  const float* bias;
  const int32_t* cu;
  int M, N, K, groups;
  int epilogue;
  bool swiglu;
  const int32_t* a_rows = nullptr;  // when set, row m of A is row a_rows[m] of the A matrix
};
int launch_simt_gemm(const SimtGemmArgs& a, int in_dtype_a, int in_dtype_b, int out_dtype,
                     cudaStream_t s);

}  // namespace moe
