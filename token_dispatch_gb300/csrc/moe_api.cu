// The C ABI: argument validation, workspace sizing and launches.
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

// Per-device error word: kernels that bound a wait or check an index write a
// status code here instead of trapping.
__device__ unsigned g_moe_device_error;

unsigned long long g_kernel_launches = 0;

static std::atomic<unsigned*> g_err_ptr[64];
static std::mutex g_err_mu;

// The device address of the error word, looked up once per device under a lock
// (two host threads making their first call at the same time both get it);
// later calls read the published address without locking.
unsigned* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned* known = g_err_ptr[dev].load(std::memory_order_acquire);
  if (known) return known;
  std::lock_guard<std::mutex> lock(g_err_mu);
  known = g_err_ptr[dev].load(std::memory_order_relaxed);
  if (!known) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_device_error) != cudaSuccess) return nullptr;
    known = static_cast<unsigned*>(p);
    g_err_ptr[dev].store(known, std::memory_order_release);
  }
  return known;
}

}  // namespace moe

using namespace moe;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// all non-null pointers 16-byte aligned
inline bool all_aligned(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p && !aligned16(p)) return false;
  return true;
}

inline bool valid_dtype(int dt) { return dt == MOE_F32 || dt == MOE_BF16; }
inline int vec_elems(int dt) { return dt == MOE_BF16 ? 8 : 4; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* moe_status_str(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_version(void) { return 100; }

unsigned long long moe_kernel_launches(void) { return __atomic_load_n(&g_kernel_launches, __ATOMIC_RELAXED); }

size_t moe_workspace_bytes(int op, int T, int H, int E, int K, int Hp) {
  if (T < 0 || H < 0 || E < 0 || K < 0) return 0;
  switch (op) {
    case MOE_OP_ROUTE: return (E > 0 && H > 0) ? route_ws_bytes(T, H, E) : 0;
    case MOE_OP_DISPATCH: return E > 0 ? dispatch_ws_bytes(T, E, K) : 0;
    case MOE_OP_ROUTE_BWD: return (E > 0 && H > 0) ? route_bwd_ws_bytes(T, H, E) : 0;
    case MOE_OP_EXPERT_FFN: return expert_ffn_ws_bytes();
    case MOE_OP_EXPERT_FFN_BWD: return Hp > 0 ? expert_ffn_bwd_ws_bytes((int)((long long)T * K), Hp) : 0;
    default: return 0;
  }
}

int moe_check_wait_timeout(unsigned long long wait_cycles, void* stream) {
  if (wait_cycles == 0 || wait_cycles > (1ull << 31)) return MOE_ERR_INVALID_ARG;
  return launch_wait_probe(wait_cycles, as_stream(stream));
}

int moe_last_device_error(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned* p = device_error_word();
  if (!p) return MOE_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    unsigned z = 0;
    if (cudaMemcpy(p, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return (int)v;
}

int moe_route_ex(const void* x, const void* w_router, const float* logit_bias, int T, int H, int E, int K,
                 int dtype, int flags, float* logits, int32_t* topk_idx, float* topk_gate, void* ws,
                 size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || E < 1 || E > 1024 || K < 1 || K > E || K > 16)
    return MOE_ERR_INVALID_ARG;
  if (flags & ~(MOE_ROUTE_RENORM | MOE_ROUTE_BIAS_SELECT)) return MOE_ERR_INVALID_ARG;
  if ((T > 0 && (!x || !logits || !topk_idx || !topk_gate)) || !w_router) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, w_router, logit_bias, logits, topk_idx, topk_gate, ws})) return MOE_ERR_MISALIGNED;
  if (H % vec_elems(dtype) != 0 || E % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_BF16 && E % 8 != 0) return MOE_ERR_UNSUPPORTED;  // 16-byte rows of W_r for TMA
  if (T == 0) return MOE_OK;
  const size_t need = dtype == MOE_BF16 ? route_ws_bytes(T, H, E) : 0;
  if (need > 0 && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  return launch_route(x, w_router, logit_bias, T, H, E, K, dtype, flags, logits, topk_idx, topk_gate, ws,
                      as_stream(stream));
}

int moe_route(const void* x, const void* w_router, const float* logit_bias, int T, int H, int E,
              int K, int dtype, float* logits, int32_t* topk_idx, float* topk_gate, void* ws,
              size_t ws_bytes, void* stream) {
  return moe_route_ex(x, w_router, logit_bias, T, H, E, K, dtype, 0, logits, topk_idx, topk_gate, ws, ws_bytes,
                      stream);
}

int moe_dispatch(const void* x, const int32_t* topk_idx, int T, int H, int E, int K, int dtype,
                 int32_t* cu_seqlens, int32_t* dst_row, int32_t* src_tok, void* xs, void* ws,
                 size_t ws_bytes, void* stream) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || E < 1 || E > 1024 || K < 1 || K > E || K > 16)
    return MOE_ERR_INVALID_ARG;
  if ((long long)T * K > 0x7fffffffll) return MOE_ERR_UNSUPPORTED;
  if (!cu_seqlens || (T > 0 && (!topk_idx || !dst_row || !src_tok || (xs && !x))))
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, topk_idx, cu_seqlens, dst_row, src_tok, xs, ws})) return MOE_ERR_MISALIGNED;
  if (H % vec_elems(dtype) != 0) return MOE_ERR_UNSUPPORTED;
  size_t need = dispatch_ws_bytes(T, E, K);
  if (need > 0 && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  return launch_dispatch(x, topk_idx, T, H, E, K, dtype, cu_seqlens, dst_row, src_tok, xs, ws,
                         as_stream(stream));
}

int moe_dispatch_noalloc(const void* x, const int32_t* topk_idx, int T, int H, int E, int K, int dtype,
                         int32_t* cu_seqlens, int32_t* dst_row, int32_t* src_tok, void* xs, void* stream) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || E < 1 || E > 1024 || K < 1 || K > E || K > 16)
    return MOE_ERR_INVALID_ARG;
  if ((long long)T * K > 0x7fffffffll) return MOE_ERR_UNSUPPORTED;
  if (!cu_seqlens || (T > 0 && (!topk_idx || !dst_row || !src_tok || (xs && !x))))
    return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, topk_idx, cu_seqlens, dst_row, src_tok, xs})) return MOE_ERR_MISALIGNED;
  if (H % vec_elems(dtype) != 0) return MOE_ERR_UNSUPPORTED;
  if (dispatch_scratch_ints(T, E) > dispatch_static_scratch_ints()) return MOE_ERR_WORKSPACE;
  return launch_dispatch_static(x, topk_idx, T, H, E, K, dtype, cu_seqlens, dst_row, src_tok, xs,
                                as_stream(stream));
}

static int check_expert_ffn(const void* xs, const int32_t* cu_seqlens, int rows, const void* w_gate,
                            const void* w_up, const void* w_down, int E, int H, int Hp, int dtype) {
  if (!valid_dtype(dtype) || rows < 0 || E < 1 || H < 1 || Hp < 1) return MOE_ERR_INVALID_ARG;
  if (!cu_seqlens || !w_gate || !w_up || !w_down || (rows > 0 && !xs)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({xs, cu_seqlens, w_gate, w_up, w_down})) return MOE_ERR_MISALIGNED;
  if (H % vec_elems(dtype) != 0 || Hp % vec_elems(dtype) != 0) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_BF16 && (H % 64 != 0 || Hp % 64 != 0 || E > 1024)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int moe_expert_ffn_ex(const void* xs, const int32_t* cu_seqlens, int rows, const void* w_gate, const void* w_up,
                      const void* w_down, int E, int H, int Hp, int dtype, void* act, void* gu, void* h, void* ws,
                      size_t ws_bytes, void* stream) {
  int st = check_expert_ffn(xs, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype);
  if (st != MOE_OK) return st;
  if (rows > 0 && (!act || !h)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({act, gu, h, ws})) return MOE_ERR_MISALIGNED;
  if (gu && dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  return launch_expert_ffn(xs, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype, act, gu, h,
                           as_stream(stream), nullptr, 0, ws, ws_bytes);
}

int moe_expert_ffn_gather(const void* x, const int32_t* src_tok, int T, const int32_t* cu_seqlens, int rows,
                          const void* w_gate, const void* w_up, const void* w_down, int E, int H, int Hp, int dtype,
                          void* act, void* gu, void* h, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0) return MOE_ERR_INVALID_ARG;
  int st = check_expert_ffn(x, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype);
  if (st != MOE_OK) return st;
  if (rows > 0 && (!act || !h || !src_tok || T < 1)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({act, gu, h, src_tok, ws})) return MOE_ERR_MISALIGNED;
  if (gu && dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  return launch_expert_ffn(x, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype, act, gu, h,
                           as_stream(stream), src_tok, T, ws, ws_bytes);
}

int moe_expert_ffn(const void* xs, const int32_t* cu_seqlens, int rows, const void* w_gate,
                   const void* w_up, const void* w_down, int E, int H, int Hp, int dtype, void* act,
                   void* h, void* ws, size_t ws_bytes, void* stream) {
  return moe_expert_ffn_ex(xs, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype, act, nullptr, h, ws,
                           ws_bytes, stream);
}

int moe_expert_ffn_bwd(const void* xs, const int32_t* cu_seqlens, int rows, const void* w_gate, const void* w_up,
                       const void* w_down, int E, int H, int Hp, int dtype, const void* gu, const void* act,
                       const void* dh, void* dxs, float* dw_gate, float* dw_up, float* dw_down, void* ws,
                       size_t ws_bytes, void* stream) {
  int st = check_expert_ffn(xs, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype);
  if (st != MOE_OK) return st;
  if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (rows > 0 && (!gu || !act || !dh)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({gu, act, dh, dxs, dw_gate, dw_up, dw_down, ws})) return MOE_ERR_MISALIGNED;
  if (rows > 0 && (!ws || ws_bytes < expert_ffn_bwd_ws_bytes(rows, Hp))) return MOE_ERR_WORKSPACE;
  return launch_expert_ffn_bwd(xs, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, gu, act, dh, dxs, dw_gate,
                               dw_up, dw_down, ws, as_stream(stream));
}

int moe_combine(const void* h, const float* gate, const int32_t* dst_row, const float* row_scale,
                const void* residual, const int32_t* out_row, int T, int H, int K, int dtype,
                void* y, void* stream) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || K < 1 || K > 16) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!h || !gate || !y)) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({h, gate, dst_row, row_scale, residual, out_row, y})) return MOE_ERR_MISALIGNED;
  if (H % vec_elems(dtype) != 0) return MOE_ERR_UNSUPPORTED;
  return launch_combine(h, gate, dst_row, row_scale, residual, out_row, T, H, K, dtype, y,
                        as_stream(stream));
}

int moe_route_bwd(int mode, const float* d_gate, const float* logits, const int32_t* topk_idx,
                  const void* x, const void* w_router, int T, int H, int E, int K, int dtype,
                  float* d_logits, float* dw_router, void* dx, void* ws, size_t ws_bytes,
                  void* stream) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || E < 1 || E > 1024 || K < 1 || K > E || K > 16)
    return MOE_ERR_INVALID_ARG;
  const bool dx_write = (mode & MOE_ROUTE_DX_WRITE) != 0;
  const bool renorm = (mode & MOE_ROUTE_GATE_RENORM) != 0;
  mode &= ~(MOE_ROUTE_DX_WRITE | MOE_ROUTE_GATE_RENORM);
  if (renorm && mode != MOE_ROUTE_SOFTMAX_TOPK) return MOE_ERR_INVALID_ARG;
  if (mode == MOE_ROUTE_SOFTMAX_TOPK) {
    if (T > 0 && (!logits || !topk_idx)) return MOE_ERR_INVALID_ARG;
    if (E % 4 != 0) return MOE_ERR_UNSUPPORTED;
  } else if (mode == MOE_ROUTE_MOD_LINEAR) {
    if (E != 1 || K != 1) return MOE_ERR_INVALID_ARG;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  if (T > 0 && !d_gate) return MOE_ERR_INVALID_ARG;
  if ((dw_router || dx) && (T > 0 && !x)) return MOE_ERR_INVALID_ARG;
  if (dx && !w_router) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({d_gate, logits, topk_idx, x, w_router, d_logits, dw_router, dx, ws}))
    return MOE_ERR_MISALIGNED;
  if (H % vec_elems(dtype) != 0) return MOE_ERR_UNSUPPORTED;
  size_t need = route_bwd_ws_bytes(T, H, E);
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  return launch_route_bwd(mode, d_gate, logits, topk_idx, x, w_router, T, H, E, K, dtype, d_logits,
                          dw_router, dx, dx_write, renorm, ws, as_stream(stream));
}

int moe_permute_bwd(const void* dy, const void* h, const float* gate, const int32_t* dst_row,
                    const float* row_scale, const int32_t* out_row, const void* dxs, int T, int H,
                    int K, int dtype, void* dh, float* d_gate, float* d_scale, void* dx,
                    void* stream) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || K < 1 || K > 16) return MOE_ERR_INVALID_ARG;
  if (T > 0 && !gate) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (dh || d_gate || d_scale) && !dy) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (d_gate || d_scale) && !h) return MOE_ERR_INVALID_ARG;
  if (dx && !dxs) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({dy, h, gate, dst_row, row_scale, out_row, dxs, dh, d_gate, d_scale, dx}))
    return MOE_ERR_MISALIGNED;
  if (H % vec_elems(dtype) != 0) return MOE_ERR_UNSUPPORTED;
  return launch_permute_bwd(dy, h, gate, dst_row, row_scale, out_row, dxs, T, H, K, dtype, dh,
                            d_gate, d_scale, dx, as_stream(stream));
}

int mod_select(const void* x, const void* w_mod, int B, int L, int H, int C, int dtype,
               float* score, int32_t* sel, float* sel_score, uint8_t* mask, void* x_sel,
               void* y_skip, void* ws, size_t ws_bytes, void* stream) {
  (void)ws; (void)ws_bytes;
  if (!valid_dtype(dtype) || B < 0 || L < 1 || L > 8192 || H < 1 || C < 0 || C > L)
    return MOE_ERR_INVALID_ARG;
  if (B > 0 && (!x || !w_mod || !score || !mask || (C > 0 && !sel))) return MOE_ERR_INVALID_ARG;
  if (!all_aligned({x, w_mod, score, sel, sel_score, mask, x_sel, y_skip})) return MOE_ERR_MISALIGNED;
  if (H % vec_elems(dtype) != 0) return MOE_ERR_UNSUPPORTED;
  return launch_mod_select(x, w_mod, B, L, H, C, dtype, score, sel, sel_score, mask, x_sel, y_skip,
                           as_stream(stream));
}

}  // extern "C"
