"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Each function has the name and argument order of the C entry point.  Tensor
arguments may be torch tensors (their ``data_ptr()`` is passed), raw integer
addresses, or None for nullable pointers.  ``stream`` defaults to torch's
current CUDA stream.  A non-zero status raises ``MoEError``.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_MISALIGNED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_UNSUPPORTED = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_DEVICE_BOUNDS = 7

MOE_F32 = 0
MOE_BF16 = 1

MOE_OP_ROUTE = 0
MOE_OP_DISPATCH = 1
MOE_OP_EXPERT_FFN = 2
MOE_OP_ROUTE_BWD = 3
MOE_OP_MOD_SELECT = 4
MOE_OP_EXPERT_FFN_BWD = 5

MOE_ROUTE_SOFTMAX_TOPK = 0
MOE_ROUTE_MOD_LINEAR = 1
MOE_ROUTE_DX_WRITE = 0x100
MOE_ROUTE_GATE_RENORM = 0x200

MOE_ROUTE_RENORM = 0x1
MOE_ROUTE_BIAS_SELECT = 0x2

EXPORTS = ("moe_status_str", "moe_version", "moe_kernel_launches", "moe_workspace_bytes", "moe_last_device_error",
           "moe_check_wait_timeout",
           "moe_route", "moe_route_ex", "moe_dispatch", "moe_dispatch_noalloc", "moe_expert_ffn",
           "moe_expert_ffn_ex", "moe_expert_ffn_gather", "moe_expert_ffn_bwd", "moe_combine", "moe_route_bwd",
           "moe_permute_bwd", "mod_select", "moe_ep_plan")


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, name: str):
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t

_SIGS = {
    "moe_status_str": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
    "moe_kernel_launches": (ctypes.c_ulonglong, []),
    "moe_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I]),
    "moe_last_device_error": (_I, [_P]),
    "moe_check_wait_timeout": (_I, [ctypes.c_ulonglong, _P]),
    "moe_route": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_route_ex": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_dispatch": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_dispatch_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_expert_ffn": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _Z, _P]),
    "moe_expert_ffn_ex": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_ffn_gather": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_ffn_bwd": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_combine": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_route_bwd": (_I, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_permute_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "mod_select": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_ep_plan": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """The loaded libmoe.  Raises if the library has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so not built at {LIB_PATH}; run "
                               "`python -m token_dispatch_gb300.build` (needs nvcc)")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != MOE_OK:
        raise MoEError(fn, st, moe_status_str(st))


def moe_status_str(status: int) -> str:
    return lib().moe_status_str(status).decode()


def moe_version() -> int:
    return lib().moe_version()


def moe_kernel_launches() -> int:
    return lib().moe_kernel_launches()


def moe_workspace_bytes(op: int, T: int, H: int, E: int, K: int, Hp: int) -> int:
    return lib().moe_workspace_bytes(op, T, H, E, K, Hp)


def moe_last_device_error(stream=None) -> int:
    return lib().moe_last_device_error(_stream(stream))


def moe_check_wait_timeout(wait_cycles, stream=None):
    _check("moe_check_wait_timeout", lib().moe_check_wait_timeout(wait_cycles, _stream(stream)))


def moe_route(x, w_router, logit_bias, T, H, E, K, dtype, logits, topk_idx, topk_gate,
              ws=None, ws_bytes=0, stream=None):
    _check("moe_route", lib().moe_route(_ptr(x), _ptr(w_router), _ptr(logit_bias), T, H, E, K, dtype,
                                        _ptr(logits), _ptr(topk_idx), _ptr(topk_gate), _ptr(ws),
                                        ws_bytes, _stream(stream)))


def moe_route_ex(x, w_router, logit_bias, T, H, E, K, dtype, flags, logits, topk_idx, topk_gate,
                 ws=None, ws_bytes=0, stream=None):
    _check("moe_route_ex", lib().moe_route_ex(_ptr(x), _ptr(w_router), _ptr(logit_bias), T, H, E, K, dtype, flags,
                                              _ptr(logits), _ptr(topk_idx), _ptr(topk_gate), _ptr(ws),
                                              ws_bytes, _stream(stream)))


def moe_dispatch(x, topk_idx, T, H, E, K, dtype, cu_seqlens, dst_row, src_tok, xs, ws, ws_bytes,
                 stream=None):
    _check("moe_dispatch", lib().moe_dispatch(_ptr(x), _ptr(topk_idx), T, H, E, K, dtype,
                                              _ptr(cu_seqlens), _ptr(dst_row), _ptr(src_tok), _ptr(xs),
                                              _ptr(ws), ws_bytes, _stream(stream)))


def moe_dispatch_noalloc(x, topk_idx, T, H, E, K, dtype, cu_seqlens, dst_row, src_tok, xs, stream=None):
    """moe_dispatch with the count table in a library-owned static device array
    (for callers that cannot allocate); see include/moe.h for its limits."""
    _check("moe_dispatch_noalloc", lib().moe_dispatch_noalloc(_ptr(x), _ptr(topk_idx), T, H, E, K, dtype,
                                                              _ptr(cu_seqlens), _ptr(dst_row), _ptr(src_tok),
                                                              _ptr(xs), _stream(stream)))


def moe_expert_ffn(xs, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype, act, h,
                   ws=None, ws_bytes=0, stream=None):
    _check("moe_expert_ffn", lib().moe_expert_ffn(_ptr(xs), _ptr(cu_seqlens), rows, _ptr(w_gate),
                                                  _ptr(w_up), _ptr(w_down), E, H, Hp, dtype, _ptr(act),
                                                  _ptr(h), _ptr(ws), ws_bytes, _stream(stream)))


def moe_expert_ffn_ex(xs, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype, act, gu, h,
                      ws=None, ws_bytes=0, stream=None):
    _check("moe_expert_ffn_ex", lib().moe_expert_ffn_ex(_ptr(xs), _ptr(cu_seqlens), rows, _ptr(w_gate), _ptr(w_up),
                                                        _ptr(w_down), E, H, Hp, dtype, _ptr(act), _ptr(gu), _ptr(h),
                                                        _ptr(ws), ws_bytes, _stream(stream)))


def moe_expert_ffn_gather(x, src_tok, T, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype, act, gu, h,
                          ws=None, ws_bytes=0, stream=None):
    _check("moe_expert_ffn_gather", lib().moe_expert_ffn_gather(
        _ptr(x), _ptr(src_tok), T, _ptr(cu_seqlens), rows, _ptr(w_gate), _ptr(w_up), _ptr(w_down), E, H, Hp, dtype,
        _ptr(act), _ptr(gu), _ptr(h), _ptr(ws), ws_bytes, _stream(stream)))


def moe_expert_ffn_bwd(xs, cu_seqlens, rows, w_gate, w_up, w_down, E, H, Hp, dtype, gu, act, dh, dxs,
                       dw_gate, dw_up, dw_down, ws, ws_bytes, stream=None):
    _check("moe_expert_ffn_bwd", lib().moe_expert_ffn_bwd(_ptr(xs), _ptr(cu_seqlens), rows, _ptr(w_gate),
                                                          _ptr(w_up), _ptr(w_down), E, H, Hp, dtype, _ptr(gu),
                                                          _ptr(act), _ptr(dh), _ptr(dxs), _ptr(dw_gate),
                                                          _ptr(dw_up), _ptr(dw_down), _ptr(ws), ws_bytes,
                                                          _stream(stream)))


def moe_combine(h, gate, dst_row, row_scale, residual, out_row, T, H, K, dtype, y, stream=None):
    _check("moe_combine", lib().moe_combine(_ptr(h), _ptr(gate), _ptr(dst_row), _ptr(row_scale),
                                            _ptr(residual), _ptr(out_row), T, H, K, dtype, _ptr(y),
                                            _stream(stream)))


def moe_route_bwd(mode, d_gate, logits, topk_idx, x, w_router, T, H, E, K, dtype, d_logits,
                  dw_router, dx, ws, ws_bytes, stream=None):
    _check("moe_route_bwd", lib().moe_route_bwd(mode, _ptr(d_gate), _ptr(logits), _ptr(topk_idx),
                                                _ptr(x), _ptr(w_router), T, H, E, K, dtype,
                                                _ptr(d_logits), _ptr(dw_router), _ptr(dx), _ptr(ws),
                                                ws_bytes, _stream(stream)))


def moe_permute_bwd(dy, h, gate, dst_row, row_scale, out_row, dxs, T, H, K, dtype, dh, d_gate,
                    d_scale, dx, stream=None):
    _check("moe_permute_bwd", lib().moe_permute_bwd(_ptr(dy), _ptr(h), _ptr(gate), _ptr(dst_row),
                                                    _ptr(row_scale), _ptr(out_row), _ptr(dxs), T, H,
                                                    K, dtype, _ptr(dh), _ptr(d_gate), _ptr(d_scale),
                                                    _ptr(dx), _stream(stream)))


def mod_select(x, w_mod, B, L, H, C, dtype, score, sel, sel_score, mask, x_sel, y_skip,
               ws=None, ws_bytes=0, stream=None):
    _check("mod_select", lib().mod_select(_ptr(x), _ptr(w_mod), B, L, H, C, dtype, _ptr(score),
                                          _ptr(sel), _ptr(sel_score), _ptr(mask), _ptr(x_sel),
                                          _ptr(y_skip), _ptr(ws), ws_bytes, _stream(stream)))


def moe_ep_plan(R, E, S, K, B, counts):
    """Host-side expert-parallel plan from the gathered per-rank expert counts
    (int32 [R, E]).  Returns numpy arrays: piece_count and piece_offset
    [R dst, R src, E], slot_expert [R, B], local_counts [R, E/R + B],
    remote_reads [R]."""
    import numpy as np
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    G = E // R if R > 0 and E % R == 0 else 0
    pc = np.zeros((R, R, E), np.int32)
    po = np.zeros((R, R, E), np.int32)
    se = np.zeros((R, max(B, 0)), np.int32)
    lc = np.zeros((R, G + max(B, 0)), np.int32)
    rr = np.zeros(R, np.int32)

    def a(x):
        return x.ctypes.data_as(ctypes.c_void_p) if x.size else None
    _check("moe_ep_plan", lib().moe_ep_plan(R, E, S, K, B, a(counts), a(pc), a(po), a(se), a(lc), a(rr)))
    return pc, po, se, lc, rr
