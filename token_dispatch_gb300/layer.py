"""Host-side composition of the libmoe calls into a layer step.

PyTorch only allocates device buffers and supplies the stream; every step of
the layer runs in libmoe's kernels.  Nothing here synchronises the host with the
device: the row split per expert stays on the device (cu_seqlens).

    MoE forward:  moe_route -> moe_dispatch -> moe_expert_ffn -> moe_combine
                  (or moe_dispatch writing index maps only -> moe_expert_ffn_gather,
                  whose gate/up GEMM reads the rows of x itself)
    backward:     moe_permute_bwd (dh, d_gate, dx from dxs) -> moe_route_bwd
    MoD front:    mod_select (scores, capacity top-C, gather, skip copy) -> MoE on the
                  selected tokens -> moe_combine(row_scale = score, residual = x,
                  out_row = selected rows); route backward through
                  moe_permute_bwd(d_scale) and moe_route_bwd(MOE_ROUTE_MOD_LINEAR).
"""
from __future__ import annotations

import torch

from . import _lib as L

_TDT = {"f32": torch.float32, "bf16": torch.bfloat16}
_CDT = {"f32": L.MOE_F32, "bf16": L.MOE_BF16}


def _ws(nbytes: int, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class MoEBuffers:
    """Device buffers of one MoE layer call (T tokens, H, E, K, Hp)."""

    def __init__(self, T, H, E, K, Hp, dtype: str, device, backward: bool = True, train: bool = False):
        self.T, self.H, self.E, self.K, self.Hp, self.dtype = T, H, E, K, Hp, dtype
        self.cdt = _CDT[dtype]
        tdt = _TDT[dtype]
        R = T * K
        dev = device
        f32, i32 = torch.float32, torch.int32
        self.logits = torch.empty((T, E), dtype=f32, device=dev)
        self.idx = torch.empty((T, K), dtype=i32, device=dev)
        self.gate = torch.empty((T, K), dtype=f32, device=dev)
        self.cu = torch.empty((E + 1,), dtype=i32, device=dev)
        self.dst_row = torch.empty((R,), dtype=i32, device=dev)
        self.src_tok = torch.empty((R,), dtype=i32, device=dev)
        self.xs = torch.empty((R, H), dtype=tdt, device=dev)
        self.act = torch.empty((R, Hp), dtype=tdt, device=dev)
        self.h = torch.empty((R, H), dtype=tdt, device=dev)
        self.y = torch.empty((T, H), dtype=tdt, device=dev)
        self.ws_dispatch_bytes = L.moe_workspace_bytes(L.MOE_OP_DISPATCH, T, H, E, K, Hp)
        self.ws_dispatch = _ws(self.ws_dispatch_bytes, dev)
        self.ws_route_bytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE, T, H, E, K, Hp)
        self.ws_route = _ws(self.ws_route_bytes, dev)
        # the expert FFN's optional workspace (bf16: the down projection's
        # last round split along K)
        self.ws_ffn_bytes = L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN, T, H, E, K, Hp) if dtype == "bf16" else 0
        self.ws_ffn = _ws(self.ws_ffn_bytes, dev)
        if backward:
            self.dh = torch.empty((R, H), dtype=tdt, device=dev)
            self.d_gate = torch.empty((T, K), dtype=f32, device=dev)
            self.d_logits = torch.empty((T, E), dtype=f32, device=dev)
            self.dw_router = torch.empty((H, E), dtype=f32, device=dev)
            self.dx = torch.empty((T, H), dtype=tdt, device=dev)
            self.ws_bwd_bytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, T, H, E, K, Hp)
            self.ws_bwd = _ws(self.ws_bwd_bytes, dev)
        self.gu = None
        if train:  # the expert backward: saved [g | u], dxs, fp32 weight gradients
            self.gu = torch.empty((R, 2 * Hp), dtype=tdt, device=dev)
            self.dxs = torch.empty((R, H), dtype=tdt, device=dev)
            self.dw_gate = torch.empty((E, H, Hp), dtype=f32, device=dev)
            self.dw_up = torch.empty((E, H, Hp), dtype=f32, device=dev)
            self.dw_down = torch.empty((E, H, Hp), dtype=f32, device=dev)
            self.ws_ffn_bwd_bytes = L.moe_workspace_bytes(L.MOE_OP_EXPERT_FFN_BWD, T, H, E, K, Hp)
            self.ws_ffn_bwd = _ws(self.ws_ffn_bwd_bytes, dev)


def moe_forward(b: MoEBuffers, x, w_router, logit_bias, w_gate, w_up, w_down, stream=None,
                row_scale=None, residual=None, out_row=None, y=None, route_flags=0, fused_gather=None):
    """One MoE forward pass into the buffers of ``b`` (y defaults to ``b.y``);
    ``route_flags``: MOE_ROUTE_RENORM / MOE_ROUTE_BIAS_SELECT gate options.
    ``fused_gather``: dispatch writes only the index maps and the expert FFN
    reads the rows of x itself (moe_expert_ffn_gather); off by default (the
    row-by-row operand fetch measured 7-11% slower than the gather kernel plus
    the FFN on the dispatched rows), and never with train=True buffers (the
    expert backward reads the dispatched rows)."""
    T, H, E, K, Hp, dt = b.T, b.H, b.E, b.K, b.Hp, b.cdt
    if fused_gather is None or b.gu is not None:
        fused_gather = False
    L.moe_route_ex(x, w_router, logit_bias, T, H, E, K, dt, route_flags, b.logits, b.idx, b.gate, b.ws_route,
                   b.ws_route_bytes, stream=stream)
    L.moe_dispatch(x, b.idx, T, H, E, K, dt, b.cu, b.dst_row, b.src_tok, None if fused_gather else b.xs,
                   b.ws_dispatch, b.ws_dispatch_bytes, stream=stream)
    if fused_gather:
        L.moe_expert_ffn_gather(x, b.src_tok, T, b.cu, T * K, w_gate, w_up, w_down, E, H, Hp, dt, b.act, b.gu, b.h,
                                b.ws_ffn, b.ws_ffn_bytes, stream=stream)
    else:
        L.moe_expert_ffn_ex(b.xs, b.cu, T * K, w_gate, w_up, w_down, E, H, Hp, dt, b.act, b.gu, b.h,
                            b.ws_ffn, b.ws_ffn_bytes, stream=stream)
    L.moe_combine(b.h, b.gate, b.dst_row, row_scale, residual, out_row, T, H, K, dt,
                  b.y if y is None else y, stream=stream)


def moe_backward(b: MoEBuffers, x, w_router, dy, dxs, stream=None, row_scale=None, out_row=None,
                 d_scale=None, route_flags=0):
    """Gate and dispatch/combine backward: dh, d_gate, d_logits, dw_router and
    dx = (adjoint of the gather applied to dxs) + router contribution."""
    T, H, E, K, dt = b.T, b.H, b.E, b.K, b.cdt
    L.moe_permute_bwd(dy, b.h, b.gate, b.dst_row, row_scale, out_row, dxs, T, H, K, dt, b.dh,
                      b.d_gate, d_scale, b.dx, stream=stream)
    renorm = L.MOE_ROUTE_GATE_RENORM if route_flags & L.MOE_ROUTE_RENORM else 0
    L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | renorm, b.d_gate, b.logits, b.idx, x, w_router, T, H, E, K, dt,
                    b.d_logits, b.dw_router, b.dx, b.ws_bwd, b.ws_bwd_bytes, stream=stream)


def moe_train_backward(b: MoEBuffers, x, w_router, w_gate, w_up, w_down, dy, stream=None, route_flags=0):
    """Full backward of the layer (buffers made with train=True, forward run
    with them): dh and d_gate, the expert backward (dxs and the three weight
    gradients), dx = sum_k dxs[row(t,k)] plus the router's share, dw_router."""
    T, H, E, K, Hp, dt = b.T, b.H, b.E, b.K, b.Hp, b.cdt
    L.moe_permute_bwd(dy, b.h, b.gate, b.dst_row, None, None, None, T, H, K, dt, b.dh, b.d_gate, None, None,
                      stream=stream)
    L.moe_expert_ffn_bwd(b.xs, b.cu, T * K, w_gate, w_up, w_down, E, H, Hp, dt, b.gu, b.act, b.dh, b.dxs,
                         b.dw_gate, b.dw_up, b.dw_down, b.ws_ffn_bwd, b.ws_ffn_bwd_bytes, stream=stream)
    L.moe_permute_bwd(None, None, b.gate, b.dst_row, None, None, b.dxs, T, H, K, dt, None, None, None, b.dx,
                      stream=stream)
    renorm = L.MOE_ROUTE_GATE_RENORM if route_flags & L.MOE_ROUTE_RENORM else 0
    L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | renorm, b.d_gate, b.logits, b.idx, x, w_router, T, H, E, K, dt,
                    b.d_logits, b.dw_router, b.dx, b.ws_bwd, b.ws_bwd_bytes, stream=stream)


class MoDBuffers:
    """Buffers of the MoD front end: B sequences of L tokens, capacity C."""

    def __init__(self, B, Lseq, C, H, E, K, Hp, dtype: str, device, backward: bool = True):
        self.B, self.L, self.C, self.H = B, Lseq, C, H
        self.cdt = _CDT[dtype]
        tdt = _TDT[dtype]
        n = B * Lseq
        self.score = torch.empty((n,), dtype=torch.float32, device=device)
        self.sel = torch.empty((B * C,), dtype=torch.int32, device=device)  # flat token rows
        self.sel_score = torch.empty((B * C,), dtype=torch.float32, device=device)
        self.mask = torch.empty((n,), dtype=torch.uint8, device=device)
        self.x_sel = torch.empty((B * C, H), dtype=tdt, device=device)
        self.y = torch.empty((n, H), dtype=tdt, device=device)
        self.moe = MoEBuffers(B * C, H, E, K, Hp, dtype, device, backward=backward)
        if backward:
            self.d_score = torch.empty((B * C,), dtype=torch.float32, device=device)
            self.dw_mod = torch.empty((H,), dtype=torch.float32, device=device)
            self.ws_lin_bytes = L.moe_workspace_bytes(L.MOE_OP_ROUTE_BWD, B * C, H, 1, 1, 0)
            self.ws_lin = _ws(self.ws_lin_bytes, device)


def mod_forward(m: MoDBuffers, x, w_mod, w_router, w_gate, w_up, w_down, stream=None):
    """MoD + MoE forward: y = x + s * MoE(x) on the selected tokens, y = x elsewhere."""
    b = m.moe
    L.mod_select(x, w_mod, m.B, m.L, m.H, m.C, m.cdt, m.score, m.sel, m.sel_score, m.mask, m.x_sel,
                 m.y, stream=stream)
    moe_forward(b, m.x_sel, w_router, None, w_gate, w_up, w_down, stream=stream,
                row_scale=m.sel_score, residual=x, out_row=m.sel, y=m.y)


def mod_route_backward(m: MoDBuffers, w_router, w_mod, dy, stream=None):
    """Route backward of the MoD + MoE layer with the expert outputs held fixed:
    d_gate of the MoE router, d_score = <dy, MoE(x)> of the MoD router, dw_router,
    dw_mod and their input gradients accumulated into m.moe.dx."""
    b = m.moe
    T, H, E, K, dt = b.T, b.H, b.E, b.K, b.cdt
    L.moe_permute_bwd(dy, b.h, b.gate, b.dst_row, m.sel_score, m.sel, None, T, H, K, dt, b.dh,
                      b.d_gate, m.d_score, None, stream=stream)
    L.moe_route_bwd(L.MOE_ROUTE_SOFTMAX_TOPK | L.MOE_ROUTE_DX_WRITE, b.d_gate, b.logits, b.idx, m.x_sel, w_router, T, H, E,
                    K, dt, b.d_logits, b.dw_router, b.dx, b.ws_bwd, b.ws_bwd_bytes, stream=stream)
    L.moe_route_bwd(L.MOE_ROUTE_MOD_LINEAR, m.d_score, None, None, m.x_sel, w_mod, T, H, 1, 1, dt,
                    None, m.dw_mod, b.dx, m.ws_lin, m.ws_lin_bytes, stream=stream)
