/*
 * libmoe — C ABI of the GB300 (sm_103a) MoE / MoD layer hot path.
 *
 * Sources, cited by page title and section:
 *   [FW] "PyTorch MoE/MoD Training Framework: custom CUDA kernels, DeepSpeed and
 *        7x speed-up on T4", section "What's in the box" (routing/gating =
 *        softmax over experts + top-k in one launch; dispatch and combine;
 *        sparse backward of gating and dispatch) and its Mixture-of-Depths
 *        paragraph (part of the tokens skips the layer).
 *   [EP] "Moonshot AI released MoonEP: Mixture-of-Experts training without GPU
 *        idle time", section "Step-by-step" (one contiguous [E(+B), H, H'] weight
 *        tensor per projection, experts addressed by row index; dispatch returns
 *        cu_seqlens) and section "What problem it solves" (maxvio skew; no
 *        per-layer CPU synchronisation).
 *   [T4] "MoE on T4: how to find and remove bottlenecks in training", table
 *        "RMSNorm, RoPE, SwiGLU" (SwiGLU = three matrix products).
 *
 * Conventions for every call:
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller owns all memory.  The library never allocates, frees or
 *     synchronises (except moe_last_device_error, which synchronises `stream`).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously on it.
 *   - Tensors are dense and row-major.  Activation/weight tensors use the
 *     storage type `dtype` (MOE_F32 = float, MOE_BF16 = bfloat16); router logits,
 *     gates, scores and their gradients are always float; indices are int32.
 *   - Every pointer must be 16-byte aligned (MOE_ERR_MISALIGNED otherwise) and
 *     the hidden size H must be a multiple of 8 (bf16) or 4 (fp32).
 *   - Argument errors are reported before anything is launched and nothing is
 *     written.  A CUDA launch error returns MOE_ERR_CUDA.  Kernels never trap:
 *     a device-side wait that exceeds its bound, or an index found out of range,
 *     sets a per-device error word that moe_last_device_error() returns.
 *   - Results are deterministic: the same inputs give bitwise-identical outputs.
 *   - T = tokens, H = hidden size, E = experts, K = experts per token,
 *     Hp = H' = expert FFN intermediate size, R = T*K routed rows.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* bad size, null required pointer, bad enum */
  MOE_ERR_MISALIGNED = 2,     /* a pointer is not 16-byte aligned */
  MOE_ERR_WORKSPACE = 3,      /* workspace missing or smaller than moe_workspace_bytes() */
  MOE_ERR_UNSUPPORTED = 4,    /* valid but unsupported shape/dtype combination */
  MOE_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 6,        /* device: a bounded wait gave up (reported by moe_last_device_error) */
  MOE_ERR_DEVICE_BOUNDS = 7   /* device: an index was out of range (reported by moe_last_device_error) */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* operation ids for moe_workspace_bytes */
enum { MOE_OP_ROUTE = 0, MOE_OP_DISPATCH = 1, MOE_OP_EXPERT_FFN = 2, MOE_OP_ROUTE_BWD = 3, MOE_OP_MOD_SELECT = 4,
       MOE_OP_EXPERT_FFN_BWD = 5 };

/* moe_route_bwd modes; MOE_ROUTE_DX_WRITE may be or-ed in to overwrite dx instead
 * of accumulating into it, MOE_ROUTE_GATE_RENORM when the forward renormalised the
 * gates (moe_route_ex with MOE_ROUTE_RENORM) */
enum { MOE_ROUTE_SOFTMAX_TOPK = 0, MOE_ROUTE_MOD_LINEAR = 1, MOE_ROUTE_DX_WRITE = 0x100,
       MOE_ROUTE_GATE_RENORM = 0x200 };

/* moe_route_ex gate options (bit flags) */
enum { MOE_ROUTE_RENORM = 0x1, MOE_ROUTE_BIAS_SELECT = 0x2 };

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char* moe_status_str(int status);

/* ABI version (major*10000 + minor*100 + patch). */
MOE_API int moe_version(void);

/* Number of CUDA kernels this library has launched in this process (a host-side
 * counter; no device work).  Lets a caller count the launches of a region. */
MOE_API unsigned long long moe_kernel_launches(void);

/* Bytes of device workspace `op` needs for these sizes (0 = none; `ws` may then be
 * NULL).  Sizes not used by `op` are ignored.  Returns 0 for invalid sizes.
 * MOE_OP_EXPERT_FFN: the workspace is optional (see moe_expert_ffn). */
MOE_API size_t moe_workspace_bytes(int op, int T, int H, int E, int K, int Hp);

/* Synchronises `stream`, then returns and clears the current device's error word:
 * MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_BOUNDS (MOE_ERR_CUDA if the
 * synchronisation itself failed). */
MOE_API int moe_last_device_error(void* stream);

/* Diagnostic of the device-side failure detection.  Launches one kernel whose
 * single thread waits, with the same bounded wait every pipelined kernel of this
 * library uses, on a barrier that nothing ever arrives at.  After `wait_cycles` SM
 * clock cycles (1 .. 2^31) it gives up and records MOE_ERR_TIMEOUT in the device
 * error word, as a stalled copy or MMA pipeline would; nothing traps and the
 * context stays usable.  Returns the launch status (MOE_ERR_INVALID_ARG for
 * wait_cycles out of range); read the outcome with moe_last_device_error. */
MOE_API int moe_check_wait_timeout(unsigned long long wait_cycles, void* stream);

/*
 * Router: GEMM, softmax over experts and top-K gate       [FW "What's in the box"]
 *
 *   logits[t,e] = sum_h x[t,h] * w_router[h,e] + logit_bias[e]
 *   p[t,:]      = softmax(logits[t,:])
 *   topk_idx[t,:]  = the K experts with the largest logits, ordered by decreasing
 *                    logit, equal logits by increasing expert index
 *   topk_gate[t,k] = p[t, topk_idx[t,k]]   (no renormalisation after top-k)
 *
 *   x          [T,H]   dtype           w_router [H,E] dtype
 *   logit_bias [E]     float, nullable (added before softmax and selection)
 *   logits     [T,E]   float out (kept for moe_route_bwd)
 *   topk_idx   [T,K]   int32 out;  topk_gate [T,K] float out
 *   1 <= K <= E <= 1024, K <= 16.  bf16 needs E % 8 == 0.
 *   Workspace: moe_workspace_bytes(MOE_OP_ROUTE, T, H, E, K, 0) bytes (bf16 only):
 *   partial sums of the router GEMM over slices of H, added in a fixed order, for
 *   shapes whose token tiles alone would leave SMs idle; 0 (ws may be NULL) when the
 *   token tiles fill the GPU and for E = 8 or 16 with H a multiple of 512 up to 4096
 *   (those stream x through registers in one launch).  Results are the same bits on
 *   every run for the same inputs.
 */
MOE_API int moe_route(const void* x, const void* w_router, const float* logit_bias,
              int T, int H, int E, int K, int dtype,
              float* logits, int32_t* topk_idx, float* topk_gate,
              void* ws, size_t ws_bytes, void* stream);

/*
 * Router with gate options, for a drop-in replacement of a Mixtral-style sparse
 * MoE block                              [FW "How it looks in practice"]
 *
 * moe_route with `flags`, a bitwise or of
 *   MOE_ROUTE_RENORM       topk_gate[t,k] = p[t,topk_idx[t,k]] / sum_k' p[t,topk_idx[t,k']]
 *                          (the K gates of a token sum to 1, as in the Mixtral block);
 *   MOE_ROUTE_BIAS_SELECT  logit_bias shifts only the selection: topk_idx = the top K of
 *                          x w_router + logit_bias (same order and ties as above), while
 *                          logits, p and the gates are those of x w_router alone.
 * flags = 0 is exactly moe_route; other bits return MOE_ERR_INVALID_ARG.  Arguments,
 * layouts, workspace and errors as moe_route.  The backward of renormalised gates is
 * moe_route_bwd with MOE_ROUTE_GATE_RENORM; the selection-only bias needs no flag there
 * (the stored logits are unbiased).
 */
MOE_API int moe_route_ex(const void* x, const void* w_router, const float* logit_bias,
              int T, int H, int E, int K, int dtype, int flags,
              float* logits, int32_t* topk_idx, float* topk_gate,
              void* ws, size_t ws_bytes, void* stream);

/*
 * Dispatch: expert histogram, prefix sum, permutation, gather
 *                              [FW "What's in the box"; EP "Step-by-step"]
 *
 *   cu_seqlens[0] = 0, cu_seqlens[e+1] = cu_seqlens[e] + #{(t,k): topk_idx[t,k] = e},
 *   so cu_seqlens[E] = T*K.  Rows of expert e are [cu_seqlens[e], cu_seqlens[e+1])
 *   of one contiguous expert-sorted buffer, in increasing token order (stable).
 *   dst_row[t*K+k] = row of pair (t,k);  src_tok[row] = t;  xs[row,:] = x[t,:].
 *
 *   x [T,H] dtype; topk_idx [T,K] int32 with distinct experts per token in [0,E)
 *   cu_seqlens [E+1], dst_row [T*K], src_tok [T*K] int32 out; xs [T*K,H] dtype out,
 *   nullable: without xs only the index maps are written (x may then be NULL)
 *   and moe_expert_ffn_gather reads the rows of x itself.
 *   An expert id outside [0,E) sets MOE_ERR_DEVICE_BOUNDS; its pair is dropped.
 *   Workspace: moe_workspace_bytes(MOE_OP_DISPATCH, T, 0, E, K, 0) bytes.
 */
MOE_API int moe_dispatch(const void* x, const int32_t* topk_idx, int T, int H, int E, int K, int dtype,
                 int32_t* cu_seqlens, int32_t* dst_row, int32_t* src_tok, void* xs,
                 void* ws, size_t ws_bytes, void* stream);

/*
 * moe_dispatch without a workspace argument.  The source pages have no
 * counterpart for this call; it exists for callers that cannot allocate device
 * memory: code whose device memory is owned by someone else (a framework
 * allocator or a fixed arena planned ahead of time) and that has no scratch
 * buffer to hand over, or code that must not call cudaMalloc on its hot path,
 * where it can synchronise the device or fail under memory pressure.
 *
 * Same arguments, results and errors as moe_dispatch, minus ws/ws_bytes.  The
 * scratch it needs (a ceil(T/256) x E table of int32 counts and E int32 totals)
 * is a library-owned static device array of 65536 ints (256 KB), present on
 * every GPU that loads the library until the process exits.  Sizes with
 * ceil(T/256) * E + E > 65536 return MOE_ERR_WORKSPACE before anything is
 * launched.  The call allocates
 * nothing (no cudaMalloc/cudaFree, no allocating library routine).
 *
 * The first call on a device looks up the array's device address (one
 * cudaGetSymbolAddress with that device current); make that first call before
 * any stream capture.  Every call shares the one array: nothing in it needs
 * clearing between calls, but calls whose kernels may overlap on the GPU (e.g.
 * on two streams with no ordering between them) race and must be serialised
 * by the caller.
 */
MOE_API int moe_dispatch_noalloc(const void* x, const int32_t* topk_idx, int T, int H, int E, int K,
                                 int dtype, int32_t* cu_seqlens, int32_t* dst_row, int32_t* src_tok,
                                 void* xs, void* stream);

/*
 * Grouped SwiGLU expert FFN over contiguous weights
 *                [EP "Step-by-step" (weights [E,H,H'], rows by index); T4 SwiGLU]
 *
 *   For every expert e and row r in [cu_seqlens[e], cu_seqlens[e+1]):
 *     act[r,:] = silu(xs[r,:] . w_gate[e]) * (xs[r,:] . w_up[e])     silu(z) = z/(1+exp(-z))
 *     h[r,:]   = act[r,:] . w_down[e]^T
 *   xs [rows,H]; w_gate, w_up, w_down each one contiguous [E,H,Hp] tensor (dtype);
 *   act [rows,Hp] and h [rows,H] dtype out.  Accumulation is fp32; bf16 outputs
 *   are rounded to nearest-even (silu in fp32 with exp and divide of a few ulp;
 *   moe_expert_ffn_ex with gu divides exactly, so its act may differ from this
 *   call's in the last bit).  The row split is read on the device from
 *   cu_seqlens (no host synchronisation); cu_seqlens[E] must equal `rows`.
 *   bf16 needs H % 64 == 0 and Hp % 64 == 0.
 *   Workspace (optional, bf16): with ws 16-byte aligned and ws_bytes >=
 *   moe_workspace_bytes(MOE_OP_EXPERT_FFN, ...) (about 32 MB, independent of the
 *   sizes), when the down projection's last round of 256 x 256 tiles holds at
 *   most half as many tiles as the GPU runs CTA pairs, each of those tiles is
 *   computed as two K halves on two pairs whose fp32 partials are added (once,
 *   in fp32) before the bf16 rounding; the workspace holds the partials and
 *   arrival counters (the gate/up kernel of the same call zeroes them; no
 *   state carries between calls).  h then differs from a call without the
 *   workspace by that one extra fp32 rounding in those tiles; for the same
 *   inputs on the same GPU model it is deterministic.  NULL or fewer bytes:
 *   whole tiles only.  Concurrent calls need distinct workspaces.
 */
MOE_API int moe_expert_ffn(const void* xs, const int32_t* cu_seqlens, int rows,
                   const void* w_gate, const void* w_up, const void* w_down,
                   int E, int H, int Hp, int dtype, void* act, void* h,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * Grouped SwiGLU expert FFN with the dispatch gather fused into its input load
 *                      [FW "What's in the box": dispatch reads the buffers
 *                       directly; EP "Step-by-step": rows addressed by index]
 *
 *   moe_expert_ffn_ex with xs[r,:] = x[src_tok[r],:] read straight from x: in
 *   the gate/up GEMM (CTA pairs, 256-row tiles) eight extra warps per CTA copy
 *   the CTA's 128 rows of each tile from x by src_tok (as written by
 *   moe_dispatch) into its operand stages, so the expert-sorted copy of the
 *   input is never written or read.  The results are bit-identical to
 *   moe_expert_ffn_ex on the rows moe_dispatch writes (with the same
 *   workspace argument).  x [T,H] dtype; src_tok [rows] int32 in [0,T) (an
 *   index outside sets MOE_ERR_DEVICE_BOUNDS and reads row 0); the rest as
 *   moe_expert_ffn_ex.
 *   Workspace: optional, as moe_expert_ffn (the down projection's tail split).
 */
MOE_API int moe_expert_ffn_gather(const void* x, const int32_t* src_tok, int T, const int32_t* cu_seqlens,
                                  int rows, const void* w_gate, const void* w_up, const void* w_down, int E,
                                  int H, int Hp, int dtype, void* act, void* gu, void* h, void* ws,
                                  size_t ws_bytes, void* stream);

/*
 * Expert FFN forward that also keeps the SwiGLU pre-activations for the backward
 *
 * moe_expert_ffn plus gu [rows, 2*Hp] dtype out (nullable): gu[r, 0:Hp] = g =
 * xs[r,:] . w_gate[e] and gu[r, Hp:2Hp] = u = xs[r,:] . w_up[e], rounded to dtype.
 * gu needs bf16 (MOE_ERR_UNSUPPORTED otherwise).  gu = NULL is moe_expert_ffn.
 */
MOE_API int moe_expert_ffn_ex(const void* xs, const int32_t* cu_seqlens, int rows,
                   const void* w_gate, const void* w_up, const void* w_down,
                   int E, int H, int Hp, int dtype, void* act, void* gu, void* h,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * Expert FFN backward         [T4 "RMSNorm, RoPE, SwiGLU": SwiGLU = three matrix
 *                              products; FW "What's in the box": the layer trains]
 *
 * Given dh = dL/dh [rows,H] for the forward above (gu and act as the forward wrote
 * them), for every expert e and its rows:
 *   da  = dh . w_down[e]                        [rows_e, Hp]
 *   dg  = da * u * s(g) * (1 + g (1 - s(g)))    du = da * g * s(g)      s = logistic
 *   dxs = dg . w_gate[e]^T + du . w_up[e]^T     [rows_e, H]   dtype out (nullable)
 *   dw_gate[e] = xs_e^T dg,  dw_up[e] = xs_e^T du,  dw_down[e] = dh_e^T act_e
 *                                               [E,H,Hp] float out each (nullable);
 *                                               zero for experts without rows
 * bf16 only (MOE_ERR_UNSUPPORTED otherwise), same shape rules as moe_expert_ffn.
 * Workspace: moe_workspace_bytes(MOE_OP_EXPERT_FFN_BWD, T, H, E, K, Hp) bytes with
 * T*K = rows (it holds [dg | du], bf16).  Weight gradients are written, not
 * accumulated, each element reduced over its expert's rows in one fp32 accumulator.
 */
MOE_API int moe_expert_ffn_bwd(const void* xs, const int32_t* cu_seqlens, int rows,
                   const void* w_gate, const void* w_up, const void* w_down,
                   int E, int H, int Hp, int dtype, const void* gu, const void* act, const void* dh,
                   void* dxs, float* dw_gate, float* dw_up, float* dw_down,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * Combine: gate-weighted sum back to token order        [FW "What's in the box"]
 *
 *   y[o(t),:] = residual[o(t),:] + s_t * sum_k gate[t,k] * h[dst_row[t*K+k],:]
 *   o(t) = out_row[t] (nullable: o(t) = t);  s_t = row_scale[t] (nullable: 1);
 *   residual nullable (then 0), indexed like y.  Accumulated in fp32 in k order.
 *   dst_row nullable: then dst_row[j] = j.
 *   h [T*K,H] dtype; gate [T,K] float; y dtype out; only rows o(t) are written.
 */
MOE_API int moe_combine(const void* h, const float* gate, const int32_t* dst_row,
                const float* row_scale, const void* residual, const int32_t* out_row,
                int T, int H, int K, int dtype, void* y, void* stream);

/*
 * Router backward                         [FW "What's in the box", sparse backward]
 *
 * mode MOE_ROUTE_SOFTMAX_TOPK (gate[t,k] = softmax(logits[t])[topk_idx[t,k]]):
 *   d_logits[t,j] = p_j * (G_j - sum_k d_gate[t,k] * p[topk_idx[t,k]]),
 *                   G_j = d_gate[t,k] if j = topk_idx[t,k] else 0  (no gradient
 *                   through the selection itself)
 *   dw_router[h,e] = sum_t x[t,h] * d_logits[t,e]      (float, nullable)
 *   dx[t,h]       += sum_e d_logits[t,e] * w_router[h,e] (dtype, nullable, accumulated;
 *                   written instead when mode has MOE_ROUTE_DX_WRITE)
 * with MOE_ROUTE_GATE_RENORM or-ed in (gate[t,k] = q_k = p[topk_idx[t,k]] / sum_k' p[topk_idx[t,k']]):
 *   d_logits[t,topk_idx[t,k]] = q_k * (d_gate[t,k] - sum_k' d_gate[t,k'] * q_k'), 0 elsewhere
 * mode MOE_ROUTE_MOD_LINEAR (scalar score s[t] = x[t] . w; pass E = K = 1,
 *   w_router = w [H], d_gate = d_score [T], logits/topk_idx unused):
 *   d_logits = d_score (nullable), dw_router[h] = sum_t d_score[t] x[t,h],
 *   dx[t,h] += d_score[t] * w[h].
 * The weight gradient is reduced deterministically through the workspace:
 *   moe_workspace_bytes(MOE_OP_ROUTE_BWD, T, H, E, K, 0) bytes.
 */
MOE_API int moe_route_bwd(int mode, const float* d_gate, const float* logits, const int32_t* topk_idx,
                  const void* x, const void* w_router, int T, int H, int E, int K, int dtype,
                  float* d_logits, float* dw_router, void* dx,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * Backward of combine (and of the dispatch gather)  [FW "What's in the box"]
 *
 * With g(t) = dy[o(t)] (o, s_t as in moe_combine):
 *   dh[dst_row[t*K+k]] = s_t * gate[t,k] * g(t)                 (dtype, nullable)
 *   d_gate[t,k]        = s_t * <g(t), h[dst_row[t*K+k]]>        (float, nullable)
 *   d_scale[t]         = sum_k gate[t,k] * <g(t), h[dst_row[t*K+k]]> (float, nullable)
 *   dx[t]              = sum_k dxs[dst_row[t*K+k]]              (dtype, written; nullable,
 *                                                                requires dxs)
 * Dot products and sums accumulate in fp32.
 */
MOE_API int moe_permute_bwd(const void* dy, const void* h, const float* gate, const int32_t* dst_row,
                    const float* row_scale, const int32_t* out_row, const void* dxs,
                    int T, int H, int K, int dtype,
                    void* dh, float* d_gate, float* d_scale, void* dx, void* stream);

/*
 * Mixture-of-Depths capacity router                       [FW, MoD paragraph]
 *
 *   score[b*L+i] = x[b*L+i,:] . w_mod                              (float out)
 *   per sequence b: the C positions with the highest score (equal scores -> lower
 *   position) are selected; sel[b*C+j] = the j-th selected position, ascending
 *   as a flat token index b*L + position (int32 out); mask[b*L+i] = 1 if selected
 *   (u8 out).
 *   Optional outputs (nullable):
 *     sel_score[b*C+j] = score of that token (float)  -> row_scale of moe_combine
 *     x_sel[b*C+j,:]   = x[sel[b*C+j],:]               -> input of the MoE
 *     y_skip: y[b*L+i,:] = x[b*L+i,:] for every unselected token (the skip path)
 *   x [B*L,H], w_mod [H] dtype.  1 <= L <= 8192, 0 <= C <= L.  Workspace: none.
 */
MOE_API int mod_select(const void* x, const void* w_mod, int B, int L, int H, int C, int dtype,
               float* score, int32_t* sel, float* sel_score, uint8_t* mask,
               void* x_sel, void* y_skip, void* ws, size_t ws_bytes, void* stream);

/*
 * Expert-parallel dispatch plan (host only)      [EP "Step-by-step": the S x K
 *                      rows per rank invariant, the preload pool of B slots,
 *                      the [E+B, H, H'] weights addressed by row index]
 *
 *   R ranks, E experts (E % R == 0; rank r owns experts [rG, rG+G), G = E/R),
 *   S tokens per rank, K experts per token, B preload slots per rank.
 *   counts [R][E] int32: pairs that source rank s routes to expert e; every row
 *   must sum to S*K (MOE_ERR_INVALID_ARG otherwise).
 *   Outputs (caller-owned host arrays):
 *     piece_count [R][R][E], piece_offset [R][R][E]: destination rank d
 *       processes pairs [offset, offset + count) of source s's pairs for expert
 *       e (in the source's (t, k) order);
 *     slot_expert [R][B]: the expert whose weights slot j of rank d holds, or -1;
 *     local_counts [R][G + B]: rows of each local expert (home experts, then
 *       the slots) -- the local cu_seqlens is their exclusive scan;
 *     remote_reads [R]: rows of remote experts left without a slot (weights
 *       read from the home rank).
 *   Every destination gets exactly S*K rows.  The plan depends on the counts
 *   only (deterministic), so every rank computes the same plan from gathered
 *   counts.  No device work; returns MOE_OK or an argument error.
 */
MOE_API int moe_ep_plan(int R, int E, int S, int K, int B, const int32_t* counts, int32_t* piece_count,
                        int32_t* piece_offset, int32_t* slot_expert, int32_t* local_counts,
                        int32_t* remote_reads);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
