/*
 * moe_expert.h - C ABI of the GB300 MoE expert-block library
 * (libmoe_gb300.so, built from moe_expert_dispatch_gb300/csrc).
 *
 * The library computes, on one GPU, the expert block of an MoE layer as the
 * ep_mc2_forward data flow of "NPU Training Operators - MC2" (section
 * "execution path", steps 2-10) states it: per-expert token counts (histc),
 * the offset scan, the stable permute of routed rows into expert-contiguous
 * order, grouped GEMM fc1 (gate and up) with a SwiGLU epilogue, grouped GEMM
 * fc2 and the probability-weighted unpermute. Around that path: a top-k
 * router fused with the counts, the backward of the block, MXFP8 variants of
 * the dispatch, the forward and the backward, and a micro-batch pipelined
 * forward. On one GPU the two AllToAllv of the MC2 fusion collapse into the
 * permute gather and the unpermute gather.
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise, owned by the
 *    caller, and at least 16-byte aligned (the grouped GEMMs read them with
 *    TMA). The library allocates no device memory: scratch space comes from
 *    a caller-provided workspace whose size the *_workspace_size calls give.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*,
 *    NULL = the legacy default stream) and never synchronises the host.
 *  - Matrices are row-major. bf16 is IEEE-style bfloat16 (2 bytes). Rounding
 *    to bf16 is round-to-nearest-even.
 *  - Host-detectable errors (null pointer, bad size, small workspace,
 *    unsupported shape) return a status immediately and launch nothing.
 *    Errors found on the device (an expert id outside [0, E), an in-kernel
 *    wait that ran out of time) set a device error word and the affected work
 *    stops early; moe_get_error() reports them. Nothing traps.
 *  - The library built with MOE_DEBUG (libmoe_gb300_debug.so) also checks,
 *    on the device, every row index it takes from a row map against the rows
 *    of the buffer it indexes, wherever the library knows that count (its
 *    own workspaces, moe_permute's padded rows); an index outside sets
 *    MOE_ERR_BOUNDS in the error word and its access is skipped. The release
 *    build relies on the row maps being right by construction.
 *  - T = 0 (no tokens) is valid. The block's calls then launch nothing, or
 *    only what writes outputs that do not depend on the tokens: the counting
 *    calls (moe_counts, moe_counts_static, moe_route_topk) still write zero
 *    counts and offsets, and the backward writes zero weight gradients (or
 *    leaves them as they were when accumulating).
 *  - Host threads: the first call of each entry point on a device sets that
 *    kernel's shared-memory attribute and caches device addresses, without a
 *    lock. Make one call per device from one thread (or before any stream
 *    capture) before calling from several threads at once.
 */
#ifndef MOE_EXPERT_H
#define MOE_EXPERT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, k > E, ...            */
  MOE_ERR_UNSUPPORTED = 2,   /* a shape the kernels do not handle (H, F % 128)      */
  MOE_ERR_BAD_EXPERT_ID = 3, /* device: an expert id outside [0, E)                 */
  MOE_ERR_WORKSPACE = 4,     /* workspace pointer null or smaller than required     */
  MOE_ERR_TIMEOUT = 5,       /* device: an in-kernel pipeline wait hit its limit    */
  MOE_ERR_CUDA = 6,          /* a CUDA runtime call failed (launch, attribute, ...) */
  MOE_ERR_BOUNDS = 7         /* device, MOE_DEBUG build only: a row index taken from a
                                row map fell outside the buffer it indexes; the access
                                was skipped (see moe_get_error)                       */
} moe_status;

typedef enum moe_precision { MOE_BF16 = 0, MOE_MXFP8 = 1 } moe_precision;

/* Tuning and debug knobs of the fused path. moe_config_init() fills the
 * defaults; a NULL config pointer means the defaults. */
typedef struct moe_config {
  int ring_stages;         /* depth of the shared-memory ring that feeds the tensor
                              cores: 0 (default) = the deepest that fits, 4 slots of
                              48 KB for BF16 and 6 slots of 34 KB for MXFP8; 1..6 to
                              choose (BF16 caps at 4); 1 = no overlap, the serial
                              baseline of the "tileCnt = 1" knob in "MC2 通算融合架构总览"
                              section 6                                               */
  int save_for_backward;   /* forward keeps Xp, A_g, A_u, h and O in its workspace
                              and zero-fills the padding rows (default 0)              */
  int num_sms;             /* persistent grid size of the grouped GEMMs; 0 = all SMs   */
  int fuse_gather;         /* 1: fc1 gathers routed rows of x itself instead of reading
                              a materialised permuted copy (default 0)                  */
  long long wait_limit_ns; /* bound of every in-kernel wait (default 0 = 2 s)           */
  void** step_events;      /* optional: array of num_step_events cudaEvent_t (as void*)
                              recorded on `stream` at step boundaries; NULL = none.
                              Forward (5): start, after routing (counts, row map,
                              permute), fc1+SwiGLU, fc2, unpermute.
                              Backward (7): start, after dO+dprobs, dH+SwiGLU
                              backward, dXp, dX, dW1, dW2. MXFP8 backward (9): see
                              moe_expert_backward_mxfp8.                               */
  int num_step_events;     /* entries of step_events (events past it are not recorded) */
  int mxfp8_tile_n;        /* MMA N of the MXFP8 GEMMs: 128 (two accumulators, the
                              epilogue overlaps the next tile) or 256 (one accumulator,
                              half the A traffic per FLOP); 0 (default) = automatic  */
  int cta_pairs;           /* grouped GEMMs over routed rows (fc1, fc2, dH, dXp; BF16,
                              and MXFP8 with 256-wide N tiles): 2 = pairs of CTAs on
                              two SMs share M = 256 tiles (tcgen05 cta_group::2, each
                              SM loading half of B); 1 = one CTA per 128-row tile;
                              0 (default) = pairs for BF16 when the experts average
                              at least 512 routed rows, one CTA per tile for MXFP8.
                              Results are bit-identical either way.                   */
  int mx_scales_pretiled;  /* moe_expert_forward_mxfp8: 1 = wg_s and wd_s already hold
                              the weights' scales in the block-scaled MMA's layout,
                              written by moe_tile_weight_scales_mxfp8 with the same
                              mxfp8_tile_n and the same H, F, E (wu_s is not read and
                              may be NULL), so the forward does not re-tile them on
                              every call; 0 (default) = row-major scales as
                              moe_quantize_mxfp8 writes them                          */
} moe_config;

#define MOE_STEP_EVENTS 5
#define MOE_BWD_STEP_EVENTS 7
#define MOE_MX_BWD_STEP_EVENTS 9

void moe_config_init(moe_config* cfg);

/* Readable name of a status. Never NULL. */
const char* moe_status_string(moe_status s);

/* Synchronises `stream`, then returns and clears the device error word
 * (MOE_OK when no kernel reported an error). The word is per device and is
 * shared by every stream, so concurrent users see each other's errors. */
moe_status moe_get_error(void* stream);

/* Number of streaming multiprocessors of the current device (0 on error). */
int moe_num_sms(void);

/* ------------------------------------------------------------------------
 * moe_counts - per-expert token counts and the offset scan.
 * Follows steps 2 and 4-5 of ep_mc2_forward ("NPU Training Operators - MC2",
 * section "execution path"): torch.histc(selected_experts, bins=E, min=0,
 * max=E), with send_counts = recv_counts = the local counts on one GPU.
 *
 *  expert_ids  int32 [n_ids]   flattened [T, k] routing ids (t-major)
 *  counts      int32 [E]       out: c_e = #{i : expert_ids[i] == e}
 *  offsets     int32 [E + 1]   out: offsets[0] = 0, offsets[e+1] = offsets[e] + c_e
 *  workspace   >= moe_counts_workspace_size(n_ids, E) bytes of scratch
 *              (per-chunk histograms); every call overwrites all of it, so
 *              nothing needs clearing and one workspace may serve every call
 *              on a stream.
 * Ids outside [0, E) are not counted and raise MOE_ERR_BAD_EXPERT_ID on the
 * device. Requires 1 <= E <= 1024 and n_ids < 2^31.
 * ------------------------------------------------------------------------ */
size_t moe_counts_workspace_size(int64_t n_ids, int E);
moe_status moe_counts(const int32_t* expert_ids, int64_t n_ids, int E, int32_t* counts,
                      int32_t* offsets, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * moe_counts_static - moe_counts without a workspace, for callers that
 * cannot allocate device memory at call time (a serving runtime that fixes
 * its memory footprint at start-up and forbids allocation afterwards, or a
 * plugin interface that hands an operator no scratch buffer). It computes
 * the histc step of ep_mc2_forward ("NPU Training Operators - MC2", section
 * "execution path", step 2) exactly as moe_counts does; the pages have no
 * counterpart of the workspace-free form, which exists for those callers.
 *
 * Same arguments and results as moe_counts minus the workspace. The scratch
 * (per-chunk histograms and bases) lives in a fixed 512 KB array of device
 * memory owned by the library, held by every GPU that loads the library
 * until the process exits. Limits: ceil(n_ids / 2048) * E <= 65536 (16 M ids
 * at E = 8, 1 M ids at E = 128); larger requests return MOE_ERR_WORKSPACE and
 * launch nothing. The call allocates nothing. Its first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture. Every
 * call overwrites the whole scratch it uses, so nothing needs clearing
 * between calls, but all calls on a device share the one array: calls that
 * overlap on the GPU (other streams, other threads) race and must be
 * serialised by the caller.
 * ------------------------------------------------------------------------ */
moe_status moe_counts_static(const int32_t* expert_ids, int64_t n_ids, int E, int32_t* counts,
                             int32_t* offsets, void* stream);

/* ------------------------------------------------------------------------
 * moe_route_topk - the gate ahead of the block, fused with its counts.
 * The block's routing weights and selected experts (arguments of the
 * dispatcher call in "NPU Training Operators - MC2", section "suggested
 * configuration") come from the gate computation that the MC2 for MoE
 * All-to-All article lists as the first part of a training step (section on
 * why communication is the bottleneck). The pages do not spell the gate
 * out; this call computes the usual top-k softmax gate. One kernel (after
 * one memset of its scratch) picks every token's experts and weights and,
 * for the batch, the per-expert counts and the offset scan.
 *
 *  logits      float [T, E]  router logits, row-major
 *  expert_ids  int32 [T, k]  out: the k experts with the largest logits in
 *                            descending order; equal logits rank the lower
 *                            index first (-0.0 equals +0.0); a NaN logit
 *                            ranks as -inf
 *  probs       float [T, k]  out: exp(l_j - l_0) / sum_i exp(l_i - l_0) over
 *                            the chosen k, l_0 the largest (float arithmetic);
 *                            NaN when l_0 is infinite
 *  counts      int32 [E]     out: as moe_counts of expert_ids
 *  offsets     int32 [E + 1] out: as moe_counts
 *  workspace   >= moe_route_topk_workspace_size(T, k, E) bytes, 16-byte
 *              aligned; the call clears what it uses, so one workspace may
 *              serve consecutive calls on a stream (not overlapping ones).
 * Requires 1 <= k <= E <= 1024, k <= 32 and T*k < 2^31; T = 0 gives zero
 * counts and offsets. Never reports a device error.
 * ------------------------------------------------------------------------ */
size_t moe_route_topk_workspace_size(int64_t T, int k, int E);
moe_status moe_route_topk(const float* logits, int64_t T, int E, int k, int32_t* expert_ids,
                          float* probs, int32_t* counts, int32_t* offsets, void* workspace,
                          size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * moe_permute - gather routed rows into expert-contiguous order.
 * Step 6 of ep_mc2_forward, permute(hidden_states, selected_experts): on one
 * GPU this is also the dispatch AllToAllv of all2all_grouped_matmul.
 * Rows of one expert keep the order of their flat slot index t*k + j.
 *
 *  x           [T, row_bytes]  token rows (any element type; row_bytes % 16 == 0)
 *  expert_ids  int32 [T, k]    routing ids
 *  probs       float [T, k]    routing weights, or NULL
 *  row_align   1 = dense rows (row of slot = offsets[e] + rank); 128 = each
 *              expert's segment starts at a multiple of 128 rows (the layout
 *              the grouped GEMMs tile), padding rows are left untouched
 *  x_perm      [R_cap, row_bytes] out: permuted rows, R_cap = T*k for
 *              row_align 1, else moe_padded_rows(T*k, E, row_align)
 *  row_of      int32 [T, k]    out: row of slot (t, j)
 *  token_of    int32 [R_cap]   out: token of each row (padding rows untouched)
 *  prob_of     float [R_cap]   out: probs[t, j] of each row (may be NULL)
 *  offsets     int32 [E + 1]   out: first row of each expert (aligned when
 *              row_align > 1; offsets[E] is then the padded row total)
 *  counts      int32 [E]       out: c_e
 * ------------------------------------------------------------------------ */
int64_t moe_padded_rows(int64_t n_rows, int E, int row_align);
size_t moe_permute_workspace_size(int64_t T, int k, int E);
moe_status moe_permute(const void* x, int64_t T, int64_t row_bytes, const int32_t* expert_ids,
                       const float* probs, int k, int E, int row_align, void* x_perm,
                       int32_t* row_of, int32_t* token_of, float* prob_of, int32_t* offsets,
                       int32_t* counts, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * moe_unpermute - probability-weighted combine back to token order.
 * Step 10 of ep_mc2_forward, unpermute(hidden_states, unpermute_indices,
 * probs=routing_weights); on one GPU also the combine AllToAllv of
 * grouped_matmul_all2all.
 *   y[t] = bf16( sum_{j<k} probs[t, j] * o_perm[row_of[t, j]] ), j in order,
 * accumulated in float. probs NULL means 1. Rows < 0 contribute nothing.
 *  o_perm  bf16 [*, H]    y  bf16 [T, H]    H % 8 == 0
 * ------------------------------------------------------------------------ */
moe_status moe_unpermute(const void* o_perm, const int32_t* row_of, const float* probs, int64_t T,
                         int k, int H, void* y, void* stream);

/* ------------------------------------------------------------------------
 * moe_quantize_mxfp8 - MXFP8 quantisation of bf16 rows.
 * The quantised AllToAll+Matmul of "MC2 通算融合架构总览" (section 1; scales
 * in a buffer of their own, section 5), in the OCP Microscaling (MX) v1.0
 * form: per 32 consecutive elements of a row, the shared scale
 * X = 2^(floor(log2(amax)) - 8) as an E8M0 code (exponent + 127, clamped to
 * [0, 254]; an all-zero block gets code 0), and each element E4M3(v / X),
 * round-to-nearest-even, saturating at +-448.
 *  in      bf16 [rows, K]   q  uint8 [rows, K]   scales  uint8 [rows, K/32]
 *  K % 32 == 0.
 * ------------------------------------------------------------------------ */
moe_status moe_quantize_mxfp8(const void* in, int64_t rows, int K, uint8_t* q, uint8_t* scales,
                              void* stream);

/* ------------------------------------------------------------------------
 * moe_permute_quantize_mxfp8 - the MXFP8 dispatch: each token's bf16 row is
 * quantised once, by the rule of moe_quantize_mxfp8, and its codes are
 * written to each of the token's k permuted rows. This is the quantised
 * AllToAll of "MC2 通算融合架构总览" (section 1) on one GPU, the permute of
 * moe_permute with MXFP8 rows. The scales are written once per token, in
 * token order; the block-scaled GEMMs take them per permuted row.
 *  x       bf16 [T, H]       token rows, 16-byte aligned
 *  row_of  int32 [T, k]      permuted row of slot (t, j), as moe_permute
 *                            writes it; a negative row is skipped. Rows are
 *                            not checked against the size of xq.
 *  xq      uint8 [rows, H]   out: E4M3 codes of token t at every row_of[t, j];
 *                            other rows are left untouched
 *  xs      uint8 [T, H/32]   out: E8M0 scales of token t, row-major
 *  H % 32 == 0, 1 <= k <= 32. T == 0 does nothing.
 * ------------------------------------------------------------------------ */
moe_status moe_permute_quantize_mxfp8(const void* x, int64_t T, int H, const int32_t* row_of,
                                      int k, uint8_t* xq, uint8_t* xs, void* stream);

/* ------------------------------------------------------------------------
 * moe_expert_forward - the whole block in one call:
 *   y = unpermute(fc2(swiglu(fc1(permute(x)))), probs)
 * with, per expert e over its rows, A_g = Xp_e W1g_e, A_u = Xp_e W1u_e
 * (float accumulation), h = bf16(silu(A_g) * A_u), O = bf16(h_e W2_e).
 * The argument order follows torch_npu.npu.mc2_fused_expert of the MC2 for
 * MoE All-to-All article (section "usage"), without its communication
 * group, plus the routing weights of unpermute.
 *
 *  x        bf16 [T, H]
 *  w_gate   bf16 [E, H, F]   (N contiguous, as the pages' weights_gate)
 *  w_up     bf16 [E, H, F]
 *  w_down   bf16 [E, F, H]
 *  expert_ids int32 [T, k],  probs float [T, k]
 *  y        bf16 [T, H]      out
 *  workspace >= moe_workspace_size(T, H, F, E, k, cfg, 0) bytes. With
 *           cfg->save_for_backward the workspace afterwards holds what
 *           moe_expert_backward needs; keep it unchanged until then.
 * Requires H % 128 == 0, F % 128 == 0, 1 <= k <= E <= 1024.
 * ------------------------------------------------------------------------ */
size_t moe_workspace_size(int64_t T, int H, int F, int E, int k, const moe_config* cfg,
                          int for_backward);
moe_status moe_expert_forward(const void* x, const void* w_gate, const void* w_up,
                              const void* w_down, const int32_t* expert_ids, const float* probs,
                              int64_t T, int H, int F, int E, int k, void* y, void* workspace,
                              size_t ws_bytes, const moe_config* cfg, void* stream);

/* ------------------------------------------------------------------------
 * moe_expert_forward_from_logits - moe_expert_forward with the gate fused
 * in front: the routing comes from router logits through the kernel of
 * moe_route_topk, whose counts and offsets replace the block's own counting
 * step. This is the gate whose routing_weights and selected_experts the
 * dispatcher call of "NPU Training Operators - MC2" (section "suggested
 * configuration") takes. y equals moe_expert_forward's on the expert_ids /
 * probs written here, bit for bit.
 *
 *  router_logits  float [T, E]
 *  expert_ids     int32 [T, k]  out (as moe_route_topk; the backward needs it)
 *  probs          float [T, k]  out (as moe_route_topk)
 *  everything else as moe_expert_forward, with the same workspace size.
 * ------------------------------------------------------------------------ */
moe_status moe_expert_forward_from_logits(const void* x, const void* w_gate, const void* w_up,
                                          const void* w_down, const float* router_logits,
                                          int64_t T, int H, int F, int E, int k,
                                          int32_t* expert_ids, float* probs, void* y,
                                          void* workspace, size_t ws_bytes,
                                          const moe_config* cfg, void* stream);

/* ------------------------------------------------------------------------
 * moe_expert_forward_pipelined - moe_expert_forward over n_chunks
 * contiguous token chunks of ceil(T / n_chunks) tokens (the last one
 * ragged), pipelined over two streams: the routing (counts, row map,
 * permute) of chunk c+1 and the combine of chunk c run on aux_stream while
 * the grouped GEMMs run on stream. This is the micro-batch pipeline of the
 * MC2 for MoE All-to-All article (section "pipeline design"), where the
 * dispatch of the next micro-batch overlaps the expert compute of the
 * current one; on one GPU the dispatch is the permute gather. Each chunk is
 * an independent forward, and the block's result does not depend on the
 * split, so y equals moe_expert_forward's bit for bit.
 *
 *  arguments as moe_expert_forward, plus
 *  n_chunks    >= 1 (n_chunks = 1 still runs routing and combine on aux)
 *  workspace   >= moe_workspace_size_pipelined(T, H, F, E, k, n_chunks)
 *              bytes: two per-chunk workspaces, used alternately
 *  aux_stream  a second stream, not equal to stream. It first waits for the
 *              work already queued on stream, and stream waits for all of
 *              the call's work on it before anything queued later, so the
 *              call is ordered on stream like any other.
 * cfg->save_for_backward is not supported (MOE_ERR_UNSUPPORTED): the
 * backward reads one whole-batch workspace. cfg->step_events are ignored.
 * The first call on a host thread and device creates six CUDA events that
 * the library keeps for the life of the process; make that call outside
 * stream capture. Later calls create nothing and may be captured.
 * ------------------------------------------------------------------------ */
size_t moe_workspace_size_pipelined(int64_t T, int H, int F, int E, int k, int n_chunks);
moe_status moe_expert_forward_pipelined(const void* x, const void* w_gate, const void* w_up,
                                        const void* w_down, const int32_t* expert_ids,
                                        const float* probs, int64_t T, int H, int F, int E, int k,
                                        void* y, int n_chunks, void* workspace, size_t ws_bytes,
                                        const moe_config* cfg, void* stream, void* aux_stream);

/* ------------------------------------------------------------------------
 * moe_expert_backward - gradients of moe_expert_forward.
 * The autograd Functions AllToAllGroupedMatmul / GroupedMatmulAllToAll of
 * "NPU Training Operators - MC2" (section "PR changes") wrap forward and
 * backward; its section "validation items" compares the fc1/fc2 gradients.
 *   dO_r  = bf16(p_r dY_t(r));          dprobs[t,j] = <dY_t, O_row(t,j)>
 *   dH    = dO_e W2_e^T (float);        dA_g = bf16(dH A_u silu'(A_g)),
 *   dA_u  = bf16(dH silu(A_g));         dXp = bf16(dA_g W1g_e^T + dA_u W1u_e^T)
 *   dW2_e = h_e^T dO_e, dW1g_e = Xp_e^T dA_g, dW1u_e = Xp_e^T dA_u (float)
 *   dX_t  = bf16(sum_j dXp[row_of[t, j]]), j in order, summed in float
 * A_g and A_u enter as saved by the forward (bf16). dXp, like O in the
 * forward, is a tensor of its own between two of the page's ops (the
 * grouped matmul's backward and the permute's backward), so it is bf16.
 *
 *  dy          bf16 [T, H]
 *  fwd_ws      the workspace of a forward call made with save_for_backward=1
 *              on the same inputs
 *  dx          bf16 [T, H]         out
 *  dw_gate     float [E, H, F]     out (accumulated into when accumulate_dw)
 *  dw_up       float [E, H, F]     out
 *  dw_down     float [E, F, H]     out
 *  dprobs      float [T, k]        out
 *  workspace   >= moe_workspace_size(T, H, F, E, k, cfg, 1) bytes
 * Experts that receive no token get dW = 0 (or are left as they were when
 * accumulate_dw).
 * ------------------------------------------------------------------------ */
moe_status moe_expert_backward(const void* dy, const void* x, const void* w_gate, const void* w_up,
                               const void* w_down, const int32_t* expert_ids, const float* probs,
                               int64_t T, int H, int F, int E, int k, const void* fwd_ws,
                               size_t fwd_ws_bytes, void* dx, float* dw_gate, float* dw_up,
                               float* dw_down, float* dprobs, int accumulate_dw, void* workspace,
                               size_t ws_bytes, const moe_config* cfg, void* stream);

/* ------------------------------------------------------------------------
 * moe_expert_forward_mxfp8 - the block with MXFP8 operands: the quantised
 * AllToAll+Matmul of "MC2 通算融合架构总览" (section 1, MX FP8; scales in
 * buffers of their own, section 5) on one GPU.
 * x arrives in bf16 and is quantised on the fly (per 32 along H) while it is
 * permuted; the weights arrive already quantised (moe_quantize_mxfp8) in a
 * K-contiguous layout so that each 32-block lies along the reduction:
 *  wg_q, wu_q  uint8 [E, F, H], wg_s, wu_s  uint8 [E, F, H/32]
 *  wd_q        uint8 [E, H, F], wd_s        uint8 [E, H, F/32]
 * fc1 accumulates in float, h = bf16(silu(A_g) A_u) is quantised per 32
 * along F for fc2, O = bf16(fc2) and y = bf16(combine), as in BF16 mode.
 * With cfg->save_for_backward the workspace (moe_workspace_size_mxfp8 with
 * the same cfg) also keeps A_g, A_u and h in bf16 for
 * moe_expert_backward_mxfp8, and the padding rows of the quantised x are
 * zeroed. Requires H % 128 == 0, F % 128 == 0. With cfg->mx_scales_pretiled
 * the scales come from moe_tile_weight_scales_mxfp8 (wg_s = its wgu_tiled,
 * wd_s = its wd_tiled, wu_s unused).
 * ------------------------------------------------------------------------ */
size_t moe_workspace_size_mxfp8(int64_t T, int H, int F, int E, int k, const moe_config* cfg);

/* ------------------------------------------------------------------------
 * moe_tile_weight_scales_mxfp8 - the weights' scales of moe_expert_forward_mxfp8
 * laid out once for its block-scaled MMAs, for a forward run with
 * cfg->mx_scales_pretiled = 1 (weights held in MXFP8 across calls: the
 * scales are re-tiled only when the weights change). "MC2 通算融合架构总览"
 * section 5 keeps the scales in buffers of their own, put once outside the
 * pipeline; this is that put for the weights.
 *  wg_s, wu_s  uint8 [E, F, H/32]  in (moe_quantize_mxfp8 of W1g^T, W1u^T)
 *  wd_s        uint8 [E, H, F/32]  in (moe_quantize_mxfp8 of W2^T)
 *  wgu_tiled   uint8 [E * 2F * H/32] out: pass as the forward's wg_s
 *  wd_tiled    uint8 [E * H * F/32]  out: pass as the forward's wd_s
 * The layout: atoms of 128 rows x 4 blocks of 32 (512 bytes), row blocks of
 * the gate and up scales interleaved per N tile of fc1 (half of the MMA N
 * each, which cfg->mxfp8_tile_n and H, F decide as the forward decides
 * them). The forward must get the same cfg->mxfp8_tile_n. Pointers are
 * device memory owned by the caller: the inputs 4-byte aligned, the outputs
 * 16-byte aligned (the forward reads them with bulk copies and requires the
 * same). Same argument checks as the forward (H % 128 == 0, F % 128 == 0,
 * 1 <= E <= 1024); MOE_ERR_CUDA if a launch fails.
 * ------------------------------------------------------------------------ */
moe_status moe_tile_weight_scales_mxfp8(const uint8_t* wg_s, const uint8_t* wu_s,
                                        const uint8_t* wd_s, int H, int F, int E,
                                        const moe_config* cfg, uint8_t* wgu_tiled,
                                        uint8_t* wd_tiled, void* stream);
moe_status moe_expert_forward_mxfp8(const void* x, const uint8_t* wg_q, const uint8_t* wg_s,
                                    const uint8_t* wu_q, const uint8_t* wu_s, const uint8_t* wd_q,
                                    const uint8_t* wd_s, const int32_t* expert_ids,
                                    const float* probs, int64_t T, int H, int F, int E, int k,
                                    void* y, void* workspace, size_t ws_bytes,
                                    const moe_config* cfg, void* stream);

/* ------------------------------------------------------------------------
 * moe_quantize_mxfp8_t - MXFP8 quantisation along the rows of a batch of
 * bf16 matrices (the transposed orientation of moe_quantize_mxfp8): for each
 * z < batch and column c of in[z] [rows, cols], the 32-row blocks of the
 * column become 32 consecutive codes of q[z][c] and one scale, by the rule
 * of moe_quantize_mxfp8 (the MX FP8 of "MC2 通算融合架构总览", section 1,
 * in OCP Microscaling v1.0 form). It turns the forward-layout weights into the
 * backward's: W1g, W1u [E, F, H] -> [E, H, F] quantised along F, and
 * W2 [E, H, F] -> [E, F, H] quantised along H.
 *  in      bf16 [batch, rows, cols]
 *  q       uint8 [batch, cols, rows]        out (16-byte aligned)
 *  scales  uint8 [batch, cols, rows / 32]   out
 *  rows % 32 == 0, cols % 8 == 0, in 16-byte aligned.
 * ------------------------------------------------------------------------ */
moe_status moe_quantize_mxfp8_t(const void* in, int64_t batch, int rows, int cols, uint8_t* q,
                                uint8_t* scales, void* stream);

/* ------------------------------------------------------------------------
 * moe_quantize_mxfp8_dual - both orientations of a batch of bf16 matrices
 * from one read: q_rows [batch, rows, cols] with scales [batch, rows, cols/32]
 * as moe_quantize_mxfp8 gives them, and q_cols [batch, cols, rows] with
 * scales [batch, cols, rows/32] as moe_quantize_mxfp8_t gives them, by the
 * MX FP8 rule of "MC2 通算融合架构总览" (section 1). A training
 * step quantises its weights both ways: the forward's layout and the
 * backward's. rows % 32 == 0, cols % 128 == 0, 16-byte aligned pointers.
 * ------------------------------------------------------------------------ */
moe_status moe_quantize_mxfp8_dual(const void* in, int64_t batch, int rows, int cols,
                                   uint8_t* q_rows, uint8_t* s_rows, uint8_t* q_cols,
                                   uint8_t* s_cols, void* stream);

/* ------------------------------------------------------------------------
 * moe_expert_backward_mxfp8 - gradients of moe_expert_forward_mxfp8: FP8
 * training of the expert block, the quantised AllToAll+Matmul of "MC2
 * 通算融合架构总览" (section 1) carried to the backward. Every GEMM runs on the
 * block-scaled tensor cores with both operands quantised per 32 along its
 * own reduction, and the rounding points are those of moe_expert_backward:
 *   dO_r = bf16(p_r dY_t(r)), dprobs[t,j] = <dY_t, O_row(t,j)> (float)
 *   dH   = deq(dO along H) deq(W2 as [F, H], along H)^T (float)
 *   dA_g, dA_u = the SwiGLU backward of dH on A_g, A_u as saved (bf16)
 *   dXp  = bf16(deq(dA_g along F) deq(W1g as [H, F], along F)^T + the same for up)
 *   dX_t = bf16(sum_j dXp[row_of[t, j]]), j in order, summed in float
 *   dW1g^T_e = deq(dA_g,e)^T deq(Xp_e), dW1u^T_e likewise, dW2^T_e =
 *   deq(dO_e)^T deq(h_e) (float), where the routed rows of expert e
 *   (Xp = bf16 x, h, dO, dA) are quantised along the rows in blocks of 32
 *   from the expert's first row.
 *
 *  dy               bf16 [T, H];  x  bf16 [T, H] (the forward's input)
 *  w1g_q, w1u_q     uint8 [E, H, F], scales [E, H, F/32] (moe_quantize_mxfp8_t
 *                   of the forward's wg, wu in bf16)
 *  w2_q             uint8 [E, F, H], scales [E, F, H/32] (of the forward's wd)
 *  fwd_ws           the workspace of a moe_expert_forward_mxfp8 call made with
 *                   save_for_backward on the same inputs
 *  dx               bf16 [T, H]       out
 *  dw_gate_t, dw_up_t  float [E, F, H] out, the layout of the forward's wg, wu
 *  dw_down_t        float [E, H, F]   out, the layout of the forward's wd
 *  dprobs           float [T, k]      out
 *  workspace        >= moe_workspace_size_mxfp8_backward(T, H, F, E, k) bytes
 * Experts that receive no token get dW = 0 (or are left as they were when
 * accumulate_dw). cfg->mxfp8_tile_n picks the MMA N of every GEMM (default
 * 256 where it divides the output width). cfg->step_events, when given, receive up to 9
 * events: start, after dO and its quantisations, dH, dA's quantisations,
 * dXp, dX, the quantisations of x and h, dW1, dW2.
 * Requires H % 128 == 0, F % 128 == 0.
 * ------------------------------------------------------------------------ */
size_t moe_workspace_size_mxfp8_backward(int64_t T, int H, int F, int E, int k);
moe_status moe_expert_backward_mxfp8(const void* dy, const void* x, const uint8_t* w1g_q,
                                     const uint8_t* w1g_s, const uint8_t* w1u_q,
                                     const uint8_t* w1u_s, const uint8_t* w2_q,
                                     const uint8_t* w2_s, const int32_t* expert_ids,
                                     const float* probs, int64_t T, int H, int F, int E, int k,
                                     const void* fwd_ws, size_t fwd_ws_bytes, void* dx,
                                     float* dw_gate_t, float* dw_up_t, float* dw_down_t,
                                     float* dprobs, int accumulate_dw, void* workspace,
                                     size_t ws_bytes, const moe_config* cfg, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_EXPERT_H */
