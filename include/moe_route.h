/*
 * moe_route.h -- C ABI of the MoE token routing / dispatch / combine library
 * (one GPU, sm_103a).
 *
 * The operations follow these web pages on DeepEP-style token dispatchers:
 *   [AutoEP-DeepEP]  DeepSpeed PR "Add an opt-in DeepEP transport for the AutoEP
 *                    expert all-to-all": section "Why" (dedup once per
 *                    destination rank, tokens taken before top-k expansion,
 *                    arrivals grouped by expert, weighted combine, backward =
 *                    dispatch/combine replayed on the forward handle) and the
 *                    review-fix commit text (router-score gradient must be
 *                    returned; capacity must grow or fail, not fault).
 *   [AutoEP-prep]    DeepSpeed PR "Avoid collective token preparation for
 *                    AutoEP DeepEP": "Summary" (no argsort, no [T*K,H]
 *                    expansion pass, no split-count exchange, no device-to-host
 *                    split materialisation), "Testing Done" (score-correction
 *                    bias, skewed routing, empty expert).
 *   [Titan-absorb]   torchtitan issue "[MoE] Apply router scores before W2
 *                    projection": "Motivation" and "Implementation" (scores
 *                    applied in fp32 to the W2 input, combine becomes a plain
 *                    sum; scores gathered expert-major as routed_scores_R).
 *   [NeMo-DeepEPv2]  NeMo Automodel PR "DeepEP v2 dispatcher ...":
 *                    "Performance" (one handle shared by dispatch and combine).
 *
 * Conventions for every entry point:
 *   - Every pointer named d_* is a DEVICE pointer on the device that was
 *     current when the handle was created; the caller owns all memory
 *     (tensors and workspace).  Row tensors must be 16-byte aligned and their
 *     row size (H or I times the element size) a multiple of 16 bytes.
 *   - Calls that launch work or write device memory must be made while the
 *     handle's device is current (and with a stream of that device): a call
 *     made while another device is current returns MOE_ERR_INVALID and
 *     launches nothing.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *     compute calls are asynchronous on it: none synchronises the host,
 *     allocates memory or copies device -> host.
 *   - Row dtype: MOE_BF16 (bfloat16) or MOE_F32.  Index tensors are int32,
 *     router weights fp32, row-major.
 *   - Return value: MOE_OK, or an error detected on the host before anything
 *     is launched (MOE_ERR_INVALID, MOE_ERR_CAPACITY, MOE_ERR_STATE), or
 *     MOE_ERR_CUDA if a launch failed.  Errors in the DATA (an expert index out
 *     of range, a repeated expert, a non-finite logit, a bounded wait that gave
 *     up) are found on the device: the kernel sets a bit of the handle's
 *     device status word (MOE_DEVERR_*) and skips the offending entry; read it
 *     with moe_read_device_status (which synchronises; not for the hot path).
 */
#ifndef MOE_ROUTE_H_
#define MOE_ROUTE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,  /* null / misaligned pointer, bad size or config     */
  MOE_ERR_CAPACITY = 2, /* T larger than the handle's max_tokens             */
  MOE_ERR_CUDA = 3,     /* a CUDA call or kernel launch failed               */
  MOE_ERR_STATE = 4     /* a row operation called before moe_dispatch_layout */
} moe_status;

typedef enum moe_dtype { MOE_BF16 = 0, MOE_F32 = 1 } moe_dtype;

typedef enum moe_score_fn { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;

/* Device status bits (sticky until moe_clear_device_status). */
#define MOE_DEVERR_BAD_EXPERT 0x1u /* idx entry outside [0,E): entry dropped      */
#define MOE_DEVERR_DUP_EXPERT 0x2u /* expert repeated in a token: later dropped   */
#define MOE_DEVERR_NONFINITE 0x4u  /* NaN/Inf router logit: token's route unspecified */
#define MOE_DEVERR_TIMEOUT 0x8u    /* a bounded wait inside a kernel gave up      */
#define MOE_DEVERR_INTERNAL 0x10u  /* layout counts inconsistent: writes skipped  */
#define MOE_DEVERR_BAD_LAYOUT 0x20u /* a row index or offset read from the layout
                                       lies outside the row tensors (a corrupted
                                       or foreign layout): entry skipped         */

/* Limits checked by moe_handle_create. */
#define MOE_MAX_EXPERTS 512
#define MOE_MAX_TOPK 16

/* Tokens per tile of the layout kernels (one thread block per tile). */
#define MOE_LAYOUT_TILE_TOKENS 512

/*
 * Router and layout configuration, fixed for the life of a handle.
 *   num_experts E (1..512), top_k K (1..min(E,16)), num_ranks R (virtual
 *   destination ranks; E % R == 0; rank(e) = e / (E/R)).
 *   score_fn: MOE_SCORE_SOFTMAX selects the top-K logits (softmax is strictly
 *     increasing) and weights them by softmax; MOE_SCORE_SIGMOID selects on
 *     key_e = sigmoid(l_e) + bias_e in fp64 and weights by the unbiased
 *     sigmoid ([AutoEP-prep] "score-correction bias").
 *   num_groups / topk_groups / group_score_topk: group-limited selection
 *     (sigmoid only): experts form num_groups contiguous groups; a group's
 *     score is the sum of its top group_score_topk keys; only the best
 *     topk_groups groups are eligible.  num_groups = 1 disables it.
 *   renorm: 1 = divide the K selected weights by their sum.
 *   route_scale: multiplies the weights (1.0 = none).
 *   max_tokens: capacity T_max; a larger batch is rejected with
 *     MOE_ERR_CAPACITY ([AutoEP-DeepEP] review fix: a batch that outgrows the
 *     buffer must not fault).
 *   pad_align: 0 or 1 = receive segments packed; A > 1 = every expert's
 *     segment of receive rows is rounded up to a multiple of A rows (a
 *     grouped-GEMM tile), off_e[e+1] = off_e[e] + ceil(cnt_e[e]/A)*A, as in the
 *     padded permute of [Titan-absorb] "Implementation".  Pad rows have
 *     recv_token = recv_k = recv_send_row = -1, and every kernel that writes
 *     receive rows (dispatch, expand, combine_bwd, scale_rows_bwd) writes
 *     zeros there (zero rows, zero score).  Receive-row tensors then hold
 *     T*K + E*(A-1) rows (1..4096).
 */
typedef struct moe_config {
  int32_t num_experts;
  int32_t top_k;
  int32_t num_ranks;
  int32_t score_fn;
  int32_t num_groups;
  int32_t topk_groups;
  int32_t group_score_topk;
  int32_t renorm;
  double route_scale;
  int32_t max_tokens;
  int32_t pad_align;
} moe_config;

/*
 * Device pointers into the handle's workspace, filled by moe_dispatch_layout
 * for the last layout's T tokens (all int32):
 *   cnt_e[E], off_e[E+1]              per-expert counts, exclusive offsets
 *   cnt_send_r[R], off_send_r[R+1]    token-deduplicated rows per rank
 *   cnt_recv_r[R], off_recv_r[R+1]    rows arriving at each rank (pads not
 *                                     counted) and where its region of receive
 *                                     rows starts (padded when pad_align > 1)
 *   pos[T*K]          receive row of entry (t,k), -1 if dropped
 *   recv_token[RR]    token of receive row p, recv_k[RR] its k (pad rows and
 *                     tail: -1); RR = T*K + E*(pad_align-1) receive rows
 *   send_token[T*min(K,R)]  token of send row s (tail beyond S: -1)
 *   send_row_of[T*K]  send row of entry (t,k), -1 if dropped
 *   recv_send_row[RR] send row that receive row p expands from (pad, tail: -1)
 *   S[1]              number of send rows (device scalar)
 */
typedef struct moe_layout {
  int32_t* cnt_e;
  int32_t* off_e;
  int32_t* cnt_send_r;
  int32_t* off_send_r;
  int32_t* cnt_recv_r;
  int32_t* off_recv_r;
  int32_t* pos;
  int32_t* recv_token;
  int32_t* recv_k;
  int32_t* send_token;
  int32_t* send_row_of;
  int32_t* recv_send_row;
  int32_t* S;
  int32_t num_tokens; /* T of the last layout, -1 before the first */
  int32_t pad_align;  /* receive segments padded to multiples of this (1: none) */
} moe_layout;

typedef struct moe_handle moe_handle;

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/*
 * Bytes of device workspace a handle with configuration `c` needs (0 if the
 * configuration is invalid).  The workspace holds the layout arrays above
 * plus per-tile histograms; allocate it 256-byte aligned.
 */
size_t moe_workspace_bytes(const moe_config* c);

/*
 * Creates a handle over caller-owned device workspace `d_workspace`
 * (`workspace_bytes` >= moe_workspace_bytes(c)) on the current device.  The
 * handle is a small host object holding the configuration and pointers into
 * the workspace.  The layout it holds is the state that the combine and both
 * backward passes reuse, so the backward never recomputes the layout
 * ([AutoEP-DeepEP] "Why"; [NeMo-DeepEPv2] "Performance", the paired handle).  Set-up call: it clears the workspace's
 * status word synchronously.  Not thread-safe: use one handle per stream.
 */
moe_status moe_handle_create(const moe_config* c, void* d_workspace, size_t workspace_bytes,
                             moe_handle** out);
moe_status moe_handle_destroy(moe_handle* h);

/*
 * Routing: per token, the top-K experts and their weights ([AutoEP-prep]
 * "Testing Done": the parity list covers exact routes, the score-correction
 * bias, routing scores, skewed routing and an empty expert; NeMo Automodel PR
 * "use the DeepEP dispatcher in the DiffusionGemma recipes", "Why hybridep +
 * activation checkpointing fails": a recomputed gate reproduces its top-k
 * indices exactly).
 *   d_logits [T,E] fp32 router logits; d_bias [E] fp32 score-correction bias
 *   (sigmoid only; NULL = none).  Outputs d_idx [T,K] int32 in descending key
 *   order, equal keys to the lower expert index; d_w [T,K] fp32.
 *   The selection is that of fp64 keys exactly.  Weights follow the fp64
 *   definition: computed in float-float arithmetic (about 2^-44 relative;
 *   fp64 for out-of-range logits) and rounded once to fp32, so each is the
 *   fp64 weight's rounding or one ulp from it.
 */
moe_status moe_route_topk(moe_handle* h, const float* d_logits, const float* d_bias, int32_t T,
                          int32_t* d_idx, float* d_w, void* stream);

/*
 * Router backward to the logits ([AutoEP-prep] "Testing Done": the parity
 * list covers routing-score and router-parameter gradients): given the
 * router-score gradient d_gw [T,K] fp32 (from moe_combine_bwd or
 * moe_scale_rows_bwd) and the selection d_idx [T,K] of d_logits [T,E],
 * writes d_glogits [T,E] fp32 = dL/dlogits with the selection held fixed:
 *   softmax, renorm:     c q_j (gw_j - sum_k q_k gw_k) for the selected j,
 *                        q = softmax over the selected logits, 0 elsewhere;
 *   softmax, no renorm:  c p_e (gw_e - sum_k p_k gw_k) for every e, p the
 *                        full softmax, gw_e = 0 for unselected e;
 *   sigmoid, renorm:     s_j (1 - s_j) (c / S) (gw_j - sum_k gw_k s_k / S),
 *                        S = sum of the selected sigmoids;
 *   sigmoid, no renorm:  c gw_j s_j (1 - s_j).
 * c = route_scale.  The correction bias only selects and has no gradient.
 * Computed in fp64 (sums in k order), rounded once to fp32.
 */
moe_status moe_route_bwd(const moe_handle* h, const float* d_logits, const int32_t* d_idx,
                         const float* d_gw, int32_t T, float* d_glogits, void* stream);

/*
 * Dispatch layout ([AutoEP-DeepEP] "Why"; [AutoEP-prep] "Summary"): from
 * d_idx [T,K] computes every array of moe_layout on the device, with no host
 * synchronisation.  Receive rows are grouped by expert, stable by token then
 * k; send rows by rank, one per (token, rank), stable by token.  The result
 * depends only on d_idx (bit-identical on replay).  Records T in the handle.
 * Returns MOE_ERR_CAPACITY if T > max_tokens.
 */
moe_status moe_dispatch_layout(moe_handle* h, const int32_t* d_idx, int32_t T, void* stream);

/*
 * Number of kernel launches moe_dispatch_layout makes for T tokens on the
 * handle's device: 1 when all its 512-token tiles can be resident at once
 * (a single cooperative launch), else 2.  Host-only query; *n_launches is
 * written on MOE_OK.
 */
moe_status moe_dispatch_layout_launches(const moe_handle* h, int32_t T, int32_t* n_launches);

/*
 * Allocation-free dispatch layout.  The web pages have no counterpart: this
 * entry point exists for callers that are not allowed to allocate device
 * memory, for example a plugin whose host framework hands it only its input
 * and output buffers and forbids cudaMalloc on the execution path (a
 * cudaMalloc there would synchronise the device and is illegal while the
 * framework captures the stream), so it cannot own the workspace that
 * moe_handle_create needs.
 *
 * Computes exactly what moe_dispatch_layout computes, for configuration `c`
 * (validated as in moe_workspace_bytes; max_tokens is not used) and the T
 * rows of d_idx [T,K], into the caller's arrays named in `out` (the layout of
 * moe_layout: counts and offsets always; pos, recv_token, recv_k,
 * send_row_of, recv_send_row [T*K] and send_token [T*min(K,R)] when T > 0;
 * out->num_tokens is ignored).  Data errors set bits in *d_status
 * (MOE_DEVERR_*) when d_status is not NULL.
 *
 * It allocates nothing: its scratch (an arrival counter and per-tile
 * counters) is a static device array of MOE_LAYOUT_STATIC_COUNTERS + 64
 * int32 (about 256 KiB), which every GPU that loads the library holds until
 * the process exits.  Limit: (E + R) * ceil(T / MOE_LAYOUT_TILE_TOKENS) must
 * not exceed MOE_LAYOUT_STATIC_COUNTERS, else MOE_ERR_CAPACITY (for E = 256,
 * R = 64: T up to 104448).  The first call on a device looks up the array's device
 * address and sets kernel attributes for that device, so make that first
 * call outside any stream capture.  All calls share the one array: calls
 * that overlap on the GPU (on different streams without ordering) race and
 * give wrong layouts; order them on one stream.  Asynchronous on `stream`.
 */
#define MOE_LAYOUT_STATIC_COUNTERS 65536
moe_status moe_dispatch_layout_static(const moe_config* c, const int32_t* d_idx, int32_t T,
                                      const moe_layout* out, uint32_t* d_status, void* stream);

/* Device pointers of the current layout (no device access). */
moe_status moe_layout_view(const moe_handle* h, moe_layout* out);

/*
 * Dispatch: permute token rows to expert-grouped receive rows
 * ([AutoEP-DeepEP] "Why": tokens taken before top-k expansion and replicated
 * by the dispatch itself).
 *   d_x [T,H] rows -> d_recv [T*K,H]: d_recv[pos[t,k]] = d_x[t] (bit copy).
 *   d_w [T,K] and d_recv_w [T*K] (both NULL or both set):
 *     d_recv_w[pos[t,k]] = d_w[t,k]   ([Titan-absorb] routed_scores_R).
 *   d_send [T*min(K,R),H] or NULL: d_send[send_row_of[t,k]] = d_x[t], the
 *     token-deduplicated rank-major rows.
 * Rows of d_recv beyond off_e[E] (only when entries were dropped) are not
 * written.
 */
moe_status moe_dispatch(const moe_handle* h, const void* d_x, int32_t H, int32_t dtype,
                        const float* d_w, void* d_recv, float* d_recv_w, void* d_send,
                        void* stream);

/*
 * Combine ([AutoEP-DeepEP] "Why": reduces the weighted sum back to token
 * order; [Titan-absorb]: a plain sum when scores are absorbed):
 *   d_out[t] = round( sum_k w[t,k] * d_y[pos[t,k]] ), accumulated in fp32 in
 *   k order with fused multiply-add, rounded once to the row dtype.
 *   d_w [T,K] fp32, or NULL for the plain sum.
 */
moe_status moe_combine(const moe_handle* h, const void* d_y, int32_t H, int32_t dtype,
                       const float* d_w, void* d_out, void* stream);

/*
 * Combine backward = a dispatch of the output gradient, plus the router-score
 * gradient ([AutoEP-DeepEP] "Why" and review fix):
 *   d_gy[pos[t,k]] = round(w[t,k] * d_g[t])   (fp32 product; d_w NULL: copy)
 *   d_gw[t,k] = <d_g[t], d_y[pos[t,k]]>       (fp32 accumulation; 0 for a
 *                                             dropped entry; skipped if d_gw
 *                                             or d_w is NULL)
 *   d_g [T,H], d_y [T*K,H] (the forward's expert output), d_gy [T*K,H].
 */
moe_status moe_combine_bwd(const moe_handle* h, const void* d_g, const void* d_y, int32_t H,
                           int32_t dtype, const float* d_w, void* d_gy, float* d_gw,
                           void* stream);

/*
 * Dispatch backward = a unit-weight combine ([AutoEP-DeepEP] "Why"):
 *   d_gx[t] = round( sum_k d_grecv[pos[t,k]] ), fp32 in k order.
 */
moe_status moe_dispatch_bwd(const moe_handle* h, const void* d_grecv, int32_t H, int32_t dtype,
                            void* d_gx, void* stream);

/*
 * Dispatch backward with the router backward to the logits fused in
 * ([AutoEP-prep] "Testing Done": router-parameter gradients): computes
 * exactly what moe_dispatch_bwd and moe_route_bwd compute, bit for bit, in
 * one launch:
 *   d_gx [T,H]           as moe_dispatch_bwd(d_grecv);
 *   d_glogits [T,E] fp32 as moe_route_bwd(d_logits, d_idx, d_gw),
 * where d_gw [T,K] is the complete router-score gradient (moe_combine_bwd or
 * moe_scale_rows_bwd, earlier on the stream) and d_logits [T,E], d_idx [T,K]
 * the forward routing's logits and selection, for the T of the handle's
 * layout.  The router's fp64 work runs beside the row traffic of the
 * dispatch backward, which has no cross-warp dependency (the combine
 * backward would hold it behind its per-token reduction).  Softmax routing
 * without renormalisation moves every logit of the row and runs as the two
 * separate kernels (moe_dispatch_bwd_route_launches says which).  All
 * pointers are required.
 */
moe_status moe_dispatch_bwd_route(const moe_handle* h, const void* d_grecv, int32_t H,
                                  int32_t dtype, const float* d_logits, const int32_t* d_idx,
                                  const float* d_gw, void* d_gx, float* d_glogits, void* stream);

/* Launches moe_dispatch_bwd_route makes for the handle's routing: 1, or 2 for
 * softmax without renormalisation.  Host-only query. */
moe_status moe_dispatch_bwd_route_launches(const moe_handle* h, int32_t* n_launches);

/*
 * Staged (wire-faithful) mode ([AutoEP-DeepEP] "Why": a token is sent once
 * per destination rank rather than once per selected expert, the receiving
 * side groups arrivals by expert, and the combine brings back one reduced row
 * per (token, rank)).  The send rows d_send [T*min(K,R),H] come from
 * moe_dispatch; the virtual ranks are expert partitions of this one GPU.
 *
 * moe_expand: the receiving side's expansion of arrived rows to expert rows,
 *   d_recv[pos[t,k]] = d_send[send_row_of[t,k]]  (each send row read once).
 * moe_combine_partial: stage 1, one partial row per send row s,
 *   d_partial[s] = round( fp32 sum, in k order, of w[t,k] * d_y[pos[t,k]]
 *   over the entries with send_row_of[t,k] == s )  (d_w NULL: plain sum);
 *   d_partial [T*min(K,R),H] in the row dtype (what travels back).
 * moe_combine_reduce: stage 2, d_out[t] = round( fp32 sum of the token's
 *   partial rows, each send row once, in the order of its first entry ).
 */
moe_status moe_expand(const moe_handle* h, const void* d_send, int32_t H, int32_t dtype,
                      void* d_recv, void* stream);
moe_status moe_combine_partial(const moe_handle* h, const void* d_y, int32_t H, int32_t dtype,
                               const float* d_w, void* d_partial, void* stream);
moe_status moe_combine_reduce(const moe_handle* h, const void* d_partial, int32_t H,
                              int32_t dtype, void* d_out, void* stream);

/*
 * Router-score absorption ([Titan-absorb] "Implementation": the W2 input is
 * scaled in float32 and restored to its dtype before the grouped GEMM):
 *   d_hs[r] = round(d_h[r] * d_recv_w[r]) for the T*K receive rows r of the
 *   current layout.  d_h, d_hs [T*K, I].
 */
moe_status moe_scale_rows(const moe_handle* h, const void* d_h, int32_t I, int32_t dtype,
                          const float* d_recv_w, void* d_hs, void* stream);

/*
 * Backward of moe_scale_rows:
 *   d_gh[r] = round(d_recv_w[r] * d_ghs[r])
 *   d_gw[t,k] = <d_ghs[pos[t,k]], d_h[pos[t,k]]>  (fp32 accumulation; 0 if
 *   the entry was dropped).
 */
moe_status moe_scale_rows_bwd(const moe_handle* h, const void* d_ghs, const void* d_h, int32_t I,
                              int32_t dtype, const float* d_recv_w, void* d_gh, float* d_gw,
                              void* stream);

/*
 * Router-score absorption fused into the W2 grouped GEMM ([Titan-absorb]
 * "Implementation": GroupedLinear scales the W2 input by the routed score in
 * float32 and restores the input dtype before the grouped GEMM; the same
 * page's "FusedMOE" section points at an SM100+ fused MoE backend).  For each
 * receive row r of expert e's segment in the current layout:
 *   hs[r,i] = round_bf16(d_h[r,i] * d_recv_w[r])          (fp32 product)
 *   d_y[r,n] = round_bf16(sum_i hs[r,i] * d_w2[e][n,i])    (fp32 accumulation)
 * The scaled rows hs exist only on chip (the GEMM's prologue); the products
 * run on the tensor cores.  A pad row of a padded layout gets d_y = 0.
 *   d_h     bf16 [T*K + E*(pad_align-1), I] receive rows (expert-grouped)
 *   d_recv_w fp32 per receive row (as written by moe_dispatch)
 *   d_w2    bf16 [E, H, I]: row n of expert e holds the I weights of output n
 *   d_y     bf16 [T*K + E*(pad_align-1), H]; rows outside the segments untouched
 * All device pointers caller-owned and 16-byte aligned.  Requires I % 8 == 0,
 * H % 256 == 0 and E*H < 2^31, else MOE_ERR_INVALID; MOE_ERR_STATE before the
 * first layout.  bf16 only.
 */
moe_status moe_w2_absorbed(const moe_handle* h, const void* d_h, int32_t I, const float* d_recv_w,
                           const void* d_w2, int32_t H, void* d_y, void* stream);

/*
 * Copies the device status word to *host_flags (MOE_DEVERR_* bits).  This
 * SYNCHRONISES the handle's device; keep it off the hot path.
 */
moe_status moe_read_device_status(const moe_handle* h, uint32_t* host_flags);

/*
 * Clears the device status word and re-arms the layout's arrival counter
 * (asynchronous on `stream`).  After a MOE_DEVERR_TIMEOUT, call it before the
 * next moe_dispatch_layout on this handle: a layout whose grid-wide hand-over
 * gave up leaves that counter where no later layout would complete.
 */
moe_status moe_clear_device_status(moe_handle* h, void* stream);

/*
 * Time limit, in nanoseconds, of every bounded wait inside this handle's
 * kernels: the single-launch layout's wait for all tiles' counts, and the
 * pipeline waits of moe_w2_absorbed ([AutoEP-DeepEP] review fix: a transport
 * that runs out of what it needs must fail, not fault).  A wait that gives up
 * sets MOE_DEVERR_TIMEOUT, and the kernel stops writing and returns (the W2
 * GEMM first waits, within the same limit, for the copies it has in flight
 * and releases its tensor memory).  limit_ns = 0 restores the default, one
 * second; a short limit is for tests that make a wait run out.  Host-only:
 * applies to launches made after the call.
 */
moe_status moe_set_wait_limit(moe_handle* h, uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H_ */
