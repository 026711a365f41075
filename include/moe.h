/*
 * moe.h -- C ABI of the GB300 (sm_103a) deterministic top-k SwiGLU
 * mixture-of-experts layer: routing, device-side schedule, dispatch, grouped
 * expert FFN, combine, their backward, and the MXFP8 quantiser.
 *
 * Sources of the operations (page title, section):
 *  [MoK]  "Mixture-of-Kittens (MoK)" project summary -- "use the functional
 *         API" (workspace created once per model, build_schedule from the
 *         router's top-k experts, forward -> (out, ctx), backward(ctx) ->
 *         grads) and "core concepts" (the ops layer leaves every tensor to the
 *         caller; MXFP8 weights are pre-quantised by a quantise op).
 *  [Clip] "Mixture-of-Kittens: Cursor open-sources an MoE training
 *         megakernel" -- key points 2-5 (pull dispatch / push combine and the
 *         mirrored backward rounds; minibatch granularity; ring token buffer
 *         and schedule built on the GPU with no host sync and no token
 *         dropping; SwiGLU expert FFN; bitwise determinism) and the key
 *         flowchart (router top-k -> dispatch -> expert FFN + SwiGLU ->
 *         combine -> weighted-sum output).
 *
 * General rules for every entry point:
 *  - Ownership: the caller allocates and frees every buffer (device memory
 *    unless stated otherwise). The library never allocates, frees or
 *    synchronises; each call only enqueues kernels on `stream` (a
 *    cudaStream_t, NULL = legacy default stream) and returns.
 *  - Errors detectable on the host (NULL pointer, unsupported size,
 *    misaligned pointer) return a moe_status immediately and enqueue nothing.
 *    Errors found by the kernels (expert id out of range, NaN router logit,
 *    a barrier wait that exceeded its time limit) are recorded in a sticky
 *    device error word inside the workspace; read it with
 *    moe_get_device_error after synchronising the stream.
 *  - Determinism: identical inputs give bitwise-identical outputs. No
 *    floating-point atomics are used; every reduction has a fixed order.
 *  - Pointers to device buffers must be 16-byte aligned; row-major layouts.
 *  - Stream capture: the first call of each kernel family on a device does
 *    one-time host setup (shared-memory attributes, cluster occupancy query,
 *    the scratch address of moe_build_schedule_noalloc). After one eager call
 *    of the same entry points, a sequence of calls can be captured into a
 *    CUDA graph and replayed; the graph reads its buffers at replay time.
 *    The schedule is rebuilt on the device, so new routing needs no new
 *    capture. moe_get_device_error copies to host memory, so call it outside
 *    a capture.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* NULL / inconsistent / misaligned argument */
  MOE_ERR_UNSUPPORTED = 2, /* size or dtype outside what the kernels support */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
  MOE_ERR_DEVICE = 4       /* reserved: device error word was set */
} moe_status;

/* Codes of the device error word (first error wins). */
enum {
  MOE_DEVERR_NONE = 0,
  MOE_DEVERR_BAD_EXPERT = 1, /* a top-k id outside [0, E) reached the schedule */
  MOE_DEVERR_NAN_LOGIT = 2,  /* a router logit (+ bias) was NaN */
  MOE_DEVERR_TIMEOUT = 3     /* a kernel's barrier wait ran out of time */
};

typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1 } moe_dtype;

/* Problem size. N tokens, H hidden, I expert intermediate, E experts,
 * k experts per token. Supported: N >= 0, 1 <= k <= min(E, 32), E <= 1024,
 * H and I multiples of 256. dtype MOE_BF16, or MOE_MXFP8: every operand of
 * every expert GEMM is quantised to MXFP8 (1x32 blocks along that GEMM's K,
 * E8M0 scale, E4M3 values; token-axis blocks restart per expert) and the
 * GEMMs multiply those numbers with fp32 accumulation -- as block-scaled FP8
 * MMAs when moe_weights.mx is given, else on their exact bf16 values;
 * moe_forward / moe_backward insert the activation quantisations.
 * minibatch_rows T ([Clip] key point 3, minibatch granularity; the "tokens
 * per expert slot" of the large-batch sweep): each expert's rows are grouped
 * and padded to a multiple of T. T = 128 (also for 0), 256, 512 or 1024.
 * Larger T only adds padding rows on one GPU (the expert GEMMs run on SM
 * pairs at every T); it is kept as the pages' minibatch knob.
 * pipeline_stages: depth of the shared-memory ring that the bf16 expert
 * GEMMs stream operands through (4, 5 or 6 stages of 32 KB per SM; 0 = the
 * library's choice per shape, from sweeps on a GB300). The results do not
 * depend on it (same MMAs in the same order).
 * tile_n: width in N of the pair tiles of the token-row expert GEMMs (gate/up,
 * down and their data gradients): 256, or 512 (two N tiles share each staged
 * A k-block, one TMEM accumulator, a 4-stage ring of 48 KB; needs an even
 * number of N tiles, else 256 is used); 0 = the library's choice per shape.
 * The results do not depend on it either.
 * The pages' knobs ([MoK] core concepts) that apply on one GPU are
 * minibatch_rows, the ring depth and the tile width. */
typedef struct {
  int64_t N;
  int32_t H, I, E, k;
  int32_t dtype;
  int32_t minibatch_rows;
  int32_t pipeline_stages;
  int32_t tile_n;
} moe_problem;

/* One MXFP8 operand as the block-scaled tensor-core GEMMs read it (see
 * mxfp8_quantize_mma): q = E4M3 codes of a K-major [rows, K] matrix, s = its
 * E8M0 scales (rows * K / 32 bytes) in the tensor-memory chunk layout. */
typedef struct {
  const uint8_t* q;
  const uint8_t* s;
} moe_mxfp8_operand;

/* MXFP8 expert weights for the tensor-core path, each made by
 * mxfp8_quantize_mma from the bf16 weights viewed as 2-D matrices:
 *   gate, up   [E*I, H] (transpose 0: K = H)  -- gate/up forward
 *   down       [E*H, I] (transpose 0: K = I)  -- down forward
 *   gate_t, up_t [H, E*I] (transpose 1 of [E*I, H]: K = I) -- gate/up data gradient
 *   down_t     [I, E*H] (transpose 1 of [E*H, I]: K = H)   -- down data gradient
 * A NULL q in gate_t / up_t / down_t makes moe_backward run those GEMMs on the
 * bf16 values in w_*_bwd instead. */
typedef struct {
  moe_mxfp8_operand gate, up, down;
  moe_mxfp8_operand gate_t, up_t, down_t;
} moe_mxfp8_weights;

/* Expert weights, bf16, K dimension contiguous:
 *   w_gate [E][I][H], w_up [E][I][H], w_down [E][H][I].
 * The *_bwd pointers are the same tensors as the backward data-gradient GEMMs
 * read them; NULL means "same as the forward ones" (MOE_BF16). For MOE_MXFP8
 * the forward pointers hold the weights quantised along their K (H for
 * gate/up, I for down) and the *_bwd pointers the weights quantised along the
 * backward GEMMs' K (I for gate/up, H for down), both as exact bf16 values of
 * the MXFP8 numbers (see mxfp8_qdq). */
typedef struct {
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const void* w_gate_bwd;
  const void* w_up_bwd;
  const void* w_down_bwd;
  /* MOE_MXFP8 only: the weights as E4M3 codes + E8M0 scales. Non-NULL makes
   * moe_forward / moe_forward_inference run the expert GEMMs as block-scaled
   * FP8 MMAs (tcgen05 kind::mxf8f6f4, fp32 accumulation) on the codes, with
   * the activations quantised to E4M3 + E8M0 by the library; NULL runs them
   * on the bf16 values of the MXFP8 numbers in w_gate / w_up / w_down. Both
   * compute the same products of the same MXFP8 numbers. moe_backward uses
   * the tensor-core path when mx->gate_t.q is non-NULL (then gate_t, up_t,
   * down_t must all be set), else the bf16 values in w_*_bwd. */
  const moe_mxfp8_weights* mx;
} moe_weights;

/* Rows of every expert-grouped buffer: each expert's segment of the buffer is
 * rounded up to a multiple of T = minibatch_rows, so the buffer needs at most
 * N*k + E*(T-1) rows, rounded up to T. Padding rows hold zeros. */
int64_t moe_grouped_rows(const moe_problem* p);

/* Bytes of the workspace (schedule tables, scratch, backward buffers, device
 * error word). Created once per problem size and reused across calls. */
moe_status moe_workspace_bytes(const moe_problem* p, size_t* bytes);

/* Bytes of the forward context ("fwd_ctx" of [MoK]) that moe_forward fills
 * and moe_backward reads: Xe [R,H], G [R,I], U [R,I], Act [R,I], Ye [R,H],
 * all bf16, R = moe_grouped_rows(p), in that order, each 256-byte aligned. */
moe_status moe_saved_bytes(const moe_problem* p, size_t* bytes);

typedef struct {
  void *xe, *g, *u, *act, *ye;
} moe_saved_view;
moe_status moe_saved_layout(const moe_problem* p, void* saved, moe_saved_view* out);

/* Device pointers to the schedule tables inside a workspace (host-side
 * address arithmetic only; nothing is launched):
 *  counts[E]        assignments per expert
 *  offsets[E+1]     exclusive prefix sum of counts (offsets[E] = N*k)
 *  pad_offsets[E+1] exclusive prefix sum of counts rounded up to T
 *  slot_of[N*k]     row of the expert-grouped buffer holding assignment
 *                   (t, j) = pad_offsets[e] + #{t' < t routed to e}
 *  src_of_row[R]    t*k + j of the assignment in row r, -1 on padding rows
 *                   (valid for r < pad_offsets[E])
 *  tiles[R/128][3]  (expert, first row, valid rows >= 0) of each 128-row tile
 *                   (the tensor-core tile height), in row order
 *  n_tiles[1]       number of tiles = pad_offsets[E] / 128 */
typedef struct {
  int32_t *counts, *offsets, *pad_offsets, *slot_of, *src_of_row, *tiles, *n_tiles;
} moe_schedule;
moe_status moe_schedule_view(const moe_problem* p, void* ws, moe_schedule* out);

/* [Clip] flowchart "Router picks top-k experts". logits fp32 [N,E], bias fp32
 * [E] or NULL. z = fl32(logit + bias); topk_ids int32 [N,k] = the k largest z
 * ordered by (z descending, expert index ascending); topk_w fp32 [N,k] =
 * softmax of the selected z (the full softmax renormalised over the top-k).
 * A NaN z sets MOE_DEVERR_NAN_LOGIT. ws is needed only for the error word. */
moe_status moe_route_topk(const moe_problem* p, const float* logits, const float* bias,
                          int32_t* topk_ids, float* topk_w, void* ws, void* stream);

/* [Clip] key point 4 / [MoK] build_schedule: per-expert counts, exclusive
 * prefix sums, token->row permutation and tile list, built on the device from
 * topk_ids int32 [N,k] with no host synchronisation and no token dropping.
 * Writes the tables of moe_schedule_view into ws. Ids outside [0,E) set
 * MOE_DEVERR_BAD_EXPERT (the tables are then unspecified). */
moe_status moe_build_schedule(const moe_problem* p, const int32_t* topk_ids, void* ws,
                              void* stream);

/* Allocation-free variant of moe_build_schedule (the pages have no
 * counterpart; it exists for callers of this library). For callers that
 * cannot allocate device memory -- e.g. a plugin whose host application owns
 * the whole device memory pool, or a loop that must never call the
 * allocator -- and so cannot provide the scan scratch moe_build_schedule
 * takes from the workspace. It writes these tables, with the same values as
 * moe_build_schedule, to the caller's arrays in *out (device pointers,
 * 4-byte aligned): counts[E], offsets[E+1], pad_offsets[E+1], slot_of[N*k],
 * src_of_row[moe_grouped_rows(p)], tiles[3 * moe_grouped_rows(p) / 128],
 * n_tiles[1]; device-detected errors go to *err_word (device int32). It does
 * NOT build the SM-pair work list that moe_build_schedule also writes into the
 * workspace for the expert GEMMs, so its output cannot stand in for a
 * workspace schedule in moe_forward, moe_backward or the expert-GEMM phase
 * calls: it serves callers that consume the routing tables themselves.
 * The scratch is a static device array owned by the library: 524288 int32
 * (2 MiB), held on every device that loads the library until the process
 * exits. Problems needing more than E * ceil(N*k / 256) = 524288 entries
 * return MOE_ERR_UNSUPPORTED. Allocates and frees nothing. The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress); the
 * address is cached with the id of the device's context and looked up again
 * in a new context (after cudaDeviceReset). Make the first call on a device,
 * and the first after a reset, before any stream capture. Every call shares
 * the array, so calls whose kernels overlap on the GPU (e.g. on two streams)
 * race. */
moe_status moe_build_schedule_noalloc(const moe_problem* p, const int32_t* topk_ids,
                                      const moe_schedule* out, int32_t* err_word, void* stream);

/* ---- forward phases (the ws must hold the schedule of this call) ---- */

/* Dispatch ([Clip] key point 2, pull dispatch; on one GPU an HBM copy):
 * xe[slot_of[t,j]] = x[t] for every assignment, padding rows = 0.
 * x bf16 [N,H] -> xe bf16 [R,H]. */
moe_status moe_dispatch(const moe_problem* p, const void* ws, const void* x, void* xe,
                        void* stream);

/* moe_dispatch with the MXFP8 row quantisation of Xe fused in (the MXFP8
 * forward's first step): xe as moe_dispatch writes it, plus q_e4m3 [R, H] and
 * s_e8m0 (R*H/32 bytes) exactly as mxfp8_quantize_mma(xe, R, H, 0, ...) writes
 * them on every row of the used expert segments (padding rows: codes and
 * scales 0; rows past the last segment are not written). x is read once and
 * each token's blocks are quantised once for its k copies. All pointers
 * 16-byte aligned. */
moe_status moe_dispatch_mxfp8(const moe_problem* p, const void* ws, const void* x, void* xe,
                              uint8_t* q_e4m3, uint8_t* s_e8m0, void* stream);

/* The workspace buffers that the MXFP8 tensor-core forward quantises its
 * activations into (host-only, no GPU work): xe_rows = Xe's row form (the
 * gate/up GEMM's A, written by the dispatch), act_rows = Act's row form (the
 * down GEMM's A, written by the gate/up epilogue), both [R, K] E4M3 codes with
 * scales in the mxfp8_quantize_mma chunk layout. Valid after moe_forward or
 * moe_forward_inference until the next call that reuses the workspace.
 * MOE_MXFP8 problems only. */
moe_status moe_mxfp8_forward_operands(const moe_problem* p, void* ws, moe_mxfp8_operand* xe_rows,
                                      moe_mxfp8_operand* act_rows);

/* The workspace buffers where the MXFP8 tensor-core backward leaves dG and dU
 * (host-only address arithmetic, no GPU work): their bf16 values (dg, du:
 * [R, I], written by the down data-gradient GEMM) and the two MXFP8 forms of
 * each that it quantises them into for the later GEMMs (E4M3 codes, scales in
 * the mxfp8_quantize_mma chunk layout): the row form (dg_rows, du_rows: [R, I], K = I, read by the gate/up
 * data-gradient GEMM) and the transposed form (dg_cols, du_cols: [I, R],
 * K = the token axis, read by the gate/up weight-gradient GEMM). Valid after
 * moe_backward on the FP8 tensor cores until the next call that reuses the
 * workspace. Any output pointer but dg_rows and du_rows may be NULL (not
 * written). For inspecting the quantised operands (error accounting, parity
 * of the fused quantisation); MOE_MXFP8 only. */
moe_status moe_mxfp8_backward_operands(const moe_problem* p, void* ws, moe_mxfp8_operand* dg_rows,
                                       moe_mxfp8_operand* du_rows, moe_mxfp8_operand* dg_cols,
                                       moe_mxfp8_operand* du_cols, void** dg, void** du);

/* Expert gate/up GEMM with the SwiGLU epilogue ([Clip] key point 5): per
 * expert e and its rows, G = Xe Wg[e]^T, U = Xe Wu[e]^T (fp32 accumulation on
 * the tensor cores), Act = silu(G) * U. Writes G, U, Act bf16 [R,I]; g and u
 * both NULL skip G and U (inference). */
moe_status moe_expert_gate_up(const moe_problem* p, const void* ws, const void* xe,
                              const moe_weights* w, void* g, void* u, void* act, void* stream);

/* Expert down GEMM: Ye = Act Wd[e]^T, bf16 [R,H]. */
moe_status moe_expert_down(const moe_problem* p, const void* ws, const void* act,
                           const moe_weights* w, void* ye, void* stream);

/* Combine ([Clip] key point 2 push combine; flowchart "weighted-sum output"):
 * y[t] = sum_{j=0..k-1} topk_w[t,j] * ye[slot_of[t,j]], accumulated in fp32
 * in ascending j, rounded once to bf16. y bf16 [N,H]. */
moe_status moe_combine(const moe_problem* p, const void* ws, const void* ye, const float* topk_w,
                       void* y, void* stream);

/* Dispatch + expert FFN in one persistent launch ([Clip] key point 5 and the
 * key flowchart: the producer pulls a minibatch of token rows and local
 * counters wake the expert FFN): side warps of every CTA copy token rows into
 * xe (as moe_dispatch) and count the finished rows of each 128-row tile; the
 * SM-pair GEMM roles run gate/up + SwiGLU (as moe_expert_gate_up) on a tile
 * once its rows are there, and the down GEMM (as moe_expert_down) on a group
 * of rows once all of its Act columns are stored. Bit-identical to
 * moe_dispatch, moe_expert_gate_up and moe_expert_down in sequence. x bf16
 * [N,H] -> xe [R,H], g, u, act [R,I], ye [R,H]; g and u both NULL skip G and
 * U (inference). xe and ye may be the same buffer (a row group's Xe is read
 * completely before its Ye is written). MOE_BF16 only; the grid holds only
 * co-resident CTA pairs, and every wait is bounded (MOE_DEVERR_TIMEOUT). */
moe_status moe_dispatch_expert_ffn(const moe_problem* p, const void* ws, const void* x,
                                   const moe_weights* w, void* xe, void* g, void* u, void* act,
                                   void* ye, void* stream);

/* Forward without a context (inference): dispatch, gate/up (Act only) and
 * down in one persistent launch (MOE_MXFP8: separate launches), then the
 * combine; same y as moe_forward. MOE_BF16: the dispatch fills, and the GEMMs
 * drain, a ring of 256-row minibatch slots for Xe and Act ("ring token
 * buffer", [Clip] key points 3-4): item p of the schedule's SM-pair items
 * uses slot p mod S, and a slot is refilled once the GEMM that reads it has
 * loaded it (per-item counters, bounded waits). S is set from the number of
 * co-resident CTA pairs, so the ring holds S * 256 * (H + I) bf16 values
 * whatever N is; a problem with fewer expert-grouped rows than the ring needs
 * runs with Xe and Ye sharing one scratch buffer instead.
 * Uses the workspace's backward buffers as scratch for Xe/Ye and Act, so it
 * must not run between a moe_forward and its moe_backward. */
moe_status moe_forward_inference(const moe_problem* p, const void* x, const moe_weights* w,
                                 const float* topk_w, void* y, void* ws, void* stream);

/* Whole forward: dispatch, gate/up, down, combine; saved = forward context. */
moe_status moe_forward(const moe_problem* p, const void* x, const moe_weights* w,
                       const float* topk_w, void* y, void* saved, void* ws, void* stream);

/* ---- backward phases ([Clip] key point 2: pull reverse-combine, push
 *      reverse-dispatch), for the loss gradient dy with routing held fixed */

/* Reverse-combine: dye[slot_of[t,j]] = bf16(topk_w[t,j] * dy[t]); padding
 * rows = 0; d_topk_w[t,j] = <dy[t], ye[slot_of[t,j]]> (fp32, fixed-order
 * reduction). dy bf16 [N,H], ye bf16 [R,H] -> dye bf16 [R,H], fp32 [N,k]. */
moe_status moe_reverse_combine(const moe_problem* p, const void* ws, const void* dy,
                               const void* ye, const float* topk_w, void* dye, float* d_topk_w,
                               void* stream);

/* Down backward, data gradient, with the SwiGLU backward epilogue:
 * dAct = dYe Wd[e]; s = sigmoid(G); dG = dAct * U * s * (1 + G (1 - s));
 * dU = dAct * G * s. dye, g, u bf16 [R,H] / [R,I] -> dg, du bf16 [R,I]. */
moe_status moe_expert_down_dgrad(const moe_problem* p, const void* ws, const void* dye,
                                 const void* g, const void* u, const moe_weights* w, void* dg,
                                 void* du, void* stream);

/* Down backward, weight gradient: dw_down[e] = dYe_e^T Act_e summed over the
 * expert's rows (fp32 [E][H][I]; experts without tokens get zeros). */
moe_status moe_expert_down_wgrad(const moe_problem* p, const void* ws, const void* dye,
                                 const void* act, float* dw_down, void* stream);

/* Gate/up backward, data gradient: dXe = dG Wg[e] + dU Wu[e] (bf16 [R,H]). */
moe_status moe_expert_gate_up_dgrad(const moe_problem* p, const void* ws, const void* dg,
                                    const void* du, const moe_weights* w, void* dxe,
                                    void* stream);

/* Gate/up backward, weight gradients: dw_gate[e] = dG_e^T Xe_e and
 * dw_up[e] = dU_e^T Xe_e (fp32 [E][I][H]; experts without tokens get 0). */
moe_status moe_expert_gate_up_wgrad(const moe_problem* p, const void* ws, const void* dg,
                                    const void* du, const void* xe, float* dw_gate,
                                    float* dw_up, void* stream);

/* Reverse-dispatch: dx[t] = sum_{j=0..k-1} dxe[slot_of[t,j]] (fp32, ascending
 * j, rounded once to bf16). dxe bf16 [R,H] -> dx bf16 [N,H]. */
moe_status moe_reverse_dispatch(const moe_problem* p, const void* ws, const void* dxe, void* dx,
                                void* stream);

/* Whole backward from the forward context. Outputs dx bf16 [N,H], dw_gate,
 * dw_up fp32 [E][I][H], dw_down fp32 [E][H][I], d_topk_w fp32 [N,k]. Uses
 * the workspace for dYe/dXe (shared buffer), dG and dU. */
moe_status moe_backward(const moe_problem* p, const void* saved, const moe_weights* w,
                        const float* topk_w, const void* dy, void* dx, float* dw_gate,
                        float* dw_up, float* dw_down, float* d_topk_w, void* ws, void* stream);

/* moe_backward with the reverse-combine overlapped with the down
 * data-gradient GEMM ([Clip] key point 2: the backward rounds mirror the
 * forward ones and reuse one schedule; overlapping a round's data movement
 * with the next round's GEMM tile by tile): the GEMM kernel's side warps claim
 * 8-row chunks of the expert-grouped buffer in row order, write dYe and
 * d_topk_w exactly as moe_reverse_combine does, and count the finished rows
 * of each 128-row tile; the GEMM loads a tile's dYe only after its count is
 * complete (bounded wait; on expiry MOE_DEVERR_TIMEOUT). Same arguments and
 * bit-identical results as moe_backward. MOE_BF16 only; for MOE_MXFP8 it runs
 * moe_backward (its quantisation sits between the two rounds). */
moe_status moe_backward_overlap(const moe_problem* p, const void* saved, const moe_weights* w,
                                const float* topk_w, const void* dy, void* dx, float* dw_gate,
                                float* dw_up, float* dw_down, float* d_topk_w, void* ws,
                                void* stream);

/* Router ([Clip] key flowchart, Router node: the router picks the top-k
 * experts of each token from its logits). logits = x . w_router^T with x bf16
 * [N, H], w_router bf16 [E][H] (K contiguous), fp32 accumulation on the
 * tensor cores, then the top-k and weights of moe_route_topk on
 * fl32(logit + bias). logits (fp32 [N, E], 16-byte aligned) receives the
 * logits if non-NULL (else the workspace holds them). E <= 256 and
 * E % 4 == 0, else MOE_ERR_UNSUPPORTED. Not in the layer's timed path: the
 * layer's routing input is top-k ids ([MoK] use the functional API). */
moe_status moe_route(const moe_problem* p, const void* x, const void* w_router, const float* bias,
                     float* logits, int32_t* topk_ids, float* topk_w, void* ws, void* stream);

/* Router backward, the selection held fixed (top-k is piecewise constant).
 * With w = topk_w (the softmax over the k selected logits) and
 * dw = d_topk_w (from moe_backward):
 *   dz[t,j] = w[t,j] * (dw[t,j] - sum_i w[t,i] * dw[t,i])   (dL/d logit),
 *   dx[t]  += sum_j dz[t,j] * w_router[topk_ids[t,j]]       (bf16 in place: fp32
 *             sum in j order onto the current value, one rounding),
 *   dw_router[e] = sum over the tokens routed to e of dz * x (fp32 [E][H],
 *             written whole; fixed order: 128-row tiles of the expert-grouped
 *             Xe in `saved`, then the tiles of each expert in order).
 * Uses the schedule in `ws` and Xe in `saved` from this batch's moe_forward. */
moe_status moe_router_backward(const moe_problem* p, const void* saved, const void* w_router,
                               const int32_t* topk_ids, const float* topk_w,
                               const float* d_topk_w, void* dx, float* dw_router, void* ws,
                               void* stream);

/* [MoK] core concepts, MXFP8 row: quantise bf16 [rows, cols] (cols % 32 == 0)
 * to MXFP8 along each row: per 1x32 block, E8M0 scale code =
 * clamp(floor(log2(amax)) - 8 + 127, 0, 254) (0 for an all-zero block), and
 * E4M3 elements = round-to-nearest-even(v / 2^(code-127)), saturating to
 * +-448 (OCP Microscaling Formats v1.0). q u8 [rows, cols], scale u8
 * [rows, cols/32]. */
moe_status mxfp8_quantize(const void* src_bf16, int64_t rows, int64_t cols, uint8_t* q_e4m3,
                          uint8_t* scale_e8m0, void* stream);

/* MXFP8 quantiser for the block-scaled tensor-core GEMMs (same rounding rule
 * as mxfp8_quantize), rows % 128 == 0 and cols % 128 == 0; src, q and s
 * 16-byte aligned (else MOE_ERR_INVALID_ARG).
 *   transpose 0: q [rows, cols], blocks of 32 consecutive columns of a row
 *                (the operand's K = cols);
 *   transpose 1: q [cols, rows] = src^T, blocks of 32 consecutive source rows
 *                of a column (the operand's K = rows).
 * s (rows * cols / 32 bytes) holds the scales of the K-major operand
 * [R', K'] (R' = rows or cols) in 512-byte chunks, one per (128 K, 128 rows):
 * chunk (K'/128 index kc, row block rb) at byte ((kc * R'/128) + rb) * 512; in
 * it the scale of (operand row r, 32-wide K block j) at byte
 * (r % 32) * 16 + ((r / 32) % 4) * 4 + j % 4 -- the order in which the
 * tensor-memory copy (tcgen05.cp 32x128b, warpx4) places scales for the MMA.
 * Not in the pages: the layout is fixed by the tensor-core instruction. */
moe_status mxfp8_quantize_mma(const void* src_bf16, int64_t rows, int64_t cols, int transpose,
                              uint8_t* q_e4m3, uint8_t* s_e8m0, void* stream);

/* MXFP8 quantise-dequantise of bf16 [rows, cols]: each value replaced by the
 * bf16 form of its MXFP8 number (the rule of mxfp8_quantize). axis 0: blocks
 * of 32 consecutive columns of a row (cols % 32 == 0); axis 1: blocks of 32
 * consecutive rows of a column (rows % 32 == 0, cols even). src == dst is
 * allowed. Used to prepare MXFP8 weights and by the MXFP8 layer. */
moe_status mxfp8_qdq(const void* src_bf16, void* dst_bf16, int64_t rows, int64_t cols, int axis,
                     void* stream);

/* Enqueue an asynchronous copy of the device error word of `ws` into
 * *code_out (host memory; pinned memory keeps the copy asynchronous). The
 * value is valid after the caller synchronises the stream. */
moe_status moe_get_device_error(const moe_problem* p, const void* ws, int32_t* code_out,
                                void* stream);
/* Enqueue a reset of the device error word to MOE_DEVERR_NONE. */
moe_status moe_clear_device_error(const moe_problem* p, void* ws, void* stream);

/* Test of the failure detection: launches one CTA whose barrier wait can never
 * complete; the wait's time limit (about one second) runs out, the kernel
 * records MOE_DEVERR_TIMEOUT in the workspace error word and returns, and the
 * context stays usable. No counterpart in the pages. */
moe_status moe_test_wait_timeout(const moe_problem* p, void* ws, void* stream);

/* Static description of a status code (never NULL). */
const char* moe_status_string(moe_status s);

/* Number of kernels this library has launched in the calling process (all
 * devices, all streams); for launch accounting in benchmarks. */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
