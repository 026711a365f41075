/*
 * moe_oracle.h -- plain, slow, fp64 CPU oracle of the top-k SwiGLU
 * mixture-of-experts layer (forward + backward), its device-side schedule
 * tables and the MXFP8 (E4M3 + E8M0, 1x32 blocks) weight quantiser.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this library: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it. It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it follows (page titles as cited throughout this directory):
 *  - "Mixture-of-Kittens: Cursor open-sources an MoE training megakernel"
 *    (clip, key-points bullets 2-5 and the key flowchart): the router picks
 *    top-k experts; tokens are dispatched to experts with per-expert counts
 *    and no token dropping; each expert is a SwiGLU FFN (gate/up, silu*mul,
 *    down); the combine forms the routing-weighted sum; the backward runs the
 *    mirrored reverse-combine / reverse-dispatch; reductions run in a fixed
 *    order so results are bitwise reproducible.
 *  - "Mixture-of-Kittens (MoK)" project summary, "core concepts" table:
 *    MXFP8 weight format, weights pre-quantised by a quantise op.
 *  - OCP Microscaling Formats (MX) v1.0 for the E8M0 shared-scale rule and
 *    the OFP8 E4M3 element format (public definitions; the pages only name
 *    the format).
 *
 * Every floating-point quantity below is computed in fp64 from the exact
 * values of the inputs, with no intermediate rounding, except where a step
 * is defined in fp32 (the router add, fl32(logit + bias), which the GPU
 * performs identically so that the selection is comparable bit for bit).
 *
 * Conventions: row-major arrays; bf16 arrays are passed as their uint16 bit
 * patterns. Return value 0 = OK, nonzero = error (see ORC_ERR_*).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_NAN = 2 };

/* Top-k routing. z[t,e] = fl32(logits[t,e] + bias[e]) (bias may be NULL).
 * ids[t,0..k) = the k experts with the largest z, ordered by (z descending,
 * expert index ascending). w[t,j] = softmax over the k selected z (equal to
 * the softmax over all E renormalised on the selected k). Any NaN in z ->
 * ORC_ERR_NAN. */
int orc_route_topk(int64_t N, int32_t E, int32_t k, const float* logits,
                   const float* bias, int32_t* ids, double* w);

/* Schedule tables for the expert-grouped token buffer.
 *  counts[e]          number of assignments (t,j) with ids[t,j] == e
 *  offsets[0..E]      exclusive prefix sum of counts (offsets[E] = N*k)
 *  pad_offsets[0..E]  exclusive prefix sum of counts rounded up to tile_m
 *  slot_of[t*k+j]     pad_offsets[e] + #{t' < t routed to e}: the row of the
 *                     expert-grouped buffer that holds assignment (t,j)
 *  src_of_row[r]      inverse map, r < pad_offsets[E]: t*k+j, or -1 for the
 *                     padding rows that round each segment up to tile_m
 *  tiles[3*i..]       (expert, first row, valid rows) of each tile_m-row tile
 *                     in row order; *n_tiles = pad_offsets[E] / tile_m
 * rows_cap / tiles_cap bound the output arrays (ORC_ERR_ARG if too small). */
int orc_build_schedule(int64_t N, int32_t k, int32_t E, int32_t tile_m,
                       const int32_t* ids, int32_t* counts, int32_t* offsets,
                       int32_t* pad_offsets, int32_t* slot_of,
                       int32_t* src_of_row, int64_t rows_cap, int32_t* tiles,
                       int64_t tiles_cap, int32_t* n_tiles);
/* Same tables with each expert's segment padded to a multiple of pad_m (a
 * multiple of tile_m; the minibatch granularity) while tiles stay tile_m rows
 * high; a tile lying wholly in padding has 0 valid rows. */
int orc_build_schedule_padded(int64_t N, int32_t k, int32_t E, int32_t tile_m, int32_t pad_m,
                              const int32_t* ids, int32_t* counts, int32_t* offsets,
                              int32_t* pad_offsets, int32_t* slot_of,
                              int32_t* src_of_row, int64_t rows_cap, int32_t* tiles,
                              int64_t tiles_cap, int32_t* n_tiles);

/* Layer forward. Inputs either all fp64 (the *_f64 entry points, used for
 * finite differences) or bf16 bit patterns (x, wg, wu, wd).
 *   x [N,H], wg [E,I,H], wu [E,I,H], wd [E,H,I], ids [N,k], w [N,k]
 *   y [N,H] = sum_j w[t,j] * Wd[e] (silu(Wg[e] x_t) * (Wu[e] x_t)),
 *   accumulated over j = 0..k-1 in order.
 * ye_out (optional, may be NULL) [N*k, H] receives each assignment's expert
 * output, indexed by t*k+j. threads <= 0 -> hardware concurrency. */
int orc_forward_f64(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                    const double* x, const double* wg, const double* wu,
                    const double* wd, const int32_t* ids, const double* w,
                    double* y, double* ye_out, int threads);
int orc_forward_bf16(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                     const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                     const uint16_t* wd, const int32_t* ids, const double* w,
                     double* y, double* ye_out, int threads);

/* Layer backward for the loss L = <dy, y> with the routing held fixed.
 * Outputs: dx [N,H], dwg [E,I,H], dwu [E,I,H], dwd [E,H,I], dw [N,k]
 * (dw[t,j] = dL/dw[t,j] = <dy_t, ye_{t,j}>). Weight gradients sum the
 * assignments of each expert in ascending token order. */
int orc_backward_f64(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                     const double* x, const double* wg, const double* wu,
                     const double* wd, const int32_t* ids, const double* w,
                     const double* dy, double* dx, double* dwg, double* dwu,
                     double* dwd, double* dw, int threads);
int orc_backward_bf16(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                      const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                      const uint16_t* wd, const int32_t* ids, const double* w,
                      const uint16_t* dy, double* dx, double* dwg, double* dwu,
                      double* dwd, double* dw, int threads);

/* Sampled forms for workloads too large to run whole on a CPU.
 * orc_tokens_bf16: y, dx rows [n_tok,H] and dw [n_tok,k] for the listed
 * tokens only (each needs only its own k assignments).
 * orc_expert_wgrad_bf16: the weight gradients of expert e restricted to the
 * listed rows: dwg_rows/dwu_rows [n_i,H] hold dWg[e][i_list[r]][:],
 * dwd_rows [n_h,I] hold dWd[e][h_list[r]][:]; every assignment routed to e
 * contributes, in ascending token order. */
int orc_tokens_bf16(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                    const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                    const uint16_t* wd, const int32_t* ids, const double* w,
                    const uint16_t* dy, int64_t n_tok, const int64_t* tok,
                    double* y, double* dx, double* dw, int threads);
int orc_expert_wgrad_bf16(int64_t N, int32_t H, int32_t I, int32_t E,
                          int32_t k, const uint16_t* x, const uint16_t* wg,
                          const uint16_t* wu, const uint16_t* wd,
                          const int32_t* ids, const double* w,
                          const uint16_t* dy, int32_t e, int64_t n_i,
                          const int32_t* i_list, int64_t n_h,
                          const int32_t* h_list, double* dwg_rows,
                          double* dwu_rows, double* dwd_rows, int threads);

/* Router (the GEMM in front of the routing): logits[t][e] = x[t] . Wr[e]
 * over H, x bf16 [N][H], Wr bf16 [E][H], in fp64. */
int orc_router_logits(int64_t N, int32_t H, int32_t E, const uint16_t* x, const uint16_t* wr,
                      double* logits, int threads);

/* Router backward with the top-k selection held fixed (it is piecewise
 * constant): the routing weights are the softmax over the k selected logits,
 * so with dw = dL/d(routing weights) [N][k]:
 *   dz[t][j] = w[t][j] * (dw[t][j] - sum_i w[t][i] * dw[t][i])   (dL/d logit of
 *              the j-th selected expert; the other logits get 0),
 *   dwr[e][h] = sum over (t, j) with ids[t][j] = e of dz[t][j] * x[t][h],
 *   dx[t][h]  = sum_j dz[t][j] * Wr[ids[t][j]][h]   (the router's share of dL/dx).
 * All fp64; dz [N][k], dwr [E][H], dx [N][H] are outputs. */
int orc_router_backward(int64_t N, int32_t H, int32_t E, int32_t k, const uint16_t* x,
                        const uint16_t* wr, const int32_t* ids, const double* w,
                        const double* dw, double* dz, double* dwr, double* dx, int threads);

/* MXFP8 layer (the MXFP8 workload): the layer forward + backward with every
 * operand of every GEMM quantised to MXFP8 along that GEMM's K and
 * dequantised exactly (rule of orc_mxfp8_quantize):
 *   gate/up fwd: Xe rows and Wg/Wu rows along H; down fwd: Act rows and Wd
 *   rows along I; down bwd: dYe rows and Wd columns along H; gate/up bwd:
 *   dG/dU rows and Wg/Wu columns along I; weight gradients: both operands
 *   along the token axis in blocks of 32 consecutive assignments of one
 *   expert (slot order), restarting per expert, zero-padded.
 * Intermediates that are quantised (Act, dYe, dG, dU) are first rounded to
 * bf16. quantize = 0 skips every quantisation and rounding (then the result
 * equals orc_backward_bf16 / orc_forward_bf16 exactly). Outputs as in
 * orc_forward_bf16 / orc_backward_bf16 (y, dx, dwg, dwu, dwd, dw). */
int orc_layer_mxfp8(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k, const uint16_t* x,
                    const uint16_t* wg, const uint16_t* wu, const uint16_t* wd,
                    const int32_t* ids, const double* w, const uint16_t* dy, int quantize,
                    double* y, double* dx, double* dwg, double* dwu, double* dwd, double* dw,
                    int threads);

/* The weight half of orc_layer_mxfp8, done once per set of weights: the six
 * copies the GEMMs read, each [E, I, H] (wg_h, wu_h, wg_i, wu_i) or [E, H, I]
 * (wd_i, wd_h) in fp64, the suffix naming the quantisation axis (h: blocks
 * along H, i: blocks along I). quantize = 0 gives the plain bf16 values. */
int orc_mxfp8_weights(int32_t H, int32_t I, int32_t E, const uint16_t* wg, const uint16_t* wu,
                      const uint16_t* wd, int quantize, double* wg_h, double* wu_h, double* wd_i,
                      double* wd_h, double* wg_i, double* wu_i, int threads);

/* The per-batch half of orc_layer_mxfp8 on weights from orc_mxfp8_weights
 * (orc_layer_mxfp8 = orc_mxfp8_weights followed by this). */
int orc_layer_mxfp8_prepared(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                             const uint16_t* x, const double* wg_h, const double* wu_h,
                             const double* wd_i, const double* wd_h, const double* wg_i,
                             const double* wu_i, const int32_t* ids, const double* w,
                             const uint16_t* dy, int quantize, double* y, double* dx, double* dwg,
                             double* dwu, double* dwd, double* dw, int threads);

/* orc_layer_mxfp8_prepared with two diagnostics for error accounting (never
 * used by a parity check): gu_bf16 = 1 rounds G and U to bf16 before the
 * SwiGLU backward reads them (as a layer that stores G and U in bf16 reads
 * them back; 0 keeps the fp64 values, which is orc_layer_mxfp8_prepared), and
 * dg_rows / du_rows (NULL: not written) receive the quantised dG and dU rows
 * [N*k, I] that the data-gradient GEMM of gate/up reads, in assignment order
 * t*k + j. */
int orc_layer_mxfp8_trace(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                          const uint16_t* x, const double* wg_h, const double* wu_h,
                          const double* wd_i, const double* wd_h, const double* wg_i,
                          const double* wu_i, const int32_t* ids, const double* w,
                          const uint16_t* dy, int quantize, int gu_bf16, double* y, double* dx,
                          double* dwg, double* dwu, double* dwd, double* dw, double* dg_rows,
                          double* du_rows, int threads);

/* The weight gradients of orc_layer_mxfp8 for expert e at sampled entries
 * (sampled parity where the whole layer is too large for the oracle):
 * dwg[r][c] = dWg[e][i_list[r]][h_list[c]], dwu likewise (both [n_i, n_h]),
 * dwd[c][r] = dWd[e][h_list[c]][i_list[r]] ([n_h, n_i]). Same steps, same
 * token-axis blocks and same summation order as orc_layer_mxfp8, so the
 * values are equal to its entries; cost grows with e's assignments times
 * (n_i + n_h) rows, not with H * I. */
int orc_expert_wgrad_mxfp8(int64_t N, int32_t H, int32_t I, int32_t E, int32_t k,
                           const uint16_t* x, const uint16_t* wg, const uint16_t* wu,
                           const uint16_t* wd, const int32_t* ids, const double* w,
                           const uint16_t* dy, int32_t e, int64_t n_i, const int32_t* i_list,
                           int64_t n_h, const int32_t* h_list, int quantize, double* dwg,
                           double* dwu, double* dwd, int threads);

/* MXFP8 quantiser (OCP MX v1.0, MXFP8 E4M3): for each block of 32
 * consecutive values along a row, X = 2^(floor(log2(amax)) - 8) (8 = the
 * largest E4M3 exponent), scale code = that exponent + 127 clamped to
 * [0, 254] (an all-zero block gets code 0); each element is V / 2^(code-127)
 * rounded to the nearest E4M3 value, ties to even, magnitudes above 448
 * saturating to 448. src [rows, cols] bf16, cols % 32 == 0;
 * q [rows, cols], scale [rows, cols/32]. */
int orc_mxfp8_quantize(int64_t rows, int64_t cols, const uint16_t* src,
                       uint8_t* q, uint8_t* scale);
/* Element rule alone: E4M3 code of v (double), RNE, saturating. */
uint8_t orc_e4m3_encode(double v);
/* Exact value of an E4M3 code (NaN codes return NaN). */
double orc_e4m3_decode(uint8_t code);

#ifdef __cplusplus
}
#endif
#endif
