// moe_internal.h -- host-side layout of the workspace and forward context,
// and the kernel launchers shared between the translation units of the CUDA
// library. Not part of the public ABI (see include/moe.h).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kTileM = 128;          // rows per expert tile (tcgen05 M)
constexpr int kSchedSub = 256;       // assignments per warp in the schedule scans
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
  int64_t N, A, R;        // tokens, assignments, expert-grouped rows
  int32_t H, I, E, k;
  int32_t T;              // per-expert row granularity (minibatch rows)
  int32_t dtype;          // MOE_BF16 or MOE_MXFP8
  int32_t stages;         // SM-pair GEMM ring stages requested (0: the library's choice)
  int32_t tile_n;         // token-row GEMM pair-tile width requested (0: the library's choice)
  int64_t n_warps;        // schedule warps = ceil(A / kSchedSub)
  // workspace byte offsets
  size_t err, counts, offsets, pad_offsets, slot_of, src_of_row, tiles, n_tiles, ptiles, n_ptiles,
      warp_counts,
      expert_order,
      mx_rh, mx_ri1, mx_ri2, mx_ch, mx_ci1, mx_ci2,  // MXFP8 quantised operands (bf16 values)
      // MXFP8 E4M3 codes + scale chunks (tensor-core path): token rows [R, H] and
      // [R, I] x2 quantised along K; transposed [H, R] and [I, R] x2 along tokens
      mq_rh, ms_rh, mq_ri, ms_ri, mq_ri2, ms_ri2, mq_th, ms_th, mq_ti, ms_ti, mq_ti2, ms_ti2,
      router_logits, router_dz, router_partial,  // router: logits scratch [N,E], dz [A], tile partials
      rc_sync,  // fused reverse-combine: chunk ticket + finished rows per 128-row tile
      ff_sync,  // fused forward: dispatch ticket, rows per 128-row tile, gate/up and down units per item
      dyxe, dg, du, ws_bytes;
  // forward-context byte offsets
  size_t xe, g, u, act, ye, saved_bytes;
};

// Validates the problem (sizes the kernels support) and fills the layout.
moe_status make_layout(const moe_problem* p, Layout* L);

template <class T>
inline T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}
template <class T>
inline const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

// ---- launchers (return the launch error, if any) ----
cudaError_t launch_route_topk(const Layout& L, const float* logits, const float* bias,
                              int32_t* ids, float* w, int32_t* err, cudaStream_t s);
cudaError_t launch_build_schedule(const Layout& L, const int32_t* ids, void* ws, cudaStream_t s);
cudaError_t launch_build_schedule_with_scratch(const Layout& L, const int32_t* ids, void* ws,
                                               int32_t* warp_counts, cudaStream_t s);
cudaError_t launch_dispatch(const Layout& L, const void* ws, const void* x, void* xe,
                            cudaStream_t s);
// Dispatch plus the MXFP8 row quantisation of Xe (codes q [R, H], scales sf in
// the tensor-memory chunk layout), as launch_mxfp8_quantize_mma(xe, R, H, 0)
// would write them on every row of a used expert segment.
cudaError_t launch_dispatch_quant(const Layout& L, const void* ws, const void* x, void* xe,
                                  uint8_t* q, uint8_t* sf, cudaStream_t s);
cudaError_t launch_combine(const Layout& L, const void* ws, const void* ye, const float* w,
                           void* y, cudaStream_t s);
cudaError_t launch_reverse_combine(const Layout& L, const void* ws, const void* dy,
                                   const void* ye, const float* w, void* dye, float* dw,
                                   cudaStream_t s);
cudaError_t launch_reverse_dispatch(const Layout& L, const void* ws, const void* dxe, void* dx,
                                    cudaStream_t s);
cudaError_t launch_mxfp8_qdq(const void* src, void* dst, int64_t rows, int64_t cols, int axis,
                             cudaStream_t s);
// Both MMA-layout MXFP8 forms of bf16 [rows, cols] from one read: the row
// form (q_r, sf_r; blocks along cols) and the transposed form (q_t, sf_t;
// blocks along rows). Either pair may be NULL. rows, cols multiples of 128.
cudaError_t launch_mxfp8_quantize_mma_forms(const void* src, int64_t rows, int64_t cols,
                                            uint8_t* q_r, uint8_t* sf_r, uint8_t* q_t,
                                            uint8_t* sf_t, cudaStream_t s);
cudaError_t launch_mxfp8_quantize_mma(const void* src, int64_t rows, int64_t cols, int transpose,
                                      uint8_t* q, uint8_t* sf, cudaStream_t s);
cudaError_t launch_mxfp8_quantize(const void* src, int64_t rows, int64_t cols, uint8_t* q,
                                  uint8_t* scale, cudaStream_t s);

// Grouped GEMMs (tcgen05). Return MOE_ERR_CUDA on a driver/launch failure.
moe_status gemm_gate_up(const Layout& L, const void* ws, const void* xe, const void* wg,
                        const void* wu, void* g, void* u, void* act, cudaStream_t s);
moe_status gemm_down(const Layout& L, const void* ws, const void* act, const void* wd, void* ye,
                     cudaStream_t s);
// Dispatch + gate/up + SwiGLU + down in one persistent launch (bit-identical
// to launch_dispatch, gemm_gate_up and gemm_down in sequence). g, u may both
// be NULL (inference: Act only). ring = 0: xe and act hold all R rows;
// ring > 0 (g, u NULL): xe and act are rings of `ring` slots of 256 rows
// (ring * 256 * H and ring * 256 * I bf16 values), ring from fused_ring_slots.
moe_status gemm_fused_forward(const Layout& L, const void* ws, const void* x, const void* wg,
                              const void* wu, const void* wd, void* xe, void* g, void* u,
                              void* act, void* ye, int ring, cudaStream_t s);
// Slots of the fused forward's Xe/Act ring on this device (0 if the
// occupancy query fails).
int fused_ring_slots(const Layout& L);
moe_status gemm_down_dgrad(const Layout& L, const void* ws, const void* dye, const void* g,
                           const void* u, const void* wd, void* dg, void* du, cudaStream_t s);
// DACT with the reverse-combine fused in: dYe (written here, then read by the
// GEMM) and d_topk_w from dY, Ye and the routing weights, as
// launch_reverse_combine computes them.
moe_status gemm_down_dgrad_rc(const Layout& L, const void* ws, const void* dy, const void* ye,
                              const float* topk_w, const void* dye, float* d_topk_w,
                              const void* g, const void* u, const void* wd, void* dg, void* du,
                              cudaStream_t s);
moe_status gemm_down_wgrad(const Layout& L, const void* ws, const void* dye, const void* act,
                           float* dw_down, cudaStream_t s);
moe_status gemm_gate_up_dgrad(const Layout& L, const void* ws, const void* dg, const void* du,
                              const void* wg, const void* wu, void* dxe, cudaStream_t s);
moe_status gemm_gate_up_wgrad(const Layout& L, const void* ws, const void* dg, const void* du,
                              const void* xe, float* dw_gate, float* dw_up, cudaStream_t s);

// Experts ranked by row count, descending (ties: ascending index), into the
// workspace's expert_order (the weight-gradient tile order).
moe_status launch_expert_order(const Layout& L, const void* ws, cudaStream_t s);

// Block-scaled FP8 grouped GEMMs (tcgen05 kind::mxf8f6f4) of the MXFP8 layer.
// Every operand is an E4M3 K-major matrix with its scale chunks
// (moe_mxfp8_operand): token rows [R, K] quantised along K, transposed
// weights, or transposed activations [C, R] quantised along the token axis.
moe_status gemm_mx_gate_up(const Layout& L, const void* ws, moe_mxfp8_operand xe,
                           const moe_mxfp8_operand& wg, const moe_mxfp8_operand& wu, void* g,
                           void* u, void* act, const moe_mxfp8_operand* act_q, cudaStream_t s);
moe_status gemm_mx_down(const Layout& L, const void* ws, moe_mxfp8_operand act,
                        const moe_mxfp8_operand& wd, void* ye, cudaStream_t s);
// dG, dU = SwiGLU backward of dYe . Wd[e] (B = Wd transposed, [I, E*H]).
moe_status gemm_mx_down_dgrad(const Layout& L, const void* ws, moe_mxfp8_operand dye,
                              const moe_mxfp8_operand& wd_t, const void* g, const void* u,
                              void* dg, void* du, cudaStream_t s);
// dXe = dG . Wg[e] + dU . Wu[e] (B = Wg, Wu transposed, [H, E*I]).
moe_status gemm_mx_gate_up_dgrad(const Layout& L, const void* ws, moe_mxfp8_operand dg,
                                 moe_mxfp8_operand du, const moe_mxfp8_operand& wg_t,
                                 const moe_mxfp8_operand& wu_t, void* dxe, cudaStream_t s);
// dWd[e] = dYe_e^T . Act_e from dYe^T [H, R] and Act^T [I, R] (token-axis blocks).
moe_status gemm_mx_down_wgrad(const Layout& L, const void* ws, moe_mxfp8_operand dye_t,
                              moe_mxfp8_operand act_t, float* dw_down, cudaStream_t s);
// dWg[e] = dG_e^T . Xe_e, dWu[e] = dU_e^T . Xe_e from dG^T, dU^T [I, R], Xe^T [H, R].
moe_status gemm_mx_gate_up_wgrad(const Layout& L, const void* ws, moe_mxfp8_operand dg_t,
                                 moe_mxfp8_operand du_t, moe_mxfp8_operand xe_t, float* dw_gate,
                                 float* dw_up, cudaStream_t s);

// Router GEMM: logits [N, E] fp32 = x [N, H] . w_router [E, H]^T (E <= 256, E % 4 == 0).
moe_status gemm_router(const Layout& L, const void* ws, const void* x, const void* w_router,
                       float* logits, cudaStream_t s);
// Router backward (see router.cu): dx += router share, dw_router [E, H] fp32.
cudaError_t launch_router_backward(const Layout& L, const void* ws, const void* xe,
                                   const void* w_router, const int32_t* ids, const float* w,
                                   const float* dw, void* dx, float* dw_router, cudaStream_t s);

// Launch accounting (every kernel launch of the library calls note_launch).
void note_launch();

}  // namespace moe
