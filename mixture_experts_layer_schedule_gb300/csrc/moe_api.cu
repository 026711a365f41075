// moe_api.cu -- the C ABI (include/moe.h): argument validation, workspace and
// forward-context layout, and the order of the phases of the layer.
//
// The shape of the interface follows the functional API described in the
// project summary "Mixture-of-Kittens (MoK)" (section "use the functional
// API"): a workspace created once per model, build_schedule from the router's
// top-k experts, forward returning the output and a context, backward taking
// that context; and its ops layer, where the caller owns every tensor.
#include <algorithm>
#include <atomic>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

namespace {
std::atomic<uint64_t> g_launches{0};
}
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

moe_status make_layout(const moe_problem* p, Layout* L) {
  if (!p || !L) return MOE_ERR_INVALID_ARG;
  if (p->N < 0 || p->H <= 0 || p->I <= 0 || p->E <= 0 || p->k <= 0) return MOE_ERR_INVALID_ARG;
  if (p->k > p->E) return MOE_ERR_INVALID_ARG;
  if (p->E > kMaxE || p->k > kMaxK) return MOE_ERR_UNSUPPORTED;
  if (p->H % 256 != 0 || p->I % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (p->dtype != MOE_BF16 && p->dtype != MOE_MXFP8) return MOE_ERR_UNSUPPORTED;
  const int32_t T = p->minibatch_rows == 0 ? kTileM : p->minibatch_rows;
  if (T != 128 && T != 256 && T != 512 && T != 1024) return MOE_ERR_UNSUPPORTED;
  if (p->pipeline_stages != 0 && (p->pipeline_stages < 4 || p->pipeline_stages > 6))
    return MOE_ERR_UNSUPPORTED;
  if (p->tile_n != 0 && p->tile_n != 256 && p->tile_n != 512) return MOE_ERR_UNSUPPORTED;
  // rows, slots and tile coordinates are int32 on the device; bound N before
  // forming N * k so that the product cannot overflow
  if (p->N > (1LL << 31) / p->k) return MOE_ERR_UNSUPPORTED;
  const int64_t A = p->N * p->k;
  const int64_t R = (A + static_cast<int64_t>(p->E) * (T - 1) + T - 1) / T * T;
  if (R >= (1LL << 31) - 1) return MOE_ERR_UNSUPPORTED;
  L->N = p->N;
  L->A = A;
  L->R = R;
  L->H = p->H;
  L->I = p->I;
  L->E = p->E;
  L->k = p->k;
  L->T = T;
  L->dtype = p->dtype;
  L->stages = p->pipeline_stages;
  L->tile_n = p->tile_n;
  L->n_warps = (A + kSchedSub - 1) / kSchedSub;
  size_t o = 0;
  auto take = [&o](size_t bytes) {
    const size_t here = o;
    o = align256(o + bytes);
    return here;
  };
  L->err = take(sizeof(int32_t));
  L->counts = take(sizeof(int32_t) * p->E);
  L->offsets = take(sizeof(int32_t) * (p->E + 1));
  L->pad_offsets = take(sizeof(int32_t) * (p->E + 1));
  L->slot_of = take(sizeof(int32_t) * std::max<int64_t>(A, 1));
  L->src_of_row = take(sizeof(int32_t) * R);
  L->tiles = take(sizeof(int32_t) * 3 * (R / kTileM));
  L->n_tiles = take(sizeof(int32_t));
  L->ptiles = take(sizeof(int32_t) * 3 * (R / kTileM));  // SM-pair items (at most one per tile)
  L->n_ptiles = take(sizeof(int32_t));
  L->rc_sync = take(sizeof(int32_t) * (1 + R / kTileM));
  L->ff_sync = take(sizeof(int32_t) * (1 + 3 * (R / kTileM)));
  L->warp_counts = take(sizeof(int32_t) * p->E * std::max<int64_t>(L->n_warps, 1));
  L->expert_order = take(sizeof(int32_t) * p->E);
  L->router_logits = take(sizeof(float) * std::max<int64_t>(p->N, 1) * p->E);
  L->router_dz = take(sizeof(float) * std::max<int64_t>(A, 1));
  L->router_partial = take(sizeof(float) * static_cast<size_t>(R / kTileM) * p->H);
  L->dyxe = take(static_cast<size_t>(R) * p->H * 2);
  L->dg = take(static_cast<size_t>(R) * p->I * 2);
  L->du = take(static_cast<size_t>(R) * p->I * 2);
  const bool mx = p->dtype == MOE_MXFP8;
  L->mx_rh = mx ? take(static_cast<size_t>(R) * p->H * 2) : 0;
  L->mx_ri1 = mx ? take(static_cast<size_t>(R) * p->I * 2) : 0;
  L->mx_ri2 = mx ? take(static_cast<size_t>(R) * p->I * 2) : 0;
  L->mx_ch = mx ? take(static_cast<size_t>(R) * p->H * 2) : 0;
  L->mx_ci1 = mx ? take(static_cast<size_t>(R) * p->I * 2) : 0;
  L->mx_ci2 = mx ? take(static_cast<size_t>(R) * p->I * 2) : 0;
  L->mq_rh = mx ? take(static_cast<size_t>(R) * p->H) : 0;
  L->ms_rh = mx ? take(static_cast<size_t>(R) * p->H / 32) : 0;
  L->mq_ri = mx ? take(static_cast<size_t>(R) * p->I) : 0;
  L->ms_ri = mx ? take(static_cast<size_t>(R) * p->I / 32) : 0;
  L->mq_ri2 = mx ? take(static_cast<size_t>(R) * p->I) : 0;
  L->ms_ri2 = mx ? take(static_cast<size_t>(R) * p->I / 32) : 0;
  L->mq_th = mx ? take(static_cast<size_t>(R) * p->H) : 0;
  L->ms_th = mx ? take(static_cast<size_t>(R) * p->H / 32) : 0;
  L->mq_ti = mx ? take(static_cast<size_t>(R) * p->I) : 0;
  L->ms_ti = mx ? take(static_cast<size_t>(R) * p->I / 32) : 0;
  L->mq_ti2 = mx ? take(static_cast<size_t>(R) * p->I) : 0;
  L->ms_ti2 = mx ? take(static_cast<size_t>(R) * p->I / 32) : 0;
  L->ws_bytes = o;
  o = 0;
  L->xe = take(static_cast<size_t>(R) * p->H * 2);
  L->g = take(static_cast<size_t>(R) * p->I * 2);
  L->u = take(static_cast<size_t>(R) * p->I * 2);
  L->act = take(static_cast<size_t>(R) * p->I * 2);
  L->ye = take(static_cast<size_t>(R) * p->H * 2);
  L->saved_bytes = o;
  return MOE_OK;
}

// Failure-detection check: one CTA waits, through the bounded wait every
// kernel uses, on an mbarrier nothing arrives at. The wait runs out (about
// kWaitBudgetCycles), records MOE_DEVERR_TIMEOUT in the error word and the
// kernel returns normally, leaving the context usable.
__global__ void wait_timeout_kernel(int32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_wait(&bar, 0, &abort_flag, err);  // phase 0 never completes: expected to time out
  }
}

}  // namespace moe

using namespace moe;

namespace {

inline bool aligned(const void* p, uintptr_t a) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}
inline cudaStream_t S(void* s) { return static_cast<cudaStream_t>(s); }
inline moe_status cu(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                      \
  do {                                     \
    moe_status st_ = (expr);               \
    if (st_ != MOE_OK) return st_;         \
  } while (0)

moe_status prep(const moe_problem* p, const void* ws, Layout* L) {
  MOE_TRY(make_layout(p, L));
  if (!aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

bool weights_ok(const moe_weights* w) {
  return w && aligned(w->w_gate, 16) && aligned(w->w_up, 16) && aligned(w->w_down, 16);
}

bool operand_ok(const moe_mxfp8_operand& o) { return aligned(o.q, 16) && aligned(o.s, 16); }

// The forward MXFP8 tensor-core operands are present and aligned.
bool mx_forward_ok(const moe_weights* w) {
  return w && w->mx && operand_ok(w->mx->gate) && operand_ok(w->mx->up) &&
         operand_ok(w->mx->down);
}

// The backward MXFP8 tensor-core operands (transposed weights) are present.
bool mx_backward_ok(const moe_weights* w) {
  return mx_forward_ok(w) && operand_ok(w->mx->gate_t) && operand_ok(w->mx->up_t) &&
         operand_ok(w->mx->down_t);
}

// A workspace MXFP8 operand buffer: codes at `q`, scale chunks at `s`.
moe_mxfp8_operand ws_operand(void* ws, size_t q, size_t s) {
  return moe_mxfp8_operand{at<uint8_t>(ws, q), at<uint8_t>(ws, s)};
}


// Quantise bf16 [rows, cols] into the row form (K = cols) and/or the
// transposed form (K = rows) in one pass; a NULL operand is skipped.
moe_status quantize_forms(const void* src, int64_t rows, int64_t cols,
                          const moe_mxfp8_operand* row_form, const moe_mxfp8_operand* t_form,
                          cudaStream_t s) {
  auto q = [](const moe_mxfp8_operand* o) { return o ? const_cast<uint8_t*>(o->q) : nullptr; };
  auto sf = [](const moe_mxfp8_operand* o) { return o ? const_cast<uint8_t*>(o->s) : nullptr; };
  return cu(launch_mxfp8_quantize_mma_forms(src, rows, cols, q(row_form), sf(row_form),
                                            q(t_form), sf(t_form), s));
}

// MXFP8 forward on the block-scaled tensor cores: Xe quantised along H feeds
// gate/up, Act quantised along I feeds down. g/u may be NULL (inference).
// The dispatch with the row quantisation of Xe fused in: Xe bf16 and its
// E4M3 codes + scales (the gate/up GEMM's A operand, in the workspace) from
// one read of x.
moe_status mx_dispatch(const Layout& L, void* ws, const void* x, void* xe, cudaStream_t s) {
  if ((L.N > 0 && !aligned(x, 16)) || !aligned(xe, 16)) return MOE_ERR_INVALID_ARG;
  const moe_mxfp8_operand xq = ws_operand(ws, L.mq_rh, L.ms_rh);
  return cu(launch_dispatch_quant(L, ws, x, xe, const_cast<uint8_t*>(xq.q),
                                  const_cast<uint8_t*>(xq.s), s));
}

// After mx_dispatch: gate/up reads Xe's codes, Act is quantised for down.
moe_status mx_forward_gemms(const Layout& L, void* ws, const moe_mxfp8_weights& mx, void* g,
                            void* u, void* act, void* ye, cudaStream_t s) {
  const moe_mxfp8_operand xq = ws_operand(ws, L.mq_rh, L.ms_rh);
  const moe_mxfp8_operand aq = ws_operand(ws, L.mq_ri, L.ms_ri);
  // the gate/up epilogue also quantises Act's rows for the down GEMM
  MOE_TRY(gemm_mx_gate_up(L, ws, xq, mx.gate, mx.up, g, u, act, &aq, s));
  return gemm_mx_down(L, ws, aq, mx.down, ye, s);
}

// MXFP8 backward on the block-scaled tensor cores. Each GEMM operand is
// quantised along that GEMM's K: dYe rows along H (data gradient of down),
// dG/dU rows along I (data gradient of gate/up), and for the weight
// gradients dYe, Act, dG, dU, Xe along the token axis (transposed, blocks of
// 32 rows of one expert segment; segments start at multiples of T >= 128).
moe_status mx_backward_gemms(const Layout& L, void* ws, const moe_mxfp8_weights& mx,
                             const moe_saved_view& v, void* dyxe, void* dg, void* du,
                             float* dw_gate, float* dw_up, float* dw_down, cudaStream_t s) {
  const moe_mxfp8_operand rh = ws_operand(ws, L.mq_rh, L.ms_rh);
  const moe_mxfp8_operand ri = ws_operand(ws, L.mq_ri, L.ms_ri);
  const moe_mxfp8_operand ri2 = ws_operand(ws, L.mq_ri2, L.ms_ri2);
  const moe_mxfp8_operand th = ws_operand(ws, L.mq_th, L.ms_th);
  const moe_mxfp8_operand ti = ws_operand(ws, L.mq_ti, L.ms_ti);
  const moe_mxfp8_operand ti2 = ws_operand(ws, L.mq_ti2, L.ms_ti2);
  MOE_TRY(quantize_forms(dyxe, L.R, L.H, &rh, &th, s));
  MOE_TRY(quantize_forms(v.act, L.R, L.I, nullptr, &ti, s));
  MOE_TRY(gemm_mx_down_dgrad(L, ws, rh, mx.down_t, v.g, v.u, dg, du, s));
  MOE_TRY(gemm_mx_down_wgrad(L, ws, th, ti, dw_down, s));
  // Act^T's last reader ran above: dG^T and dU^T reuse its buffers.
  MOE_TRY(quantize_forms(dg, L.R, L.I, &ri, &ti, s));
  MOE_TRY(quantize_forms(du, L.R, L.I, &ri2, &ti2, s));
  // dXe overwrites dYe in the shared buffer: dYe's last readers ran above.
  MOE_TRY(gemm_mx_gate_up_dgrad(L, ws, ri, ri2, mx.gate_t, mx.up_t, dyxe, s));
  MOE_TRY(quantize_forms(v.xe, L.R, L.H, nullptr, &th, s));
  return gemm_mx_gate_up_wgrad(L, ws, ti, ti2, th, dw_gate, dw_up, s);
}

}  // namespace

namespace {

moe_status backward_impl(const moe_problem* p, const void* saved, const moe_weights* w,
                         const float* topk_w, const void* dy, void* dx, float* dw_gate,
                         float* dw_up, float* dw_down, float* d_topk_w, void* ws, void* stream,
                         bool overlap) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  moe_saved_view v;
  MOE_TRY(moe_saved_layout(p, const_cast<void*>(saved), &v));
  void* dyxe = at<char>(ws, L.dyxe);
  void* dg = at<char>(ws, L.dg);
  void* du = at<char>(ws, L.du);
  if (p->dtype == MOE_MXFP8 && w && w->mx && w->mx->gate_t.q) {
    if (!mx_backward_ok(w) || !aligned(dw_gate, 16) || !aligned(dw_up, 16) ||
        !aligned(dw_down, 16))
      return MOE_ERR_INVALID_ARG;
    MOE_TRY(moe_reverse_combine(p, ws, dy, v.ye, topk_w, dyxe, d_topk_w, stream));
    MOE_TRY(mx_backward_gemms(L, ws, *w->mx, v, dyxe, dg, du, dw_gate, dw_up, dw_down,
                              S(stream)));
    return moe_reverse_dispatch(p, ws, dyxe, dx, stream);
  }
  if (p->dtype == MOE_MXFP8) {
    // Each GEMM operand quantised along that GEMM's K: rows of dYe along H,
    // rows of dG/dU along I; for the weight gradients both operands along the
    // token axis (blocks of 32 rows; expert segments start at multiples of T).
    // The backward weight pointers hold Wd quantised along H, Wg/Wu along I.
    if (!w || !w->w_gate_bwd || !w->w_up_bwd || !w->w_down_bwd) return MOE_ERR_INVALID_ARG;
    moe_weights wb = *w;
    wb.w_gate = w->w_gate_bwd;
    wb.w_up = w->w_up_bwd;
    wb.w_down = w->w_down_bwd;
    void* rh = at<char>(ws, L.mx_rh);
    void* ri1 = at<char>(ws, L.mx_ri1);
    void* ri2 = at<char>(ws, L.mx_ri2);
    void* ch = at<char>(ws, L.mx_ch);
    void* ci1 = at<char>(ws, L.mx_ci1);
    void* ci2 = at<char>(ws, L.mx_ci2);
    MOE_TRY(moe_reverse_combine(p, ws, dy, v.ye, topk_w, dyxe, d_topk_w, stream));
    MOE_TRY(mxfp8_qdq(dyxe, rh, L.R, L.H, 0, stream));
    MOE_TRY(moe_expert_down_dgrad(p, ws, rh, v.g, v.u, &wb, dg, du, stream));
    MOE_TRY(mxfp8_qdq(dyxe, ch, L.R, L.H, 1, stream));
    MOE_TRY(mxfp8_qdq(v.act, ci1, L.R, L.I, 1, stream));
    MOE_TRY(moe_expert_down_wgrad(p, ws, ch, ci1, dw_down, stream));
    MOE_TRY(mxfp8_qdq(dg, ri1, L.R, L.I, 0, stream));
    MOE_TRY(mxfp8_qdq(du, ri2, L.R, L.I, 0, stream));
    MOE_TRY(moe_expert_gate_up_dgrad(p, ws, ri1, ri2, &wb, dyxe, stream));
    MOE_TRY(mxfp8_qdq(dg, ci1, L.R, L.I, 1, stream));
    MOE_TRY(mxfp8_qdq(du, ci2, L.R, L.I, 1, stream));
    MOE_TRY(mxfp8_qdq(v.xe, ch, L.R, L.H, 1, stream));
    MOE_TRY(moe_expert_gate_up_wgrad(p, ws, ci1, ci2, ch, dw_gate, dw_up, stream));
    return moe_reverse_dispatch(p, ws, dyxe, dx, stream);
  }
  if (overlap) {
    // reverse-combine (dYe, d_topk_w) run by side warps of the down
    // data-gradient GEMM, which consumes dYe tile by tile as it is finished
    if (!aligned(v.ye, 16) || !aligned(dyxe, 16) || !weights_ok(w) || !aligned(dg, 16) ||
        !aligned(du, 16))
      return MOE_ERR_INVALID_ARG;
    if (L.N > 0 && (!aligned(dy, 16) || !aligned(topk_w, 4) || !aligned(d_topk_w, 4)))
      return MOE_ERR_INVALID_ARG;
    MOE_TRY(gemm_down_dgrad_rc(L, ws, dy, v.ye, topk_w, dyxe, d_topk_w, v.g, v.u, w->w_down, dg,
                               du, S(stream)));
  } else {
    MOE_TRY(moe_reverse_combine(p, ws, dy, v.ye, topk_w, dyxe, d_topk_w, stream));
    MOE_TRY(moe_expert_down_dgrad(p, ws, dyxe, v.g, v.u, w, dg, du, stream));
  }
  MOE_TRY(moe_expert_down_wgrad(p, ws, dyxe, v.act, dw_down, stream));
  // dXe overwrites dYe in the shared buffer: dYe's last reader ran above.
  MOE_TRY(moe_expert_gate_up_dgrad(p, ws, dg, du, w, dyxe, stream));
  MOE_TRY(moe_expert_gate_up_wgrad(p, ws, dg, du, v.xe, dw_gate, dw_up, stream));
  return moe_reverse_dispatch(p, ws, dyxe, dx, stream);
}

}  // namespace

extern "C" {

int64_t moe_grouped_rows(const moe_problem* p) {
  Layout L;
  return make_layout(p, &L) == MOE_OK ? L.R : -1;
}

moe_status moe_workspace_bytes(const moe_problem* p, size_t* bytes) {
  Layout L;
  MOE_TRY(make_layout(p, &L));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = L.ws_bytes;
  return MOE_OK;
}

moe_status moe_saved_bytes(const moe_problem* p, size_t* bytes) {
  Layout L;
  MOE_TRY(make_layout(p, &L));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = L.saved_bytes;
  return MOE_OK;
}

moe_status moe_saved_layout(const moe_problem* p, void* saved, moe_saved_view* out) {
  Layout L;
  MOE_TRY(make_layout(p, &L));
  if (!aligned(saved, 256) || !out) return MOE_ERR_INVALID_ARG;
  out->xe = at<char>(saved, L.xe);
  out->g = at<char>(saved, L.g);
  out->u = at<char>(saved, L.u);
  out->act = at<char>(saved, L.act);
  out->ye = at<char>(saved, L.ye);
  return MOE_OK;
}

moe_status moe_schedule_view(const moe_problem* p, void* ws, moe_schedule* out) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (!out) return MOE_ERR_INVALID_ARG;
  out->counts = at<int32_t>(ws, L.counts);
  out->offsets = at<int32_t>(ws, L.offsets);
  out->pad_offsets = at<int32_t>(ws, L.pad_offsets);
  out->slot_of = at<int32_t>(ws, L.slot_of);
  out->src_of_row = at<int32_t>(ws, L.src_of_row);
  out->tiles = at<int32_t>(ws, L.tiles);
  out->n_tiles = at<int32_t>(ws, L.n_tiles);
  return MOE_OK;
}

moe_status moe_route_topk(const moe_problem* p, const float* logits, const float* bias,
                          int32_t* topk_ids, float* topk_w, void* ws, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (L.N > 0 && (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)))
    return MOE_ERR_INVALID_ARG;
  if (bias && !aligned(bias, 4)) return MOE_ERR_INVALID_ARG;
  return cu(launch_route_topk(L, logits, bias, topk_ids, topk_w, at<int32_t>(ws, L.err), S(stream)));
}

moe_status moe_route(const moe_problem* p, const void* x, const void* w_router, const float* bias,
                     float* logits, int32_t* topk_ids, float* topk_w, void* ws, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (L.E > 256 || L.E % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned(w_router, 16) || (logits && !aligned(logits, 16)) || (bias && !aligned(bias, 4)))
    return MOE_ERR_INVALID_ARG;
  if (L.N > 0 && (!aligned(x, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)))
    return MOE_ERR_INVALID_ARG;
  float* lg = logits ? logits : at<float>(ws, L.router_logits);
  MOE_TRY(gemm_router(L, ws, x, w_router, lg, S(stream)));
  return cu(launch_route_topk(L, lg, bias, topk_ids, topk_w, at<int32_t>(ws, L.err), S(stream)));
}

moe_status moe_router_backward(const moe_problem* p, const void* saved, const void* w_router,
                               const int32_t* topk_ids, const float* topk_w,
                               const float* d_topk_w, void* dx, float* dw_router, void* ws,
                               void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  moe_saved_view v;
  MOE_TRY(moe_saved_layout(p, const_cast<void*>(saved), &v));
  if (!aligned(w_router, 16) || !aligned(dw_router, 16)) return MOE_ERR_INVALID_ARG;
  if (L.N > 0 && (!aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(d_topk_w, 4) ||
                  !aligned(dx, 16)))
    return MOE_ERR_INVALID_ARG;
  return cu(launch_router_backward(L, ws, v.xe, w_router, topk_ids, topk_w, d_topk_w, dx,
                                   dw_router, S(stream)));
}

moe_status moe_build_schedule(const moe_problem* p, const int32_t* topk_ids, void* ws,
                              void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (L.N > 0 && !aligned(topk_ids, 4)) return MOE_ERR_INVALID_ARG;
  return cu(launch_build_schedule(L, topk_ids, ws, S(stream)));
}

moe_status moe_dispatch(const moe_problem* p, const void* ws, const void* x, void* xe,
                        void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if ((L.N > 0 && !aligned(x, 16)) || !aligned(xe, 16)) return MOE_ERR_INVALID_ARG;
  return cu(launch_dispatch(L, ws, x, xe, S(stream)));
}

moe_status moe_mxfp8_forward_operands(const moe_problem* p, void* ws, moe_mxfp8_operand* xe_rows,
                                      moe_mxfp8_operand* act_rows) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (p->dtype != MOE_MXFP8 || !xe_rows || !act_rows) return MOE_ERR_INVALID_ARG;
  *xe_rows = ws_operand(ws, L.mq_rh, L.ms_rh);
  *act_rows = ws_operand(ws, L.mq_ri, L.ms_ri);
  return MOE_OK;
}

moe_status moe_mxfp8_backward_operands(const moe_problem* p, void* ws, moe_mxfp8_operand* dg_rows,
                                       moe_mxfp8_operand* du_rows, moe_mxfp8_operand* dg_cols,
                                       moe_mxfp8_operand* du_cols, void** dg, void** du) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (p->dtype != MOE_MXFP8 || !dg_rows || !du_rows) return MOE_ERR_INVALID_ARG;
  // the buffers mx_backward_gemms passes to gemm_mx_down_dgrad
  *dg_rows = ws_operand(ws, L.mq_ri, L.ms_ri);
  *du_rows = ws_operand(ws, L.mq_ri2, L.ms_ri2);
  if (dg_cols) *dg_cols = ws_operand(ws, L.mq_ti, L.ms_ti);
  if (du_cols) *du_cols = ws_operand(ws, L.mq_ti2, L.ms_ti2);
  if (dg) *dg = at<char>(ws, L.dg);
  if (du) *du = at<char>(ws, L.du);
  return MOE_OK;
}

moe_status moe_dispatch_mxfp8(const moe_problem* p, const void* ws, const void* x, void* xe,
                              uint8_t* q_e4m3, uint8_t* s_e8m0, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if ((L.N > 0 && !aligned(x, 16)) || !aligned(xe, 16) || !aligned(q_e4m3, 16) ||
      !aligned(s_e8m0, 16))
    return MOE_ERR_INVALID_ARG;
  return cu(launch_dispatch_quant(L, ws, x, xe, q_e4m3, s_e8m0, S(stream)));
}

moe_status moe_expert_gate_up(const moe_problem* p, const void* ws, const void* xe,
                              const moe_weights* w, void* g, void* u, void* act, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  const bool no_gu = g == nullptr && u == nullptr;  // inference: Act only
  if (!aligned(xe, 16) || !weights_ok(w) || !aligned(act, 16) ||
      (!no_gu && (!aligned(g, 16) || !aligned(u, 16))))
    return MOE_ERR_INVALID_ARG;
  return gemm_gate_up(L, ws, xe, w->w_gate, w->w_up, g, u, act, S(stream));
}

moe_status moe_expert_down(const moe_problem* p, const void* ws, const void* act,
                           const moe_weights* w, void* ye, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (!aligned(act, 16) || !weights_ok(w) || !aligned(ye, 16)) return MOE_ERR_INVALID_ARG;
  return gemm_down(L, ws, act, w->w_down, ye, S(stream));
}

moe_status moe_combine(const moe_problem* p, const void* ws, const void* ye, const float* topk_w,
                       void* y, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (L.N > 0 && (!aligned(ye, 16) || !aligned(topk_w, 4) || !aligned(y, 16)))
    return MOE_ERR_INVALID_ARG;
  return cu(launch_combine(L, ws, ye, topk_w, y, S(stream)));
}

moe_status moe_dispatch_expert_ffn(const moe_problem* p, const void* ws, const void* x,
                                   const moe_weights* w, void* xe, void* g, void* u, void* act,
                                   void* ye, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (p->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const bool no_gu = g == nullptr && u == nullptr;
  if ((L.N > 0 && !aligned(x, 16)) || !weights_ok(w) || !aligned(xe, 16) || !aligned(act, 16) ||
      !aligned(ye, 16) || (!no_gu && (!aligned(g, 16) || !aligned(u, 16))))
    return MOE_ERR_INVALID_ARG;
  return gemm_fused_forward(L, ws, x, w->w_gate, w->w_up, w->w_down, xe, g, u, act, ye, 0,
                            S(stream));
}

moe_status moe_forward_inference(const moe_problem* p, const void* x, const moe_weights* w,
                                 const float* topk_w, void* y, void* ws, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  void* act = at<char>(ws, L.dg);    // [R, I] scratch
  void* ye = at<char>(ws, L.dyxe);   // [R, H] scratch
  if (p->dtype == MOE_MXFP8) {
    // Xe must exist to be quantised along H: dispatch into scratch first.
    void* xe = at<char>(ws, L.mx_ch);
    if (mx_forward_ok(w)) {
      MOE_TRY(mx_dispatch(L, ws, x, xe, S(stream)));
      MOE_TRY(mx_forward_gemms(L, ws, *w->mx, nullptr, nullptr, act, ye, S(stream)));
    } else {
      MOE_TRY(moe_dispatch(p, ws, x, xe, stream));
      void* xq = at<char>(ws, L.mx_rh);
      void* aq = at<char>(ws, L.mx_ri1);
      MOE_TRY(mxfp8_qdq(xe, xq, L.R, L.H, 0, stream));
      MOE_TRY(moe_expert_gate_up(p, ws, xq, w, at<char>(ws, L.mx_ci1), at<char>(ws, L.mx_ci2),
                                 act, stream));
      MOE_TRY(mxfp8_qdq(act, aq, L.R, L.I, 0, stream));
      MOE_TRY(moe_expert_down(p, ws, aq, w, ye, stream));
    }
    return moe_combine(p, ws, ye, topk_w, y, stream);
  }
  // Dispatch, gate/up (Act only) and down in one launch, Xe and Act in a ring
  // of minibatch slots carved from the Act scratch.
  if ((L.N > 0 && !aligned(x, 16)) || !weights_ok(w)) return MOE_ERR_INVALID_ARG;
  const int ring = fused_ring_slots(L);
  const size_t ring_x = static_cast<size_t>(ring) * 2 * kTileM * L.H * 2;
  const size_t ring_a = static_cast<size_t>(ring) * 2 * kTileM * L.I * 2;
  if (ring > 0 && ring_x + ring_a <= static_cast<size_t>(L.R) * L.I * 2) {
    char* xe = static_cast<char*>(act);
    MOE_TRY(gemm_fused_forward(L, ws, x, w->w_gate, w->w_up, w->w_down, xe, nullptr, nullptr,
                               xe + ring_x, ye, ring, S(stream)));
  } else {
    // too few rows for the ring: Xe and Ye share the scratch rows (a row
    // group's Xe is consumed before its Ye is written)
    MOE_TRY(moe_dispatch_expert_ffn(p, ws, x, w, ye, nullptr, nullptr, act, ye, stream));
  }
  return moe_combine(p, ws, ye, topk_w, y, stream);
}

moe_status moe_forward(const moe_problem* p, const void* x, const moe_weights* w,
                       const float* topk_w, void* y, void* saved, void* ws, void* stream) {
  moe_saved_view v;
  MOE_TRY(moe_saved_layout(p, saved, &v));
  if (p->dtype == MOE_MXFP8 && w && w->mx) {
    Layout L;
    MOE_TRY(prep(p, ws, &L));
    if (!mx_forward_ok(w)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(mx_dispatch(L, ws, x, v.xe, S(stream)));
    MOE_TRY(mx_forward_gemms(L, ws, *w->mx, v.g, v.u, v.act, v.ye, S(stream)));
    return moe_combine(p, ws, v.ye, topk_w, y, stream);
  }
  if (p->dtype == MOE_BF16) {
    // Four launches: measured faster than moe_dispatch_expert_ffn (the same
    // work in one persistent launch), whose dispatch competes with the GEMMs
    // for the same memory system instead of overlapping a separate resource.
    MOE_TRY(moe_dispatch(p, ws, x, v.xe, stream));
    MOE_TRY(moe_expert_gate_up(p, ws, v.xe, w, v.g, v.u, v.act, stream));
    MOE_TRY(moe_expert_down(p, ws, v.act, w, v.ye, stream));
    return moe_combine(p, ws, v.ye, topk_w, y, stream);
  }
  // MXFP8 on bf16 MMAs: gate/up reads Xe quantised along H, down reads Act
  // quantised along I, as exact bf16 values
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  MOE_TRY(moe_dispatch(p, ws, x, v.xe, stream));
  void* xq = at<char>(ws, L.mx_rh);
  void* aq = at<char>(ws, L.mx_ri1);
  MOE_TRY(mxfp8_qdq(v.xe, xq, L.R, L.H, 0, stream));
  MOE_TRY(moe_expert_gate_up(p, ws, xq, w, v.g, v.u, v.act, stream));
  MOE_TRY(mxfp8_qdq(v.act, aq, L.R, L.I, 0, stream));
  MOE_TRY(moe_expert_down(p, ws, aq, w, v.ye, stream));
  return moe_combine(p, ws, v.ye, topk_w, y, stream);
}

moe_status moe_reverse_combine(const moe_problem* p, const void* ws, const void* dy,
                               const void* ye, const float* topk_w, void* dye, float* d_topk_w,
                               void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (!aligned(ye, 16) || !aligned(dye, 16)) return MOE_ERR_INVALID_ARG;
  if (L.N > 0 && (!aligned(dy, 16) || !aligned(topk_w, 4) || !aligned(d_topk_w, 4)))
    return MOE_ERR_INVALID_ARG;
  return cu(launch_reverse_combine(L, ws, dy, ye, topk_w, dye, d_topk_w, S(stream)));
}

moe_status moe_expert_down_dgrad(const moe_problem* p, const void* ws, const void* dye,
                                 const void* g, const void* u, const moe_weights* w, void* dg,
                                 void* du, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (!aligned(dye, 16) || !aligned(g, 16) || !aligned(u, 16) || !weights_ok(w) ||
      !aligned(dg, 16) || !aligned(du, 16))
    return MOE_ERR_INVALID_ARG;
  return gemm_down_dgrad(L, ws, dye, g, u, w->w_down, dg, du, S(stream));
}

moe_status moe_expert_down_wgrad(const moe_problem* p, const void* ws, const void* dye,
                                 const void* act, float* dw_down, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (!aligned(dye, 16) || !aligned(act, 16) || !aligned(dw_down, 16))
    return MOE_ERR_INVALID_ARG;
  return gemm_down_wgrad(L, ws, dye, act, dw_down, S(stream));
}

moe_status moe_expert_gate_up_dgrad(const moe_problem* p, const void* ws, const void* dg,
                                    const void* du, const moe_weights* w, void* dxe,
                                    void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (!aligned(dg, 16) || !aligned(du, 16) || !weights_ok(w) || !aligned(dxe, 16))
    return MOE_ERR_INVALID_ARG;
  return gemm_gate_up_dgrad(L, ws, dg, du, w->w_gate, w->w_up, dxe, S(stream));
}

moe_status moe_expert_gate_up_wgrad(const moe_problem* p, const void* ws, const void* dg,
                                    const void* du, const void* xe, float* dw_gate,
                                    float* dw_up, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (!aligned(dg, 16) || !aligned(du, 16) || !aligned(xe, 16) || !aligned(dw_gate, 16) ||
      !aligned(dw_up, 16))
    return MOE_ERR_INVALID_ARG;
  return gemm_gate_up_wgrad(L, ws, dg, du, xe, dw_gate, dw_up, S(stream));
}

moe_status moe_reverse_dispatch(const moe_problem* p, const void* ws, const void* dxe, void* dx,
                                void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (L.N > 0 && (!aligned(dxe, 16) || !aligned(dx, 16))) return MOE_ERR_INVALID_ARG;
  return cu(launch_reverse_dispatch(L, ws, dxe, dx, S(stream)));
}

moe_status moe_backward(const moe_problem* p, const void* saved, const moe_weights* w,
                        const float* topk_w, const void* dy, void* dx, float* dw_gate,
                        float* dw_up, float* dw_down, float* d_topk_w, void* ws, void* stream) {
  return backward_impl(p, saved, w, topk_w, dy, dx, dw_gate, dw_up, dw_down, d_topk_w, ws, stream,
                       false);
}

moe_status moe_backward_overlap(const moe_problem* p, const void* saved, const moe_weights* w,
                                const float* topk_w, const void* dy, void* dx, float* dw_gate,
                                float* dw_up, float* dw_down, float* d_topk_w, void* ws,
                                void* stream) {
  return backward_impl(p, saved, w, topk_w, dy, dx, dw_gate, dw_up, dw_down, d_topk_w, ws, stream,
                       p && p->dtype == MOE_BF16);
}

moe_status mxfp8_qdq(const void* src_bf16, void* dst_bf16, int64_t rows, int64_t cols, int axis,
                     void* stream) {
  if (rows < 0 || cols < 0 || (axis != 0 && axis != 1)) return MOE_ERR_INVALID_ARG;
  if (axis == 0 && cols % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (axis == 1 && (rows % 32 != 0 || cols % 2 != 0)) return MOE_ERR_INVALID_ARG;
  if (rows * cols == 0) return MOE_OK;
  if (!aligned(src_bf16, 16) || !aligned(dst_bf16, 16)) return MOE_ERR_INVALID_ARG;
  return cu(launch_mxfp8_qdq(src_bf16, dst_bf16, rows, cols, axis, S(stream)));
}

moe_status mxfp8_quantize_mma(const void* src_bf16, int64_t rows, int64_t cols, int transpose,
                              uint8_t* q_e4m3, uint8_t* s_e8m0, void* stream) {
  if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (transpose != 0 && transpose != 1) return MOE_ERR_INVALID_ARG;
  if (rows * cols == 0) return MOE_OK;
  if (!aligned(src_bf16, 16) || !aligned(q_e4m3, 16) || !aligned(s_e8m0, 16))
    return MOE_ERR_INVALID_ARG;
  return cu(launch_mxfp8_quantize_mma(src_bf16, rows, cols, transpose, q_e4m3, s_e8m0,
                                      S(stream)));
}

moe_status mxfp8_quantize(const void* src_bf16, int64_t rows, int64_t cols, uint8_t* q_e4m3,
                          uint8_t* scale_e8m0, void* stream) {
  if (rows < 0 || cols < 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (rows * cols == 0) return MOE_OK;
  if (!aligned(src_bf16, 16) || !aligned(q_e4m3, 16) || !scale_e8m0) return MOE_ERR_INVALID_ARG;
  return cu(launch_mxfp8_quantize(src_bf16, rows, cols, q_e4m3, scale_e8m0, S(stream)));
}

moe_status moe_get_device_error(const moe_problem* p, const void* ws, int32_t* code_out,
                                void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  if (!code_out) return MOE_ERR_INVALID_ARG;
  return cu(cudaMemcpyAsync(code_out, at<int32_t>(ws, L.err), sizeof(int32_t),
                            cudaMemcpyDeviceToHost, S(stream)));
}

moe_status moe_clear_device_error(const moe_problem* p, void* ws, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  return cu(cudaMemsetAsync(at<int32_t>(ws, L.err), 0, sizeof(int32_t), S(stream)));
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status moe_test_wait_timeout(const moe_problem* p, void* ws, void* stream) {
  Layout L;
  MOE_TRY(prep(p, ws, &L));
  wait_timeout_kernel<<<1, 32, 0, S(stream)>>>(at<int32_t>(ws, L.err));
  note_launch();
  return cu(cudaGetLastError());
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or dtype";
    case MOE_ERR_CUDA: return "CUDA runtime or driver error";
    case MOE_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

}  // extern "C"
