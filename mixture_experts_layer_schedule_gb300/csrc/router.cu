// router.cu -- the router's backward (the router GEMM itself is a mode of the
// grouped GEMM, grouped_gemm.cu; its top-k is topk_kernel).
//
// The router sits in front of the layer ("Mixture-of-Kittens: Cursor
// open-sources an MoE training megakernel", key flowchart, Router node):
// logits = x . Wr^T, routing weights w = softmax over the k selected logits.
// With the selection held fixed (top-k is piecewise constant) and
// dw = dL/dw from the reverse-combine:
//   dz[t,j] = w[t,j] * (dw[t,j] - sum_i w[t,i] * dw[t,i])       (dL/d logit)
//   dx[t]  += sum_j dz[t,j] * Wr[ids[t,j]]                       (in place)
//   dWr[e]  = sum over the rows of expert e of dz[row] * Xe[row]  (fp32)
// dWr is a segmented reduction over the expert-grouped Xe of the forward
// context: one partial per 128-row tile (rows in order), then per expert the
// partials of its tiles in tile order -- a fixed order, no atomics.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

// One CTA per token: dz of its k assignments (one thread, j order), then the
// router's share of dx added to the row, fp32 in j order, one rounding.
__global__ void __launch_bounds__(kThreads) router_dx_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, const float* __restrict__ dw,
    const uint4* __restrict__ wr, int64_t N, int k, int E, int hv, float* __restrict__ dz,
    uint4* __restrict__ dx, int32_t* err) {
  __shared__ float dzs[kMaxK];
  __shared__ int32_t es[kMaxK];
  const int64_t t = blockIdx.x;
  if (threadIdx.x == 0) {
    float s = 0.0f;
    for (int j = 0; j < k; ++j) s = fmaf(w[t * k + j], dw[t * k + j], s);
    for (int j = 0; j < k; ++j) {
      const float d = w[t * k + j] * (dw[t * k + j] - s);
      int32_t e = ids[t * k + j];
      if (e < 0 || e >= E) {
        set_dev_error(err, MOE_DEVERR_BAD_EXPERT);
        e = -1;
      }
      dzs[j] = d;
      es[j] = e;
      dz[t * k + j] = d;
    }
  }
  __syncthreads();
  for (int v = threadIdx.x; v < hv; v += blockDim.x) {
    const uint4 cur = dx[t * hv + v];
    float acc[8] = {bf16lo(cur.x), bf16hi(cur.x), bf16lo(cur.y), bf16hi(cur.y),
                    bf16lo(cur.z), bf16hi(cur.z), bf16lo(cur.w), bf16hi(cur.w)};
    for (int j = 0; j < k; ++j) {
      if (es[j] < 0) continue;
      const uint4 r = wr[static_cast<int64_t>(es[j]) * hv + v];
      const float f[8] = {bf16lo(r.x), bf16hi(r.x), bf16lo(r.y), bf16hi(r.y),
                          bf16lo(r.z), bf16hi(r.z), bf16lo(r.w), bf16hi(r.w)};
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(dzs[j], f[q], acc[q]);
    }
    dx[t * hv + v] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

// Partial of one 128-row tile of the expert-grouped buffer over 1024 columns:
// thread i owns 8 columns; rows in order (padding rows: dz 0 and Xe 0).
__global__ void __launch_bounds__(128) router_wgrad_partial_kernel(
    const uint4* __restrict__ xe, const int32_t* __restrict__ src_of_row,
    const int32_t* __restrict__ pad_offsets, const float* __restrict__ dz, int E, int64_t A,
    int hv, float* __restrict__ partial) {
  __shared__ float dz_row[128];  // dz of each row of the tile (0 for padding rows)
  const int64_t tile = blockIdx.x;
  const int v = blockIdx.y * blockDim.x + threadIdx.x;  // 8-column vector index
  const int64_t row0 = tile * 128;
  if (row0 >= pad_offsets[E]) return;  // past the last segment: never read (whole CTA)
  {
    const int32_t a = src_of_row[row0 + threadIdx.x];  // blockDim.x == 128 rows
    dz_row[threadIdx.x] = (a >= 0 && a < A) ? dz[a] : 0.0f;
  }
  __syncthreads();
  if (v >= hv) return;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll 8
  for (int r = 0; r < 128; ++r) {
    const float d = dz_row[r];  // padding rows hold zeros in Xe as well
    const uint4 x = xe[(row0 + r) * hv + v];
    const float f[8] = {bf16lo(x.x), bf16hi(x.x), bf16lo(x.y), bf16hi(x.y),
                        bf16lo(x.z), bf16hi(x.z), bf16lo(x.w), bf16hi(x.w)};
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = fmaf(d, f[q], acc[q]);
  }
  float4* out = reinterpret_cast<float4*>(partial + tile * (hv * 8) + v * 8);
  out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// dWr[e] = the partials of expert e's tiles, in tile order.
__global__ void __launch_bounds__(128) router_wgrad_reduce_kernel(
    const float* __restrict__ partial, const int32_t* __restrict__ pad_offsets, int64_t n_row_tiles,
    int hv, float* __restrict__ dwr) {
  const int e = blockIdx.x;
  const int v = blockIdx.y * blockDim.x + threadIdx.x;
  if (v >= hv) return;
  int64_t t0 = pad_offsets[e] / 128, t1 = pad_offsets[e + 1] / 128;
  t0 = t0 < 0 ? 0 : t0;
  t1 = t1 > n_row_tiles ? n_row_tiles : t1;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int64_t tt = t0; tt < t1; ++tt) {
    const float4* p = reinterpret_cast<const float4*>(partial + tt * (hv * 8) + v * 8);
    const float4 a = p[0], b = p[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  float4* out = reinterpret_cast<float4*>(dwr + static_cast<int64_t>(e) * (hv * 8) + v * 8);
  out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

}  // namespace

cudaError_t launch_router_backward(const Layout& L, const void* ws, const void* xe,
                                   const void* w_router, const int32_t* ids, const float* w,
                                   const float* dw, void* dx, float* dw_router, cudaStream_t s) {
  const int hv = L.H / 8;
  float* dz = const_cast<float*>(at<float>(ws, L.router_dz));
  float* partial = const_cast<float*>(at<float>(ws, L.router_partial));
  int32_t* err = const_cast<int32_t*>(at<int32_t>(ws, L.err));
  if (L.N > 0) {
    router_dx_kernel<<<static_cast<unsigned>(L.N), kThreads, 0, s>>>(
        ids, w, dw, static_cast<const uint4*>(w_router), L.N, L.k, L.E, hv, dz,
        static_cast<uint4*>(dx), err);
    note_launch();
  }
  const int64_t n_row_tiles = L.R / 128;
  const dim3 pgrid(static_cast<unsigned>(n_row_tiles), static_cast<unsigned>((hv + 127) / 128));
  router_wgrad_partial_kernel<<<pgrid, 128, 0, s>>>(
      static_cast<const uint4*>(xe), at<int32_t>(ws, L.src_of_row), at<int32_t>(ws, L.pad_offsets),
      dz, L.E, L.A, hv, partial);
  note_launch();
  const dim3 rgrid(static_cast<unsigned>(L.E), static_cast<unsigned>((hv + 127) / 128));
  router_wgrad_reduce_kernel<<<rgrid, 128, 0, s>>>(partial, at<int32_t>(ws, L.pad_offsets),
                                                   n_row_tiles, hv, dw_router);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
