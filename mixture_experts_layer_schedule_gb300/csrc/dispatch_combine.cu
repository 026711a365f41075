// dispatch_combine.cu -- the HBM-bound data-movement phases of the layer.
//
// On one GPU the pages' NVLink rounds ("Mixture-of-Kittens: Cursor
// open-sources an MoE training megakernel", key point 2: pull dispatch, push
// combine, pull reverse-combine, push reverse-dispatch) become copies between
// the token-ordered tensors and the expert-grouped buffer:
//   dispatch         xe[slot(t,j)] = x[t]
//   combine          y[t] = sum_j w[t,j] * ye[slot(t,j)]           (fp32, j order)
//   reverse-combine  dye[slot(t,j)] = w[t,j] * dy[t];  dw[t,j] = <dy[t], ye[slot(t,j)]>
//   reverse-dispatch dx[t] = sum_j dxe[slot(t,j)]                  (fp32, j order)
// Each CTA owns one token and walks its row in 16-byte vectors, so every row
// of x / dy / y / dx is read or written exactly once and each expert row is
// touched by exactly one CTA. Extra CTAs at the front of the grid (kPadSplit per
// expert) zero the padding rows that round each expert segment up to T rows. Slots are
// bounds-checked: an unplaced assignment (bad expert id) is skipped.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
// CTAs per expert that zero its padding rows. They come first in the grid so
// that their writes overlap the token CTAs instead of forming a tail.
constexpr int kPadSplit = 8;

// Zero every kPadSplit-th padding row of expert e's segment, from the part-th.
__device__ __forceinline__ void zero_padding(int e, int part, const int32_t* __restrict__ counts,
                                             const int32_t* __restrict__ pad_offsets,
                                             int64_t R, int hv, uint4* __restrict__ buf) {
  const int64_t r0 = static_cast<int64_t>(pad_offsets[e]) + counts[e];
  const int64_t r1 = pad_offsets[e + 1];
  for (int64_t r = r0 + part; r < r1 && r < R; r += kPadSplit)
    for (int v = threadIdx.x; v < hv; v += blockDim.x) buf[r * hv + v] = make_uint4(0, 0, 0, 0);
}

__global__ void __launch_bounds__(kThreads) dispatch_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ slot_of,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ pad_offsets, int64_t N, int k,
    int hv, int64_t R, int E, uint4* __restrict__ xe) {
  const int64_t b = blockIdx.x;
  if (b < static_cast<int64_t>(E) * kPadSplit) {
    zero_padding(static_cast<int>(b / kPadSplit), static_cast<int>(b % kPadSplit), counts,
                 pad_offsets, R, hv, xe);
    return;
  }
  const int64_t t = b - static_cast<int64_t>(E) * kPadSplit;
  __shared__ int32_t slots[kMaxK];
  if (threadIdx.x < k) slots[threadIdx.x] = slot_of[t * k + threadIdx.x];
  __syncthreads();
  for (int v = threadIdx.x; v < hv; v += blockDim.x) {
    const uint4 val = x[t * hv + v];
    for (int j = 0; j < k; ++j)
      if (slots[j] >= 0 && slots[j] < R) xe[static_cast<int64_t>(slots[j]) * hv + v] = val;
  }
}

__global__ void __launch_bounds__(kThreads) combine_kernel(
    const uint4* __restrict__ ye, const float* __restrict__ w, const int32_t* __restrict__ slot_of,
    int64_t N, int k, int hv, int64_t R, uint4* __restrict__ y) {
  const int64_t t = blockIdx.x;
  __shared__ int32_t slots[kMaxK];
  __shared__ float wt[kMaxK];
  if (threadIdx.x < k) {
    slots[threadIdx.x] = slot_of[t * k + threadIdx.x];
    wt[threadIdx.x] = w ? w[t * k + threadIdx.x] : 1.0f;
  }
  __syncthreads();
  for (int v = threadIdx.x; v < hv; v += blockDim.x) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j = 0; j < k; ++j) {
      if (slots[j] < 0 || slots[j] >= R) continue;
      float f[8];
      unpack8(ye[static_cast<int64_t>(slots[j]) * hv + v], f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(wt[j], f[q], acc[q]);
    }
    y[t * hv + v] = pack8(acc);
  }
}

__global__ void __launch_bounds__(kThreads) reverse_combine_kernel(
    const uint4* __restrict__ dy, const uint4* __restrict__ ye, const float* __restrict__ w,
    const int32_t* __restrict__ slot_of, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ pad_offsets, int64_t N, int k, int hv, int64_t R,
    int E, uint4* __restrict__ dye, float* __restrict__ dw) {
  __shared__ float red[kThreads / 32][kMaxK];
  const int64_t b = blockIdx.x;
  if (b < static_cast<int64_t>(E) * kPadSplit) {
    zero_padding(static_cast<int>(b / kPadSplit), static_cast<int>(b % kPadSplit), counts,
                 pad_offsets, R, hv, dye);
    return;
  }
  const int64_t t = b - static_cast<int64_t>(E) * kPadSplit;
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  for (int j = 0; j < k; ++j) {
    const int32_t slot = slot_of[t * k + j];
    const bool ok = slot >= 0 && slot < R;
    const float wj = w[t * k + j];
    float part = 0.0f;
    for (int v = threadIdx.x; v < hv; v += blockDim.x) {
      float g[8];
      unpack8(dy[t * hv + v], g);
      if (ok) {
        float s[8], e8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) s[q] = wj * g[q];
        dye[static_cast<int64_t>(slot) * hv + v] = pack8(s);
        unpack8(ye[static_cast<int64_t>(slot) * hv + v], e8);
#pragma unroll
        for (int q = 0; q < 8; ++q) part = fmaf(g[q], e8[q], part);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_down_sync(0xffffffffu, part, off);
    if (lane == 0) red[wib][j] = part;
  }
  __syncthreads();
  if (threadIdx.x < k) {
    float s = 0.0f;
    for (int q = 0; q < kThreads / 32; ++q) s += red[q][threadIdx.x];  // fixed order
    dw[t * k + threadIdx.x] = s;
  }
}

}  // namespace

cudaError_t launch_dispatch(const Layout& L, const void* ws, const void* x, void* xe,
                            cudaStream_t s) {
  const int64_t blocks = L.N + static_cast<int64_t>(L.E) * kPadSplit;
  dispatch_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
      static_cast<const uint4*>(x), at<int32_t>(ws, L.slot_of), at<int32_t>(ws, L.counts),
      at<int32_t>(ws, L.pad_offsets), L.N, L.k, L.H / 8, L.R, L.E, static_cast<uint4*>(xe));
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine(const Layout& L, const void* ws, const void* ye, const float* w,
                           void* y, cudaStream_t s) {
  if (L.N == 0) return cudaSuccess;
  combine_kernel<<<static_cast<unsigned>(L.N), kThreads, 0, s>>>(
      static_cast<const uint4*>(ye), w, at<int32_t>(ws, L.slot_of), L.N, L.k, L.H / 8, L.R,
      static_cast<uint4*>(y));
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_reverse_combine(const Layout& L, const void* ws, const void* dy,
                                   const void* ye, const float* w, void* dye, float* dw,
                                   cudaStream_t s) {
  const int64_t blocks = L.N + static_cast<int64_t>(L.E) * kPadSplit;
  reverse_combine_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
      static_cast<const uint4*>(dy), static_cast<const uint4*>(ye), w,
      at<int32_t>(ws, L.slot_of), at<int32_t>(ws, L.counts), at<int32_t>(ws, L.pad_offsets), L.N,
      L.k, L.H / 8, L.R, L.E, static_cast<uint4*>(dye), dw);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_reverse_dispatch(const Layout& L, const void* ws, const void* dxe, void* dx,
                                    cudaStream_t s) {
  if (L.N == 0) return cudaSuccess;
  combine_kernel<<<static_cast<unsigned>(L.N), kThreads, 0, s>>>(
      static_cast<const uint4*>(dxe), nullptr, at<int32_t>(ws, L.slot_of), L.N, L.k, L.H / 8, L.R,
      static_cast<uint4*>(dx));
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
