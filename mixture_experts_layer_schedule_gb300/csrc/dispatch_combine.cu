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

// Dispatch with the MXFP8 row quantisation of Xe fused in (the MXFP8 forward):
// besides xe[slot] = x[t] it writes, for every copy, the row's E4M3 codes
// q[slot] (blocks of 32 along H) and E8M0 scales in the tensor-memory chunk
// layout. A token's blocks are the same for all k copies, so each is
// quantised once: thread i holds 8 values (one 16-byte vector), four
// neighbouring threads form a 32-value block (amax by shuffles), and the 4
// scales of one 512-byte-chunk word (16 neighbouring threads) go out as one
// 32-bit store per copy. Same rounding as quant32. Padding rows get zero codes
// and scales (the front CTAs, as for xe).
__global__ void __launch_bounds__(kThreads) dispatch_quant_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ slot_of,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ pad_offsets, int64_t N, int k,
    int hv, int64_t R, int E, uint4* __restrict__ xe, uint2* __restrict__ q,
    uint8_t* __restrict__ sf) {
  const int64_t b = blockIdx.x;
  const int64_t rows_chunks = R >> 7;
  if (b < static_cast<int64_t>(E) * kPadSplit) {
    const int e = static_cast<int>(b / kPadSplit), part = static_cast<int>(b % kPadSplit);
    zero_padding(e, part, counts, pad_offsets, R, hv, xe);
    const int64_t r0 = static_cast<int64_t>(pad_offsets[e]) + counts[e];
    const int64_t r1 = pad_offsets[e + 1];
    for (int64_t r = r0 + part; r < r1 && r < R; r += kPadSplit) {
      for (int v = threadIdx.x; v < hv; v += blockDim.x) q[r * hv + v] = make_uint2(0u, 0u);
      for (int w = threadIdx.x; w < hv / 16; w += blockDim.x)
        *reinterpret_cast<uint32_t*>(sf + (w * rows_chunks + (r >> 7)) * 512 + (r & 31) * 16 +
                                     ((r >> 5) & 3) * 4) = 0u;
    }
    return;
  }
  const int64_t t = b - static_cast<int64_t>(E) * kPadSplit;
  __shared__ int32_t slots[kMaxK];
  if (threadIdx.x < k) slots[threadIdx.x] = slot_of[t * k + threadIdx.x];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  for (int v = threadIdx.x; v < hv; v += blockDim.x) {  // hv % 32 == 0: whole warps
    const uint4 val = x[t * hv + v];
    float f[8];
    unpack8(val, f);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int biased = (__float_as_uint(amax) >> 23) & 0xFF;
    const int code = biased == 0 ? 0 : max(0, biased - 8);
    const float inv = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
    const uint32_t lo = e4m3x2(f[0] * inv, f[1] * inv) | (e4m3x2(f[2] * inv, f[3] * inv) << 16);
    const uint32_t hi = e4m3x2(f[4] * inv, f[5] * inv) | (e4m3x2(f[6] * inv, f[7] * inv) << 16);
    // the chunk word of blocks 4w..4w+3 (vectors 16w..16w+15) from lanes 0 / 16
    const int base = lane & 16;
    const uint32_t word = static_cast<uint32_t>(__shfl_sync(0xffffffffu, code, base)) |
                          (static_cast<uint32_t>(__shfl_sync(0xffffffffu, code, base + 4)) << 8) |
                          (static_cast<uint32_t>(__shfl_sync(0xffffffffu, code, base + 8)) << 16) |
                          (static_cast<uint32_t>(__shfl_sync(0xffffffffu, code, base + 12)) << 24);
    const int w = v >> 4;
    for (int j = 0; j < k; ++j) {
      const int64_t r = slots[j];
      if (r < 0 || r >= R) continue;
      xe[r * hv + v] = val;
      q[r * hv + v] = make_uint2(lo, hi);
      if ((lane & 15) == 0)
        *reinterpret_cast<uint32_t*>(sf + (w * rows_chunks + (r >> 7)) * 512 + (r & 31) * 16 +
                                     ((r >> 5) & 3) * 4) = word;
    }
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

cudaError_t launch_dispatch_quant(const Layout& L, const void* ws, const void* x, void* xe,
                                  uint8_t* q, uint8_t* sf, cudaStream_t s) {
  const int64_t blocks = L.N + static_cast<int64_t>(L.E) * kPadSplit;
  dispatch_quant_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
      static_cast<const uint4*>(x), at<int32_t>(ws, L.slot_of), at<int32_t>(ws, L.counts),
      at<int32_t>(ws, L.pad_offsets), L.N, L.k, L.H / 8, L.R, L.E, static_cast<uint4*>(xe),
      reinterpret_cast<uint2*>(q), sf);
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
