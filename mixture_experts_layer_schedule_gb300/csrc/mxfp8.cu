// mxfp8.cu -- MXFP8 quantiser for expert weights and activations.
//
// The project summary "Mixture-of-Kittens (MoK)" (core concepts, MXFP8 row)
// says weights are pre-quantised to MXFP8 by a quantise op before they reach
// the kernel. The format is OCP Microscaling (MX) v1.0 with E4M3 elements:
// per block of 32 consecutive values of a row, the shared scale is
// 2^(floor(log2(amax)) - 8) stored as an E8M0 code (exponent + 127), and each
// element is v / scale rounded to nearest-even E4M3, saturating at +-448.
//
// One thread per 32-value block: it reads 64 contiguous bytes and writes 32
// code bytes plus one scale byte, so consecutive threads stream consecutive
// memory. The scale exponent comes straight from the fp32 exponent field of
// amax (bf16 values are exact in fp32); v / scale is a power-of-two product,
// exact in fp32 for every value that does not round to zero in E4M3.
#include <cuda_fp16.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(const uint4* __restrict__ src,
                                                             int64_t n_blocks,
                                                             uint4* __restrict__ q,
                                                             uint8_t* __restrict__ scale) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= n_blocks) return;
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) raw[i] = src[b * 4 + i];
  float f[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[8 * i + 0] = bf16lo(raw[i].x); f[8 * i + 1] = bf16hi(raw[i].x);
    f[8 * i + 2] = bf16lo(raw[i].y); f[8 * i + 3] = bf16hi(raw[i].y);
    f[8 * i + 4] = bf16lo(raw[i].z); f[8 * i + 5] = bf16hi(raw[i].z);
    f[8 * i + 6] = bf16lo(raw[i].w); f[8 * i + 7] = bf16hi(raw[i].w);
  }
  uint32_t packed[8];
  scale[b] = quant32(f, packed);
  q[b * 2 + 0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  q[b * 2 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
}

// Quantise-dequantise: the MXFP8 value of each element, written back as bf16
// (exact: an E4M3 value times a power of two fits bf16 for every scale the
// quantiser produces from bf16 data of normal magnitude).
__device__ __forceinline__ void qdq32(float (&f)[32]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const int biased = (__float_as_uint(amax) >> 23) & 0xFF;
  const int code = biased == 0 ? 0 : max(0, biased - 8);
  const float inv = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);  // 2^(127-code)
  // 2^(code-127) as a product of two normal floats (code may be < 1)
  const float sc_hi = __uint_as_float(static_cast<uint32_t>(max(code, 1)) << 23);
  const float sc_lo = code >= 1 ? 1.0f : 0.5f;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint32_t q = e4m3x2(f[i] * inv, f[i + 1] * inv);
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(q)));
    const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
    f[i] = __low2float(hv) * sc_hi * sc_lo;
    f[i + 1] = __high2float(hv) * sc_hi * sc_lo;
  }
}

// Blocks of 32 consecutive columns of a row; one thread per block.
__global__ void __launch_bounds__(256) qdq_rows_kernel(const uint4* __restrict__ src,
                                                       int64_t n_blocks, uint4* __restrict__ dst) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= n_blocks) return;
  float f[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 r = src[b * 4 + i];
    f[8 * i + 0] = bf16lo(r.x); f[8 * i + 1] = bf16hi(r.x);
    f[8 * i + 2] = bf16lo(r.y); f[8 * i + 3] = bf16hi(r.y);
    f[8 * i + 4] = bf16lo(r.z); f[8 * i + 5] = bf16hi(r.z);
    f[8 * i + 6] = bf16lo(r.w); f[8 * i + 7] = bf16hi(r.w);
  }
  qdq32(f);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    dst[b * 4 + i] = make_uint4(pack_bf16x2(f[8 * i], f[8 * i + 1]), pack_bf16x2(f[8 * i + 2], f[8 * i + 3]),
                                pack_bf16x2(f[8 * i + 4], f[8 * i + 5]), pack_bf16x2(f[8 * i + 6], f[8 * i + 7]));
}

// Blocks of 32 consecutive rows of a column; one thread per (row block, column
// pair), so a warp reads 128 contiguous bytes of each row.
__global__ void __launch_bounds__(256) qdq_cols_kernel(const uint32_t* __restrict__ src,
                                                       int64_t rows, int64_t cols2,
                                                       uint32_t* __restrict__ dst) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n = (rows / 32) * cols2;
  if (idx >= n) return;
  const int64_t rb = idx / cols2, c = idx % cols2;
  float lo[32], hi[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const uint32_t v = src[(rb * 32 + r) * cols2 + c];
    lo[r] = bf16lo(v);
    hi[r] = bf16hi(v);
  }
  qdq32(lo);
  qdq32(hi);
#pragma unroll
  for (int r = 0; r < 32; ++r) dst[(rb * 32 + r) * cols2 + c] = pack_bf16x2(lo[r], hi[r]);
}

// Row form: blocks of 32 consecutive values of a row; q [rows, cols].
__global__ void __launch_bounds__(256) quant_mma_rows_kernel(const uint4* __restrict__ src,
                                                             int64_t rows, int64_t cols,
                                                             uint4* __restrict__ q,
                                                             uint8_t* __restrict__ sf) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_row = cols / 32;
  if (b >= rows * per_row) return;
  float f[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 r = src[b * 4 + i];
    f[8 * i + 0] = bf16lo(r.x); f[8 * i + 1] = bf16hi(r.x);
    f[8 * i + 2] = bf16lo(r.y); f[8 * i + 3] = bf16hi(r.y);
    f[8 * i + 4] = bf16lo(r.z); f[8 * i + 5] = bf16hi(r.z);
    f[8 * i + 6] = bf16lo(r.w); f[8 * i + 7] = bf16hi(r.w);
  }
  uint32_t packed[8];
  const uint8_t code = quant32(f, packed);
  q[b * 2 + 0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  q[b * 2 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  sf[sf_mma_index(b / per_row, b % per_row, rows)] = code;
}

// Transposed form: q [cols, rows] = src^T, blocks of 32 consecutive source
// rows of a column (the K of the transposed operand). A CTA stages a
// 128-row x 64-column tile in shared memory (coalesced 128-byte row reads);
// thread (column c, block b) quantises rows 32b..32b+31 of column c into the
// shared output tile (64 output rows of 128 code bytes), which the warps then
// write out with coalesced 16-byte stores (8 lanes per 128-byte output row).
constexpr int kQtRows = 128, kQtCols = 64;

__global__ void __launch_bounds__(256) quant_mma_t_kernel(const uint16_t* __restrict__ src,
                                                          int64_t rows, int64_t cols,
                                                          uint8_t* __restrict__ q,
                                                          uint8_t* __restrict__ sf) {
  __shared__ __align__(16) uint16_t tile[kQtRows][kQtCols];
  __shared__ __align__(16) uint8_t out[kQtCols][kQtRows + 16];  // +16: conflict-free rows
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kQtRows;
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kQtCols;
  for (int i = threadIdx.x; i < kQtRows * kQtCols / 8; i += blockDim.x) {
    const int r = i / (kQtCols / 8), cv = i % (kQtCols / 8);
    *reinterpret_cast<uint4*>(&tile[r][cv * 8]) =
        *reinterpret_cast<const uint4*>(src + (r0 + r) * cols + c0 + cv * 8);
  }
  __syncthreads();
  const int c = threadIdx.x % kQtCols, b = threadIdx.x / kQtCols;
  float f[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) f[r] = __uint_as_float(static_cast<uint32_t>(tile[32 * b + r][c]) << 16);
  uint32_t packed[8];
  const uint8_t code = quant32(f, packed);
  uint4* o = reinterpret_cast<uint4*>(&out[c][32 * b]);
  o[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  o[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  sf[sf_mma_index(c0 + c, (r0 >> 5) + b, cols)] = code;
  __syncthreads();
  for (int i = threadIdx.x; i < kQtCols * kQtRows / 16; i += blockDim.x) {
    const int oc = i / (kQtRows / 16), piece = i % (kQtRows / 16);
    *reinterpret_cast<uint4*>(q + (c0 + oc) * rows + r0 + 16 * piece) =
        *reinterpret_cast<const uint4*>(&out[oc][16 * piece]);
  }
}

}  // namespace

cudaError_t launch_mxfp8_quantize_mma(const void* src, int64_t rows, int64_t cols, int transpose,
                                      uint8_t* q, uint8_t* sf, cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (!transpose) {
    const int64_t n = rows * (cols / 32);
    quant_mma_rows_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
        static_cast<const uint4*>(src), rows, cols, reinterpret_cast<uint4*>(q), sf);
  } else {
    const dim3 grid(static_cast<unsigned>(rows / kQtRows), static_cast<unsigned>(cols / kQtCols));
    quant_mma_t_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(src), rows, cols, q, sf);
  }
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_qdq(const void* src, void* dst, int64_t rows, int64_t cols, int axis,
                             cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (axis == 0) {
    const int64_t n_blocks = rows * (cols / 32);
    qdq_rows_kernel<<<static_cast<unsigned>((n_blocks + 255) / 256), 256, 0, s>>>(
        static_cast<const uint4*>(src), n_blocks, static_cast<uint4*>(dst));
  } else {
    const int64_t n = (rows / 32) * (cols / 2);
    qdq_cols_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
        static_cast<const uint32_t*>(src), rows, cols / 2, static_cast<uint32_t*>(dst));
  }
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_quantize(const void* src, int64_t rows, int64_t cols, uint8_t* q,
                                  uint8_t* scale, cudaStream_t s) {
  const int64_t n_blocks = rows * (cols / 32);
  if (n_blocks == 0) return cudaSuccess;
  const int64_t grid = (n_blocks + 255) / 256;
  mxfp8_quantize_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(
      static_cast<const uint4*>(src), n_blocks, reinterpret_cast<uint4*>(q), scale);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
