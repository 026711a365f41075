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

// Row form alone: blocks of 32 consecutive values of a row; q [rows, cols].
// One thread per block streams 64 bytes in and 32 code bytes out; this
// measured faster than the tile kernel below when only this form is wanted.
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

// Both MMA-layout forms of bf16 src [rows, cols] (rows, cols multiples of
// 128), one 128 x 128 tile per CTA, read from HBM once:
//   row form (ROWF): q_r [rows, cols], blocks of 32 consecutive values of a
//     row (K = cols); the tile's 512 scales fill chunk (c0/128, r0/128);
//   transposed form (TF): q_t [cols, rows] = src^T, blocks of 32 consecutive
//     source rows of a column (K = rows); its scales fill chunk (r0/128, c0/128).
// The tile lands in shared memory by cp.async (16-byte pieces, coalesced
// 256-byte row reads), its 16-byte chunks XOR-swizzled by the row so that
// both the row-wise and the column-wise reads below are conflict-free. The
// codes and scales of both forms are staged in shared memory again and
// written out as whole 128-byte rows and whole 512-byte scale chunks.
constexpr int kQtTile = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

template <bool ROWF, bool TF>
__global__ void __launch_bounds__(256, 3) quant_mma_tile_kernel(
    const uint4* __restrict__ src, int64_t rows, int64_t cols, uint8_t* __restrict__ q_r,
    uint8_t* __restrict__ sf_r, uint8_t* __restrict__ q_t, uint8_t* __restrict__ sf_t) {
  // tile: 128 rows x 16 chunks (16 bytes = 8 bf16); chunk c of row r at
  // r * 16 + (c ^ (r & 15)). Reused after the reads for the code staging:
  // row form [128 rows][8 chunks] at uint4 0, transposed [128][8] at 1024.
  __shared__ __align__(16) uint4 tile[kQtTile * 16];
  __shared__ __align__(16) uint8_t sfs[2][512];
  const int tid = threadIdx.x;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kQtTile;
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kQtTile;
  const int64_t src_ld = cols / 8;  // uint4 per source row
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = tid + 256 * k, r = i >> 4, c = i & 15;
    cp_async16(smem_u32(&tile[r * 16 + (c ^ (r & 15))]), src + (r0 + r) * src_ld + c0 / 8 + c);
  }
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  uint32_t pr[2][8], pt[2][8];
  uint8_t cr[2] = {0, 0}, ct[2] = {0, 0};
  const int rr = tid & 127, bp = tid >> 7;  // row form: row rr, column blocks 2bp, 2bp+1
  const int cp = tid & 63, rb = tid >> 6;   // transposed: columns 2cp, 2cp+1, rows 32rb..+31
  if constexpr (ROWF) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float f[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = 8 * bp + 4 * j + q;
        const uint4 w = tile[rr * 16 + (c ^ (rr & 15))];
        f[8 * q + 0] = bf16lo(w.x); f[8 * q + 1] = bf16hi(w.x);
        f[8 * q + 2] = bf16lo(w.y); f[8 * q + 3] = bf16hi(w.y);
        f[8 * q + 4] = bf16lo(w.z); f[8 * q + 5] = bf16hi(w.z);
        f[8 * q + 6] = bf16lo(w.w); f[8 * q + 7] = bf16hi(w.w);
      }
      cr[j] = quant32(f, pr[j]);
    }
  }
  if constexpr (TF) {
    const uint32_t* tw = reinterpret_cast<const uint32_t*>(tile);
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // column 2cp + h: the low / high bf16 of each word
      float f[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const int row = 32 * rb + r;
        const uint32_t w = tw[row * 64 + (((cp >> 2) ^ (row & 15)) << 2) + (cp & 3)];
        f[r] = h ? bf16hi(w) : bf16lo(w);
      }
      ct[h] = quant32(f, pt[h]);
    }
  }
  __syncthreads();  // every read of the bf16 tile is done

  if constexpr (ROWF) {
    // row rr, code bytes [64 bp, +64) = chunks 4bp..4bp+3, swizzled by rr & 7
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = 4 * bp + 2 * j + h;
        tile[rr * 8 + (c ^ (rr & 7))] =
            make_uint4(pr[j][4 * h], pr[j][4 * h + 1], pr[j][4 * h + 2], pr[j][4 * h + 3]);
      }
    // scales of (row rr, blocks 2bp, 2bp+1): adjacent bytes of the chunk
    *reinterpret_cast<uint16_t*>(&sfs[0][(rr & 31) * 16 + ((rr >> 5) & 3) * 4 + 2 * bp]) =
        static_cast<uint16_t>(cr[0] | (cr[1] << 8));
  }
  if constexpr (TF) {
    // output row (column) 2cp + h, code bytes [32 rb, +32) = chunks 2rb, 2rb+1,
    // swizzled by (row >> 1) & 7 so that 8 neighbouring threads hit 8 chunks
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int orow = 2 * cp + h;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c = 2 * rb + q;
        tile[1024 + orow * 8 + (c ^ ((orow >> 1) & 7))] =
            make_uint4(pt[h][4 * q], pt[h][4 * q + 1], pt[h][4 * q + 2], pt[h][4 * q + 3]);
      }
      sfs[1][(orow & 31) * 16 + ((orow >> 5) & 3) * 4 + rb] = ct[h];
    }
  }
  __syncthreads();

  if constexpr (ROWF) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = tid + 256 * k, r = i >> 3, c = i & 7;
      *reinterpret_cast<uint4*>(q_r + (r0 + r) * cols + c0 + 16 * c) = tile[r * 8 + (c ^ (r & 7))];
    }
    if (tid < 32)
      reinterpret_cast<uint4*>(sf_r + (static_cast<int64_t>(blockIdx.y) * (rows / kQtTile) +
                                       blockIdx.x) * 512)[tid] =
          reinterpret_cast<const uint4*>(sfs[0])[tid];
  }
  if constexpr (TF) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = tid + 256 * k, r = i >> 3, c = i & 7;
      *reinterpret_cast<uint4*>(q_t + (c0 + r) * rows + r0 + 16 * c) =
          tile[1024 + r * 8 + (c ^ ((r >> 1) & 7))];
    }
    if (tid >= 32 && tid < 64)
      reinterpret_cast<uint4*>(sf_t + (static_cast<int64_t>(blockIdx.x) * (cols / kQtTile) +
                                       blockIdx.y) * 512)[tid - 32] =
          reinterpret_cast<const uint4*>(sfs[1])[tid - 32];
  }
}

}  // namespace

cudaError_t launch_mxfp8_quantize_mma_forms(const void* src, int64_t rows, int64_t cols,
                                            uint8_t* q_r, uint8_t* sf_r, uint8_t* q_t,
                                            uint8_t* sf_t, cudaStream_t s) {
  if (rows == 0 || cols == 0 || (!q_r && !q_t)) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(rows / kQtTile), static_cast<unsigned>(cols / kQtTile));
  const uint4* in = static_cast<const uint4*>(src);
  if (q_r && q_t) {
    quant_mma_tile_kernel<true, true><<<grid, 256, 0, s>>>(in, rows, cols, q_r, sf_r, q_t, sf_t);
  } else if (q_r) {
    const int64_t n = rows * (cols / 32);
    quant_mma_rows_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
        in, rows, cols, reinterpret_cast<uint4*>(q_r), sf_r);
  } else {
    quant_mma_tile_kernel<false, true><<<grid, 256, 0, s>>>(in, rows, cols, q_r, sf_r, q_t, sf_t);
  }
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_quantize_mma(const void* src, int64_t rows, int64_t cols, int transpose,
                                      uint8_t* q, uint8_t* sf, cudaStream_t s) {
  return transpose ? launch_mxfp8_quantize_mma_forms(src, rows, cols, nullptr, nullptr, q, sf, s)
                   : launch_mxfp8_quantize_mma_forms(src, rows, cols, q, sf, nullptr, nullptr, s);
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
