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
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  // first source goes to the upper byte, second to the lower byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

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
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  // floor(log2(amax)) = biased exponent - 127 for normal amax; zero and
  // subnormal amax give code 0 after the clamp.
  const int biased = (__float_as_uint(amax) >> 23) & 0xFF;
  const int code = biased == 0 ? 0 : max(0, biased - 8);  // (biased-127) - 8 + 127
  scale[b] = static_cast<uint8_t>(code);
  const float inv = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);  // 2^(127-code)
  uint32_t packed[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = e4m3x2(f[4 * i + 0] * inv, f[4 * i + 1] * inv);
    const uint32_t hi = e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv);
    packed[i] = lo | (hi << 16);
  }
  q[b * 2 + 0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  q[b * 2 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
}

}  // namespace

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
