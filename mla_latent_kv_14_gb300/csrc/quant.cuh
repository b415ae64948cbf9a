// quant.cuh -- writer of the 656-byte FP8 cache rows
// ("FlashMLA 实战：MLA 注意力加速指南", §FP8 缓存怎么把 KV 压掉四成; "矩阵、注意力与
// GPU：拆解 DeepGEMM 与 FlashMLA", §八 '格式'): per 128 latent values one fp32
// scale = amax/448 (1.0 for an all-zero block), e4m3 code = round-to-nearest-
// even of x/scale saturated to +-448, both divisions IEEE round-to-nearest;
// then the 4 scales; then the 64 RoPE dims as bf16.
#pragma once
#include <cuda_bf16.h>

#include "params.h"
#include "ptx.cuh"

namespace mla {

// two fp32 -> two e4m3 bytes, `lo` in the low byte
__device__ __forceinline__ uint16_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One warp per row; lane l owns values [4l, 4l+4) of each 128-value block.
__global__ void __launch_bounds__(256) mla_quant_fp8_kernel(const uint16_t* __restrict__ kv,
                                                            uint8_t* __restrict__ out, int64_t n) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n; row += warps) {
    const uint16_t* src = kv + row * kDK;
    uint8_t* dst = out + row * kRowBytesFp8;
    float scales[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint2 raw = *reinterpret_cast<const uint2*>(src + j * 128 + lane * 4);
      float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                    __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
      float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float scale = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
      scales[j] = scale;
      const uint16_t c01 = e4m3x2_rn_sat(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
      const uint16_t c23 = e4m3x2_rn_sat(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
      *reinterpret_cast<uint32_t*>(dst + j * 128 + lane * 4) = (uint32_t)c01 | ((uint32_t)c23 << 16);
    }
    if (lane == 0)
      *reinterpret_cast<float4*>(dst + 512) = make_float4(scales[0], scales[1], scales[2], scales[3]);
    // RoPE: 64 bf16 = 128 bytes, 4 per lane
    *reinterpret_cast<uint32_t*>(dst + 528 + lane * 4) =
        *reinterpret_cast<const uint32_t*>(src + 512 + lane * 2);
  }
}

}  // namespace mla

// ---------------------------------------------------------------------------
// Writers of the V4.1 rows of 512 values ("矩阵、注意力与 GPU：拆解 DeepGEMM 与
// FlashMLA", §八 '版本漂移' and the §十 format table; §三 'UE8M0': a scale is a
// power of two, rounded up). Input: bf16 rows [n, 512].
// ---------------------------------------------------------------------------
namespace mla {

// sixteen bf16 values from 32 bytes at src
__device__ __forceinline__ void load_bf16x16(const uint16_t* src, float* x) {
  const uint4 a = *reinterpret_cast<const uint4*>(src);
  const uint4 b = *reinterpret_cast<const uint4*>(src + 8);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

// 528-byte rows: 512 e4m3 codes, then 16 UE8M0 scales (byte k + 127 for the
// scale 2^k of values [32j, 32j + 32)). k is the smallest integer >= -127 with
// 448 * 2^k >= amax, found from amax's fp32 fields: amax = f * 2^e, f in
// [1, 2), gives k = e - 8 when f <= 1.75 (448 = 1.75 * 2^8) and e - 7 above.
// One warp per row; lane l owns values [16l, 16l + 16) (two lanes per block).
__global__ void __launch_bounds__(256) mla_quant_fp8_528_kernel(const uint16_t* __restrict__ kv,
                                                                uint8_t* __restrict__ out, int64_t n) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n; row += warps) {
    float x[16];
    load_bf16x16(kv + row * kDV41 + 16 * lane, x);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const uint32_t bits = __float_as_uint(amax);
    const int e_field = (int)(bits >> 23);  // amax >= 0; 0 for zero and fp32 subnormals
    int k = -127;                           // zero and subnormal blocks: 448 * 2^-127 covers them
    if (e_field > 0) {
      k = (e_field - 127) - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
      k = k < -127 ? -127 : k;
    }
    // 2^-k: -k in [-120, 127], a normal fp32 value; x * 2^-k is exact
    const float inv = __uint_as_float((uint32_t)(127 - k) << 23);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint16_t c01 = e4m3x2_rn_sat(x[4 * q] * inv, x[4 * q + 1] * inv);
      const uint16_t c23 = e4m3x2_rn_sat(x[4 * q + 2] * inv, x[4 * q + 3] * inv);
      w[q] = (uint32_t)c01 | ((uint32_t)c23 << 16);
    }
    uint8_t* dst = out + row * kRowBytesFp8_528;
    *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
    // the 16 scale bytes, gathered into lanes 0..3 (one word each)
    const uint32_t ue = (uint32_t)(k + 127);
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) word |= __shfl_sync(0xffffffffu, ue, (8 * lane + 2 * b) & 31) << (8 * b);
    if (lane < 4) *reinterpret_cast<uint32_t*>(dst + 512 + 4 * lane) = word;
  }
}

// value of a non-negative e4m3 code (0x00 .. 0x7E) as fp32, from its fields
__device__ __forceinline__ float e4m3_pos_value(uint32_t c) {
  const uint32_t e = c >> 3, m = c & 7u;
  return e == 0 ? (float)m * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// 288-byte rows: 512 e2m1 codes (value 2i in the low nibble of byte i), then 32
// e4m3 scales (values [16j, 16j + 16)). The scale v is the smallest
// non-negative e4m3 value with 6 v >= amax (448 when none is large enough);
// the code is the nearest e2m1 magnitude of |x| / v, ties to the even code,
// with the sign of x. The decision is taken against the midpoints of the e2m1
// magnitudes times v (at most 7 significant bits: exact in fp32), so no
// division rounds. One warp per row; lane l owns block l.
__global__ void __launch_bounds__(256) mla_quant_fp4_288_kernel(const uint16_t* __restrict__ kv,
                                                                uint8_t* __restrict__ out, int64_t n) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  // midpoints between consecutive e2m1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6
  const float mids[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < n; row += warps) {
    float x[16];
    load_bf16x16(kv + row * kDV41 + 16 * lane, x);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
    // a first guess from the rounded quotient, then corrected by exact tests
    // (6 v is exact: at most 6 significant bits)
    uint32_t c = e4m3x2_rn_sat(amax / 6.0f, 0.f) & 0x7Fu;
    if (c > 0x7Eu) c = 0x7Eu;
    for (int it = 0; it < 4 && c < 0x7Eu && 6.0f * e4m3_pos_value(c) < amax; ++it) ++c;
    for (int it = 0; it < 4 && c > 0u && 6.0f * e4m3_pos_value(c - 1u) >= amax; ++it) --c;
    const float v = e4m3_pos_value(c);
    float t[7];
#pragma unroll
    for (int j = 0; j < 7; ++j) t[j] = mids[j] * v;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float a = fabsf(x[k]);
      uint32_t mag = 0;
#pragma unroll
      for (int j = 0; j < 7; ++j) mag += (a > t[j] || (a == t[j] && (j & 1))) ? 1u : 0u;
      if (v == 0.f) mag = 0;
      const uint32_t code = mag | ((__float_as_uint(x[k]) >> 31) << 3);
      if (k < 8) lo |= code << (4 * k);
      else hi |= code << (4 * (k - 8));
    }
    uint8_t* dst = out + row * kRowBytesFp4_288;
    *reinterpret_cast<uint2*>(dst + 8 * lane) = make_uint2(lo, hi);
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) word |= __shfl_sync(0xffffffffu, c, (4 * lane + b) & 31) << (8 * b);
    if (lane < 8) *reinterpret_cast<uint32_t*>(dst + 256 + 4 * lane) = word;
  }
}

}  // namespace mla
