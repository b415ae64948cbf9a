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
