// convert.cuh -- int8 -> binary16 operand conversion for the exact integer
// path. Every int8 value is a binary16 value exactly, so this is a widening
// copy with no rounding. Memory-bound: 16 bytes in, 32 bytes out per thread
// step, grid-stride over the array.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace sptg {

__global__ void __launch_bounds__(256) s8_to_f16_kernel(const int4* __restrict__ src,
                                                        uint4* __restrict__ dst, int64_t n16) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int4 v = __ldcs(src + i);  // streamed once
    const uint32_t w[4] = {static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y),
                           static_cast<uint32_t>(v.z), static_cast<uint32_t>(v.w)};
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int8_t b0 = static_cast<int8_t>(w[j] & 0xff);
      const int8_t b1 = static_cast<int8_t>((w[j] >> 8) & 0xff);
      const int8_t b2 = static_cast<int8_t>((w[j] >> 16) & 0xff);
      const int8_t b3 = static_cast<int8_t>((w[j] >> 24) & 0xff);
      __half2 lo = __halves2half2(__short2half_rn(b0), __short2half_rn(b1));
      __half2 hi = __halves2half2(__short2half_rn(b2), __short2half_rn(b3));
      h[2 * j] = *reinterpret_cast<uint32_t*>(&lo);
      h[2 * j + 1] = *reinterpret_cast<uint32_t*>(&hi);
    }
    dst[2 * i] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[2 * i + 1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

}  // namespace sptg
