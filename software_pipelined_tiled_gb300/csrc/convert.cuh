// convert.cuh -- int8 -> binary16 operand conversion for the exact integer
// path. Every int8 value is a binary16 value exactly, so this is a widening
// copy with no rounding. Memory-bound: one launch widens both operands, each
// thread keeping eight 16-byte loads in flight.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace sptg {

// 16 int8 values -> 16 binary16 values (8 words, lower address first).
// Flipping the sign bit of a byte b gives the unsigned byte b + 128; placed
// under the exponent byte 0x64 it is the binary16 number 1024 + (b + 128)
// (ulp 1 in [1024, 2048)), and one subtraction of 1152 leaves b. Both steps
// are exact.
__device__ __forceinline__ void widen16(const int4 v, uint32_t h[8]) {
  const uint32_t w[4] = {static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y),
                         static_cast<uint32_t>(v.z), static_cast<uint32_t>(v.w)};
  const __half2 bias = __halves2half2(__float2half_rn(1152.0f), __float2half_rn(1152.0f));
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t u = w[j] ^ 0x80808080u;
    const uint32_t p0 = __byte_perm(u, 0x64646464u, 0x4140);  // bytes 0, 1 under 0x64
    const uint32_t p1 = __byte_perm(u, 0x64646464u, 0x4342);  // bytes 2, 3 under 0x64
    const __half2 r0 = __hsub2(*reinterpret_cast<const __half2*>(&p0), bias);
    const __half2 r1 = __hsub2(*reinterpret_cast<const __half2*>(&p1), bias);
    h[2 * j] = *reinterpret_cast<const uint32_t*>(&r0);
    h[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&r1);
  }
}

// Groups of 16 values: [0, na16) of A, then [0, nb16) of B. A block lets
// the dependent GEMM launch once its own share is done (earlier, the GEMM's
// CTAs could take the SM slots that this grid's last blocks still need); the
// GEMM waits for this grid's completion before it reads the widened
// operands.
__global__ void __launch_bounds__(256) s8_to_f16_kernel(const int4* __restrict__ srcA,
                                                        uint4* __restrict__ dstA, int64_t na16,
                                                        const int4* __restrict__ srcB,
                                                        uint4* __restrict__ dstB, int64_t nb16) {
  grid_dependency_wait();  // the previous GEMM may still read the scratch
  constexpr int U = 8;
  const int64_t n = na16 + nb16;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += U * stride) {
    int4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = i + u * stride;
      if (k < n) v[u] = __ldcs(k < na16 ? srcA + k : srcB + (k - na16));  // streamed once
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = i + u * stride;
      if (k < n) {
        uint32_t h[8];
        widen16(v[u], h);
        uint4* d = k < na16 ? dstA + 2 * k : dstB + 2 * (k - na16);
        d[0] = make_uint4(h[0], h[1], h[2], h[3]);
        d[1] = make_uint4(h[4], h[5], h[6], h[7]);
      }
    }
  }
  grid_launch_dependents();
}

}  // namespace sptg
