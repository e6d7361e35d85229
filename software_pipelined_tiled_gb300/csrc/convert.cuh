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

// Groups of 16 values: the rows x (K / 16) groups of A, then those of B,
// each written densely (row pitch K) whatever the source's row pitch (lda,
// ldb bytes, multiples of 16). A block lets the dependent GEMM launch once
// its own share is done (earlier, the GEMM's CTAs could take the SM slots
// that this grid's last blocks still need); the GEMM waits for this grid's
// completion before it reads the widened operands.
struct WidenParams {
  const int4* srcA;
  const int4* srcB;
  uint4* dstA;
  uint4* dstB;
  int64_t lda16, ldb16;  // source row pitches in 16-byte groups
  int64_t na16, nb16;    // groups of A and of B
  int64_t k16;           // groups per row (K / 16)
};

__global__ void __launch_bounds__(256) s8_to_f16_kernel(const WidenParams p) {
  grid_dependency_wait();  // the previous GEMM may still read the scratch
  constexpr int U = 8;
  const int64_t n = p.na16 + p.nb16;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += U * stride) {
    int4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = i + u * stride;
      if (k < n) {
        const bool is_a = k < p.na16;
        const int64_t g = is_a ? k : k - p.na16;
        const int64_t row = g / p.k16, col = g - row * p.k16;
        const int4* src = is_a ? p.srcA + row * p.lda16 + col : p.srcB + row * p.ldb16 + col;
        v[u] = __ldcs(src);  // streamed once
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = i + u * stride;
      if (k < n) {
        uint32_t h[8];
        widen16(v[u], h);
        uint4* d = k < p.na16 ? p.dstA + 2 * k : p.dstB + 2 * (k - p.na16);
        d[0] = make_uint4(h[0], h[1], h[2], h[3]);
        d[1] = make_uint4(h[4], h[5], h[6], h[7]);
      }
    }
  }
  grid_launch_dependents();
}

}  // namespace sptg
