// convert.cuh -- int8 -> binary16 operand conversion for the exact integer
// path. Every int8 value is a binary16 value exactly, so this is a widening
// copy with no rounding. Memory-bound: one launch widens both operands, each
// thread keeping eight 8-byte loads in flight.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace sptg {

// 8 int8 values -> 8 binary16 values (4 words, lower address first).
// Flipping the sign bit of a byte b gives the unsigned byte b + 128; placed
// under the exponent byte 0x64 it is the binary16 number 1024 + (b + 128)
// (ulp 1 in [1024, 2048)), and one subtraction of 1152 leaves b. Both steps
// are exact.
__device__ __forceinline__ uint4 widen8(const int2 v) {
  const uint32_t w[2] = {static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y)};
  const __half2 bias = __halves2half2(__float2half_rn(1152.0f), __float2half_rn(1152.0f));
  uint32_t h[4];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t u = w[j] ^ 0x80808080u;
    const uint32_t p0 = __byte_perm(u, 0x64646464u, 0x4140);  // bytes 0, 1 under 0x64
    const uint32_t p1 = __byte_perm(u, 0x64646464u, 0x4342);  // bytes 2, 3 under 0x64
    const __half2 r0 = __hsub2(*reinterpret_cast<const __half2*>(&p0), bias);
    const __half2 r1 = __hsub2(*reinterpret_cast<const __half2*>(&p1), bias);
    h[2 * j] = *reinterpret_cast<const uint32_t*>(&r0);
    h[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&r1);
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

// Groups of 8 values: the rows x (K / 8) groups of A, then those of B, each
// written densely (row pitch K) whatever the source's row pitch (lda, ldb
// bytes, multiples of 16). A lane reads 8 bytes and writes 16, so the
// consecutive lanes of a warp read 256 and write 512 contiguous bytes per
// instruction (measured: 64 MB of binary16 written as two 16-byte halves 32
// bytes apart per lane took ~40 % longer than fully coalesced stores). A
// block lets the dependent GEMM launch once its own share is done (earlier,
// the GEMM's CTAs could take the SM slots that this grid's last blocks still
// need); the GEMM waits for this grid's completion before it reads the
// widened operands.
struct WidenParams {
  const int2* srcA;
  const int2* srcB;
  uint4* dstA;
  uint4* dstB;
  int64_t lda8, ldb8;  // source row pitches in 8-byte groups
  int64_t na8, nb8;    // groups of A and of B
  int64_t k8;          // groups per row (K / 8)
};

__global__ void __launch_bounds__(256) s8_to_f16_kernel(const WidenParams p) {
  grid_dependency_wait();  // the previous GEMM may still read the scratch
  constexpr int U = 8;
  const int64_t n = p.na8 + p.nb8;
  const bool dense = p.lda8 == p.k8 && p.ldb8 == p.k8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += U * stride) {
    int2 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = i + u * stride;
      if (k < n) {
        const bool is_a = k < p.na8;
        const int64_t g = is_a ? k : k - p.na8;
        int64_t off = g;
        if (!dense) {
          const int64_t row = g / p.k8;
          off = row * (is_a ? p.lda8 : p.ldb8) + (g - row * p.k8);
        }
        v[u] = __ldcs((is_a ? p.srcA : p.srcB) + off);  // streamed once
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = i + u * stride;
      if (k < n) {
        if (k < p.na8)
          p.dstA[k] = widen8(v[u]);
        else
          p.dstB[k - p.na8] = widen8(v[u]);
      }
    }
  }
  grid_launch_dependents();
}

}  // namespace sptg
