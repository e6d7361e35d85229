// square_s8.cu -- the square kernel in exact-integer mode (int8 operands held
// as binary16, fp32 chunk accumulators of at most 1024 products, int32 sums in
// the epilogue's registers), and the int8 -> binary16 widening kernel it runs
// after.
#include <cstring>

#include "convert.cuh"
#include "square_variants.cuh"

namespace sptg {

// Tile widths 128-256 in steps of 32, one CTA or a CTA pair, each at the
// deepest ring that fits: tensor memory holds the two accumulators of a float
// tile, and the epilogue keeps the int32 sums in registers.
bool square_variant_s8(int bn, int stages, bool pair, KernelVariant* v) {
#define SPTG_S8(BNV)                                                                           \
  if (bn == BNV) {                                                                             \
    if (!pair && (stages == 0 || stages == square_max_stages<BNV, false, 4, true>())) {         \
      *v = make_square<BNV, square_max_stages<BNV, false, 4, true>(), false, OUT_S32, true, false>(); \
      return true;                                                                             \
    }                                                                                          \
    if (pair && (stages == 0 || stages == square_max_stages<BNV, true, 4, true>())) {           \
      *v = make_square<BNV, square_max_stages<BNV, true, 4, true>(), false, OUT_S32, true, true>();   \
      return true;                                                                             \
    }                                                                                          \
    return false;                                                                              \
  }
  SPTG_S8(128)
  SPTG_S8(160)
  SPTG_S8(192)
  SPTG_S8(224)
  SPTG_S8(256)
#undef SPTG_S8
  return false;
}

cudaError_t launch_s8_to_f16(const void* srcA, int64_t lda, int64_t rows_a, const void* srcB,
                             int64_t ldb, int64_t rows_b, int64_t K, void* dstA, void* dstB,
                             int blocks, cudaStream_t stream, bool overlap_previous) {
  WidenParams p;
  p.srcA = static_cast<const int2*>(srcA);
  p.srcB = static_cast<const int2*>(srcB);
  p.dstA = static_cast<uint4*>(dstA);
  p.dstB = static_cast<uint4*>(dstB);
  p.lda8 = lda / 8;
  p.ldb8 = ldb / 8;
  p.k8 = K / 8;
  p.na8 = rows_a * p.k8;
  p.nb8 = rows_b * p.k8;
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(blocks, 1, 1);
  lc.blockDim = dim3(256, 1, 1);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = overlap_previous ? attr : nullptr;
  lc.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&lc, s8_to_f16_kernel, p);
}

}  // namespace sptg
