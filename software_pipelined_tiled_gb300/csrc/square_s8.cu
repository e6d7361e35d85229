// square_s8.cu -- the square kernel in exact-integer mode (int8 operands held
// as binary16, fp32 chunk accumulators of at most 1024 products, int32 sums),
// and the int8 -> binary16 widening kernel it runs after.
#include "convert.cuh"
#include "square_variants.cuh"

namespace sptg {

// Tile widths 128 and 160: two accumulators and the int32 running sum,
// 3 x BN tensor-memory columns, fit the 512 columns up to BN = 160.
bool square_variant_s8(int bn, int stages, bool pair, KernelVariant* v) {
#define SPTG_S8(BNV)                                                                      \
  if (bn == BNV) {                                                                        \
    if (!pair && (stages == 0 || stages == square_max_stages<BNV, false, 4>())) {          \
      *v = make_square<BNV, square_max_stages<BNV, false, 4>(), false, OUT_S32, true, false>(); \
      return true;                                                                        \
    }                                                                                     \
    if (pair && (stages == 0 || stages == square_max_stages<BNV, true, 4>())) {            \
      *v = make_square<BNV, square_max_stages<BNV, true, 4>(), false, OUT_S32, true, true>();   \
      return true;                                                                        \
    }                                                                                     \
    return false;                                                                         \
  }
  SPTG_S8(128)
  SPTG_S8(160)
#undef SPTG_S8
  return false;
}

cudaError_t launch_s8_to_f16(const void* src, void* dst, int64_t n16, int blocks,
                             cudaStream_t stream) {
  s8_to_f16_kernel<<<blocks, 256, 0, stream>>>(static_cast<const int4*>(src),
                                               static_cast<uint4*>(dst), n16);
  return cudaGetLastError();
}

}  // namespace sptg
