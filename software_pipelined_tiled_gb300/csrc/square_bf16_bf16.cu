// square_bf16_bf16.cu -- square-kernel instantiations for the bf16_bf16 dtype pair.
#include "square_variants.cuh"

namespace sptg {

bool square_variant_bf16_bf16(int bn, int stages, bool pair, KernelVariant* v, int kch) {
  return square_float_variant<true, OUT_BF16>(bn, stages, pair, v, kch);
}

}  // namespace sptg
