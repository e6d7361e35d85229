// square_f16_f16.cu -- square-kernel instantiations for the f16_f16 dtype pair.
#include "square_variants.cuh"

namespace sptg {

bool square_variant_f16_f16(int bn, int stages, bool pair, KernelVariant* v, int kch) {
  return square_float_variant<false, OUT_F16>(bn, stages, pair, v, kch);
}

}  // namespace sptg
