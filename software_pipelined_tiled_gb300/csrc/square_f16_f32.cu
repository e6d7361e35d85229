// square_f16_f32.cu -- square-kernel instantiations for the f16_f32 dtype pair.
#include "square_variants.cuh"

namespace sptg {

bool square_variant_f16_f32(int bn, int stages, bool pair, KernelVariant* v, int kch) {
  return square_float_variant<false, OUT_F32>(bn, stages, pair, v, kch);
}

}  // namespace sptg
