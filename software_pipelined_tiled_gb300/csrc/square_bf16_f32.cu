// square_bf16_f32.cu -- square-kernel instantiations for the bf16_f32 dtype pair.
#include "square_variants.cuh"

namespace sptg {

bool square_variant_bf16_f32(int bn, int stages, bool pair, KernelVariant* v) {
  return square_float_variant<true, OUT_F32>(bn, stages, pair, v);
}

}  // namespace sptg
