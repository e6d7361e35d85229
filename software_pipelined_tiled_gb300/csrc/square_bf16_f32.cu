// square_bf16_f32.cu -- square-kernel instantiations for the bf16_f32 dtype pair.
#include "square_variants.cuh"

namespace sptg {

// Besides the deepest rings, the shallower rings 1-5 of the 256-wide pair
// tile, for the pipelining ablation on the long K-loop (K = 16384).
bool square_variant_bf16_f32(int bn, int stages, bool pair, KernelVariant* v, int kch) {
  if (square_float_variant<true, OUT_F32>(bn, stages, pair, v, kch)) return true;
  if (kch != 1 || !pair || bn != 256) return false;
  switch (stages) {
    case 1: *v = make_square<256, 1, true, OUT_F32, false, true>(); return true;
    case 2: *v = make_square<256, 2, true, OUT_F32, false, true>(); return true;
    case 3: *v = make_square<256, 3, true, OUT_F32, false, true>(); return true;
    case 4: *v = make_square<256, 4, true, OUT_F32, false, true>(); return true;
    case 5: *v = make_square<256, 5, true, OUT_F32, false, true>(); return true;
    default: return false;
  }
}

}  // namespace sptg
