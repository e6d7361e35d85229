// square_variants.cuh -- the instantiation table of the square kernel,
// included by one translation unit per dtype pair.
#pragma once

#include "square_gemm.cuh"
#include "variants.h"

namespace sptg {

template <int BN, int ST, bool BF, int OUT, bool IE, bool PAIR, int KCH = 1>
KernelVariant make_square() {
  KernelVariant v{
      reinterpret_cast<const void*>(&square_gemm_kernel<BN, ST, BF, OUT, IE, PAIR, KCH>), BN, ST,
      SquareLayout<BN, ST, IE, PAIR, OutTraits<OUT>::bytes, KCH>::SMEM_BYTES, PAIR,
      IE ? SQUARE_THREADS_INT : SQUARE_THREADS};
  v.ksub = KCH;
  return v;
}

// Tile widths BN from 112 to 256 in steps of 16, one CTA or a CTA pair per
// tile, each at the deepest ring that fits (square_max_stages). For
// binary16 -> binary16 also the shallower rings of BN 256 and 224 (one CTA)
// and of BN 224 (pair) for the pipelining ablation (1 = load, then compute,
// no overlap).
template <bool BF, int OUT>
bool square_float_variant(int bn, int stages, bool pair, KernelVariant* v, int kch = 1) {
  constexpr int OB = OutTraits<OUT>::bytes;
  if (kch == 2) {
    // two 64-wide K-chunks per ring stage, at the deepest ring that fits
    if (stages != 0) return false;
#define SPTG_SQ2(BNV)                                                                           \
  case BNV:                                                                                     \
    if (pair)                                                                                   \
      *v = make_square<BNV, square_max_stages<BNV, true, OB, false, 2>(), BF, OUT, false, true, 2>(); \
    else                                                                                        \
      *v = make_square<BNV, square_max_stages<BNV, false, OB, false, 2>(), BF, OUT, false, false, 2>(); \
    return true;
    switch (bn) {
      SPTG_SQ2(256)
      SPTG_SQ2(240)
      SPTG_SQ2(224)
      SPTG_SQ2(208)
      SPTG_SQ2(192)
      SPTG_SQ2(176)
      SPTG_SQ2(160)
      SPTG_SQ2(144)
      SPTG_SQ2(128)
      SPTG_SQ2(112)
      default:
        return false;
    }
#undef SPTG_SQ2
  }
  if (kch != 1) return false;
  if (bn == 512) {
    // 256 x 512 CTA-pair tiles: two 256-column MMAs per K-step, one accumulator
    if (!pair || (stages != 0 && stages != square_max_stages<512, true, OB>())) return false;
    *v = make_square<512, square_max_stages<512, true, OB>(), BF, OUT, false, true>();
    return true;
  }
#define SPTG_SQ(BNV)                                                                     \
  case BNV:                                                                              \
    if (!pair && (stages == 0 || stages == square_max_stages<BNV, false, OB>())) {       \
      *v = make_square<BNV, square_max_stages<BNV, false, OB>(), BF, OUT, false, false>(); \
      return true;                                                                       \
    }                                                                                    \
    if (pair && (stages == 0 || stages == square_max_stages<BNV, true, OB>())) {         \
      *v = make_square<BNV, square_max_stages<BNV, true, OB>(), BF, OUT, false, true>();   \
      return true;                                                                       \
    }                                                                                    \
    break;
  switch (bn) {
    SPTG_SQ(256)
    SPTG_SQ(240)
    SPTG_SQ(224)
    SPTG_SQ(208)
    SPTG_SQ(192)
    SPTG_SQ(176)
    SPTG_SQ(160)
    SPTG_SQ(144)
    SPTG_SQ(128)
    SPTG_SQ(112)
    default:
      return false;
  }
#undef SPTG_SQ
  if constexpr (!BF && OUT == OUT_F16) {
    if (!pair && (bn == 256 || bn == 224) && stages >= 1 && stages <= 3) {
      if (bn == 256)
        *v = stages == 1 ? make_square<256, 1, false, OUT_F16, false, false>()
                         : stages == 2 ? make_square<256, 2, false, OUT_F16, false, false>()
                                       : make_square<256, 3, false, OUT_F16, false, false>();
      else
        *v = stages == 1 ? make_square<224, 1, false, OUT_F16, false, false>()
                         : stages == 2 ? make_square<224, 2, false, OUT_F16, false, false>()
                                       : make_square<224, 3, false, OUT_F16, false, false>();
      return true;
    }
    if (pair && bn == 224 && stages >= 1 && stages <= 6) {
      switch (stages) {
        case 1: *v = make_square<224, 1, false, OUT_F16, false, true>(); return true;
        case 2: *v = make_square<224, 2, false, OUT_F16, false, true>(); return true;
        case 3: *v = make_square<224, 3, false, OUT_F16, false, true>(); return true;
        case 4: *v = make_square<224, 4, false, OUT_F16, false, true>(); return true;
        case 5: *v = make_square<224, 5, false, OUT_F16, false, true>(); return true;
        default: *v = make_square<224, 6, false, OUT_F16, false, true>(); return true;
      }
    }
  }
  return false;
}

}  // namespace sptg
