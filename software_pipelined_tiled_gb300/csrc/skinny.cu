// skinny.cu -- instantiations of the skinny kernels (swap-AB stream-K,
// swap-AB cluster split, swap-AB CTA pairs, and one CTA per strip of output
// columns).
#include "skinny_cluster_gemm.cuh"
#include "skinny_gemm.cuh"
#include "skinny_pair_gemm.cuh"
#include "skinny_rows_gemm.cuh"
#include "variants.h"

namespace sptg {

template <int MN, int ST, bool BF, int OUT, int KSUB>
KernelVariant make_skinny() {
  KernelVariant v{reinterpret_cast<const void*>(&skinny_gemm_kernel<MN, ST, BF, OUT, KSUB>), MN,
                  ST, SkinnyLayout<MN, ST, KSUB>::SMEM_BYTES, false};
  v.ksub = KSUB;
  return v;
}

// MMA N = 64 (up to 64 rows of A), two 64-wide K-chunks per stage (each B
// row read 256 contiguous bytes at a time) at a 4-stage ring for every float
// dtype pair; bfloat16 -> bfloat16 also at rings 1, 2 and 3 for the ablation.
bool skinny_variant(bool in_bf16, int out_kind, int stages, KernelVariant* v) {
  const int s = stages ? stages : 4;
  if (s == 4) {
    if (out_kind == OUT_BF16 && in_bf16) *v = make_skinny<64, 4, true, OUT_BF16, 2>();
    else if (out_kind == OUT_F16 && !in_bf16) *v = make_skinny<64, 4, false, OUT_F16, 2>();
    else if (out_kind == OUT_F32 && in_bf16) *v = make_skinny<64, 4, true, OUT_F32, 2>();
    else if (out_kind == OUT_F32 && !in_bf16) *v = make_skinny<64, 4, false, OUT_F32, 2>();
    else return false;
    return true;
  }
  if (!(in_bf16 && out_kind == OUT_BF16)) return false;
  switch (s) {
    case 1: *v = make_skinny<64, 1, true, OUT_BF16, 2>(); return true;
    case 2: *v = make_skinny<64, 2, true, OUT_BF16, 2>(); return true;
    case 3: *v = make_skinny<64, 3, true, OUT_BF16, 2>(); return true;
    default: return false;
  }
}

template <int MN, int ST, bool BF, int OUT, int KSUB>
KernelVariant make_skinny_cluster_at() {
  constexpr int OB = OutTraits<OUT>::bytes;
  KernelVariant v{reinterpret_cast<const void*>(&skinny_cluster_gemm_kernel<MN, ST, BF, OUT, KSUB>),
                  MN, ST, SkinnyClusterLayout<MN, ST, OB, KSUB>::SMEM_BYTES, false};
  v.ksub = KSUB;
  return v;
}

template <int MN, bool BF, int OUT, int KSUB>
KernelVariant make_skinny_cluster() {
  return make_skinny_cluster_at<MN, skinny_cluster_stages<MN, OutTraits<OUT>::bytes, KSUB>(), BF,
                                OUT, KSUB>();
}

// MMA N = 64 (M <= 64) at the deepest ring next to the receive buffer, for
// every float dtype pair. Two 64-wide K-chunks per stage (4 stages of 48 KB):
// each stage then reads 256 contiguous bytes of every B row instead of 128,
// which measured 5.6 TB/s against 5.2 TB/s for 8 stages of one chunk on
// 64 x 8192 x 8192 (4 chunks leave room for only 2 stages: 5.2 TB/s).
// MMA N = 128 (64 < M <= 128): two chunks per stage at 3 stages of 64 KB for
// 16-bit outputs; one chunk at 5 stages of 32 KB for fp32 outputs, whose
// 64 KB output staging leaves no room for a third 64 KB stage.
constexpr int kSkinnyClusterKsub = 2;
bool skinny_cluster_variant(bool in_bf16, int out_kind, int stages, int M, KernelVariant* v) {
  constexpr int K = kSkinnyClusterKsub;
  KernelVariant c;
  if (M > 64) {
    if (M > 128 || stages != 0) return false;
    if (out_kind == OUT_BF16 && in_bf16) c = make_skinny_cluster<128, true, OUT_BF16, K>();
    else if (out_kind == OUT_F16 && !in_bf16) c = make_skinny_cluster<128, false, OUT_F16, K>();
    else if (out_kind == OUT_F32 && in_bf16) c = make_skinny_cluster<128, true, OUT_F32, 1>();
    else if (out_kind == OUT_F32 && !in_bf16) c = make_skinny_cluster<128, false, OUT_F32, 1>();
    else return false;
    *v = c;
    return true;
  }
  if (out_kind == OUT_BF16 && in_bf16) c = make_skinny_cluster<64, true, OUT_BF16, K>();
  else if (out_kind == OUT_F16 && !in_bf16) c = make_skinny_cluster<64, false, OUT_F16, K>();
  else if (out_kind == OUT_F32 && in_bf16) c = make_skinny_cluster<64, true, OUT_F32, K>();
  else if (out_kind == OUT_F32 && !in_bf16) c = make_skinny_cluster<64, false, OUT_F32, K>();
  else return false;
  if (stages != 0 && stages != c.stages) {
    // shallower rings of the bfloat16 -> bfloat16 variant, for the
    // pipelining ablation of the memory-bound shape
    if (!(out_kind == OUT_BF16 && in_bf16)) return false;
    switch (stages) {
      case 1: c = make_skinny_cluster_at<64, 1, true, OUT_BF16, K>(); break;
      case 2: c = make_skinny_cluster_at<64, 2, true, OUT_BF16, K>(); break;
      case 3: c = make_skinny_cluster_at<64, 3, true, OUT_BF16, K>(); break;
      default: return false;
    }
  }
  *v = c;
  return true;
}

// One CTA per strip of output columns (M <= 64), the ring depth and strip
// width set per call: two 64-wide K-chunks per stage up to 160 columns (a ring
// of 4 or more stages), one chunk past that, where two leave room for only
// 2-3 stages (64 x 24576 x 4096, 168 columns: 31.8 us at 7 stages of one
// chunk against 32.3 us at 3 of two; 64 x 38912 x 2048, 256 columns: 25.6
// against 27.7 us; 64 x 19456 x 4096, 128 columns: 25.1 us with two chunks
// against 25.7 us with one).
template <bool BF, int OUT, int KS>
KernelVariant make_skinny_rows() {
  KernelVariant v{reinterpret_cast<const void*>(&skinny_rows_gemm_kernel<BF, OUT, KS>), 64, 0, 0,
                  false};
  v.ksub = KS;
  return v;
}

template <int KS>
bool skinny_rows_variant_k(bool in_bf16, int out_kind, KernelVariant* v) {
  if (out_kind == OUT_BF16 && in_bf16) *v = make_skinny_rows<true, OUT_BF16, KS>();
  else if (out_kind == OUT_F16 && !in_bf16) *v = make_skinny_rows<false, OUT_F16, KS>();
  else if (out_kind == OUT_F32 && in_bf16) *v = make_skinny_rows<true, OUT_F32, KS>();
  else if (out_kind == OUT_F32 && !in_bf16) *v = make_skinny_rows<false, OUT_F32, KS>();
  else return false;
  return true;
}

bool skinny_rows_variant(bool in_bf16, int out_kind, int n_tile, KernelVariant* v) {
  return n_tile > 160 ? skinny_rows_variant_k<1>(in_bf16, out_kind, v)
                      : skinny_rows_variant_k<2>(in_bf16, out_kind, v);
}

// CTA pairs with the 2-SM MMA over the whole of K. Up to 64 rows (MN = 64):
// four 64-wide K-chunks per stage, so each stage reads 512 contiguous bytes of
// every Bcm row (64 x 8192 x 8192: 22.6 us against 23.3 us with two chunks at
// twice the ring depth, 36.9 us with one). 65-128 rows (MN = 128), whose rows
// of A take twice the room: two chunks per stage (128 x 8192 x 8192: 25.2 us
// against 26.4 us with four chunks at 3 stages), four up to 40 columns per CTA
// (128 x 4096 x 8192: 17.5 against 22.3 us). Past 64 columns per CTA (two
// 64-row blocks of Bcm rows, two MMAs per K-step) two chunks per stage for
// either MN. 129-256 rows (MN = 256): two chunks per stage. The ring depth
// and each CTA's column count are set per call.
template <int MN, bool BF, int OUT, int KS>
KernelVariant make_skinny_pair() {
  KernelVariant v{reinterpret_cast<const void*>(&skinny_pair_gemm_kernel<MN, BF, OUT, KS>), MN, 0,
                  0, true};
  v.ksub = KS;
  return v;
}

template <int MN, int KS>
bool skinny_pair_variant_mn(bool in_bf16, int out_kind, KernelVariant* v) {
  if (out_kind == OUT_BF16 && in_bf16) *v = make_skinny_pair<MN, true, OUT_BF16, KS>();
  else if (out_kind == OUT_F16 && !in_bf16) *v = make_skinny_pair<MN, false, OUT_F16, KS>();
  else if (out_kind == OUT_F32 && in_bf16) *v = make_skinny_pair<MN, true, OUT_F32, KS>();
  else if (out_kind == OUT_F32 && !in_bf16) *v = make_skinny_pair<MN, false, OUT_F32, KS>();
  else return false;
  return true;
}

bool skinny_pair_variant(bool in_bf16, int out_kind, int M, int n_cta, KernelVariant* v) {
  if (M <= 64) {
    // past 64 columns four chunks would leave room for only 2-3 stages
    if (n_cta <= 64) return skinny_pair_variant_mn<64, 4>(in_bf16, out_kind, v);
    return skinny_pair_variant_mn<64, 2>(in_bf16, out_kind, v);
  }
  if (M <= 128) {
    if (n_cta <= 40) return skinny_pair_variant_mn<128, 4>(in_bf16, out_kind, v);
    return skinny_pair_variant_mn<128, 2>(in_bf16, out_kind, v);
  }
  if (M <= 256) return skinny_pair_variant_mn<256, 2>(in_bf16, out_kind, v);
  return false;
}

}  // namespace sptg
