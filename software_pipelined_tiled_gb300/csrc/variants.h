// variants.h -- host-side catalogue of the compiled kernel variants.
//
// Each kernel template instantiation lives in one of the square_*.cu /
// skinny.cu translation units (compiled in parallel); the host API finds
// them through these lookups and launches them with cudaLaunchKernelExC.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sptg {

struct KernelVariant {
  const void* fn;  // the __global__ function
  int bn;          // square: tile columns; skinny: MMA N (rows of A covered)
  int stages;      // shared-memory ring depth
  int smem;        // dynamic shared memory per CTA, bytes
  bool pair;       // square: 2-SM CTA-pair variant (cluster of 2)
  int threads = 192;  // CTA size
  int ksub = 1;       // 64-wide K-chunks per ring stage (skinny kernels, square kernel)
};

// Square kernel for binary16 inputs (out_kind OUT_F16 or OUT_F32); kch =
// 64-wide K-chunks per ring stage (1, or 2 for the deepest rings of tiles up
// to 256 wide).
bool square_variant_f16_f16(int bn, int stages, bool pair, KernelVariant* v, int kch = 1);
bool square_variant_f16_f32(int bn, int stages, bool pair, KernelVariant* v, int kch = 1);
// Square kernel for bfloat16 inputs (out_kind OUT_BF16 or OUT_F32).
bool square_variant_bf16_bf16(int bn, int stages, bool pair, KernelVariant* v, int kch = 1);
bool square_variant_bf16_f32(int bn, int stages, bool pair, KernelVariant* v, int kch = 1);
// Square kernel in exact-integer mode (int8 operands widened to binary16).
bool square_variant_s8(int bn, int stages, bool pair, KernelVariant* v);
// Skinny kernel (in_bf16 selects bfloat16 inputs, else binary16).
bool skinny_variant(bool in_bf16, int out_kind, int stages, KernelVariant* v);
// Skinny kernel with K split inside a cluster (launched in clusters of 2-8).
// M picks the MMA N: 64 for M <= 64, 128 for M <= 128.
bool skinny_cluster_variant(bool in_bf16, int out_kind, int stages, int M, KernelVariant* v);
// Skinny kernel with one CTA per strip of n_tile output columns (M <= 64,
// 64-row MMA): bn = 64, ksub = K-chunks per stage; stages and smem are
// chosen per call (0 here).
bool skinny_rows_variant(bool in_bf16, int out_kind, int n_tile, KernelVariant* v);
// Skinny kernel on CTA pairs with the 2-SM MMA (M <= 256, n_cta <= 128
// output columns per CTA): bn = MMA N (64, 128 or 256 rows of A), ksub =
// K-chunks per stage; the ring depth and stage size are set per call (0 here).
bool skinny_pair_variant(bool in_bf16, int out_kind, int M, int n_cta, KernelVariant* v);
// The streaming ring out = alpha * in (bn = tile bytes).
KernelVariant stream_variant();
// int8 -> binary16 widening of both operands in one launch: rows_a rows of
// A and rows_b rows of B, K values each (a multiple of 16), read with row
// pitches lda and ldb (multiples of 16) and written densely to dstA, dstB.
cudaError_t launch_s8_to_f16(const void* srcA, int64_t lda, int64_t rows_a, const void* srcB,
                             int64_t ldb, int64_t rows_b, int64_t K, void* dstA, void* dstB,
                             int blocks, cudaStream_t stream, bool overlap_previous);

}  // namespace sptg
