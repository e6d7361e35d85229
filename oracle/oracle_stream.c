/*
 * oracle_stream.c -- plain CPU reference for the streaming pipeline:
 * out[i] = alpha * in[i] in binary32.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle_gemm.c): shares nothing with the CUDA
 * library; only tests, the smoke check and the bench's CPU legs use it.
 *
 * What it computes: the minimal working example of "Hiding Memory Latency in
 * CUDA: Asynchronous Loads and Software Pipelines" (section 8) streams a
 * vector through a multi-stage shared-memory ring and writes twice each
 * element; the pipeline changes only when data moves, so the result is the
 * element-wise product itself. Written here for any scale factor: one
 * binary32 multiplication per element (a single rounding, no contraction).
 */
#include <stdint.h>

void oracle_scale_f32(int64_t n, float alpha, const float* in, float* out) {
    for (int64_t i = 0; i < n; ++i) {
        volatile float p = alpha * in[i]; /* one IEEE binary32 multiply */
        out[i] = p;
    }
}
