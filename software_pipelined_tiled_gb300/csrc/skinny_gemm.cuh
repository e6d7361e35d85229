// skinny_gemm.cuh -- the memory-bound variant for few output rows (M <= 64).
//
// With M small the product streams B (K x N) once from HBM and does little
// arithmetic per byte: the regime where "Pipeline GPU Kernel" (when-to-use
// list, Step 2) says load latency dominates and a deep asynchronous ring pays
// most.  The kernel computes C^T = B^T * A^T ("swap AB") so that N, the long
// side, is the 128-row side of the tensor-core instruction and the few rows of
// A become its N = MN (64) side:
//
//   D^T[n, m] = sum_k Bcm[n, k] * A[m, k]      (both operands K-major)
//
// Work is the list of (n-tile, k-tile) units in n-major order, cut into one
// contiguous range per CTA (a stream-K split), so every SM streams the same
// share of B however the shape divides.  A CTA accumulates each n-tile segment
// of its range in tensor memory.  A segment that covers all of K is written to
// C directly; otherwise its fp32 partial tile goes to scratch, and the CTA
// that arrives last at that n-tile (an atomic counter) adds the partials in
// contributor order (= increasing k), converts and writes C.  The sum order
// is fixed, so results do not depend on arrival order.
//
// Roles are those of the square kernel: warp 0 loads through an S-stage ring
// (full/empty mbarriers), warp 1 issues tcgen05.mma, warps 2-5 drain tensor
// memory; two accumulators let one segment's epilogue overlap the next
// segment's loads and MMAs.
#pragma once

#include "common.cuh"

namespace sptg {

struct SkinnyParams {
  int M, N, K;
  int num_n_tiles, num_k_tiles;
  int num_ctas;
  int64_t total_units;
  int max_contrib;            // partial slots per n-tile
  void* C;                    // row-major M x N output
  int64_t ldc;                // elements between rows of C
  float* partials;            // [n_tile][max_contrib][MN][128] fp32, or null if unsplit
  unsigned long long* counters;  // [n_tile] (generation << 32 | arrivals); 0 after the call
  unsigned int generation;    // this call's tag for the counters, never 0
  unsigned int* error_word;
  uint64_t timeout_ns;
  int inject_stall;
  unsigned long long* trace;  // optional timeline (see TraceEvent), or null
};

// A ring stage holds KSUB consecutive 64-wide K-chunks (each its own
// 128-byte-swizzled sub-tile) of B^T and of A: one unit of work is one stage.
template <int MN, int STAGES, int KSUB = 1>
struct SkinnyLayout {
  static constexpr int BNT = 128;  // output columns per tile (MMA M)
  static constexpr int BK = 64;
  static constexpr int SUB_BT = BNT * BK * 2;
  static constexpr int SUB_A = MN * BK * 2;
  static constexpr int BT_STAGE = KSUB * SUB_BT;
  static constexpr int A_STAGE = KSUB * SUB_A;
  static constexpr int STAGE = BT_STAGE + A_STAGE;
  static constexpr int OFF_BAR = STAGES * STAGE;
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TMEM_COLS = 2 * MN <= 32 ? 32 : 2 * MN <= 64 ? 64 : 2 * MN <= 128 ? 128 : 256;
  static_assert(MN % 32 == 0 && MN >= 32 && MN <= 128, "MN must be 32, 64, 96 or 128");
  static_assert(BT_STAGE % 1024 == 0 && A_STAGE % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
};

// CTA whose unit range [c*T/G, (c+1)*T/G) holds unit u.
__device__ __forceinline__ int cta_of_unit(int64_t u, int G, int64_t T) {
  return static_cast<int>(((u + 1) * G - 1) / T);
}

template <int MN, int STAGES, bool IN_BF16, int OUT, int KSUB = 1>
__global__ void __launch_bounds__(192, 1)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap tmBt,
                       const __grid_constant__ CUtensorMap tmA, const SkinnyParams p) {
  using L = SkinnyLayout<MN, STAGES, KSUB>;
  constexpr int BNT = L::BNT, BK = L::BK;
  constexpr uint32_t IDESC = idesc_f16_f32acc(IN_BF16, BNT, MN);
  static_assert(OUT != OUT_S32, "the skinny kernel writes float outputs");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto stage_bt = [&](int s) { return sbase + s * L::STAGE; };
  auto stage_a = [&](int s) { return sbase + s * L::STAGE + L::BT_STAGE; };
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // kernel parameters, not written by earlier kernels: fetch them early
    prefetch_tensor_map(&tmBt);
    prefetch_tensor_map(&tmA);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int64_t u_begin0 = static_cast<int64_t>(blockIdx.x) * p.total_units / p.num_ctas;
  const int64_t u_end0 = static_cast<int64_t>(blockIdx.x + 1) * p.total_units / p.num_ctas;
  // Warm L2 with this CTA's first stages while the previous kernel drains
  // (safe: L2 is where writes become coherent; the loads proper wait).
  if (threadIdx.x == 0) {
    for (int64_t u = u_begin0; u < min(u_end0, u_begin0 + STAGES); ++u) {
      const int nt = static_cast<int>(u / p.num_k_tiles);
      const int kt = static_cast<int>(u - static_cast<int64_t>(nt) * p.num_k_tiles);
#pragma unroll
      for (int j = 0; j < KSUB; ++j) {
        tma_prefetch_l2_2d(&tmBt, (kt * KSUB + j) * L::BK, nt * L::BNT);
        tma_prefetch_l2_2d(&tmA, (kt * KSUB + j) * L::BK, 0);
      }
    }
  }
  // Set-up above may overlap the previous kernel in the stream; no global
  // memory is read for use before that kernel has completed.
  grid_dependency_wait();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_SETUP);

  const WaitCtl ctl{p.timeout_ns, p.error_word, abort_flag};
  const int G = p.num_ctas;
  const int64_t T = p.total_units;
  const int KT = p.num_k_tiles;
  const int64_t u_begin = static_cast<int64_t>(blockIdx.x) * T / G;
  const int64_t u_end = static_cast<int64_t>(blockIdx.x + 1) * T / G;

  // Producer and MMA issuer run as whole warps; one elected lane issues the
  // copies, MMAs and commits (a lane alone in its warp pays a large fixed
  // cost per loop trip).
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    {  // the whole warp
      const bool leader = elect_one_sync();
      const uint64_t pol_stream = policy_evict_first();  // B is read once
      const uint64_t pol_keep = policy_evict_last();     // A is read by every CTA
      int issued_round[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_round[s] = -1;
      bool ok = true;
      uint32_t it = 0;
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int nt = static_cast<int>(u / KT);
        const int kt = static_cast<int>(u - static_cast<int64_t>(nt) * KT);
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        if (!__all_sync(0xffffffffu,
                        wait_bounded(empty_bar(s), (round & 1u) ^ 1u, ctl, WAIT_PRODUCER_EMPTY))) {
          ok = false;
          break;
        }
        if (p.inject_stall && it == 1) continue;  // test hook: this stage never fills
        issued_round[s] = static_cast<int>(round);
        if (!leader) continue;
        mbar_arrive_expect_tx(full_bar(s), L::STAGE);
#pragma unroll
        for (int j = 0; j < KSUB; ++j) {
          tma_load_2d(stage_bt(s) + j * L::SUB_BT, &tmBt, full_bar(s), (kt * KSUB + j) * BK,
                      nt * BNT, pol_stream);
          tma_load_2d(stage_a(s) + j * L::SUB_A, &tmA, full_bar(s), (kt * KSUB + j) * BK, 0,
                      pol_keep);
        }
        if (it == 0) trace_mark(p.trace, TR_FIRST_LOAD);
        trace_ktile(p.trace, 0, it);
      }
      if (leader) trace_mark(p.trace, TR_LAST_LOAD);
      grid_launch_dependents();  // the next kernel may start its set-up
      if (!ok) {
        for (int s = 0; s < STAGES; ++s) {
          if (issued_round[s] < 0) continue;
          const uint32_t par = static_cast<uint32_t>(issued_round[s]) & 1u;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(full_bar(s), par) && global_timer_ns() - t0 < ctl.timeout_ns) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    {  // the whole warp
      const bool leader = elect_one_sync();
      bool ok = true;
      uint32_t it = 0, seg = 0;
      int64_t u = u_begin;
      while (ok && u < u_end) {
        const int nt = static_cast<int>(u / KT);
        const int64_t seg_end = min(u_end, static_cast<int64_t>(nt + 1) * KT);
        const uint32_t b = seg & 1u;
        const uint32_t use = seg >> 1;
        if (!__all_sync(0xffffffffu,
                        wait_bounded(tempty_bar(b), (use & 1u) ^ 1u, ctl, WAIT_MMA_TMEM_EMPTY))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * MN;
        for (int64_t v = u; v < seg_end; ++v, ++it) {
          const int s = it % STAGES;
          const uint32_t round = it / STAGES;
          if (!__all_sync(0xffffffffu, wait_bounded(full_bar(s), round & 1u, ctl, WAIT_MMA_FULL))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (leader) {
            if (it == 0) trace_mark(p.trace, TR_FIRST_DATA);
            trace_ktile(p.trace, 1, it);
#pragma unroll
            for (int j = 0; j < KSUB; ++j) {
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                mma_f16(d_tmem, sdesc_k_major_sw128(stage_bt(s) + j * L::SUB_BT + 32 * k),
                        sdesc_k_major_sw128(stage_a(s) + j * L::SUB_A + 32 * k), IDESC,
                        (v > u || j > 0 || k > 0) ? 1u : 0u);
              }
            }
            mma_commit(empty_bar(s));
          }
          __syncwarp();
        }
        if (ok && leader) mma_commit(tfull_bar(b));
        __syncwarp();
        u = seg_end;
        ++seg;
      }
      if (leader) {
        trace_mark(p.trace, TR_LAST_MMA);
        mma_commit(drain_bar);
      }
      __syncwarp();
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < ctl.timeout_ns) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int n_local = 32 * q + lane;  // this thread's row of D^T (an output column)
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const int M = p.M;
    uint32_t seg = 0;
    int64_t u = u_begin;
    bool ok = true;
    while (ok && u < u_end) {
      const int nt = static_cast<int>(u / KT);
      const int64_t seg_end = min(u_end, static_cast<int64_t>(nt + 1) * KT);
      const uint32_t b = seg & 1u;
      const uint32_t use = seg >> 1;
      // The four epilogue warps take one decision: they meet at named barriers below.
      ok = named_barrier_and(1, 128, wait_bounded(tfull_bar(b), use & 1u, ctl, WAIT_EPI_TMEM_FULL));
      if (!ok) break;
      tc_fence_after();
      float acc[MN];
#pragma unroll
      for (int cb = 0; cb < MN / 32; ++cb) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_lane + b * MN + 32 * cb, r);
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[32 * cb + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(b));  // accumulator b may be reused

      const int n = nt * BNT + n_local;
      const int c_first = cta_of_unit(static_cast<int64_t>(nt) * KT, G, T);
      const int c_last = cta_of_unit(static_cast<int64_t>(nt + 1) * KT - 1, G, T);
      const int count = c_last - c_first + 1;
      if (count == 1) {
        if (n < p.N) {
#pragma unroll
          for (int m = 0; m < MN; ++m)
            if (m < M) store_out<OUT>(p.C, static_cast<int64_t>(m) * p.ldc + n, acc[m]);
        }
      } else if (p.partials == nullptr || count > p.max_contrib) {
        // the host planned no room for this split: report instead of writing
        if (threadIdx.x == 64) atomicOr(p.error_word, WAIT_PLAN);
      } else {
        const int j = static_cast<int>(blockIdx.x) - c_first;
        float* slot = p.partials + (static_cast<int64_t>(nt) * p.max_contrib + j) * (MN * BNT);
#pragma unroll
        for (int m = 0; m < MN; ++m) __stcg(slot + m * BNT + n_local, acc[m]);
        __threadfence();
        named_barrier_sync(1, 128);
        if (threadIdx.x == 64) {
          *last_flag = arrive_generation(p.counters + nt, p.generation, count, p.error_word);
          // the last arrival is the last use of the counter in this call
          if (*last_flag) atomicExch(p.counters + nt, 0ull);
        }
        named_barrier_sync(1, 128);
        if (*last_flag) {
          // Sum the partial tiles in contributor order (increasing k), 16-byte
          // loads with every contributor's loads in flight together.
          __threadfence();
          constexpr int F4_PER_ROW = BNT / 4;
          constexpr int PER_THREAD = MN * F4_PER_ROW / 128;
          const int tid = threadIdx.x - 64;
          const float4* base = reinterpret_cast<const float4*>(
              p.partials + static_cast<int64_t>(nt) * p.max_contrib * (MN * BNT));
          // two halves of the tile; in each, the loads of up to four
          // contributors are issued together, then added in order
          constexpr int HALF = PER_THREAD / 2;
          constexpr int64_t SLOT4 = MN * BNT / 4;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float4 v[4][HALF];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              if (jj < count) {
#pragma unroll
                for (int i = 0; i < HALF; ++i)
                  v[jj][i] = __ldcg(base + jj * SLOT4 + tid + 128 * (h * HALF + i));
              }
            }
            float4 sum[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) sum[i] = v[0][i];
#pragma unroll
            for (int jj = 1; jj < 4; ++jj) {
              if (jj < count) {
#pragma unroll
                for (int i = 0; i < HALF; ++i) {
                  sum[i].x += v[jj][i].x;
                  sum[i].y += v[jj][i].y;
                  sum[i].z += v[jj][i].z;
                  sum[i].w += v[jj][i].w;
                }
              }
            }
            for (int jj = 4; jj < count; ++jj) {  // more than four contributors: rare
#pragma unroll
              for (int i = 0; i < HALF; ++i) {
                const float4 w = __ldcg(base + jj * SLOT4 + tid + 128 * (h * HALF + i));
                sum[i].x += w.x;
                sum[i].y += w.y;
                sum[i].z += w.z;
                sum[i].w += w.w;
              }
            }
#pragma unroll
            for (int i = 0; i < HALF; ++i) {
              const int f = tid + 128 * (h * HALF + i);
              const int m = f / F4_PER_ROW;
              const int n0 = nt * BNT + 4 * (f % F4_PER_ROW);
              if (m < M && n0 < p.N) store_out4<OUT>(p.C, static_cast<int64_t>(m) * p.ldc + n0, sum[i]);
            }
          }
          if (threadIdx.x == 64) trace_mark(p.trace, TR_FIXUP_DONE);
        }
        named_barrier_sync(1, 128);  // last_flag is reused by the next segment
      }
      u = seg_end;
      ++seg;
    }
    if (threadIdx.x == 64) trace_mark(p.trace, TR_EPI_DONE);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace sptg
