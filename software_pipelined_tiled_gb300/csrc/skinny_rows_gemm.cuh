// skinny_rows_gemm.cuh -- the memory-bound skinny product (M <= 64) with one
// CTA per strip of output columns and no reduction at all.
//
// C = A * B with A (M x K, M <= 64) and B given as Bcm (N x K). The MMA's M
// side is the 64 rows of A (rows past M are zero-filled by the copies and
// never stored); its N side is a strip of n_tile output columns, a multiple
// of 8 up to 256 chosen by the host so that the strips cover the SMs about
// once (16384 columns over 152 SMs: strips of 112, 147 CTAs). Each CTA streams its
// n_tile rows of Bcm over the whole of K through a TMA ring whose stages hold
// KSUB consecutive 64-wide K-chunks of A and of Bcm, accumulates in tensor
// memory, and its four epilogue warps store the 64 x n_tile block straight
// from registers to C.
//
// Compared with the cluster split (skinny_cluster_gemm.cuh), nothing is
// exchanged between SMs and no cluster is launched; the price is that every
// CTA reads all of A (M x K, from L2: A is read once from DRAM) instead of
// its share of K.
//
// Tensor-memory layout of a 64-row accumulator (cta_group::1, M = 64): row i
// of D sits in lane 32 * (i / 16) + i % 16, i.e. lanes 0-15 of each warp's
// 32-lane quarter; lanes 16-31 of each quarter are not written.
#pragma once

#include "common.cuh"

namespace sptg {

struct SkinnyRowsParams {
  void* C;
  int64_t ldc;          // row pitch of C, elements
  int M, N, K;
  int n_tile;           // output columns per CTA: a multiple of 8, 8 ... 256
  int num_k_tiles;      // ring stages' worth of K: ceil(K / (64 * KSUB))
  int stages;           // ring depth, 1 ... SKINNY_ROWS_MAX_STAGES
  int stage_bytes;      // KSUB * (64 + n_tile) * 128, a multiple of 1024
  int load3d;           // 1: one 3-D copy per operand and stage; 0: 2-D per chunk
  int k_rotate;         // 1: strip i starts its K-loop at chunk i * num_k_tiles / strips
  unsigned int* error_word;
  uint64_t timeout_ns;
  int inject_stall;
  unsigned long long* trace;
};

constexpr int SKINNY_ROWS_MAX_STAGES = 16;
constexpr int SKINNY_ROWS_MAX_NT = 256;
// barriers (2 per stage + 2) and misc words after the ring
constexpr int SKINNY_ROWS_BAR_BYTES = (2 * SKINNY_ROWS_MAX_STAGES + 2) * 8 + 16;
// the largest ring the shared memory holds, after 1 KB of alignment slack
constexpr int SKINNY_ROWS_RING_BUDGET = 232448 - 1024 - SKINNY_ROWS_BAR_BYTES;

template <bool IN_BF16, int OUT, int KSUB>
__global__ void __launch_bounds__(192, 1)
    skinny_rows_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const SkinnyRowsParams p) {
  constexpr int BK = 64;
  constexpr int SUB_A = 64 * BK * 2;  // one 64-wide K-chunk of 64 rows of A
  static_assert(OUT != OUT_S32, "float outputs only");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int S = p.stages;
  const int nt_cols = p.n_tile;
  const int sub_b = nt_cols * 128;  // one K-chunk of the strip's Bcm rows
  const uint32_t bar0 = sbase + static_cast<uint32_t>(S * p.stage_bytes);
  auto stage_a = [&](int s) { return sbase + static_cast<uint32_t>(s * p.stage_bytes); };
  auto stage_b = [&](int s) { return stage_a(s) + KSUB * SUB_A; };
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (SKINNY_ROWS_MAX_STAGES + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * SKINNY_ROWS_MAX_STAGES);
  const uint32_t drain_bar = tfull_bar + 8u;
  uint8_t* misc = smem + S * p.stage_bytes + (2 * SKINNY_ROWS_MAX_STAGES + 2) * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* failed = reinterpret_cast<volatile int*>(misc + 8);
  // tensor-memory columns: a power of two >= 32 that holds the strip
  const uint32_t tmem_cols =
      nt_cols <= 32 ? 32u : nt_cols <= 64 ? 64u : nt_cols <= 128 ? 128u : 256u;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = static_cast<int>(blockIdx.x) * nt_cols;  // first output column
  const int KT = p.num_k_tiles;
  // With k_rotate the strips start their K-loops at evenly spaced chunks and
  // wrap around, so that at any moment they read different columns of A and
  // different K-ranges of their Bcm rows (each column's order over K is
  // fixed by the launch).
  const int k_rot = p.k_rotate ? static_cast<int>((static_cast<int64_t>(blockIdx.x) * KT) /
                                                  static_cast<int64_t>(gridDim.x))
                               : 0;
  auto kchunk = [&](int kt) {  // the chunk a strip copies at loop position kt
    const int c = kt + k_rot;
    return c >= KT ? c - KT : c;
  };
  // kind::f16, fp32 accumulation, M = 64, N = n_tile
  const uint32_t idesc = idesc_f16_f32acc(IN_BF16, 64, nt_cols);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *failed = 0;
    fence_mbar_init();
    prefetch_tensor_map(&tmA);
    prefetch_tensor_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Warm L2 with this CTA's first stages of Bcm while the previous kernel
  // drains (L2 is where writes become coherent, so this is safe even if that
  // kernel writes B; the loads proper come after the dependency wait).
  uint64_t pol_stream = 0, pol_keep = 0;
  if (warp == 0) {
    pol_stream = policy_evict_first();  // Bcm is read once
    pol_keep = policy_evict_last();     // A is read by every CTA
    for (int kt = 0; lane == 0 && kt < min(KT, S); ++kt) {
      const int kc = kchunk(kt);
      if (p.load3d) {
        tma_prefetch_l2_3d(&tmB, 0, n0, kc * KSUB);
      } else {
#pragma unroll
        for (int j = 0; j < KSUB; ++j) tma_prefetch_l2_2d(&tmB, (kc * KSUB + j) * BK, n0);
      }
    }
  }
  grid_dependency_wait();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_SETUP);

  const WaitCtl ctl{p.timeout_ns, p.error_word, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const bool leader = elect_one_sync();
    int issued_round[SKINNY_ROWS_MAX_STAGES];
    for (int s = 0; s < SKINNY_ROWS_MAX_STAGES; ++s) issued_round[s] = -1;
    bool ok = true;
    int s = 0;
    uint32_t round = 0;
    for (int kt = 0; kt < KT; ++kt) {
      // in the first round every stage is free: no wait
      if (round > 0 && !__all_sync(0xffffffffu, wait_bounded(empty_bar(s), (round & 1u) ^ 1u, ctl,
                                                              WAIT_PRODUCER_EMPTY))) {
        ok = false;
        break;
      }
      if (!(p.inject_stall && kt == 1)) {  // test hook: this stage never fills
        issued_round[s] = static_cast<int>(round);
        if (leader) {
          mbar_arrive_expect_tx(full_bar(s), static_cast<uint32_t>(p.stage_bytes));
          const int kc = kchunk(kt);
          if (p.load3d) {
            tma_load_3d(stage_a(s), &tmA, full_bar(s), 0, 0, kc * KSUB, pol_keep);
            tma_load_3d(stage_b(s), &tmB, full_bar(s), 0, n0, kc * KSUB, pol_stream);
          } else {
#pragma unroll
            for (int j = 0; j < KSUB; ++j) {
              tma_load_2d(stage_a(s) + j * SUB_A, &tmA, full_bar(s), (kc * KSUB + j) * BK, 0,
                          pol_keep);
              tma_load_2d(stage_b(s) + j * sub_b, &tmB, full_bar(s), (kc * KSUB + j) * BK, n0,
                          pol_stream);
            }
          }
          if (kt == 0) trace_mark(p.trace, TR_FIRST_LOAD);
          trace_ktile(p.trace, 0, static_cast<uint32_t>(kt));
        }
      }
      if (++s == S) {
        s = 0;
        ++round;
      }
    }
    if (leader) trace_mark(p.trace, TR_LAST_LOAD);
    grid_launch_dependents();
    if (!ok) {
      if (leader) *failed = 1;
      // let the copies in flight land before the CTA leaves
      for (int t = 0; t < S; ++t) {
        if (issued_round[t] < 0) continue;
        const uint32_t par = static_cast<uint32_t>(issued_round[t]) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(full_bar(t), par) && global_timer_ns() - t0 < ctl.timeout_ns) {
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const bool leader = elect_one_sync();
    int s = 0;
    uint32_t round = 0;
    for (int kt = 0; kt < KT; ++kt) {
      if (!__all_sync(0xffffffffu, wait_bounded(full_bar(s), round & 1u, ctl, WAIT_MMA_FULL))) {
        if (leader) *failed = 1;
        break;
      }
      tc_fence_after();
      if (leader) {
        if (kt == 0) trace_mark(p.trace, TR_FIRST_DATA);
        trace_ktile(p.trace, 1, static_cast<uint32_t>(kt));
#pragma unroll
        for (int j = 0; j < KSUB; ++j) {
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            mma_f16(tmem_base, sdesc_k_major_sw128(stage_a(s) + j * SUB_A + 32 * k),
                    sdesc_k_major_sw128(stage_b(s) + j * sub_b + 32 * k), idesc,
                    (kt > 0 || j > 0 || k > 0) ? 1u : 0u);
          }
        }
        mma_commit(empty_bar(s));
      }
      __syncwarp();
      if (++s == S) {
        s = 0;
        ++round;
      }
    }
    if (leader) {
      trace_mark(p.trace, TR_LAST_MMA);
      mma_commit(tfull_bar);
      mma_commit(drain_bar);
    }
    __syncwarp();
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < ctl.timeout_ns) {
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warps 2-5: the warp of lane quarter q (= warp % 4) reads lanes
    // 32q ... 32q + 31; its lanes 0-15 hold rows 16q ... 16q + 15
    const int q = warp & 3;
    const int m = 16 * q + lane;
    const bool have_row = lane < 16 && m < p.M;
    const bool done = __all_sync(0xffffffffu, wait_bounded(tfull_bar, 0, ctl, WAIT_EPI_TMEM_FULL));
    if (done && !*failed) {
      tc_fence_after();
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
      void* row_ptr = static_cast<uint8_t*>(p.C) +
                      static_cast<int64_t>(have_row ? m : 0) * p.ldc * OutTraits<OUT>::bytes;
      constexpr int G = OUT == OUT_F32 ? 4 : 8;  // outputs per 16-byte store
      for (int cb = 0; cb < nt_cols; cb += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_lane + cb, r);
        tmem_wait_ld_regs(r);
        if (have_row) {
#pragma unroll
          for (int g = 0; g < 32; g += G) {
            const int col = n0 + cb + g;
            const int n_valid = min(min(G, nt_cols - cb - g), p.N - col);
            if (n_valid <= 0) continue;
            float v[G];
#pragma unroll
            for (int i = 0; i < G; ++i) v[i] = __uint_as_float(r[g + i]);
            store_row_group<OUT>(row_ptr, col, v, n_valid);
          }
        }
      }
    }
    if (lane == 0 && q == 0) trace_mark(p.trace, TR_EPI_DONE);
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace sptg
