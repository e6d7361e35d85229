// skinny_pair_gemm.cuh -- the memory-bound skinny product (M <= 256) on CTA
// pairs with the 2-SM tensor-core instruction, K never split.
//
// Swap-AB as in skinny_gemm.cuh: D^T[n, m] = sum_k Bcm[n, k] * A[m, k]. The
// MMA's N side covers MN = 64, 128 or 256 rows of A. A pair of CTAs (a
// cluster of two) owns 2 * n_cta consecutive output columns (n_cta <= 128).
// CTA rank r loads the n_cta rows of Bcm of its own columns, in blocks of 64
// rows (one MMA each; rows past n_cta are never stored), and the MN / 2 rows
// r * MN / 2 ... of A. The leader's tcgen05.mma.cta_group::2 (M = 128 over
// the pair's 64-column blocks, N = MN over the rows of A) reads both CTAs'
// shared memory, so each SM copies only half of A per K-chunk, and each CTA's
// tensor memory receives the sums of its own columns over the whole of K.
// Nothing is exchanged between SMs after the K-loop: each CTA converts its
// MN x n_cta block of C, stages it in shared memory (the ring, idle by then)
// and writes it with one tensor copy.
//
// Per SM a K-chunk moves (n_cta + MN / 2) x 128 bytes, against (n_cta + 64)
// x 128 for one CTA per strip (skinny_rows_gemm.cuh, MN = 64) and (128 + MN)
// x 128 for half a K-range of a 128-column tile (skinny_cluster_gemm.cuh,
// which then exchanges partial sums). The host picks n_cta so that the pairs
// cover the SMs about once (8192 columns over 152 SMs: 56 per CTA, 74 pairs).
//
// Copies of both CTAs complete on the leader's "full" barrier; the leader's
// commits arrive on both CTAs' "empty" and "tmem_full" barriers.
//
// Tensor-memory layout of an accumulator (cta_group::2, M = 128, N = MN):
// each CTA holds its 64 rows of D with the N side split in halves: row i's
// sums for the rows 0 ... MN/2 - 1 of A lie in lane i, those for the rows
// MN/2 ... MN - 1 in lane 64 + i, each half in MN / 2 columns. Block h of a
// CTA's columns takes the columns h * MN / 2 ... of tensor memory.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace sptg {

struct SkinnyPairParams {
  int M, N, K;
  int n_cta;        // output columns per CTA: a multiple of 8, 8 ... 128
  int num_k_tiles;  // ring stages' worth of K: ceil(K / (64 * KSUB))
  int stages;       // ring depth, 1 ... SKINNY_PAIR_MAX_STAGES
  int stage_bytes;  // skinny_pair_stage_bytes(KSUB, n_cta, MN)
  int load3d;       // 1: one 3-D copy per operand and stage; 0: 2-D per chunk
  int k_rotate;     // 1: pair i starts its K-loop at chunk i * num_k_tiles / pairs
  unsigned int* error_word;
  uint64_t timeout_ns;
  int inject_stall;
  unsigned long long* trace;
};

constexpr int SKINNY_PAIR_MAX_STAGES = 16;
// barriers (2 per stage + 2) and misc words after the ring
constexpr int SKINNY_PAIR_BAR_BYTES = (2 * SKINNY_PAIR_MAX_STAGES + 2) * 8 + 16;
constexpr int SKINNY_PAIR_RING_BUDGET = 232448 - 1024 - SKINNY_PAIR_BAR_BYTES;

constexpr int SKINNY_PAIR_SUB_B = 64 * 128;  // the MMA's 64-row operand tile of Bcm rows
// one K-chunk of a CTA's MN / 2 rows of A
__host__ __device__ constexpr int skinny_pair_sub_a(int mn) { return mn / 2 * 128; }

// One ring stage: the KSUB K-chunks of this CTA's n_cta rows of Bcm back to
// back (as one 3-D copy writes them) -- the MMAs read 64-row tiles from the
// start of each (one per 64-row block), so the region holds (KSUB - 1) packed
// chunks and the blocks of one more -- then the KSUB chunks of its MN / 2 rows
// of A. A multiple of 1024 bytes (n_cta is a multiple of 8), which keeps
// every chunk on the swizzle pattern.
__host__ __device__ constexpr int skinny_pair_blocks(int n_cta) { return (n_cta + 63) / 64; }
__host__ __device__ constexpr int skinny_pair_b_region(int ksub, int n_cta) {
  return (ksub - 1) * n_cta * 128 + skinny_pair_blocks(n_cta) * SKINNY_PAIR_SUB_B;
}
__host__ __device__ constexpr int skinny_pair_stage_bytes(int ksub, int n_cta, int mn) {
  return skinny_pair_b_region(ksub, n_cta) + ksub * skinny_pair_sub_a(mn);
}

template <int MN, bool IN_BF16, int OUT, int KSUB>
__global__ void __launch_bounds__(192, 1)
    skinny_pair_gemm_kernel(const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmC,
                            const SkinnyPairParams p) {
  constexpr int BK = 64;
  constexpr int OBYTES = OutTraits<OUT>::bytes;
  constexpr int HALF = MN / 2;  // rows of A each CTA copies
  constexpr int SUB_A = skinny_pair_sub_a(MN);
  // kind::f16, fp32 accumulation, M = 128 (the pair), N = MN
  constexpr uint32_t IDESC = idesc_f16_f32acc(IN_BF16, 128, MN);
  static_assert(MN == 64 || MN == 128 || MN == 256, "MN must be 64, 128 or 256");
  static_assert(OUT != OUT_S32, "float outputs only");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int S = p.stages;
  const int n_cta = p.n_cta;
  const uint32_t bar0 = sbase + static_cast<uint32_t>(S * p.stage_bytes);
  auto stage_b = [&](int s) { return sbase + static_cast<uint32_t>(s * p.stage_bytes); };
  const uint32_t a_off = static_cast<uint32_t>(skinny_pair_b_region(KSUB, n_cta));
  auto stage_a = [&](int s) { return stage_b(s) + a_off; };
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (SKINNY_PAIR_MAX_STAGES + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * SKINNY_PAIR_MAX_STAGES);
  const uint32_t drain_bar = tfull_bar + 8u;
  uint8_t* misc = smem + S * p.stage_bytes + (2 * SKINNY_PAIR_MAX_STAGES + 2) * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* failed = reinterpret_cast<volatile int*>(misc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 = leader, which issues the MMAs
  // this CTA's first output column
  const int n_base =
      static_cast<int>(blockIdx.x >> 1) * 2 * n_cta + static_cast<int>(rank) * n_cta;
  const int KT = p.num_k_tiles;
  // With k_rotate the pairs start their K-loops at evenly spaced chunks and
  // wrap around, so that at any moment they read different columns of A and
  // different K-ranges of their Bcm rows (the sum's order over K differs
  // from pair to pair; each column's order is fixed by the launch).
  const int k_rot = p.k_rotate ? static_cast<int>((static_cast<int64_t>(blockIdx.x >> 1) * KT) /
                                                  static_cast<int64_t>(gridDim.x >> 1))
                               : 0;
  auto kchunk = [&](int kt) {  // the chunk a pair copies at loop position kt
    const int c = kt + k_rot;
    return c >= KT ? c - KT : c;
  };
  // bytes that complete one stage's "full" barrier: both CTAs' copies
  const uint32_t stage_tx = 2u * KSUB * static_cast<uint32_t>((n_cta + HALF) * 128);
  // A K-chunk of this CTA's Bcm rows fills n_cta rows; the chunks of a stage
  // lie back to back, so the MMA's 64-row operand tile of chunk j starts at
  // j * n_cta rows and its rows past n_cta (the next chunk's, or unused ones)
  // only reach sums that are never stored.
  const int sub_b = n_cta * 128;
  // 64-row blocks of the CTA's columns: one MMA (and one accumulator of HALF
  // tensor-memory columns) each
  const int nblk = skinny_pair_blocks(n_cta);
  const uint32_t tmem_cols =
      nblk * HALF <= 32 ? 32u : nblk * HALF <= 64 ? 64u : nblk * HALF <= 128 ? 128u : 256u;

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
    prefetch_tensor_map(&tmB);
    prefetch_tensor_map(&tmA);
    prefetch_tensor_map(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_g<true>(smem_addr(tmem_slot), tmem_cols);
    tmem_relinquish_g<true>();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Warm L2 with this CTA's first stages of Bcm while the previous kernel
  // drains (safe: L2 is where writes become coherent; the loads proper wait
  // for the dependency).
  uint64_t pol_stream = 0, pol_keep = 0;
  if (warp == 0) {
    pol_stream = policy_evict_first();  // Bcm is read once
    pol_keep = policy_evict_last();     // A is read by every pair
    for (int kt = 0; lane == 0 && kt < min(KT, S); ++kt) {
      const int kc = kchunk(kt);
      if (p.load3d) {
        tma_prefetch_l2_3d(&tmB, 0, n_base, kc * KSUB);
      } else {
#pragma unroll
        for (int j = 0; j < KSUB; ++j) tma_prefetch_l2_2d(&tmB, (kc * KSUB + j) * BK, n_base);
      }
    }
  }
  grid_dependency_wait();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_SETUP);

  const WaitCtl ctl{p.timeout_ns, p.error_word, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const bool leader = elect_one_sync();
    int issued_round[SKINNY_PAIR_MAX_STAGES];
    for (int s = 0; s < SKINNY_PAIR_MAX_STAGES; ++s) issued_round[s] = -1;
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
      if (!(p.inject_stall && kt == 1 && rank == 0)) {  // test hook: this stage never fills
        issued_round[s] = static_cast<int>(round);
        if (leader) {
          // both CTAs' copies complete on the leader's barrier; the leader
          // announces the bytes of both
          if (rank == 0) mbar_arrive_expect_tx(full_bar(s), stage_tx);
          const uint32_t leader_full = map_to_cta(full_bar(s), 0u);
          const int kc = kchunk(kt);
          if (p.load3d) {
            tma_load_3d_pair(stage_b(s), &tmB, leader_full, 0, n_base, kc * KSUB, pol_stream);
            tma_load_3d_pair(stage_a(s), &tmA, leader_full, 0, HALF * static_cast<int>(rank),
                             kc * KSUB, pol_keep);
          } else {
#pragma unroll
            for (int j = 0; j < KSUB; ++j) {
              tma_load_2d_pair(stage_b(s) + j * sub_b, &tmB, leader_full, (kc * KSUB + j) * BK,
                               n_base, pol_stream);
              tma_load_2d_pair(stage_a(s) + j * SUB_A, &tmA, leader_full, (kc * KSUB + j) * BK,
                               HALF * static_cast<int>(rank), pol_keep);
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
      if (rank == 0) {
        // let every copy already issued land before the CTA can exit
        for (int t = 0; t < S; ++t) {
          if (issued_round[t] < 0) continue;
          const uint32_t par = static_cast<uint32_t>(issued_round[t]) & 1u;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(full_bar(t), par) && global_timer_ns() - t0 < ctl.timeout_ns) {
          }
        }
      } else {
        // the copies complete on the leader's barriers, which this CTA
        // cannot wait on: give them a fixed 100 us to land
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (rank == 0) {
      const bool leader = elect_one_sync();
      // The K-loop with each stage's MMAs as straight-line code, compiled
      // for one and for two 64-row blocks (n_cta <= 128) and chosen once: a
      // loop with a runtime trip count, or a branch, run by the elected lane
      // alone costs more per stage than the MMAs it issues (64 x 4096 x 8192:
      // 20.6 us with a runtime block loop against 15.4 us straight-line).
      auto k_loop = [&](auto nb) {
        constexpr int NB = decltype(nb)::value;
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
              for (int h = 0; h < NB; ++h) {
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                  mma_f16_g<true>(tmem_base + h * HALF,
                                  sdesc_k_major_sw128(stage_b(s) + j * sub_b +
                                                      h * SKINNY_PAIR_SUB_B + 32 * k),
                                  sdesc_k_major_sw128(stage_a(s) + j * SUB_A + 32 * k), IDESC,
                                  (kt > 0 || j > 0 || k > 0) ? 1u : 0u);
                }
              }
            }
            mma_commit_g<true>(empty_bar(s));  // stage s may be refilled in both CTAs
          }
          __syncwarp();
          if (++s == S) {
            s = 0;
            ++round;
          }
        }
      };
      if (nblk == 1)
        k_loop(std::integral_constant<int, 1>{});
      else
        k_loop(std::integral_constant<int, 2>{});
      if (leader) {
        trace_mark(p.trace, TR_LAST_MMA);
        mma_commit_g<true>(tfull_bar);  // both CTAs' accumulators are complete
        mma_commit_local_g<true>(drain_bar);
      }
      __syncwarp();
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < ctl.timeout_ns) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warps 2-5: the warp of lane quarter q (= warp % 4) reads lanes
    // 32q ... 32q + 31, which hold the columns 64h + 32 (q % 2) ... + 31 of
    // block h (in tensor-memory columns h * MN / 2 ...), each with the sums
    // for the MN / 2 rows of A from (MN / 2)(q / 2) on
    const int q = warp & 3;
    const int m0 = HALF * (q >> 1);  // first row of A this warp's sums belong to
    const bool done = __all_sync(0xffffffffu, wait_bounded(tfull_bar, 0, ctl, WAIT_EPI_TMEM_FULL));
    const bool ok = named_barrier_and(1, 128, done && !*failed);
    if (ok) {
      tc_fence_after();
      // stage the MN x n_cta block of C (row m holds consecutive outputs) at
      // the start of the ring, free once every MMA has completed (the host
      // checks that the ring holds it)
      uint8_t* stage = smem;
      for (int h = 0; h < nblk; ++h) {
        const int col = 64 * h + 32 * (q & 1) + lane;  // column within the CTA's block
        const bool have_col = col < n_cta;
#pragma unroll
        for (int cb = 0; cb < HALF; cb += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + h * HALF + cb,
                             r);
          tmem_wait_ld_regs(r);
          if (have_col) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int m = m0 + cb + i;
              const float v = __uint_as_float(r[i]);
              if constexpr (OBYTES == 4) {
                reinterpret_cast<float*>(stage)[m * n_cta + col] = v;
              } else if constexpr (OUT == OUT_F16) {
                reinterpret_cast<__half*>(stage)[m * n_cta + col] = __float2half_rn(v);
              } else {
                reinterpret_cast<__nv_bfloat16*>(stage)[m * n_cta + col] = __float2bfloat16_rn(v);
              }
            }
          }
        }
      }
      fence_proxy_async_smem();
      named_barrier_sync(1, 128);
      // rows past M and columns past N clip
      if (threadIdx.x == 64 && n_base < p.N) {
        tma_store_2d(&tmC, smem_addr(stage), n_base, 0);
        bulk_commit_group();
        bulk_wait_group_read<0>();  // the staging may go once the copy has read it
      }
    }
    if (threadIdx.x == 64) trace_mark(p.trace, TR_EPI_DONE);
  }

  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the pair's MMAs may still read it
  if (threadIdx.x == 0) trace_mark(p.trace, TR_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_g<true>(tmem_base, tmem_cols);
  }
}

}  // namespace sptg
