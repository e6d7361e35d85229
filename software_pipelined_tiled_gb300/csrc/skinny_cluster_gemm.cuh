// skinny_cluster_gemm.cuh -- the memory-bound skinny product (M <= 64) with
// its K split inside a thread-block cluster.
//
// Same arithmetic as skinny_gemm.cuh (swap-AB: D^T[n, m] = sum_k Bcm[n, k] *
// A[m, k], MMA M = 128 over N, MMA N = MN over the rows of A), but the work
// is cut along whole column tiles: one cluster of CS CTAs per 128-column tile,
// CTA rank r streaming the contiguous K-range [r*KT/CS, (r+1)*KT/CS). Each
// CTA accumulates its range in tensor memory. When all have finished, ranks
// 1..CS-1 leave their fp32 partial tile in their own shared memory and rank 0
// reads them through distributed shared memory, adds them in rank order
// (= increasing k, a fixed order) to its own, converts and writes C.
//
// Compared with the stream-K kernel this needs no global scratch and no
// atomics, and the final reduction is one exchange between SMs of a cluster
// instead of a round trip through L2. The price is that the grid is
// (column tiles x CS) CTAs, which the host uses when that fills the GPU.
#pragma once

#include "common.cuh"

namespace sptg {

struct SkinnyClusterParams {
  int M, N, K;
  int num_n_tiles, num_k_tiles;
  void* C;  // row-major M x N output
  unsigned int* error_word;
  uint64_t timeout_ns;
  int inject_stall;
  unsigned long long* trace;
};

template <int MN, int STAGES>
struct SkinnyClusterLayout {
  static constexpr int BNT = 128;
  static constexpr int BK = 64;
  static constexpr int BT_STAGE = BNT * BK * 2;
  static constexpr int A_STAGE = MN * BK * 2;
  static constexpr int STAGE = BT_STAGE + A_STAGE;
  // partial tile in shared memory, rows of MN floats + 16 bytes of padding
  // so that 16-byte accesses of 8 consecutive rows hit 8 distinct bank groups
  static constexpr int PART_ROW = MN * 4 + 16;
  static constexpr int PART_BYTES = BNT * PART_ROW;
  static constexpr int OFF_BAR = STAGES * STAGE;
  static constexpr int NUM_BARS = 2 * STAGES + 2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TMEM_COLS = MN <= 32 ? 32 : MN <= 64 ? 64 : 128;
  static_assert(PART_BYTES <= STAGES * STAGE, "the partial tile reuses the ring's memory");
  static_assert(MN % 32 == 0 && MN >= 32 && MN <= 128, "MN must be 32, 64, 96 or 128");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
};

__device__ __forceinline__ float4 ld_shared_cluster_f4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}

template <int MN, int STAGES, bool IN_BF16, int OUT>
__global__ void __launch_bounds__(192, 1)
    skinny_cluster_gemm_kernel(const __grid_constant__ CUtensorMap tmBt,
                               const __grid_constant__ CUtensorMap tmA,
                               const SkinnyClusterParams p) {
  using L = SkinnyClusterLayout<MN, STAGES>;
  constexpr int BNT = L::BNT, BK = L::BK;
  constexpr uint32_t IDESC = idesc_f16_f32acc(IN_BF16, BNT, MN);
  static_assert(OUT != OUT_S32, "float outputs only");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto stage_bt = [&](int s) { return sbase + s * L::STAGE; };
  auto stage_a = [&](int s) { return sbase + s * L::STAGE + L::BT_STAGE; };
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * STAGES);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cs = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int nt = static_cast<int>(blockIdx.x / cs);
  const int KT = p.num_k_tiles;
  const int kt0 = static_cast<int>(static_cast<int64_t>(rank) * KT / cs);
  const int kt1 = static_cast<int>(static_cast<int64_t>(rank + 1) * KT / cs);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *failed = 0;
    fence_mbar_init();
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
  grid_dependency_wait();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_SETUP);

  const WaitCtl ctl{p.timeout_ns, p.error_word, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();  // B is read once
      const uint64_t pol_keep = policy_evict_last();     // A is read by every CTA
      int issued_round[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_round[s] = -1;
      bool ok = true;
      uint32_t it = 0;
      for (int kt = kt0; kt < kt1; ++kt, ++it) {
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        if (!wait_bounded(empty_bar(s), (round & 1u) ^ 1u, ctl, WAIT_PRODUCER_EMPTY)) {
          ok = false;
          break;
        }
        if (p.inject_stall && it == 1) continue;  // test hook: this stage never fills
        mbar_arrive_expect_tx(full_bar(s), L::STAGE);
        tma_load_2d(stage_bt(s), &tmBt, full_bar(s), kt * BK, nt * BNT, pol_stream);
        tma_load_2d(stage_a(s), &tmA, full_bar(s), kt * BK, 0, pol_keep);
        issued_round[s] = static_cast<int>(round);
        if (it == 0) trace_mark(p.trace, TR_FIRST_LOAD);
        trace_ktile(p.trace, 0, it);
      }
      trace_mark(p.trace, TR_LAST_LOAD);
      grid_launch_dependents();
      if (!ok) {
        *failed = 1;
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
    if (lane == 0) {
      uint32_t it = 0;
      for (int kt = kt0; kt < kt1; ++kt, ++it) {
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        if (!wait_bounded(full_bar(s), round & 1u, ctl, WAIT_MMA_FULL)) {
          *failed = 1;
          break;
        }
        tc_fence_after();
        if (it == 0) trace_mark(p.trace, TR_FIRST_DATA);
        trace_ktile(p.trace, 1, it);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          mma_f16(tmem_base, sdesc_k_major_sw128(stage_bt(s) + 32 * k),
                  sdesc_k_major_sw128(stage_a(s) + 32 * k), IDESC,
                  (kt > kt0 || k > 0) ? 1u : 0u);
        }
        mma_commit(empty_bar(s));
      }
      trace_mark(p.trace, TR_LAST_MMA);
      mma_commit(tfull_bar);  // also arrives when no MMA was issued (empty K-range)
      mma_commit(drain_bar);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < ctl.timeout_ns) {
      }
    }
  }

  // ---------------------------------------------------------- epilogue part 1
  // warps 2-5 read this CTA's partial tile (their 32 lanes each = 32 output
  // columns, MN values per column) out of tensor memory
  float acc[MN];
  const int q = warp & 3;
  const int n_local = 32 * q + lane;
  if (warp >= 2) {
    const bool done =
        __all_sync(0xffffffffu, wait_bounded(tfull_bar, 0, ctl, WAIT_EPI_TMEM_FULL));
    if (done) {
      tc_fence_after();
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
#pragma unroll
      for (int cb = 0; cb < MN / 32; ++cb) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_lane + 32 * cb, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          acc[32 * cb + i] = (kt1 > kt0) ? __uint_as_float(r[i]) : 0.0f;
      }
      if (rank != 0) {
        // leave the partial in this CTA's own shared memory (the ring is idle:
        // every stage has been consumed) for rank 0 to read
        uint8_t* row = smem + n_local * L::PART_ROW;
#pragma unroll
        for (int i = 0; i < MN / 4; ++i)
          *reinterpret_cast<float4*>(row + 16 * i) =
              make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
      }
    } else if (lane == 0) {
      *failed = 1;
    }
  }
  tc_fence_before();
  cluster_sync();  // every partial and every failure flag of the cluster is visible

  // ---------------------------------------------------------- epilogue part 2
  if (warp >= 2 && rank == 0) {
    // the result is written only when no CTA of the cluster gave up a wait
    bool all_ok = (*failed == 0);
    for (uint32_t r = 1; r < cs; ++r)
      all_ok = all_ok && ld_shared_cluster_u32(map_to_cta(smem_addr(const_cast<int*>(failed)), r)) == 0;
    if (all_ok) {
      for (uint32_t r = 1; r < cs; ++r) {  // rank order = increasing k: a fixed sum order
        const uint32_t peer_row = map_to_cta(smem_addr(smem + n_local * L::PART_ROW), r);
#pragma unroll
        for (int i = 0; i < MN / 4; ++i) {
          const float4 v = ld_shared_cluster_f4(peer_row + 16 * i);
          acc[4 * i] += v.x;
          acc[4 * i + 1] += v.y;
          acc[4 * i + 2] += v.z;
          acc[4 * i + 3] += v.w;
        }
      }
      const int n = nt * BNT + n_local;
      if (n < p.N) {
#pragma unroll
        for (int m = 0; m < MN; ++m)
          if (m < p.M) store_out<OUT>(p.C, static_cast<int64_t>(m) * p.N + n, acc[m]);
      }
    }
  }
  if (threadIdx.x == 64) trace_mark(p.trace, TR_EPI_DONE);
  cluster_sync();  // peers keep their shared memory until rank 0 has read it
  if (threadIdx.x == 0) trace_mark(p.trace, TR_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace sptg
