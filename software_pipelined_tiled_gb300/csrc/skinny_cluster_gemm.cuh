// skinny_cluster_gemm.cuh -- the memory-bound skinny product (M <= 64) with
// its K split across the CTAs of a thread-block cluster (1, 2 or 4).
//
// Same arithmetic as skinny_gemm.cuh (swap-AB: D^T[n, m] = sum_k Bcm[n, k] *
// A[m, k], MMA M = 128 over N, MMA N = MN over the rows of A), but the work
// is cut along whole column tiles: one cluster of CS (1, 2 or 4) CTAs per
// 128-column tile, CTA rank r streaming the contiguous K-range
// [r*KT/CS, (r+1)*KT/CS). Each CTA accumulates its range in tensor memory.
// Then each rank finalises 128 / CS of the columns: it pushes its partial of
// the other ranks' columns straight into their receive buffers (distributed
// shared memory stores) and arrives on a barrier there, adds the CS partials
// of its own columns in rank order (a fixed order), converts, stages its
// output block in shared memory and writes it with one tensor-copy store.
//
// Compared with the stream-K kernel this needs no global scratch and no
// atomics: the reduction is one push between the SMs of a cluster. The grid
// is (column tiles x CS) CTAs, which the host uses when that fills the GPU.
#pragma once

#include "common.cuh"

namespace sptg {

struct SkinnyClusterParams {
  int M, N, K;
  int num_n_tiles, num_k_tiles;
  // 1: the maps are 3-D (64-element K-chunk, row, chunk index) and one copy
  // per operand moves a stage's KSUB chunks; 0: 2-D maps, one copy per chunk
  int load3d;
  unsigned int* error_word;
  uint64_t timeout_ns;
  int inject_stall;
  unsigned long long* trace;
};

// One ring stage holds KSUB consecutive 64-wide K-chunks of B^T (128 rows)
// and of A (MN rows), each chunk its own 128-byte-swizzled sub-tile.
template <int MN, int STAGES, int OBYTES, int KSUB = 1>
struct SkinnyClusterLayout {
  static constexpr int BNT = 128;
  static constexpr int BK = 64;
  static constexpr int SUB_BT = BNT * BK * 2;
  static constexpr int SUB_A = MN * BK * 2;
  static constexpr int BT_STAGE = KSUB * SUB_BT;
  static constexpr int A_STAGE = KSUB * SUB_A;
  static constexpr int STAGE = BT_STAGE + A_STAGE;
  // receive buffer for the other ranks' partials: for each of the columns
  // this rank finalises, a row of MN floats from each other rank (at most
  // 3 x 32 columns, cluster of 4), plus 16 bytes per row so that 16-byte
  // accesses of 8 consecutive rows hit 8 distinct bank groups
  static constexpr int PART_ROW = MN * 4 + 16;
  // Largest cluster the receive buffer is sized for: 4 (3 x 32 columns from
  // the other ranks) for MN = 64; 2 (64 columns from the peer) for wider MN,
  // whose partial rows are twice as long.
  static constexpr int MAX_CS = MN <= 64 ? 4 : 2;
  // rows received at most: 1 x 64 (cluster of 2) or 3 x 32 (cluster of 4)
  static constexpr int RECV_ROWS = MAX_CS == 4 ? 96 : 64;
  // output staging (reuses the receive buffer once it has been read): MN rows
  // of up to 128 outputs, the layout of C
  static constexpr int OUT_BYTES = MN * BNT * OBYTES;
  static constexpr int PART_BYTES =
      RECV_ROWS * PART_ROW > OUT_BYTES ? RECV_ROWS * PART_ROW : OUT_BYTES;
  static constexpr int OFF_PART = STAGES * STAGE;
  static constexpr int OFF_BAR = OFF_PART + PART_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 3;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TMEM_COLS = MN <= 32 ? 32 : MN <= 64 ? 64 : 128;
  static_assert(OFF_PART % 1024 == 0, "receive buffer alignment");
  static_assert(PART_BYTES % 16 == 0, "barrier alignment");
  static_assert(MN % 32 == 0 && MN >= 32 && MN <= 128, "MN must be 32, 64, 96 or 128");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
};

// Deepest ring next to the receive buffer within the 227 KB budget.
template <int MN, int OBYTES, int KSUB = 1>
constexpr int skinny_cluster_stages() {
  using L1 = SkinnyClusterLayout<MN, 1, OBYTES, KSUB>;
  return (232448 - 1024 - L1::PART_BYTES - 512) / L1::STAGE;
}

// 16-byte store into the shared memory of a CTA of the cluster.
__device__ __forceinline__ void st_shared_cluster_f4(uint32_t cluster_addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}

template <int MN, int STAGES, bool IN_BF16, int OUT, int KSUB = 1>
__global__ void __launch_bounds__(192, 1)
    skinny_cluster_gemm_kernel(const __grid_constant__ CUtensorMap tmBt,
                               const __grid_constant__ CUtensorMap tmA,
                               const __grid_constant__ CUtensorMap tmC,
                               const SkinnyClusterParams p) {
  constexpr int OBYTES = OutTraits<OUT>::bytes;
  using L = SkinnyClusterLayout<MN, STAGES, OBYTES, KSUB>;
  constexpr int BNT = L::BNT, BK = L::BK;
  constexpr uint32_t IDESC = idesc_f16_f32acc(IN_BF16, BNT, MN);
  static_assert(OUT != OUT_S32, "float outputs only");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  uint8_t* part = smem + L::OFF_PART;
  auto stage_bt = [&](int s) { return sbase + s * L::STAGE; };
  auto stage_a = [&](int s) { return sbase + s * L::STAGE + L::BT_STAGE; };
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * STAGES);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 1);
  const uint32_t recv_bar = bar0 + 8u * (2 * STAGES + 2);  // the peer's half partial is in
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cs = cluster_nctarank();  // 1, 2 or 4
  if (cs > static_cast<uint32_t>(L::MAX_CS)) {
    // the receive buffer has no room for this many ranks: report, touch
    // nothing (every CTA of the cluster leaves here, before any barrier)
    if (threadIdx.x == 0) atomicOr(p.error_word, WAIT_PLAN);
    return;
  }
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
    // one arrival per pushing thread of the other ranks: (cs - 1) x 128 / cs
    mbar_init(recv_bar, cs > 1 ? static_cast<int>((cs - 1) * (128 / cs)) : 1);
    *abort_flag = 0;
    *failed = 0;
    fence_mbar_init();
    prefetch_tensor_map(&tmBt);
    prefetch_tensor_map(&tmA);
    prefetch_tensor_map(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  if (cs > 1)
    cluster_sync();  // rank 0's receive barrier exists before the peer can arrive on it
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Warm L2 with this CTA's first stages while the previous kernel drains.
  // L2 is where writes become coherent, so this is safe even if that kernel
  // writes these operands: the loads proper come after the dependency wait.
  // (every lane of the producer warp holds the policies: the lane elected
  // to issue the copies need not be lane 0)
  uint64_t pol_stream = 0, pol_keep = 0;
  if (warp == 0) {
    pol_stream = policy_evict_first();  // B is read once
    pol_keep = policy_evict_last();     // A is read by every CTA
    for (int kt = kt0; lane == 0 && kt < min(kt1, kt0 + STAGES); ++kt) {
      if (p.load3d) {
        tma_prefetch_l2_3d(&tmBt, 0, nt * BNT, kt * KSUB);
        tma_prefetch_l2_3d(&tmA, 0, 0, kt * KSUB);
      } else {
#pragma unroll
        for (int j = 0; j < KSUB; ++j) {
          tma_prefetch_l2_2d(&tmBt, (kt * KSUB + j) * BK, nt * BNT);
          tma_prefetch_l2_2d(&tmA, (kt * KSUB + j) * BK, 0);
        }
      }
    }
  }
  grid_dependency_wait();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_SETUP);

  const WaitCtl ctl{p.timeout_ns, p.error_word, abort_flag};

  // Producer and MMA issuer run as whole warps; one elected lane issues the
  // copies, MMAs and commits (a lane alone in its warp pays a large fixed
  // cost per loop trip).
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    {  // the whole warp
      const bool leader = elect_one_sync();
      int issued_round[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_round[s] = -1;
      bool ok = true;
      uint32_t it = 0;
      for (int kt = kt0; kt < kt1; ++kt, ++it) {
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        // in the first round every stage is free: no wait
        if (round > 0 && !__all_sync(0xffffffffu, wait_bounded(empty_bar(s), (round & 1u) ^ 1u, ctl,
                                                                WAIT_PRODUCER_EMPTY))) {
          ok = false;
          break;
        }
        if (p.inject_stall && it == 1) continue;  // test hook: this stage never fills
        issued_round[s] = static_cast<int>(round);
        if (!leader) continue;
        mbar_arrive_expect_tx(full_bar(s), L::STAGE);
        if (p.load3d) {
          // one copy per operand: KSUB chunks of 64 K-elements, each landing
          // as its own 128-byte-swizzled sub-tile
          tma_load_3d(stage_bt(s), &tmBt, full_bar(s), 0, nt * BNT, kt * KSUB, pol_stream);
          tma_load_3d(stage_a(s), &tmA, full_bar(s), 0, 0, kt * KSUB, pol_keep);
        } else {
#pragma unroll
          for (int j = 0; j < KSUB; ++j) {
            tma_load_2d(stage_bt(s) + j * L::SUB_BT, &tmBt, full_bar(s), (kt * KSUB + j) * BK,
                        nt * BNT, pol_stream);
            tma_load_2d(stage_a(s) + j * L::SUB_A, &tmA, full_bar(s), (kt * KSUB + j) * BK, 0,
                        pol_keep);
          }
        }
        if (it == 0) trace_mark(p.trace, TR_FIRST_LOAD);
        trace_ktile(p.trace, 0, it);
      }
      if (leader) trace_mark(p.trace, TR_LAST_LOAD);
      grid_launch_dependents();
      if (!ok) {
        if (leader) *failed = 1;
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
      uint32_t it = 0;
      for (int kt = kt0; kt < kt1; ++kt, ++it) {
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        if (!__all_sync(0xffffffffu, wait_bounded(full_bar(s), round & 1u, ctl, WAIT_MMA_FULL))) {
          if (leader) *failed = 1;
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
              mma_f16(tmem_base, sdesc_k_major_sw128(stage_bt(s) + j * L::SUB_BT + 32 * k),
                      sdesc_k_major_sw128(stage_a(s) + j * L::SUB_A + 32 * k), IDESC,
                      (kt > kt0 || j > 0 || k > 0) ? 1u : 0u);
            }
          }
          mma_commit(empty_bar(s));
        }
        __syncwarp();
      }
      if (leader) {
        trace_mark(p.trace, TR_LAST_MMA);
        mma_commit(tfull_bar);  // also arrives when no MMA was issued (empty K-range)
        mma_commit(drain_bar);
      }
      __syncwarp();
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < ctl.timeout_ns) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warps 2-5: each lane owns one output column (a row of D^T) and reads its
    // MN fp32 values out of tensor memory
    const int q = warp & 3;
    const int n_local = 32 * q + lane;
    float acc[MN];
    const bool done = __all_sync(0xffffffffu, wait_bounded(tfull_bar, 0, ctl, WAIT_EPI_TMEM_FULL));
    const bool mine_ok = __all_sync(0xffffffffu, done && !*failed);
    if (done) {
      tc_fence_after();
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
#pragma unroll
      for (int cb = 0; cb < MN / 32; ++cb) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_lane + 32 * cb, r);
        tmem_wait_ld_regs(r);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          acc[32 * cb + i] = (kt1 > kt0) ? __uint_as_float(r[i]) : 0.0f;
      }
    }
    // With cs ranks each finalises 128 / cs of the columns (rank r the block
    // r * 128 / cs ..): a warp whose 32 columns belong to another rank pushes
    // its partial into that rank's receive buffer (distributed shared memory
    // stores, one slot per sending rank) and arrives on its barrier (release,
    // cluster scope: each thread covers its own stores); all ranks' blocks
    // move at once. A rank that failed does not arrive, and the owner's
    // bounded wait gives up.
    const int cpr = BNT / static_cast<int>(cs);  // columns each rank finalises
    const int owner = (32 * q) / cpr;              // cs <= 4: whole warps
    const bool keep = owner == static_cast<int>(rank);
    const int col = n_local - owner * cpr;         // column within the owner's block
    const int keep_threads = cpr;
    if (!keep) {
      if (mine_ok) {
        const int slot = static_cast<int>(rank) < owner ? static_cast<int>(rank)
                                                        : static_cast<int>(rank) - 1;
        const uint32_t dst = map_to_cta(smem_addr(part + (slot * cpr + col) * L::PART_ROW),
                                        static_cast<uint32_t>(owner));
#pragma unroll
        for (int i = 0; i < MN / 4; ++i)
          st_shared_cluster_f4(dst + 16 * i,
                               make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]));
        mbar_arrive_cluster(map_to_cta(recv_bar, static_cast<uint32_t>(owner)));
      }
    } else {
      bool ok = mine_ok;
      if (cs > 1) {
        ok = named_barrier_and(1, keep_threads,
                               ok && wait_bounded(recv_bar, 0, ctl, WAIT_EPI_TMEM_FULL));
        if (ok && cs == 2) {
          // two partials: their fp32 sum is the same in either order; up to
          // 16 loads in flight, then the adds
          const uint8_t* row = part + col * L::PART_ROW;
          constexpr int G2 = MN / 4 < 16 ? MN / 4 : 16;
#pragma unroll
          for (int i0 = 0; i0 < MN / 4; i0 += G2) {
            float4 v[G2];
#pragma unroll
            for (int i = 0; i < G2; ++i)
              v[i] = *reinterpret_cast<const float4*>(row + 16 * (i0 + i));
#pragma unroll
            for (int i = 0; i < G2; ++i) {
              acc[4 * (i0 + i)] += v[i].x;
              acc[4 * (i0 + i) + 1] += v[i].y;
              acc[4 * (i0 + i) + 2] += v[i].z;
              acc[4 * (i0 + i) + 3] += v[i].w;
            }
          }
        } else if (ok) {
          // four partials added in rank order (= increasing k): a fixed
          // order; the three received ones are loaded 4 chunks at a time
          const int k = static_cast<int>(rank);
#pragma unroll
          for (int i0 = 0; i0 < MN / 4; i0 += 4) {
            float4 t[3][4];
#pragma unroll
            for (int sl = 0; sl < 3; ++sl)
#pragma unroll
              for (int j = 0; j < 4; ++j)
                t[sl][j] = *reinterpret_cast<const float4*>(
                    part + (sl * cpr + col) * L::PART_ROW + 16 * (i0 + j));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = i0 + j;
              const float4 own = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
              // rank r's partial: this rank's own, or receive slot r (r < k) / r - 1
              const float4 p0 = k == 0 ? own : t[0][j];
              const float4 p1 = k == 1 ? own : (k > 1 ? t[1][j] : t[0][j]);
              const float4 p2 = k == 2 ? own : (k > 2 ? t[2][j] : t[1][j]);
              const float4 p3 = k == 3 ? own : t[2][j];
              float4 s4 = p0;
              s4.x += p1.x;
              s4.y += p1.y;
              s4.z += p1.z;
              s4.w += p1.w;
              s4.x += p2.x;
              s4.y += p2.y;
              s4.z += p2.z;
              s4.w += p2.w;
              s4.x += p3.x;
              s4.y += p3.y;
              s4.z += p3.z;
              s4.w += p3.w;
              acc[4 * i] = s4.x;
              acc[4 * i + 1] = s4.y;
              acc[4 * i + 2] = s4.z;
              acc[4 * i + 3] = s4.w;
            }
          }
        }
        named_barrier_sync(1, keep_threads);  // the receive buffer is read: reuse it for staging
      } else {
        ok = named_barrier_and(1, keep_threads, ok);
      }
      if (ok) {
        // stage the kept MN x (128 / cs) block of C (row m holds consecutive
        // outputs) and store it with one tensor copy; rows past M and
        // columns past N clip
        const int width = BNT / static_cast<int>(cs);
        uint8_t* stage = part;
#pragma unroll
        for (int m = 0; m < MN; ++m) {
          if constexpr (OBYTES == 4) {
            reinterpret_cast<float*>(stage)[m * width + col] = acc[m];
          } else if constexpr (OUT == OUT_F16) {
            reinterpret_cast<__half*>(stage)[m * width + col] = __float2half_rn(acc[m]);
          } else {
            reinterpret_cast<__nv_bfloat16*>(stage)[m * width + col] = __float2bfloat16_rn(acc[m]);
          }
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, keep_threads);
        const int x0 = nt * BNT + static_cast<int>(rank) * cpr;
        if (col == 0 && x0 < p.N) {
          tma_store_2d(&tmC, smem_addr(stage), x0, 0);
          bulk_commit_group();
          bulk_wait_group_read<0>();  // the staging may go once the copy has read it
        }
      }
      if (col == 0) trace_mark(p.trace, TR_EPI_DONE);
    }
  }

  tc_fence_before();
  if (cs > 1)
    cluster_sync();  // the peer's pushes have landed before either CTA leaves
  else
    __syncthreads();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace sptg
