// stream_scale.cuh -- the pipelined ring on its own: out[i] = alpha * in[i]
// over a 1-D binary32 array.
//
// The GB300 form of the minimal working example of "Hiding Memory Latency in
// CUDA: Asynchronous Loads and Software Pipelines" (section 8): a multi-stage
// shared-memory ring whose stages the copy engine fills ahead of the threads
// that consume them. With no arithmetic worth the name, the kernel measures
// the ring itself against the HBM roofline.
//
//   warp 0     producer: for each 32 KB tile of this CTA, waits until its
//              stage is free, then one bulk copy (cp.async.bulk) global ->
//              shared completes the stage's "full" barrier by byte count.
//   warps 1-4  consumers: wait for "full", multiply every element by alpha
//              (one binary32 rounding), write 16-byte vectors to global
//              memory, and release the stage on its "empty" barrier.
//
// The persistent grid takes tiles round robin. The last n % 4 elements (past
// the 16-byte vector prefix the bulk copies cover) are done with plain loads
// by one thread.
#pragma once

#include "common.cuh"

namespace sptg {

struct StreamParams {
  const float* in;
  float* out;
  float alpha;
  int64_t n;          // elements
  int64_t n_vec;      // leading elements the bulk path covers (a multiple of 4)
  int64_t num_tiles;  // ceil(n_vec * 4 / TILE_BYTES)
  unsigned int* error_word;
  uint64_t timeout_ns;
  int inject_stall;
  unsigned long long* trace;
};

template <int TILE_BYTES, int STAGES>
struct StreamLayout {
  static constexpr int OFF_BAR = STAGES * TILE_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 2 * STAGES * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 128;
  static_assert(TILE_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
};

// 1-D bulk copy global -> shared completing `bytes` on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

template <int TILE_BYTES, int STAGES>
__global__ void __launch_bounds__(160, 1) stream_scale_kernel(const StreamParams p) {
  using L = StreamLayout<TILE_BYTES, STAGES>;
  constexpr int F4_PER_TILE = TILE_BYTES / 16;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t vec_bytes = p.n_vec * 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 4);  // one arrival per consumer warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_SETUP);
  const WaitCtl ctl{p.timeout_ns, p.error_word, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();  // every byte is read once
      int issued_round[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_round[s] = -1;
      bool ok = true;
      uint32_t it = 0;
      for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        if (!wait_bounded(empty_bar(s), (round & 1u) ^ 1u, ctl, WAIT_PRODUCER_EMPTY)) {
          ok = false;
          break;
        }
        if (p.inject_stall && it == 1) continue;  // test hook: this stage never fills
        const int64_t off = t * TILE_BYTES;
        const int64_t left = vec_bytes - off;
        const uint32_t bytes = static_cast<uint32_t>(left < TILE_BYTES ? left : TILE_BYTES);
        mbar_arrive_expect_tx(full_bar(s), bytes);
        bulk_load(sbase + s * TILE_BYTES, reinterpret_cast<const uint8_t*>(p.in) + off, bytes,
                  full_bar(s), pol);
        issued_round[s] = static_cast<int>(round);
        if (it == 0) trace_mark(p.trace, TR_FIRST_LOAD);
        trace_ktile(p.trace, 0, it);
      }
      trace_mark(p.trace, TR_LAST_LOAD);
      grid_launch_dependents();
      if (!ok) {
        for (int s = 0; s < STAGES; ++s) {
          if (issued_round[s] < 0) continue;
          const uint32_t par = static_cast<uint32_t>(issued_round[s]) & 1u;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(full_bar(s), par) && global_timer_ns() - t0 < ctl.timeout_ns) {
          }
        }
      }
    } else if (lane == 1 && blockIdx.x == 0) {
      // the ragged end past the 16-byte vector prefix
      for (int64_t i = p.n_vec; i < p.n; ++i) p.out[i] = __fmul_rn(p.alpha, p.in[i]);
    }
  } else {
    // ----------------------------------------------------------- consumers
    const int tid = threadIdx.x - 32;  // 0..127
    uint32_t it = 0;
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
      const int s = it % STAGES;
      const uint32_t round = it / STAGES;
      const bool ok =
          __all_sync(0xffffffffu, wait_bounded(full_bar(s), round & 1u, ctl, WAIT_MMA_FULL));
      if (!ok) break;
      if (it == 0 && tid == 0) trace_mark(p.trace, TR_FIRST_DATA);
      if (tid == 0) trace_ktile(p.trace, 1, it);
      const int64_t off = t * TILE_BYTES;
      const int64_t left = vec_bytes - off;
      const int f4 = static_cast<int>((left < TILE_BYTES ? left : TILE_BYTES) / 16);
      const float4* src = reinterpret_cast<const float4*>(smem + s * TILE_BYTES);
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(p.out) + off);
#pragma unroll 4
      for (int f = tid; f < F4_PER_TILE; f += 128) {
        if (f < f4) {
          float4 v = src[f];
          v.x = __fmul_rn(p.alpha, v.x);
          v.y = __fmul_rn(p.alpha, v.y);
          v.z = __fmul_rn(p.alpha, v.z);
          v.w = __fmul_rn(p.alpha, v.w);
          __stcs(dst + f, v);  // streamed: not read again
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));  // this warp is done reading the stage
    }
    if (tid == 0) trace_mark(p.trace, TR_EPI_DONE);
  }
  __syncthreads();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_EXIT);
}

}  // namespace sptg
