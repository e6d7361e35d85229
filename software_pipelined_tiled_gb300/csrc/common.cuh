// common.cuh -- shared device-side pieces of the GEMM kernels: the bounded
// mbarrier wait, the output conversions and the tile raster.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace sptg {

// Output element kinds of the epilogue.
enum OutKind : int { OUT_F32 = 0, OUT_F16 = 1, OUT_BF16 = 2, OUT_S32 = 3 };

template <int OUT>
struct OutTraits {
  static constexpr int bytes = (OUT == OUT_F16 || OUT == OUT_BF16) ? 2 : 4;
};

// Codes or-ed into the device error word when a bounded wait runs out; the
// bit names the wait that gave up.
enum WaitSite : unsigned int {
  WAIT_PRODUCER_EMPTY = 1u << 0,
  WAIT_MMA_FULL = 1u << 1,
  WAIT_MMA_TMEM_EMPTY = 1u << 2,
  WAIT_EPI_TMEM_FULL = 1u << 3,
  WAIT_DRAIN = 1u << 4,
  WAIT_PLAN = 1u << 5,  // not a wait: a launch whose scratch plan does not fit
  WAIT_FIXUP_NOTE = 1u << 6,  // reduction warps: notice of a written partial tile
  WAIT_FIXUP_SLOT = 1u << 7,  // epilogue: a free notice slot
};

// Optional timeline: with a trace buffer, chosen threads stamp %globaltimer
// (ns) at these points into trace[cta * TR_SLOTS + event] (CTAs < TR_MAX_CTAS).
enum TraceEvent : int {
  TR_SETUP = 0,       // barriers, tensor memory and the dependency wait done
  TR_FIRST_LOAD = 1,  // producer issued its first copy
  TR_FIRST_DATA = 2,  // MMA issuer saw its first full stage
  TR_LAST_LOAD = 3,   // producer issued its last copy
  TR_LAST_MMA = 4,    // MMA issuer committed its last MMA
  TR_EPI_DONE = 5,    // epilogue finished its last tile (stores complete)
  TR_EXIT = 6,        // every role of the CTA (and of its pair) is done
  TR_FIXUP_DONE = 7,  // last split-K / stream-K reduction this CTA did, if any
  TR_SLOTS = 8,
  TR_MAX_CTAS = 1024,
  // detail of CTA 0: when the producer issued K-tile i and when the MMA
  // issuer found it full, for the first TR_DETAIL K-tiles of the CTA
  TR_DETAIL = 64,
  TR_DETAIL_BASE = TR_SLOTS * TR_MAX_CTAS,
  TR_WORDS = TR_DETAIL_BASE + 2 * TR_DETAIL
};

__device__ __forceinline__ void trace_mark(unsigned long long* trace, int event) {
  if (trace != nullptr && blockIdx.x < TR_MAX_CTAS)
    trace[blockIdx.x * TR_SLOTS + event] = global_timer_ns();
}

// role 0 = producer issued K-tile `it`, role 1 = MMA issuer found it full
__device__ __forceinline__ void trace_ktile(unsigned long long* trace, int role, uint32_t it) {
  if (trace != nullptr && blockIdx.x == 0 && it < TR_DETAIL)
    trace[TR_DETAIL_BASE + role * TR_DETAIL + it] = global_timer_ns();
}

// Everything a bounded wait needs: the limit, where to report, and the
// CTA-wide abort flag that lets the other roles stop early once one gave up.
struct WaitCtl {
  uint64_t timeout_ns;
  unsigned int* error_word;
  volatile int* abort_flag;  // in shared memory
};

// Waits for the phase of `bar` with parity `parity` to complete, for at most
// ctl.timeout_ns. On time-out it records `site` in the error word, raises the
// CTA's abort flag and returns false; it also returns false as soon as
// another role of the CTA has raised the flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl& ctl,
                                             unsigned int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 63u) == 0) {
      if (*ctl.abort_flag) return false;
      if (global_timer_ns() - t0 > ctl.timeout_ns) {
        *ctl.abort_flag = 1;
        atomicOr(ctl.error_word, site);
        return false;
      }
    }
  }
}

// Barrier over `nthreads` threads (named barrier `id`) that also returns the
// AND of every participant's `pred`, so a group of warps takes one decision.
__device__ __forceinline__ bool named_barrier_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.u32 pin, %1, 0;\n\t"
      "bar.red.and.pred pout, %2, %3, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Packs two fp32 values into one 32-bit word of the 16-bit output type
// (round to nearest even; `lo` lands at the lower address).
template <int OUT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (OUT == OUT_F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// One output element of the given kind from an fp32 value (round to nearest
// even for the 16-bit kinds).
template <int OUT>
__device__ __forceinline__ void store_out(void* C, int64_t idx, float v) {
  if constexpr (OUT == OUT_F32) {
    static_cast<float*>(C)[idx] = v;
  } else if constexpr (OUT == OUT_F16) {
    static_cast<__half*>(C)[idx] = __float2half_rn(v);
  } else {
    static_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(v);
  }
}

// Four consecutive outputs; idx is a multiple of 4 and the row pitch keeps
// the group inside one row (N is a multiple of 4 for every output type).
template <int OUT>
__device__ __forceinline__ void store_out4(void* C, int64_t idx, float4 v) {
  if constexpr (OUT == OUT_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(C) + idx) = v;
  } else {
    uint2 w = make_uint2(pack2<OUT>(v.x, v.y), pack2<OUT>(v.z, v.w));
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(C) + idx) = w;
  }
}

// Stores 8 (16-bit outputs) or 4 (fp32) consecutive outputs of one row from
// fp32 values; `n_valid` of them lie inside C (all when n_valid >= the group).
template <int OUT>
__device__ __forceinline__ void store_row_group(void* row_ptr, int col, const float* v,
                                                int n_valid) {
  if constexpr (OUT == OUT_F32) {
    float* dst = static_cast<float*>(row_ptr) + col;
    if (n_valid >= 4) {
      *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
      for (int i = 0; i < n_valid; ++i) dst[i] = v[i];
    }
  } else {
    uint16_t* dst = static_cast<uint16_t*>(row_ptr) + col;
    if (n_valid >= 8) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(pack2<OUT>(v[0], v[1]), pack2<OUT>(v[2], v[3]),
                                                  pack2<OUT>(v[4], v[5]), pack2<OUT>(v[6], v[7]));
    } else {
      for (int i = 0; i < n_valid; ++i) store_out<OUT>(dst, i, v[i]);
    }
  }
}

// Counts one arrival at a tile's split-K counter and returns whether it was the
// last of `count`. The 64-bit counter holds (call generation << 32 |
// arrivals): a value left by an earlier call (or by one that gave up) carries
// another generation and is replaced, so no call has to clear the counters
// first. The last arrival sets the counter back to 0 (a CUDA graph replays a
// call with the generation it was captured with, so the next replay must not
// find this call's count). The compare-and-swap retries only when another
// contributor got in first.
__device__ __forceinline__ int arrive_generation(unsigned long long* ctr, unsigned int gen,
                                                 int count, unsigned int* error_word) {
  unsigned long long cur = atomicAdd(ctr, 0ull);
  for (int tries = 0; tries < (1 << 20); ++tries) {
    const unsigned long long base =
        (static_cast<unsigned int>(cur >> 32) == gen) ? cur : (static_cast<unsigned long long>(gen) << 32);
    const unsigned long long want = base + 1;
    const unsigned long long prev = atomicCAS(ctr, cur, want);
    if (prev == cur) return static_cast<int>(want & 0xffffull) == count;
    cur = prev;
  }
  atomicOr(error_word, WAIT_PLAN);
  return 0;
}

// Tile index -> (m tile, n tile). Tiles are visited in column strips of
// `group` m-tiles so that CTAs running at the same time share A and B tiles
// in L2.
__device__ __forceinline__ void tile_coords(int tile, int num_m_tiles, int num_n_tiles, int group,
                                            int& m_tile, int& n_tile) {
  const int per_group = group * num_n_tiles;
  const int g = tile / per_group;
  const int first_m = g * group;
  const int rows = min(group, num_m_tiles - first_m);
  const int r = tile - g * per_group;
  m_tile = first_m + r % rows;
  n_tile = r / rows;
}

}  // namespace sptg
