// square_gemm.cuh -- the software-pipelined tiled GEMM for sm_103a.
//
// C (M x N, row-major) = A (M x K, row-major) * B (K x N, column-major), i.e.
// both operands K-major.  One CTA per SM, persistent over output tiles of
// 128 x BN, with three roles in warp specialisation:
//
//   warp 0     producer: for every K-tile, waits until its ring stage is free
//              (the stage's "empty" mbarrier), then has the tensor-copy engine
//              load the A tile (128 x 64) and the B tile (BN x 64) into it;
//              the copy completes the stage's "full" mbarrier by byte count.
//   warp 1     MMA issuer: waits for "full", issues four tcgen05.mma (K = 16
//              each) into a tensor-memory accumulator, then tcgen05.commit
//              arrives on "empty" once those MMAs have read the stage.
//   warps 2-5  epilogue: wait until an accumulator is complete, read it from
//              tensor memory (each warp owns 32 of the 128 lanes), convert,
//              stage 32-row blocks in shared memory and store them with the
//              tensor-copy engine; then hand the accumulator back.
//   warps 6-9  stream-K reduction (below); when no tile is cut, they store
//              half of the CTA's last tile instead.
//   (INT_EXACT: 12 warps, 2-9 epilogue and 10-11 reduction, see below.)
//
// This is the producer/consumer ring of "Hiding Memory Latency in CUDA:
// Asynchronous Loads and Software Pipelines" (sections 5, 6 and 11): stage =
// k-tile mod STAGES, separate read and write positions each with its own
// wrap, "producer never overwrites an in-use stage" enforced by the empty
// barrier and "consumer never reads an incomplete stage" by the full barrier.
// The prologue is the producer running up to STAGES tiles ahead, the steady
// state is the overlap, and the drain is the final commit of a tile's last
// MMA ("Pipeline GPU Kernel", Step 3).  The register-fragment pipeline of the
// Ampere design (section 7) has no counterpart: tcgen05.mma reads both
// operands from shared memory and accumulates in tensor memory; its place is
// taken by two accumulators, so the epilogue of one tile overlaps the K-loop
// of the next.
//
// PAIR mode runs the same roles on a cluster of two CTAs (two SMs) with the
// 2-SM tensor-core instruction (tcgen05.mma.cta_group::2): a tile is 256 x BN,
// each CTA loads its own 128 rows of A and its own BN/2 rows of B, the leader
// CTA's MMA warp multiplies the whole 256 x BN tile reading both CTAs' shared
// memory, and each CTA's tensor memory receives its 128 rows of the result.
// Per SM this halves the B traffic of a 128 x BN tile. The copies of both
// CTAs complete on the leader's "full" barrier; the leader's commits arrive
// on both CTAs' "empty" and "tmem_full" barriers; both CTAs' epilogue warps
// release the accumulator on the leader's "tmem_empty" barrier.
//
// A pair tile may be 512 wide (BN = 512): each K-step is then two 256-column
// MMAs into the two halves of one 512-column accumulator (tensor memory holds
// no second one, so that tile's epilogue does not overlap the next K-loop),
// and each CTA copies its 128 rows of each half's B. Per FLOP this moves a
// quarter fewer operand bytes than 256-wide tiles, which pays on long
// K-loops.
//
// Work schedule (stream-K + data-parallel). With T tiles and W workers (CTAs,
// or CTA pairs), T mod W tiles would leave a last round with most SMs idle.
// Those tiles are instead cut along K into one contiguous range of
// (tile, K-tile) units per worker and done first; the remaining T - T mod W
// tiles follow round robin, every worker the same number. A worker whose range
// covers only part of a tile's K writes its fp32 (int32 in INT_EXACT mode)
// partial tile to scratch and counts its arrival (an atomic counter tagged
// with the call's generation). The contributor whose arrival completes the
// count adds up all partials of its rows in contributor order (= increasing
// k, a fixed order, so the result does not depend on which one came last) and
// writes C; the others go on at once. No CTA ever waits for another, so the
// schedule needs no co-residency of the grid: a CTA that becomes resident
// only after others have finished (the GPU shared with other work) still
// completes the product. The epilogue writes the partial, counts the arrival
// and posts a notice; four reduction warps of their own take the sum, so the
// accumulators keep draining and the K-loop of the next tiles never waits
// for a reduction.
//
// INT_EXACT mode computes an int8 product exactly on the fp16 tensor path: the
// inputs are int8 values held as binary16 (exact), every product is an integer
// of magnitude <= 2^14 and every partial sum of at most 1024 products is an
// integer of magnitude <= 2^24, which fp32 holds exactly.  The K-loop is cut
// into chunks of 1024 products, each accumulated in one of the two
// accumulators in turn; eight epilogue warps convert each chunk to int32 and
// add it to a running sum in their registers (two warps per lane quadrant,
// half of the columns each), so tensor memory holds only the two accumulators
// and int8 takes the float tile widths up to 256.
#pragma once

#include "common.cuh"

namespace sptg {

// Threads of a square-kernel CTA: producer, MMA, 4 epilogue, 4 reduction
// warps; in exact-integer mode producer, MMA, 8 epilogue, 2 reduction warps.
constexpr int SQUARE_THREADS = 320;
constexpr int SQUARE_THREADS_INT = 384;
// first thread and number of threads of the stream-K reduction warps
template <bool INT_EXACT>
struct ReductionWarps {
  static constexpr int FIRST = INT_EXACT ? 320 : 192;
  static constexpr int COUNT = INT_EXACT ? 64 : 128;
};

struct SquareParams {
  int M, N, K;
  void* C_out;   // C, for the stream-K reductions' direct stores
  int64_t ldc;   // elements between rows of C
  int num_m_tiles, num_n_tiles, num_k_tiles;
  int k_tiles_per_chunk;  // accumulation chunk (all K-tiles unless INT_EXACT)
  int group_m;            // raster strip height in m-tiles
  // stream-K part: the last sk_tiles tile indices, cut into sk_units =
  // sk_tiles * num_k_tiles units over the first sk_workers workers
  int sk_tiles;
  int sk_workers;
  int max_contrib;              // partial slots per (tile, CTA of the pair)
  // [sk_tile][rank][contributor][128 x BN] 32-bit, each 128 x BN block as
  // 16-byte groups in the order [32-column block][4-column group][row]
  uint32_t* partials;
  // [sk_tile * 2 + rank]: generation << 32 | arrivals (0 between calls)
  unsigned long long* counters;
  unsigned int generation;
  unsigned int* error_word;
  uint64_t timeout_ns;
  int inject_stall;  // test hook: withhold the load of the second K-tile
  unsigned long long* trace;  // optional timeline (see TraceEvent), or null
  int b_once;   // 1: every tile of B is read by one output tile only (one tile row)
};

template <int N>
struct IntConst {
  static constexpr int value = N;
};

// Exact-integer epilogue: reads NBLK blocks of 32 fp32 columns of this
// thread's accumulator row (exact integers, |v| <= 2^24), converts them to
// int32 and assigns (FIRST) or adds them to the running sums (as unsigned
// words: the int32 sum wraps modulo 2^32). 16 columns per tensor-memory load.
template <bool FIRST, int NBLK>
__device__ __forceinline__ void int_chunk_sums(uint32_t (&sum)[32 * NBLK], uint32_t t_acc) {
#pragma unroll
  for (int j = 0; j < 2 * NBLK; ++j) {
    uint32_t t[16];
    tmem_ld_32x32b_x16(t_acc + 16 * j, t);
    tmem_wait_ld_regs16(t);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t x = static_cast<uint32_t>(__float2int_rn(__uint_as_float(t[e])));
      if constexpr (FIRST)
        sum[16 * j + e] = x;
      else
        sum[16 * j + e] += x;
    }
  }
}

// One piece of a worker's work: K-tiles [kt0, kt1) of tile `tile`. A partial
// segment (not all of K) belongs to stream-K tile `sk`, whose contributors are
// workers c_first .. c_first + count - 1; this worker is contributor j.
struct Segment {
  int tile, kt0, kt1;
  bool partial;
  int sk, j, count;
};

// The worker holding stream-K unit u: ranges are [w*U/G, (w+1)*U/G).
__device__ __forceinline__ int sk_worker_of(int64_t u, int G, int64_t U) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

// The i-th segment of `worker` (false past the last). Stream-K segments come
// first, then the data-parallel tiles.
__device__ __forceinline__ bool square_segment(const SquareParams& p, int worker, int workers,
                                               int i, Segment& seg) {
  const int KT = p.num_k_tiles;
  const int T = p.num_m_tiles * p.num_n_tiles;
  const int T_dp = T - p.sk_tiles;
  int n_sk = 0;
  int64_t u0 = 0, u1 = 0;
  const int64_t U = static_cast<int64_t>(p.sk_tiles) * KT;
  if (p.sk_tiles > 0 && worker < p.sk_workers) {
    u0 = static_cast<int64_t>(worker) * U / p.sk_workers;
    u1 = static_cast<int64_t>(worker + 1) * U / p.sk_workers;
    if (u1 > u0) n_sk = static_cast<int>((u1 - 1) / KT - u0 / KT + 1);
  }
  if (i < n_sk) {
    const int sk = static_cast<int>(u0 / KT) + i;
    const int64_t lo = max(u0, static_cast<int64_t>(sk) * KT);
    const int64_t hi = min(u1, static_cast<int64_t>(sk + 1) * KT);
    seg.tile = T_dp + sk;
    seg.kt0 = static_cast<int>(lo - static_cast<int64_t>(sk) * KT);
    seg.kt1 = static_cast<int>(hi - static_cast<int64_t>(sk) * KT);
    seg.partial = !(seg.kt0 == 0 && seg.kt1 == KT);
    seg.sk = sk;
    const int c_first = sk_worker_of(static_cast<int64_t>(sk) * KT, p.sk_workers, U);
    const int c_last = sk_worker_of(static_cast<int64_t>(sk + 1) * KT - 1, p.sk_workers, U);
    seg.j = worker - c_first;
    seg.count = c_last - c_first + 1;
    return true;
  }
  const int tile = worker + (i - n_sk) * workers;
  if (tile >= T_dp) return false;
  seg.tile = tile;
  seg.kt0 = 0;
  seg.kt1 = KT;
  seg.partial = false;
  seg.sk = seg.j = seg.count = 0;
  return true;
}

// Epilogue staging per warp: buffers of one block of 32 rows x 32 outputs,
// used in turn, so that the tensor-copy stores of the last blocks are still
// reading while the next ones are written. The ring is sized against the
// minimum (two 4 KB buffers for 4-byte outputs, one 2 KB buffer for 16-bit
// outputs, which leaves room for one more stage in the 224-wide pair
// kernels); whatever the ring leaves over goes to more buffers, up to four.
// The exact-integer epilogue has twice the warps (eight) and one 4 KB buffer
// each at least: the same 32 KB.
// Tiles 512 wide (one accumulator, never cut along K) also drain with eight
// warps, the reduction warps storing half of every tile's blocks: their
// epilogue is not overlapped with a K-loop.
template <int OBYTES, bool INT_EXACT = false, bool WIDE = false>
struct EpiStaging {
  static constexpr int WARPS = (INT_EXACT || WIDE) ? 8 : 4;
  static constexpr int BUF = 32 * 32 * OBYTES;
  static constexpr int MIN_NBUF = (INT_EXACT || WIDE) ? 1 : OBYTES == 4 ? 2 : 1;
  static constexpr int MAX_NBUF = 4;
};

template <int BN, int STAGES, bool INT_EXACT, bool PAIR, int OBYTES = 4, int KCH = 1>
struct SquareLayout {
  static constexpr int BM = 128;         // rows of A (and of C) per CTA
  static constexpr int TILE_M = PAIR ? 256 : 128;
  static constexpr int BN_CTA = PAIR ? BN / 2 : BN;  // rows of B per CTA
  static constexpr int BK = 64;  // 64 16-bit elements = one 128-byte swizzle row
  // A ring stage holds KCH consecutive 64-wide K-chunks of each operand
  // (chunk j of A at j * A_CHUNK, of B at j * B_CHUNK within the stage)
  static constexpr int A_CHUNK = BM * BK * 2;
  static constexpr int B_CHUNK = BN_CTA * BK * 2;
  static constexpr int A_STAGE = KCH * A_CHUNK;
  static constexpr int B_STAGE = KCH * B_CHUNK;
  using Epi = EpiStaging<OBYTES, INT_EXACT, (BN > 256)>;
  static constexpr int EPI_WARPS = Epi::WARPS;
  static constexpr int EPI_BUF = Epi::BUF;
  static constexpr int RING_BYTES = STAGES * (A_STAGE + B_STAGE);
  static constexpr bool staging_fits(int nbuf) {
    return RING_BYTES + EPI_WARPS * nbuf * EPI_BUF + 256 + 1024 <= 232448;
  }
  static constexpr int EPI_NBUF = staging_fits(Epi::MAX_NBUF)                   ? Epi::MAX_NBUF
                                  : (staging_fits(2) && Epi::MIN_NBUF <= 2) ? 2
                                                                            : Epi::MIN_NBUF;
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_NBUF * EPI_BUF;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
  static constexpr int OFF_EPI = OFF_B + STAGES * B_STAGE;
  static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 1 + 4;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int BYTES_USED = OFF_MISC + 40;
  static constexpr int SMEM_BYTES = BYTES_USED + 1024;  // slack to align the base to 1024
  // tiles wider than one MMA (BN = 512: two 256-column MMAs per K-step) keep
  // a single accumulator: 512 columns fill tensor memory
  static constexpr int NACC = BN > 256 ? 1 : 2;
  // The epilogue moves whole blocks of 32 columns; a float tile may end in a
  // block of 16 (BN = 112, 144, ..., 240), stored straight from registers.
  static constexpr int NB_FULL = BN / 32;
  static constexpr bool HALF_BLOCK = BN % 32 != 0;
  // tensor-memory columns from one accumulator to the next (a multiple of 32)
  static constexpr int ACC_COLS = (BN + 31) / 32 * 32;
  static constexpr int TMEM_NEEDED = NACC == 2 ? 2 * ACC_COLS : BN;
  static constexpr int TMEM_COLS = TMEM_NEEDED <= 32    ? 32
                                   : TMEM_NEEDED <= 64  ? 64
                                   : TMEM_NEEDED <= 128 ? 128
                                   : TMEM_NEEDED <= 256 ? 256
                                                        : 512;
  // The CTA's last tile (no tile cut along K, two accumulators): the epilogue
  // warps store its first LAST_NB0 32-column blocks, the otherwise idle
  // reduction warps the rest, staged in the ring (free by then), when the
  // ring holds their buffers.
  // (a last 16-column block stays with the epilogue warps)
  static constexpr int LAST_NB0 = (NB_FULL + 1) / 2;
  static constexpr bool LAST_SPLIT =
      !INT_EXACT && NACC == 2 && NB_FULL > 1 && RING_BYTES >= 4 * (NB_FULL - LAST_NB0) * EPI_BUF;
  // exact-integer epilogue: 32-column blocks of the first and second warp of a
  // lane quadrant
  static constexpr int INT_NB0 = (BN + 63) / 64;
  static constexpr int INT_NB1 = BN / 32 - INT_NB0;
  // bytes that complete one stage's "full" barrier (both CTAs' copies in PAIR mode)
  static constexpr uint32_t STAGE_TX = (PAIR ? 2 : 1) * (A_STAGE + B_STAGE);
  static_assert(TMEM_NEEDED <= 512, "accumulators exceed tensor memory");
  static_assert((BN % 32 == 0 && BN >= 32 && BN <= 256) ||
                    (BN % 16 == 0 && BN >= 48 && BN <= 256 && !INT_EXACT) ||
                    (BN == 512 && PAIR && !INT_EXACT),
                "BN must be a multiple of 32 in [32, 256], of 16 for float tiles, or 512 for "
                "float CTA pairs");
  static_assert(!INT_EXACT || (BN >= 64 && BN <= 256),
                "the exact-integer epilogue keeps at most 128 columns per thread");
  // the 2-SM MMA with M = 256 takes N in steps of 16: half a step per CTA
  static_assert(!PAIR || BN_CTA % 8 == 0, "each CTA's B rows must be a multiple of 8");
  static_assert(STAGES >= 1, "at least one stage");
  static_assert(KCH == 1 || (KCH == 2 && !INT_EXACT && BN <= 256),
                "two K-chunks per stage: float tiles up to 256 wide");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget exceeded");
  static_assert(NUM_BARS * 8 + 40 <= 256, "barrier area");
};

template <int OUT>
__device__ __forceinline__ void store_c4(void* C, int64_t idx, uint4 bits) {
  if constexpr (OUT == OUT_S32) {
    *reinterpret_cast<uint4*>(static_cast<int32_t*>(C) + idx) = bits;
  } else {
    store_out4<OUT>(C, idx, make_float4(__uint_as_float(bits.x), __uint_as_float(bits.y),
                                        __uint_as_float(bits.z), __uint_as_float(bits.w)));
  }
}

// One block of 32 outputs of this lane's row into a staging buffer of the
// epilogue: 128-byte rows with 128-byte swizzle for 4-byte outputs, 64-byte
// rows with 64-byte swizzle for 16-bit ones (round to nearest even), the
// layout the C tensor map's store reads.
template <int OUT>
__device__ __forceinline__ void stage_block(uint8_t* buf, const uint32_t (&v)[32], uint32_t lane) {
  if constexpr (OutTraits<OUT>::bytes == 4) {
    uint8_t* row = buf + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint4 q4 = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      if constexpr (OUT == OUT_S32)
        q4 = make_uint4(static_cast<uint32_t>(__float2int_rn(__uint_as_float(q4.x))),
                        static_cast<uint32_t>(__float2int_rn(__uint_as_float(q4.y))),
                        static_cast<uint32_t>(__float2int_rn(__uint_as_float(q4.z))),
                        static_cast<uint32_t>(__float2int_rn(__uint_as_float(q4.w))));
      *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) = q4;
    }
  } else {
    uint32_t w[16];
#pragma unroll
    for (int i2 = 0; i2 < 16; ++i2)
      w[i2] = pack2<OUT>(__uint_as_float(v[2 * i2]), __uint_as_float(v[2 * i2 + 1]));
    uint8_t* row = buf + lane * 64;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 q4 = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      *reinterpret_cast<uint4*>(row + ((j ^ ((lane >> 1) & 3)) << 4)) = q4;
    }
  }
}

// Deepest ring that fits the 227 KB per-CTA budget next to the epilogue
// staging, the barriers and the 1 KB alignment slack.
template <int BN, bool PAIR = false, int OBYTES = 4, bool INT_EXACT = false, int KCH = 1>
constexpr int square_max_stages() {
  using E = EpiStaging<OBYTES, INT_EXACT, (BN > 256)>;
  return (232448 - 1024 - E::WARPS * E::MIN_NBUF * E::BUF - 256) /
         (KCH * (128 * 64 * 2 + (PAIR ? BN / 2 : BN) * 64 * 2));
}

// Adds up a cut tile's partials of this CTA's 128 rows in contributor order
// (a fixed order: increasing k) and writes them to C, with NT threads (tid in
// [0, NT)). base points at the tile's first partial slot of this CTA.
// Flat index f over the 128 rows: group g = f % 8 of four columns, row
// (f / 8) % 128, 32-column block f / (8 * 128); past the whole blocks, a last
// 16-column block takes g = f % 4, row f / 4. A warp reads 64-byte runs of
// the partials and writes whole row segments of C.
template <int BN, int OUT, bool INT_EXACT, int NT>
__device__ __forceinline__ void reduce_cut_tile(const SquareParams& p, const uint4* base, int count,
                                                int row0, int col0, int tid) {
  constexpr int nr = 128;
  constexpr int total = nr * (BN / 4);
  constexpr int full = nr * 8 * (BN / 32);  // the groups of whole 32-column blocks
  // groups per contributor in flight (fewer with 256 threads, which run beside
  // the exact-integer epilogue's running sums), contributors in flight
  constexpr int CH = NT >= 256 ? 4 : 8;
  constexpr int CB = 2;
#pragma unroll 1
  for (int f0 = 0; f0 < total; f0 += NT * CH) {
    int idx[CH];
#pragma unroll
    for (int i2 = 0; i2 < CH; ++i2) {
      const int f = f0 + tid + NT * i2;
      if (f < full) {
        const int rest = f >> 3;
        const int cb = rest / nr;
        idx[i2] = (cb * 8 + (f & 7)) * 128 + (rest - cb * nr);
      } else if (f < total) {
        idx[i2] = ((BN / 32) * 8 + ((f - full) & 3)) * 128 + ((f - full) >> 2);
      } else {
        idx[i2] = -1;
      }
    }
    uint4 acc[CH];
#pragma unroll 1
    for (int c0 = 0; c0 < count; c0 += CB) {
      // CB contributors' groups are loaded together, then added in order
      uint4 v4[CB][CH];
#pragma unroll
      for (int cc = 0; cc < CB; ++cc) {
        if (c0 + cc < count) {
          const uint4* pj = base + static_cast<int64_t>(c0 + cc) * (32 * BN);
#pragma unroll
          for (int i2 = 0; i2 < CH; ++i2)
            if (idx[i2] >= 0) v4[cc][i2] = __ldcg(pj + idx[i2]);
        }
      }
#pragma unroll
      for (int cc = 0; cc < CB; ++cc) {
        if (c0 + cc >= count) break;
#pragma unroll
        for (int i2 = 0; i2 < CH; ++i2) {
          if (idx[i2] < 0) continue;
          if (c0 + cc == 0) {
            acc[i2] = v4[cc][i2];
          } else if constexpr (INT_EXACT) {
            acc[i2].x += v4[cc][i2].x;  // int32 sums added as unsigned words (two's complement)
            acc[i2].y += v4[cc][i2].y;
            acc[i2].z += v4[cc][i2].z;
            acc[i2].w += v4[cc][i2].w;
          } else {
            acc[i2].x = __float_as_uint(__uint_as_float(acc[i2].x) + __uint_as_float(v4[cc][i2].x));
            acc[i2].y = __float_as_uint(__uint_as_float(acc[i2].y) + __uint_as_float(v4[cc][i2].y));
            acc[i2].z = __float_as_uint(__uint_as_float(acc[i2].z) + __uint_as_float(v4[cc][i2].z));
            acc[i2].w = __float_as_uint(__uint_as_float(acc[i2].w) + __uint_as_float(v4[cc][i2].w));
          }
        }
      }
    }
#pragma unroll
    for (int i2 = 0; i2 < CH; ++i2) {
      if (idx[i2] < 0) continue;
      const int g = idx[i2] >> 7;  // cb * 8 + group
      const int r = row0 + (idx[i2] & 127);
      const int col = col0 + 4 * g;
      if (r < p.M && col < p.N) {
        if constexpr (INT_EXACT || OUT == OUT_S32)
          store_c4<OUT_S32>(p.C_out, static_cast<int64_t>(r) * p.ldc + col, acc[i2]);
        else
          store_c4<OUT>(p.C_out, static_cast<int64_t>(r) * p.ldc + col, acc[i2]);
      }
    }
  }
}

template <int BN, int STAGES, bool IN_BF16, int OUT, bool INT_EXACT, bool PAIR = false, int KCH = 1>
__global__ void __launch_bounds__(INT_EXACT ? SQUARE_THREADS_INT : SQUARE_THREADS, 1)
    square_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const SquareParams p) {
  constexpr int OBYTES = OutTraits<OUT>::bytes;
  using L = SquareLayout<BN, STAGES, INT_EXACT, PAIR, OBYTES, KCH>;
  constexpr int BM = L::BM, BK = L::BK;
  // one MMA covers at most 256 columns: a 512-wide tile is two halves, each
  // half's B rows split between the CTAs of the pair like a 256-wide tile's
  constexpr int NH = BN > 256 ? 2 : 1;
  constexpr int MMA_N = BN / NH;
  constexpr int NACC = L::NACC;
  constexpr uint32_t IDESC = idesc_f16_f32acc(IN_BF16, L::TILE_M, MMA_N);
  static_assert(!INT_EXACT || OUT == OUT_S32, "exact integer mode writes int32");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sA = sbase + L::OFF_A;
  const uint32_t sB = sbase + L::OFF_B;
  uint8_t* epi_buf = smem + L::OFF_EPI;
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  // notices "partial tile written" from the epilogue to the reduction warps
  auto note_full = [&](int j) { return bar0 + 8u * (2 * STAGES + 5 + j); };
  auto note_empty = [&](int j) { return bar0 + 8u * (2 * STAGES + 7 + j); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  // the reduction warps' decision per notice (two slots, alternating)
  volatile int* fix_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 8);
  // per notice: 1 if this CTA's arrival completed the tile (it reduces it)
  volatile int* note_last = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 16);
  // the CTA's last tile for the reduction warps that help store it: m tile,
  // n tile, accumulator
  volatile int* last_tile = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 24);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA rank within the pair (0 = leader, which issues the MMAs)
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const uint32_t leader_crank = 0u;  // cluster rank of the pair's leader

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      // (a 512-wide tile cut along K, a test setting, drains with four warps:
      // the other four reduce)
      mbar_init(tempty_bar(b), (PAIR ? 2 : 1) *
                                   ((!INT_EXACT && L::EPI_WARPS == 8 && p.sk_tiles > 0) ? 4
                                                                                         : L::EPI_WARPS));
    }
    mbar_init(drain_bar, 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(note_full(j), 1);
      mbar_init(note_empty(j), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    // kernel parameters, not written by earlier kernels: fetch them early
    prefetch_tensor_map(&tmA);
    prefetch_tensor_map(&tmB);
    prefetch_tensor_map(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_g<PAIR>(smem_addr(tmem_slot), L::TMEM_COLS);
    tmem_relinquish_g<PAIR>();
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA use
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int kpc = p.k_tiles_per_chunk;
  // the persistent work unit is a CTA, or a CTA pair in PAIR mode
  constexpr int WSHIFT = PAIR ? 1 : 0;
  const int worker = static_cast<int>(blockIdx.x >> WSHIFT);
  const int workers = static_cast<int>(gridDim.x >> WSHIFT);
  // The producer warp works out its first segment and warms L2 with its
  // first stages while the previous kernel drains (safe: L2 is where writes
  // become coherent; the loads proper wait for the dependency).
  Segment seg0;
  bool have_seg0 = false;
  int mt0 = 0, nt0 = 0;
  uint64_t pol_operands = 0;
  if (warp == 0) {
    pol_operands = policy_evict_last();  // operands are re-read by other tiles
    have_seg0 = square_segment(p, worker, workers, 0, seg0);
    if (have_seg0) {
      tile_coords(seg0.tile, p.num_m_tiles, p.num_n_tiles, p.group_m, mt0, nt0);
      for (int kt = seg0.kt0; lane == 0 && kt < min(seg0.kt1, seg0.kt0 + STAGES); ++kt) {
        for (int j = 0; j < KCH; ++j) {
          tma_prefetch_l2_2d(&tmA, (kt * KCH + j) * BK, mt0 * L::TILE_M + static_cast<int>(rank) * BM);
          for (int h = 0; h < NH; ++h)
            tma_prefetch_l2_2d(&tmB, (kt * KCH + j) * BK,
                               nt0 * BN + h * MMA_N + static_cast<int>(rank) * (L::BN_CTA / NH));
        }
      }
    }
  }
  // Set-up above may overlap the previous kernel in the stream; no global
  // memory is read for use before that kernel has completed.
  grid_dependency_wait();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_SETUP);

  const WaitCtl ctl{p.timeout_ns, p.error_word, abort_flag};

  // The producer and the MMA issuer run their loops as whole warps, with one
  // elected lane issuing the copies, MMAs and commits: a lane running alone
  // in its warp pays a large fixed cost per loop trip (measured: ~470 cycles
  // per K-tile at the MMA issuer whatever the tile width, against 128 per
  // 256-wide MMA on the tensor pipe), which the converged warp does not.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    {  // the whole warp
      const bool leader = elect_one_sync();
      const uint64_t pol = pol_operands;
      // B streamed (evict-first) when no other tile reads it: 256 x 16384 x
      // 4096 bfloat16 28.7 -> 27.7 us; elsewhere kept like A
      const uint64_t pol_b = p.b_once ? policy_evict_first() : pol_operands;
      int issued_round[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_round[s] = -1;
      bool ok = true;
      uint32_t it = 0;
      Segment seg;
      for (int i = 0; ok; ++i) {
        int mt, nt;
        if (i == 0) {
          if (!have_seg0) break;
          seg = seg0;  // worked out before the dependency wait
          mt = mt0;
          nt = nt0;
        } else {
          if (!square_segment(p, worker, workers, i, seg)) break;
          tile_coords(seg.tile, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt);
        }
        const int a_row = mt * L::TILE_M + static_cast<int>(rank) * BM;
        const int b_row = nt * BN + static_cast<int>(rank) * L::BN_CTA;
        for (int kt = seg.kt0; kt < seg.kt1; ++kt, ++it) {
          const int s = it % STAGES;
          const uint32_t round = it / STAGES;
          // in the first round every stage is free: no wait; the warp
          // leaves a wait together (every lane polls, all must succeed)
          if (round > 0 && !__all_sync(0xffffffffu, wait_bounded(empty_bar(s), (round & 1u) ^ 1u,
                                                                  ctl, WAIT_PRODUCER_EMPTY))) {
            ok = false;
            break;
          }
          if (p.inject_stall && it == 1 && rank == 0) continue;  // test hook: stage never fills
          issued_round[s] = static_cast<int>(round);
          if (!leader) continue;
          if constexpr (PAIR) {
            // both CTAs' copies complete on the leader's barrier; the leader
            // announces the bytes of both
            if (rank == 0) mbar_arrive_expect_tx(full_bar(s), L::STAGE_TX);
            const uint32_t leader_full = map_to_cta(full_bar(s), leader_crank);
            if constexpr (KCH > 1) {
              // KCH consecutive K-chunks of each operand (tiles up to 256 wide)
#pragma unroll
              for (int j = 0; j < KCH; ++j) {
                tma_load_2d_pair(sA + s * L::A_STAGE + j * L::A_CHUNK, &tmA, leader_full,
                                 (kt * KCH + j) * BK, a_row, pol);
                tma_load_2d_pair(sB + s * L::B_STAGE + j * L::B_CHUNK, &tmB, leader_full,
                                 (kt * KCH + j) * BK, b_row, pol_b);
              }
            } else if constexpr (NH == 2) {
              tma_load_2d_pair(sA + s * L::A_STAGE, &tmA, leader_full, kt * BK, a_row, pol);
              // this CTA's rows of each 256-column half, one box per half
#pragma unroll
              for (int h = 0; h < NH; ++h)
                tma_load_2d_pair(sB + s * L::B_STAGE + h * (MMA_N / 2) * (BK * 2), &tmB, leader_full,
                                 kt * BK, nt * BN + h * MMA_N + static_cast<int>(rank) * (MMA_N / 2),
                                 pol_b);
            } else {
              tma_load_2d_pair(sA + s * L::A_STAGE, &tmA, leader_full, kt * BK, a_row, pol);
              tma_load_2d_pair(sB + s * L::B_STAGE, &tmB, leader_full, kt * BK, b_row, pol_b);
            }
          } else {
            mbar_arrive_expect_tx(full_bar(s), L::STAGE_TX);
#pragma unroll
            for (int j = 0; j < KCH; ++j) {
              tma_load_2d(sA + s * L::A_STAGE + j * L::A_CHUNK, &tmA, full_bar(s),
                          (kt * KCH + j) * BK, a_row, pol);
              tma_load_2d(sB + s * L::B_STAGE + j * L::B_CHUNK, &tmB, full_bar(s),
                          (kt * KCH + j) * BK, b_row, pol_b);
            }
          }
          if (it == 0) trace_mark(p.trace, TR_FIRST_LOAD);
          trace_ktile(p.trace, 0, it);
        }
      }
      if (leader) trace_mark(p.trace, TR_LAST_LOAD);
      grid_launch_dependents();  // the next kernel may start its set-up
      if (!ok) {
        // Let every copy already issued land before the CTA can exit.
        if (!PAIR || rank == 0) {
          for (int s = 0; s < STAGES; ++s) {
            if (issued_round[s] < 0) continue;
            const uint32_t bar = full_bar(s), par = static_cast<uint32_t>(issued_round[s]) & 1u;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar, par) && global_timer_ns() - t0 < ctl.timeout_ns) {
            }
          }
        } else {
          // the peer's copies complete on the leader's barriers, which this
          // CTA cannot wait on: give them a fixed 100 us to land
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 100000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (rank == 0) {
      const bool leader = elect_one_sync();
      const bool tracing = p.trace != nullptr && leader;
      const uint64_t a_desc0 = sdesc_k_major_sw128(sA);
      const uint64_t b_desc0 = sdesc_k_major_sw128(sB);
      bool ok = true;
      uint32_t it = 0, unit = 0;
      Segment seg;
      for (int i = 0; ok && square_segment(p, worker, workers, i, seg); ++i) {
        for (int c0 = seg.kt0; ok && c0 < seg.kt1; c0 += kpc, ++unit) {
          const uint32_t b = NACC == 2 ? (unit & 1u) : 0u;
          const uint32_t use = NACC == 2 ? (unit >> 1) : unit;
          if (!__all_sync(0xffffffffu,
                          wait_bounded(tempty_bar(b), (use & 1u) ^ 1u, ctl, WAIT_MMA_TMEM_EMPTY))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + b * L::ACC_COLS;
          const int c1 = min(seg.kt1, c0 + kpc);
          // Stage and phase are counted, not divided; descriptors advance by
          // adds (the 14-bit start-address field cannot carry: shared
          // addresses are below 256 KB).
          int s = static_cast<int>(it % STAGES);
          uint32_t phase = (it / STAGES) & 1u;
          for (int kt = c0; kt < c1; ++kt, ++it) {
            if (!__all_sync(0xffffffffu, wait_bounded(full_bar(s), phase, ctl, WAIT_MMA_FULL))) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (tracing) {
              if (it == 0) trace_mark(p.trace, TR_FIRST_DATA);
              trace_ktile(p.trace, 1, it);
            }
            const uint64_t adesc = a_desc0 + static_cast<uint64_t>((s * L::A_STAGE) >> 4);
            const uint64_t bdesc = b_desc0 + static_cast<uint64_t>((s * L::B_STAGE) >> 4);
            if (leader) {
#pragma unroll
              for (int j = 0; j < KCH; ++j) {  // each 64-wide K-chunk of the stage
                const uint64_t aj = adesc + static_cast<uint64_t>((j * L::A_CHUNK) >> 4);
#pragma unroll
                for (int h = 0; h < NH; ++h) {  // each 256-column half of a 512-wide tile
                  const uint64_t bd = bdesc + static_cast<uint64_t>((j * L::B_CHUNK) >> 4) +
                                      static_cast<uint64_t>((h * (MMA_N / 2) * (BK * 2)) >> 4);
                  const uint32_t dt = d_tmem + h * MMA_N;
                  mma_f16_g<PAIR>(dt, aj, bd, IDESC, (kt > c0 || j > 0) ? 1u : 0u);
#pragma unroll
                  for (int k = 1; k < BK / 16; ++k)  // +32 bytes (2 in descriptor units) per K = 16
                    mma_f16_g<PAIR>(dt, aj + 2 * k, bd + 2 * k, IDESC, 1u);
                }
              }
              // stage s may be refilled (in both CTAs of a pair)
              mma_commit_g<PAIR>(empty_bar(s));
            }
            __syncwarp();
            if (++s == STAGES) {
              s = 0;
              phase ^= 1u;
            }
          }
          if (ok && leader)  // accumulator b holds the finished chunk
            mma_commit_g<PAIR>(tfull_bar(b));
          __syncwarp();
        }
      }
      if (leader) {
        trace_mark(p.trace, TR_LAST_MMA);
        // Drain: every MMA issued above has completed before tensor memory is freed.
        mma_commit_local_g<PAIR>(drain_bar);
      }
      __syncwarp();
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < ctl.timeout_ns) {
      }
    }
  } else if (INT_EXACT && warp < 10) {
    // ------------------------------------------------ exact-integer epilogue
    if constexpr (INT_EXACT) {
      // Warps 2-9. A chunk's accumulator holds exact integers (|v| <= 2^24);
      // each thread converts its row's values to int32 and adds them to a
      // running sum in its registers (int32 sums wrap modulo 2^32), so the
      // accumulator goes back to the MMA warp as soon as it is read and tensor
      // memory holds just the two accumulators. Each lane quadrant has two
      // warps: warps 2-5 keep the first 32 * INT_NB0 columns, warps 6-9 the
      // rest (at most 128 registers of sum per thread). After a segment's last
      // chunk the sum goes to C through the tensor-copy store, or, for a piece
      // of a tile cut along K, to its scratch slot, with a notice to the two
      // reduction warps (warps 10-11) as in the float epilogue.
      const int q = warp & 3;  // tensor-memory lane quadrant this warp may access
      const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
      const int grp = (warp - 2) >> 2;
      const int etid = static_cast<int>(threadIdx.x) - 64;  // 0..255
      uint8_t* bufs = epi_buf + (warp - 2) * L::EPI_NBUF * L::EPI_BUF;
      auto run = [&](auto nblk) {
        constexpr int NBLK = decltype(nblk)::value;
        const int cb0 = grp == 0 ? 0 : L::INT_NB0;  // this warp's first 32-column block
        uint32_t sum[32 * NBLK];
        uint32_t unit = 0, stores = 0, notes = 0;
        bool ok = true;
        Segment seg;
        for (int i = 0; ok && square_segment(p, worker, workers, i, seg); ++i) {
          int mt, nt;
          tile_coords(seg.tile, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt);
          const int c_row = mt * L::TILE_M + static_cast<int>(rank) * BM + 32 * q;
          const int n_chunks = (seg.kt1 - seg.kt0 + kpc - 1) / kpc;
          // One chunk: wait for its accumulator, convert and add it into the
          // registers, hand the accumulator back. The first chunk of a segment
          // assigns the sums (peeled, so they are dead between segments).
          auto wait_chunk = [&](uint32_t& bb) {
            bb = unit & 1u;
            const uint32_t use = unit >> 1;
            ++unit;
            // the eight warps leave the wait with one decision
            const bool got = named_barrier_and(
                1, 256,
                __all_sync(0xffffffffu, wait_bounded(tfull_bar(bb), use & 1u, ctl, WAIT_EPI_TMEM_FULL)));
            if (got) tc_fence_after();
            return got;
          };
          auto release_chunk = [&](uint32_t bb) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if constexpr (PAIR)
                mbar_arrive_cluster(map_to_cta(tempty_bar(bb), leader_crank));  // the leader's barrier
              else
                mbar_arrive(tempty_bar(bb));
            }
          };
          // (a failed first wait leaves the segment loop at once: no path
          // reaches a read of the sums without passing the assignment)
          uint32_t b = 0;
          if (!wait_chunk(b)) {
            ok = false;
            break;
          }
          int_chunk_sums<true, NBLK>(sum, tmem_base + lane_base + b * L::ACC_COLS + 32 * cb0);
          release_chunk(b);
          for (int c = 1; c < n_chunks; ++c) {
            if (!wait_chunk(b)) {
              ok = false;
              break;
            }
            int_chunk_sums<false, NBLK>(sum, tmem_base + lane_base + b * L::ACC_COLS + 32 * cb0);
            release_chunk(b);
          }
          if (!ok) break;
          if (seg.partial) {
            // 16-byte groups in the order [32-column block][group of 4 columns][row]
            uint4* slot = reinterpret_cast<uint4*>(p.partials) +
                          ((static_cast<int64_t>(seg.sk) * 2 + rank) * p.max_contrib + seg.j) * (32 * BN) +
                          32 * q + lane;
  #pragma unroll
            for (int j = 0; j < NBLK; ++j)
  #pragma unroll
              for (int g = 0; g < 8; ++g)
                __stcg(slot + ((cb0 + j) * 8 + g) * 128,
                       make_uint4(sum[32 * j + 4 * g], sum[32 * j + 4 * g + 1], sum[32 * j + 4 * g + 2],
                                  sum[32 * j + 4 * g + 3]));
            // visible at GPU scope, then one thread counts the arrival and
            // posts a notice to the reduction warps saying whether this arrival
            // completed the tile
            __threadfence();
            named_barrier_sync(1, 256);
            if (etid == 0) {
              unsigned long long* ctr = p.counters + seg.sk * 2 + rank;
              const int last = arrive_generation(ctr, p.generation, seg.count, p.error_word);
              if (last) atomicExch(ctr, 0ull);  // the counter's last use in this call
              const uint32_t j = notes & 1u, use = notes >> 1;
              if (wait_bounded(note_empty(j), (use & 1u) ^ 1u, ctl, WAIT_FIXUP_SLOT)) {
                note_last[j] = last;
                mbar_arrive(note_full(j));
              }
            }
            ++notes;
          } else {
            // one 32-column block at a time through this warp's staging
            // buffers (128-byte rows, 128-byte swizzle), a tensor-copy store each
  #pragma unroll
            for (int j = 0; j < NBLK; ++j) {
              uint8_t* buf = bufs + (stores % L::EPI_NBUF) * L::EPI_BUF;
              if (lane == 0) bulk_wait_group_read<L::EPI_NBUF - 1>();
              __syncwarp();
              uint8_t* row = buf + lane * 128;
  #pragma unroll
              for (int g = 0; g < 8; ++g)
                *reinterpret_cast<uint4*>(row + ((g ^ (lane & 7)) << 4)) =
                    make_uint4(sum[32 * j + 4 * g], sum[32 * j + 4 * g + 1], sum[32 * j + 4 * g + 2],
                               sum[32 * j + 4 * g + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                // a block that starts past the matrix (ragged edge) stores nothing
                const int col = nt * BN + 32 * (cb0 + j);
                if (c_row < p.M && col < p.N) tma_store_2d(&tmC, smem_addr(buf), col, c_row);
                bulk_commit_group();
              }
              ++stores;
            }
          }
        }
        bulk_wait_group_read<0>();  // staging is free once the stores have read it
        if (warp == 2 && lane == 0) trace_mark(p.trace, TR_EPI_DONE);
      };
      if (grp == 0)
        run(IntConst<L::INT_NB0>{});
      else
        run(IntConst<L::INT_NB1>{});
    }
  } else if (!INT_EXACT &&
             (warp < 6 || (L::EPI_WARPS == 8 && warp < 10 && p.sk_tiles == 0))) {
    // ------------------------------------------------------------ epilogue
    // (eight warps for 512-wide tiles when none is cut along K: warps 2-5
    // store the first half of a tile's 32-column blocks, warps 6-9 the second)
    const bool wide8 = L::EPI_WARPS == 8 && p.sk_tiles == 0;
    const int q = warp & 3;  // tensor-memory lane quadrant this warp may access
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    uint8_t* bufs = epi_buf + (warp - 2) * L::EPI_NBUF * L::EPI_BUF;
    const int cb_first = wide8 ? ((warp - 2) >> 2) * (BN / 64) : 0;
    uint32_t unit = 0, notes = 0;
    bool ok = true;
    Segment seg;
    for (int i = 0; ok && square_segment(p, worker, workers, i, seg); ++i) {
      int mt, nt;
      tile_coords(seg.tile, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt);
      const int c_row = mt * L::TILE_M + static_cast<int>(rank) * BM + 32 * q;
      const int n_chunks = (seg.kt1 - seg.kt0 + kpc - 1) / kpc;
      // A partial segment's 32-bit values go to its scratch slot as 16-byte
      // groups in the order [32-column block][group of 4 columns][row]: the
      // 32 lanes (32 consecutive rows) of one store write 512 contiguous bytes.
      uint4* slot = nullptr;
      if (seg.partial)
        slot = reinterpret_cast<uint4*>(p.partials) +
               ((static_cast<int64_t>(seg.sk) * 2 + rank) * p.max_contrib + seg.j) * (32 * BN) +
               32 * q + lane;
      // the CTA's last tile shares its blocks with the reduction warps
      bool split = false;
      if constexpr (L::LAST_SPLIT) {
        Segment nxt;
        split = p.sk_tiles == 0 && !square_segment(p, worker, workers, i + 1, nxt);
      }
      for (int c = 0; c < n_chunks; ++c, ++unit) {
        const uint32_t b = NACC == 2 ? (unit & 1u) : 0u;
        const uint32_t use = NACC == 2 ? (unit >> 1) : unit;
        // every lane waits, and the warp leaves together: the tensor-memory
        // loads below are warp-collective
        ok = __all_sync(0xffffffffu, wait_bounded(tfull_bar(b), use & 1u, ctl, WAIT_EPI_TMEM_FULL));
        if (!ok) break;
        tc_fence_after();
        const uint32_t t_acc = tmem_base + lane_base + b * L::ACC_COLS + 32 * cb_first;
        if (split && threadIdx.x == 64) {
          last_tile[0] = mt;
          last_tile[1] = nt;
          last_tile[2] = static_cast<int>(b);
          mbar_arrive(note_full(0));  // the helpers may start
        }
        // One block = 32 output columns of this warp's 32 rows. The
        // tensor-memory load of block cb+1 is in flight while block cb is
        // converted.
        const int NB = split ? L::LAST_NB0 : (wide8 ? BN / 64 : L::NB_FULL);
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_acc, v);
        tmem_wait_ld_regs(v);
        if (seg.partial) {
#pragma unroll 1
          for (int cb = 0; cb < NB; ++cb) {
            const bool more = cb + 1 < NB;
            uint32_t nxt[32];
            if (more) tmem_ld_32x32b_x32(t_acc + 32 * (cb + 1), nxt);
            // fp32 partial straight to scratch
#pragma unroll
            for (int j = 0; j < 8; ++j)
              __stcg(slot + ((cb_first + cb) * 8 + j) * 128,
                     make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            if (more) {
              tmem_wait_ld_regs(nxt);
#pragma unroll
              for (int i2 = 0; i2 < 32; ++i2) v[i2] = nxt[i2];
            }
          }
        } else {
          // Blocks go out in groups of G = the staging buffers of the warp:
          // each block is converted into its own buffer (128-byte rows with
          // 128-byte swizzle for 4-byte outputs, 64-byte rows with 64-byte
          // swizzle for 16-bit ones), one proxy fence covers the group, and
          // lanes 0..G-1 each issue the tensor-copy store of one block.
          constexpr int G = L::EPI_NBUF;
#pragma unroll 1
          for (int cb0 = 0; cb0 < NB; cb0 += G) {
            // every lane's earlier stores are done reading the buffers
            bulk_wait_group_read<0>();
            __syncwarp();
#pragma unroll 1
            for (int g = 0; g < G; ++g) {
              const int cb = cb0 + g;
              if (cb < NB) {
                const bool more = cb + 1 < NB;
                uint32_t nxt[32];
                if (more) tmem_ld_32x32b_x32(t_acc + 32 * (cb + 1), nxt);
                stage_block<OUT>(bufs + g * L::EPI_BUF, v, lane);
                if (more) {
                  tmem_wait_ld_regs(nxt);
#pragma unroll
                  for (int i2 = 0; i2 < 32; ++i2) v[i2] = nxt[i2];
                }
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            const int cb = cb0 + lane;
            const int col = nt * BN + 32 * (cb_first + cb);
            // a block that starts past the matrix (ragged edge) stores nothing
            if (lane < G && cb < NB && c_row < p.M && col < p.N) {
              tma_store_2d(&tmC, smem_addr(bufs + lane * L::EPI_BUF), col, c_row);
              bulk_commit_group();
            }
          }
        }
        if constexpr (L::HALF_BLOCK) {
          // The tile's last 16 columns: each lane's row goes out from its
          // registers (N * sizeof(out) is a multiple of 16 bytes, so a group
          // of 8 16-bit or 4 fp32 outputs lies wholly inside or outside C),
          // or, for a partial segment, to the scratch slot's last groups.
          uint32_t h[16];
          tmem_ld_32x32b_x16(t_acc + 32 * L::NB_FULL, h);
          tmem_wait_ld_regs16(h);
          if (seg.partial) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              __stcg(slot + (L::NB_FULL * 8 + j) * 128,
                     make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]));
          } else {
            const int row = c_row + lane;
            const int col = nt * BN + 32 * L::NB_FULL;
            if (row < p.M && col < p.N) {
              float f[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(h[j]);
              void* row_ptr = static_cast<uint8_t*>(p.C_out) +
                              (static_cast<int64_t>(row) * p.ldc) * OBYTES;
              constexpr int GRP = OBYTES == 4 ? 4 : 8;
#pragma unroll
              for (int g = 0; g < 16 / GRP; ++g)
                if (col + GRP * g < p.N) store_row_group<OUT>(row_ptr, col + GRP * g, f + GRP * g, GRP);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(map_to_cta(tempty_bar(b), leader_crank));  // the leader's barrier
          else
            mbar_arrive(tempty_bar(b));
        }
      }
      if (!ok || !seg.partial) continue;
      // The partial is written: every writer makes its stores visible at GPU
      // scope, then one thread counts the arrival at the tile's counter and
      // posts a notice to the reduction warps saying whether this arrival
      // completed the tile.
      __threadfence();
      named_barrier_sync(1, 128);
      if (threadIdx.x == 64) {
        unsigned long long* ctr = p.counters + seg.sk * 2 + rank;
        const int last = arrive_generation(ctr, p.generation, seg.count, p.error_word);
        // the last arrival is the counter's last use in this call
        if (last) atomicExch(ctr, 0ull);
        const uint32_t j = notes & 1u, use = notes >> 1;
        if (wait_bounded(note_empty(j), (use & 1u) ^ 1u, ctl, WAIT_FIXUP_SLOT)) {
          note_last[j] = last;
          mbar_arrive(note_full(j));
        }
      }
      ++notes;
    }
    bulk_wait_group_read<0>();  // staging is free once every lane's stores have read it
    if (warp == 2 && lane == 0) trace_mark(p.trace, TR_EPI_DONE);
  } else if (p.sk_tiles > 0) {
    // ---------------------------------------------- stream-K reduction warps
    // For each partial tile this CTA wrote (the epilogue's notices, in
    // segment order): if this CTA's arrival completed the tile, add up this
    // CTA's 128 rows over all partials in contributor order and write them to
    // C; otherwise another contributor does.
    constexpr int NT = ReductionWarps<INT_EXACT>::COUNT;
    const int tid = static_cast<int>(threadIdx.x) - ReductionWarps<INT_EXACT>::FIRST;  // 0..NT-1
    uint32_t notes = 0;
    bool ok = true;
    Segment seg;
    for (int i = 0; ok && square_segment(p, worker, workers, i, seg); ++i) {
      if (!seg.partial) continue;
      const uint32_t j = notes & 1u, use = notes >> 1;
      if (tid == 0) {
        int flag = -1;  // -1: gave up waiting for the notice
        if (wait_bounded(note_full(j), use & 1u, ctl, WAIT_FIXUP_NOTE)) {
          flag = note_last[j];
          mbar_arrive(note_empty(j));  // the notice is consumed
        }
        fix_flag[j] = flag;
      }
      named_barrier_sync(2, NT);
      const int flag = fix_flag[j];
      ++notes;
      if (flag < 0) {
        ok = false;
        break;
      }
      if (flag == 0) continue;  // a later contributor reduces this tile
      __threadfence();
      int mt, nt;
      tile_coords(seg.tile, p.num_m_tiles, p.num_n_tiles, p.group_m, mt, nt);
      const uint4* base = reinterpret_cast<const uint4*>(p.partials) +
                          (static_cast<int64_t>(seg.sk) * 2 + rank) * p.max_contrib * (32 * BN);
      reduce_cut_tile<BN, OUT, INT_EXACT, NT>(p, base, seg.count,
                                           mt * L::TILE_M + static_cast<int>(rank) * BM, nt * BN, tid);
      if (tid == 0) trace_mark(p.trace, TR_FIXUP_DONE);
    }
  } else if constexpr (L::LAST_SPLIT) {
    // ------------------------------------------ last-tile epilogue helpers
    // With no tile cut along K the reduction warps have nothing to do. The
    // CTA's last tile has no K-loop after it to hide its epilogue behind, so
    // they store the second half of its 32-column blocks while the epilogue
    // warps store the first: warp 6 + j takes the rows of lane quadrant
    // (6 + j) mod 4. Their staging is the ring, which neither the copies nor
    // the MMAs use once that tile's accumulator is complete (the notice comes
    // after the epilogue warps have seen it complete).
    Segment s0;
    if (square_segment(p, worker, workers, 0, s0)) {
      const bool got = __all_sync(0xffffffffu, wait_bounded(note_full(0), 0, ctl, WAIT_FIXUP_NOTE));
      if (got) {
        const int mt = last_tile[0], nt = last_tile[1];
        const uint32_t b = static_cast<uint32_t>(last_tile[2]);
        tc_fence_after();
        const int q = warp & 3;
        const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * L::ACC_COLS;
        const int c_row = mt * L::TILE_M + static_cast<int>(rank) * BM + 32 * q;
        constexpr int NB1 = L::NB_FULL - L::LAST_NB0;
        uint8_t* bufs = smem + L::OFF_A + (warp - 6) * NB1 * L::EPI_BUF;
        fence_proxy_async_smem();  // the ring's async-proxy use is over
#pragma unroll 1
        for (int j = 0; j < NB1; ++j) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_acc + 32 * (L::LAST_NB0 + j), v);
          tmem_wait_ld_regs(v);
          stage_block<OUT>(bufs + j * L::EPI_BUF, v, lane);
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int cb = L::LAST_NB0 + lane;
        // a block that starts past the matrix (ragged edge) stores nothing
        if (lane < NB1 && c_row < p.M && nt * BN + 32 * cb < p.N) {
          tma_store_2d(&tmC, smem_addr(bufs + lane * L::EPI_BUF), nt * BN + 32 * cb, c_row);
          bulk_commit_group();
        }
        bulk_wait_group_read<0>();
      }
    }
  }

  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  else
    __syncthreads();
  if (threadIdx.x == 0) trace_mark(p.trace, TR_EXIT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_g<PAIR>(tmem_base, L::TMEM_COLS);
  }
}

}  // namespace sptg
