// sptgemm.cu -- the C ABI of the library (declared in include/sptgemm.h):
// argument checks, kernel choice, tensor-map encoding and launch.
//
// All device work runs in the kernels of square_gemm.cuh, skinny_gemm.cuh and
// convert.cuh; this file only validates, plans and launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <string>
#include <utility>

#include "sptgemm.h"

#include "skinny_cluster_gemm.cuh"  // SkinnyClusterParams
#include "skinny_gemm.cuh"  // SkinnyParams
#include "skinny_pair_gemm.cuh"  // SkinnyPairParams
#include "skinny_rows_gemm.cuh"  // SkinnyRowsParams
#include "square_gemm.cuh"  // SquareParams
#include "stream_scale.cuh"  // StreamParams
#include "variants.h"

// Device error word: a timed-out bounded wait ors its site code in here.
__device__ unsigned int g_sptg_error_word;

namespace {

using namespace sptg;

thread_local std::string t_last_error;
thread_local int t_launches = 0;  // kernels this library launched in the current call

// What the last call of this thread chose, formatted only when asked for
// (sptg_last_config), so that a call pays no string formatting.
struct LastConfig {
  const char* fmt = "";
  const char* name = "";
  long long v[16] = {};
  int launches = 0;
};
thread_local LastConfig t_config;

void set_config(const char* fmt, const char* name, std::initializer_list<long long> vals) {
  t_config.fmt = fmt;
  t_config.name = name;
  int i = 0;
  for (long long x : vals) {
    if (i < 16) t_config.v[i++] = x;
  }
  for (; i < 16; ++i) t_config.v[i] = 0;
  t_config.launches = t_launches;
}

std::string config_text() {
  char buf[512];
  const long long* v = t_config.v;
  snprintf(buf, sizeof(buf), t_config.fmt, t_config.name, v[0], v[1], v[2], v[3], v[4], v[5], v[6],
           v[7], v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
  return std::string(buf) + " launches=" + std::to_string(t_config.launches);
}

int cuda_fail(cudaError_t e, const char* what) {
  t_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return SPTG_ERR_LAUNCH;
}

// ------------------------------------------------------------ driver entry
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// ------------------------------------------------------------ device state
struct DeviceInfo {
  bool ok = false;
  int sm_count = 0;
  int major = 0, minor = 0;
  unsigned int* error_word = nullptr;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::set<std::pair<int, const void*>> g_smem_set;

int device_info(DeviceInfo& out, int& dev) {
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    t_last_error = std::string("cudaGetDevice: ") + cudaGetErrorString(e);
    return SPTG_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_devices.find(dev);
  if (it != g_devices.end()) {
    out = it->second;
    return out.ok ? SPTG_OK : SPTG_ERR_UNSUPPORTED;
  }
  DeviceInfo d;
  cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
  d.ok = (d.major == 10 && d.minor == 3);
  if (d.ok) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_sptg_error_word);
    if (e != cudaSuccess) {
      t_last_error = std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e);
      return SPTG_ERR_LAUNCH;
    }
    d.error_word = static_cast<unsigned int*>(p);
  } else {
    char b[128];
    snprintf(b, sizeof(b), "device %d has compute capability %d.%d; this library needs 10.3", dev,
             d.major, d.minor);
    t_last_error = b;
  }
  g_devices[dev] = d;
  out = d;
  return d.ok ? SPTG_OK : SPTG_ERR_UNSUPPORTED;
}

int ensure_smem(int dev, const void* kernel, int bytes) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem_set.count({dev, kernel})) return SPTG_OK;
  }
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  std::lock_guard<std::mutex> lk(g_mu);
  g_smem_set.insert({dev, kernel});
  return SPTG_OK;
}

// ------------------------------------------------------------ scratch space
// One stream-ordered scratch area per (device, stream), grown on demand. Its
// first kCounterArea bytes hold the split-K arrival counters of the skinny
// kernel and of the square kernel's stream-K tiles (zeroed whenever the area
// is (re)allocated; each call tags its arrivals with a new generation); the
// rest holds a call's data (int8 operands widened to binary16, split-K
// partial tiles).
constexpr size_t kCounterArea = static_cast<size_t>(1) << 16;

struct Scratch {
  void* ptr = nullptr;
  size_t bytes = 0;
  unsigned int generation = 0;  // tag of the last call that used the counters
};
std::map<std::pair<int, cudaStream_t>, Scratch> g_scratch;

struct ScratchView {
  void* data;
  unsigned long long* counters;
  unsigned int generation;  // a new non-zero tag for this call's counters
};

// Growing a stream-ordered allocation inside a CUDA graph capture would put
// the allocation into the graph (valid only while the graph runs), so under
// capture the area must already be large enough: a call made once on the
// stream before capturing sizes it.
bool stream_capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return st != cudaStreamCaptureStatusNone;
}

int capture_growth_error() {
  t_last_error =
      "the library's device buffers for this stream must exist before graph capture: make the "
      "same call once on the stream first";
  return SPTG_ERR_CONFIG;
}

int scratch_for(int dev, cudaStream_t stream, size_t data_bytes, ScratchView* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  Scratch& s = g_scratch[{dev, stream}];
  const size_t need = kCounterArea + data_bytes;
  if (s.bytes < need && stream_capturing(stream)) return capture_growth_error();
  if (s.bytes < need) {
    if (s.ptr) cudaFreeAsync(s.ptr, stream);
    s.ptr = nullptr;
    s.bytes = 0;
    size_t grow = std::max(need, static_cast<size_t>(1) << 20);
    cudaError_t e = cudaMallocAsync(&s.ptr, grow, stream);
    if (e != cudaSuccess) {
      s.ptr = nullptr;
      t_last_error = std::string("cudaMallocAsync: ") + cudaGetErrorString(e);
      return SPTG_ERR_NOMEM;
    }
    e = cudaMemsetAsync(s.ptr, 0, kCounterArea, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    s.bytes = grow;
  }
  s.generation = s.generation + 1 ? s.generation + 1 : 1;
  out->counters = static_cast<unsigned long long*>(s.ptr);
  out->data = static_cast<char*>(s.ptr) + kCounterArea;
  out->generation = s.generation;
  return SPTG_OK;
}

// Device copies of the operands and result of a host-buffer call
// (sptg_gemm_host), one area per (device, stream), grown on demand and freed
// in stream order like the scratch.
struct IoArea {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, IoArea> g_io;

int io_for(int dev, cudaStream_t stream, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  IoArea& a = g_io[{dev, stream}];
  if (a.bytes < bytes && stream_capturing(stream)) return capture_growth_error();
  if (a.bytes < bytes) {
    if (a.ptr) cudaFreeAsync(a.ptr, stream);
    a.ptr = nullptr;
    a.bytes = 0;
    cudaError_t e = cudaMallocAsync(&a.ptr, bytes, stream);
    if (e != cudaSuccess) {
      a.ptr = nullptr;
      t_last_error = std::string("cudaMallocAsync: ") + cudaGetErrorString(e);
      return SPTG_ERR_NOMEM;
    }
    a.bytes = bytes;
  }
  *out = a.ptr;
  return SPTG_OK;
}

// ------------------------------------------------------------ tensor maps
// The last tensor maps this thread encoded, keyed by everything that goes
// into them: a call on the same buffers and shape reuses them.
struct MapKey {
  const void* base;
  uint64_t inner, outer, pitch;
  uint32_t box_inner, box_outer;
  int dt, esize, swizzle;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && pitch == o.pitch &&
           box_inner == o.box_inner &&
           box_outer == o.box_outer && dt == o.dt && esize == o.esize && swizzle == o.swizzle;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool valid = false;
};
constexpr int kMapCache = 32;
thread_local MapEntry t_maps[kMapCache];
thread_local int t_map_next = 0;

int encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
                  uint64_t inner, uint64_t outer, uint64_t pitch, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle);

// A 2-D map of `outer` rows of `inner` elements, rows `pitch` elements apart
// (0: dense, pitch = inner).
int make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
                uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, uint64_t pitch = 0) {
  if (pitch == 0) pitch = inner;
  const MapKey key{base, inner, outer, pitch, box_inner, box_outer, static_cast<int>(dt), esize,
                   static_cast<int>(swizzle)};
  for (const MapEntry& e : t_maps) {
    if (e.valid && e.key == key) {
      *map = e.map;
      return SPTG_OK;
    }
  }
  int rc = encode_map_2d(map, dt, esize, base, inner, outer, pitch, box_inner, box_outer, swizzle);
  if (rc == SPTG_OK) {
    MapEntry& e = t_maps[t_map_next];
    t_map_next = (t_map_next + 1) % kMapCache;
    e.key = key;
    e.map = *map;
    e.valid = true;
  }
  return rc;
}

int encode_map_2d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
                  uint64_t inner, uint64_t outer, uint64_t pitch, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (!enc) {
    t_last_error = "cuTensorMapEncodeTiled is not available from the driver";
    return SPTG_ERR_UNSUPPORTED;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch * static_cast<uint64_t>(esize)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char b[160];
    snprintf(b, sizeof(b), "cuTensorMapEncodeTiled failed (%d) for %llux%llu box %ux%u", (int)r,
             (unsigned long long)outer, (unsigned long long)inner, box_outer, box_inner);
    t_last_error = b;
    return SPTG_ERR_ARG;
  }
  return SPTG_OK;
}

// A 3-D view of a K-major operand (rows of K 16-bit elements, `pitch`
// elements apart) as (64-element K-chunk, row, chunk index), the chunk index
// stepping 128 bytes: one box of {64, box_rows, ksub} then lands as ksub
// consecutive 128-byte-swizzled sub-tiles of box_rows x 64, the layout of
// ksub separate 2-D boxes. Needs K to be a multiple of 64. Cached like the
// 2-D maps.
struct ChunkMapEntry {
  const void* base = nullptr;
  uint64_t K = 0, rows = 0, pitch = 0;
  uint32_t box_rows = 0, ksub = 0;
  int dt = -1;
  CUtensorMap map;
};
constexpr int kChunkMapCache = 32;  // as many as the 2-D maps: rotating operand sets hit
thread_local ChunkMapEntry t_chunk_maps[kChunkMapCache];
thread_local int t_chunk_next = 0;

int make_map_kchunks(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t K,
                     uint64_t rows, uint64_t pitch, uint32_t box_rows, uint32_t ksub) {
  for (const ChunkMapEntry& e : t_chunk_maps) {
    if (e.base == base && e.K == K && e.rows == rows && e.pitch == pitch &&
        e.box_rows == box_rows && e.ksub == ksub && e.dt == static_cast<int>(dt)) {
      *map = e.map;
      return SPTG_OK;
    }
  }
  auto enc = tensor_map_encoder();
  if (!enc) {
    t_last_error = "cuTensorMapEncodeTiled is not available from the driver";
    return SPTG_ERR_UNSUPPORTED;
  }
  cuuint64_t dims[3] = {64, rows, K / 64};
  cuuint64_t strides[2] = {pitch * 2, 128};
  cuuint32_t box[3] = {64, box_rows, ksub};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return SPTG_ERR_ARG;
  ChunkMapEntry& e = t_chunk_maps[t_chunk_next];
  t_chunk_next = (t_chunk_next + 1) % kChunkMapCache;
  e.base = base;
  e.K = K;
  e.rows = rows;
  e.pitch = pitch;
  e.box_rows = box_rows;
  e.ksub = ksub;
  e.dt = static_cast<int>(dt);
  e.map = *map;
  return SPTG_OK;
}

// ------------------------------------------------------------ dtype table
struct DtypeInfo {
  int in_bytes, out_bytes;
  bool in_bf16, is_int8;
  int out_kind;
  CUtensorMapDataType in_tma, out_tma;
  const char* name;
};

bool dtype_info(int dtype, DtypeInfo& d) {
  switch (dtype) {
    case SPTG_F16_F32:
      d = {2, 4, false, false, OUT_F32, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
           CU_TENSOR_MAP_DATA_TYPE_FLOAT32, "f16_f32"};
      return true;
    case SPTG_F16_F16:
      d = {2, 2, false, false, OUT_F16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
           CU_TENSOR_MAP_DATA_TYPE_FLOAT16, "f16_f16"};
      return true;
    case SPTG_S8_S32:
      d = {1, 4, false, true, OUT_S32, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
           CU_TENSOR_MAP_DATA_TYPE_INT32, "s8_s32"};
      return true;
    case SPTG_BF16_BF16:
      d = {2, 2, true, false, OUT_BF16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
           CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, "bf16_bf16"};
      return true;
    case SPTG_BF16_F32:
      d = {2, 4, true, false, OUT_F32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
           CU_TENSOR_MAP_DATA_TYPE_FLOAT32, "bf16_f32"};
      return true;
    default:
      return false;
  }
}

// ------------------------------------------------------------ launching
// Launches a kernel variant with the given arguments; a CTA-pair variant
// goes out as clusters of two.
// Every launch allows programmatic dependent launch: the kernel may start its
// set-up while the previous kernel of the stream drains, and waits for that
// kernel (griddepcontrol.wait) before touching global memory.
cudaError_t launch_variant(const KernelVariant& v, int grid, cudaStream_t stream, void** args,
                           bool overlap_previous, int cluster = 0) {
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(grid, 1, 1);
  lc.blockDim = dim3(v.threads, 1, 1);
  lc.dynamicSmemBytes = v.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (v.pair || cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = v.pair ? 2 : cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (overlap_previous) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  lc.attrs = n ? attr : nullptr;
  lc.numAttrs = n;
  return cudaLaunchKernelExC(&lc, v.fn, args);
}

// How many CTA pairs of a pair variant can be resident at once.
// How many clusters of `cluster` CTAs of a variant can be resident at once.
std::map<std::tuple<int, const void*, int>, int> g_cluster_slots;

int cluster_slots(int dev, const KernelVariant& v, int cluster, int sm_count) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_cluster_slots.find({dev, v.fn, cluster});
    if (it != g_cluster_slots.end()) return it->second;
  }
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(cluster * (sm_count / cluster), 1, 1);
  lc.blockDim = dim3(v.threads, 1, 1);
  lc.dynamicSmemBytes = v.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, v.fn, &lc) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sm_count / cluster;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_cluster_slots[{dev, v.fn, cluster}] = n;
  return n;
}

int pair_slots(int dev, const KernelVariant& v, int sm_count) {
  return cluster_slots(dev, v, 2, sm_count);
}

// ------------------------------------------------------------ square path
bool pick_square(const DtypeInfo& d, int bn, int stages, bool pair, KernelVariant* v,
                 int kch = 1) {
  if (d.is_int8) return kch == 1 && square_variant_s8(bn, stages, pair, v);
  switch (d.out_kind) {
    case OUT_F16: return !d.in_bf16 && square_variant_f16_f16(bn, stages, pair, v, kch);
    case OUT_BF16: return d.in_bf16 && square_variant_bf16_bf16(bn, stages, pair, v, kch);
    case OUT_F32:
      return d.in_bf16 ? square_variant_bf16_f32(bn, stages, pair, v, kch)
                       : square_variant_f16_f32(bn, stages, pair, v, kch);
    default: return false;
  }
}

// 64-wide K-chunks per ring stage of a square tile: two for float CTA pairs
// over K-loops of 32 K-chunks or more whose two-chunk ring still holds four
// stages (up to 176 columns with 16-bit C, 128 with fp32 C), one elsewhere
// and with a forced ring depth. Narrow pair tiles pay a stage's barrier trips
// and MMA issue for little tensor work; two chunks halve that per FLOP. Same
// box, us, one / two chunks: 768 x 8192 x 8192 bfloat16 on 256 x 176 pairs
// 65.9 / 61.0, 256 x 8192 x 8192 on 256 x 112 pairs 34.9 / 31.1; with three
// stages it lost (4096^3 on 256 x 224 pairs 78.0 / 80.2, 512 x 8192 x 8192 on
// 256 x 224 pairs 40.9 / 44.3), and single CTAs, whose rings are half as
// deep, lost most (384 x 8192 x 8192 on 128 x 176 tiles, two stages: 40.2 /
// 52.8).
int square_kch(const DtypeInfo& d, int bn, bool pair, int64_t K, const sptg_config& cfg) {
  if (d.is_int8 || !pair || cfg.stages != 0 || (K + 63) / 64 < 32) return 1;
  KernelVariant v2;
  return (pick_square(d, bn, 0, true, &v2, 2) && v2.stages >= 4) ? 2 : 1;
}

// Per-FLOP rate of each tile shape measured on GB300 (binary16 8192 x 8192 x
// 4096 data-parallel, TFLOPS with wave quantisation and padding divided out:
// rounds x workers x tile FLOPs / time), for BN = 512 (pairs only) and 256
// down to 112 in steps of 16: the weights of the shape model below. Narrow
// tiles lose more than their share: a K-tile's copies and barrier trip cost
// about the same whatever its width. (The 512 entry was measured on another
// box and scaled by the ratio of the two boxes' 256-wide pair rates.)
constexpr int kNumWidths = 11;
constexpr int kTileWidths[kNumWidths] = {512, 256, 240, 224, 208, 192, 176, 160, 144, 128, 112};
constexpr double kRatePair[kNumWidths] = {2103, 1915, 1889, 1875, 1829, 1729, 1648, 1558, 1434, 1312, 1189};
constexpr double kRateSingle[kNumWidths] = {0, 1684, 1639, 1613, 1684, 1669, 1557, 1507, 1414, 1224, 1138};

// Stream-K part of the schedule for T tiles over W workers, KT K-tiles each:
// the tiles of a partial last round (mode 0, when that round is at most 90 %
// full), none (mode 1), or every tile (mode 2, a test setting), cut over
// enough workers that each gets at least 8 K-tiles. sk_tiles = 0: nothing
// is cut.
void plan_stream_k(int T, int W, int KT, int mode, int* sk_tiles, int* sk_workers,
                   int* max_contrib) {
  *sk_tiles = 0;
  *sk_workers = 0;
  *max_contrib = 1;
  int t = 0;
  if (mode == 2)
    t = T;
  else if (mode == 0 && T % W != 0 && T % W <= (9 * W) / 10)
    t = T % W;
  if (t == 0) return;
  const int64_t units = static_cast<int64_t>(t) * KT;
  int sw = static_cast<int>(std::min<int64_t>(W, units / 8));
  if (sw < 2) {
    if (mode != 2) return;
    sw = 1;
  }
  // every worker holds at least floor(units / sw) consecutive units, so a
  // tile of KT units meets at most ceil(KT / that) + 1 of them
  const int64_t per = units / sw;
  const int mc = static_cast<int>((KT + per - 1) / per) + 1;
  *sk_tiles = t;
  *sk_workers = sw;
  *max_contrib = std::min(mc, sw);
}

// Tile shape and schedule: one CTA (128 x BN) or a CTA pair (256 x BN) per
// tile, data-parallel or with a partial last round cut along K. The estimate
// is in microseconds: a worker (one SM or one CTA pair) does a K-tile of its
// tile in t_k = 2 x rows x BN x 64 / (rate / workers), with the measured
// per-width rate; the data-parallel schedule takes ceil(tiles / workers)
// rounds of K-tiles, the stream-K one tiles / workers rounds plus the cost
// of cutting: 8 us for the partial writes and reductions and 0.1 us per
// K-tile of the tile (fitted to stream-K against data-parallel 256 x 256
// pair schedules at 4096^3, 8192 x 8192 x 4096, 6144^3, 12288^3 and
// 8192 x 8192 x 16384: a data-parallel last round that is partly idle runs
// faster than a full one, and more so the longer the K-loop). The cheapest
// estimate wins; ties keep the wider tile and the data-parallel schedule.
double stream_k_fixed_us(int k_tiles) { return 8.0 + 0.1 * k_tiles; }

// 256 x 512 pair tiles (two 256-column MMAs per K-step) move a quarter fewer
// operand bytes per FLOP (the 2133 TFLOPS rate above, fitted to 8192 x 8192
// x {8192, 16384}) but hold one accumulator, so each round also pays its
// epilogue and refill. 4.3 us fits those two runs; 6 us also keeps 6144^3
// on 256-wide tiles, where they measured 1.5 % faster. Measured wins:
// 16384^3 5 %, 8192 x 8192 x 16384 2-3 %; 8192^3 and 12288^3 even.
constexpr double kWideEpilogueUs = 6.0;

// A CTA pair costs a fixed extra over its K-loop rate: the cluster launch,
// the pair's barrier and tensor-memory set-up and teardown, and a tail its
// halved B traffic cannot pay back within one round. Products of one round
// (CUDA-graph replay, binary16, us, single / pair): 256^3 3.71 / 4.23,
// 512^3 4.71 / 5.04, 1024^3 6.72 / 7.17, 1536^3 9.30 / 10.62, 1024 x 1024 x
// 4096 17.50 / 17.84, 1024 x 4096 x 1024 9.62 / 10.22, 2048^3 15.40 / 15.17;
// the rate model alone put the pair 0.05-1.8 us ahead in all of them. 1.4 us
// makes it pick the faster mode in each.
constexpr double kPairFixedUs = 1.4;

void choose_square_shape(int64_t M, int64_t N, int64_t K, int sm_count, const sptg_config& cfg,
                         bool int8, int* bn_out, bool* pair_out, bool* sk_out) {
  double best = 1e300;
  *bn_out = 256;
  *pair_out = false;
  *sk_out = false;
  const int KT = static_cast<int>((K + 63) / 64);
  for (int pair = 0; pair < 2; ++pair) {
    if ((cfg.cta_pair == 1 && pair) || (cfg.cta_pair == 2 && !pair)) continue;
    if (pair && M <= 128 && cfg.cta_pair != 2) continue;  // one CTA already covers all rows
    const int64_t rows = pair ? 256 : 128;
    const int W = pair ? sm_count / 2 : sm_count;
    for (int i = 0; i < kNumWidths; ++i) {
      const int bn = kTileWidths[i];
      if (cfg.bn && bn != cfg.bn) continue;
      // 512 columns: CTA pairs and float types only; int8 in 32-column steps
      if (bn == 512 && (!pair || int8)) continue;
      if (int8 && bn % 32 != 0) continue;
      const int64_t T64 = ((M + rows - 1) / rows) * ((N + bn - 1) / bn);
      const int T = static_cast<int>(std::min<int64_t>(T64, INT32_MAX));
      const double rate = (pair ? kRatePair[i] : kRateSingle[i]) * 1e6;  // FLOP per us
      const double t_k = 2.0 * rows * bn * 64 / (rate / W);            // us per K-tile
      for (int sk = 0; sk < 2; ++sk) {
        double cost = static_cast<double>((T + W - 1) / W) * KT * t_k + (pair ? kPairFixedUs : 0.0);
        if (bn == 512) {
          // one accumulator: each round's epilogue is exposed; never cut
          if (sk) continue;
          cost += static_cast<double>((T + W - 1) / W) * kWideEpilogueUs;
        }
        if (sk) {
          if (cfg.stream_k == 1) continue;
          int skt, skw, mc;
          plan_stream_k(T, W, KT, 0, &skt, &skw, &mc);
          if (skt == 0) continue;
          cost = static_cast<double>(T) / W * KT * t_k + stream_k_fixed_us(KT) +
                 (pair ? kPairFixedUs : 0.0);
        }
        if (cost < best) {
          best = cost;
          *bn_out = bn;
          *pair_out = pair != 0;
          *sk_out = sk != 0;
        }
      }
    }
  }
}

struct SquarePlan {
  KernelVariant v;
  bool pair;
  int kch;  // 64-wide K-chunks per ring stage
  int tile_m, m_tiles, n_tiles, k_tiles, workers, grid;
  int sk_tiles, sk_workers, max_contrib;
  size_t partial_bytes;  // scratch for the stream-K partial tiles (0: none)
};

int plan_square(int dev, const DeviceInfo& di, const DtypeInfo& d, int64_t M, int64_t N,
                int64_t K, const sptg_config& cfg, SquarePlan* pl) {
  int bn = 0;
  bool pair = false, sk = false;
  choose_square_shape(M, N, K, di.sm_count, cfg, d.is_int8, &bn, &pair, &sk);
  if (cfg.bn && bn != cfg.bn) {
    t_last_error = "the requested tile width does not exist for this dtype/pairing";
    return SPTG_ERR_CONFIG;
  }
  int kch = square_kch(d, bn, pair, K, cfg);
  if (!pick_square(d, bn, cfg.stages, pair, &pl->v, kch)) {
    // a forced ring depth may exist for the other tile mode only
    if (cfg.cta_pair == 0 && pick_square(d, bn, cfg.stages, !pair, &pl->v, kch)) {
      pair = !pair;
    } else if (kch != 1 && pick_square(d, bn, cfg.stages, pair, &pl->v, 1)) {
      kch = 1;
    } else {
      t_last_error = "no square-kernel variant for the requested bn/stages/pairing";
      return SPTG_ERR_CONFIG;
    }
  }
  pl->kch = pl->v.ksub;
  int rc = ensure_smem(dev, pl->v.fn, pl->v.smem);
  if (rc) return rc;
  pl->pair = pair;
  pl->tile_m = pair ? 256 : 128;
  pl->m_tiles = static_cast<int>((M + pl->tile_m - 1) / pl->tile_m);
  pl->n_tiles = static_cast<int>((N + pl->v.bn - 1) / pl->v.bn);
  pl->k_tiles = static_cast<int>((K + 64 * pl->kch - 1) / (64 * pl->kch));  // ring stages
  const int tiles = pl->m_tiles * pl->n_tiles;
  int workers = pair ? pair_slots(dev, pl->v, di.sm_count) : di.sm_count;
  if (cfg.splits > 0) workers = std::min(workers, cfg.splits);
  plan_stream_k(tiles, workers, pl->k_tiles, cfg.stream_k == 2 ? 2 : (sk ? 0 : 1), &pl->sk_tiles,
                &pl->sk_workers, &pl->max_contrib);
  if (pl->sk_tiles == 0)
    workers = std::min(workers, tiles);
  else if (pl->sk_tiles == tiles)
    workers = pl->sk_workers;  // no data-parallel tiles: idle workers are not launched
  pl->workers = workers;
  pl->grid = pair ? 2 * workers : workers;
  pl->partial_bytes =
      static_cast<size_t>(pl->sk_tiles) * 2 * pl->max_contrib * 128 * pl->v.bn * 4;
  if (static_cast<size_t>(pl->sk_tiles) * 2 * sizeof(unsigned long long) > kCounterArea) {
    t_last_error = "too many stream-K tiles for the arrival-counter area";
    return SPTG_ERR_CONFIG;
  }
  return SPTG_OK;
}

int launch_square(const DeviceInfo& di, const DtypeInfo& d, int64_t M, int64_t N, int64_t K,
                  const void* A16, int64_t lda, const void* B16, int64_t ldb, void* C,
                  int64_t ldc, cudaStream_t stream, const sptg_config& cfg, const SquarePlan& pl,
                  void* partials, unsigned long long* counters, unsigned int generation) {
  const int BM = 128, BK = 64;
  CUtensorMap ta, tb, tc;
  int rc = make_map_2d(&ta, d.in_tma, 2, A16, K, M, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B, lda);
  if (rc) return rc;
  rc = make_map_2d(&tb, d.in_tma, 2, B16, K, N, BK,
                   pl.v.bn > 256 ? pl.v.bn / 4 : pl.pair ? pl.v.bn / 2 : pl.v.bn,
                   CU_TENSOR_MAP_SWIZZLE_128B, ldb);
  if (rc) return rc;
  // C blocks of 32 columns x 32 rows: 128-byte rows for 4-byte outputs,
  // 64-byte rows for 16-bit ones (matching the kernel's staging swizzle)
  rc = make_map_2d(&tc, d.out_tma, d.out_bytes, C, N, M, 32, 32,
                   d.out_bytes == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, ldc);
  if (rc) return rc;

  SquareParams p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.C_out = C;
  p.ldc = ldc;
  p.num_m_tiles = pl.m_tiles;
  p.num_n_tiles = pl.n_tiles;
  p.num_k_tiles = pl.k_tiles;
  p.k_tiles_per_chunk = d.is_int8 ? 1024 / BK : pl.k_tiles;
  // Raster: strips of group_m tile rows, walked column by column. Measured
  // on 4096^3 .. 16384 x 16384 x 4096 and 8192 x 8192 x 16384: 16-row strips
  // are best up to K = 4096 (0.6-1.8 % over 8), 12-row strips are never
  // worse than 8 beyond (16 loses 2-3 % there: the strip's A rows outgrow
  // L2).
  p.group_m = K <= 4096 ? 16 : 12;
  p.sk_tiles = pl.sk_tiles;
  p.sk_workers = pl.sk_workers;
  p.max_contrib = pl.max_contrib;
  p.partials = static_cast<uint32_t*>(partials);
  p.counters = counters;
  p.generation = generation;
  p.error_word = di.error_word;
  p.timeout_ns = static_cast<uint64_t>(cfg.timeout_ms > 0 ? cfg.timeout_ms : 2000) * 1000000ull;
  p.inject_stall = cfg.inject_stall;
  p.trace = static_cast<unsigned long long*>(cfg.trace);
  p.b_once = pl.m_tiles == 1 ? 1 : 0;
  void* args[] = {&ta, &tb, &tc, &p};
  cudaError_t e = launch_variant(pl.v, pl.grid, stream, args, !cfg.no_overlap);
  ++t_launches;
  if (e != cudaSuccess) return cuda_fail(e, "square_gemm launch");
  set_config(
      "kernel=square dtype=%s tile_m=%lld bn=%lld bk=%lld stages=%lld pair=%lld grid=%lld "
      "tiles=%lld k_tiles=%lld chunk_k_tiles=%lld stream_k_tiles=%lld stream_k_workers=%lld "
      "kch=%lld smem=%lld",
      d.name, {pl.tile_m, pl.v.bn, BK, pl.v.stages, pl.pair ? 1 : 0, pl.grid,
               static_cast<long long>(pl.m_tiles) * pl.n_tiles, pl.k_tiles, p.k_tiles_per_chunk,
               pl.sk_tiles, pl.sk_workers, pl.kch, pl.v.smem});
  return SPTG_OK;
}

// ------------------------------------------------------------ skinny path
// Caller-provided scratch for the skinny kernel's split-K partials and
// arrival counters (used by sptg_gemm_skinny_noalloc); null = the cached
// per-stream scratch of scratch_for().
struct FixedScratch {
  void* partials;
  size_t partial_bytes;
  void* counters;
  size_t counter_bytes;
  std::atomic<unsigned int>* generation;
};

// Next non-zero call generation of a scratch area.
unsigned int next_generation(std::atomic<unsigned int>* g) {
  unsigned int v = g->fetch_add(1) + 1;
  if (v == 0) v = g->fetch_add(1) + 1;
  return v;
}

int run_skinny(int dev, const DeviceInfo& di, const DtypeInfo& d, int64_t M, int64_t N, int64_t K,
               const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
               cudaStream_t stream, const sptg_config& cfg, const FixedScratch* fixed = nullptr) {
  KernelVariant v;
  if (d.is_int8 || !skinny_variant(d.in_bf16, d.out_kind, cfg.stages, &v) || M > v.bn) {
    t_last_error = "no skinny-kernel variant for the requested dtype/stages/M";
    return SPTG_ERR_CONFIG;
  }
  const int BNT = 128, BK = 64;
  const int kstep = BK * v.ksub;  // K per ring stage (one unit of work)
  CUtensorMap tb, ta;
  // MMA operand A is the B^T tile (128 output columns x 64 k), operand B is the A tile.
  int rc = make_map_2d(&tb, d.in_tma, 2, B, K, N, BK, BNT, CU_TENSOR_MAP_SWIZZLE_128B, ldb);
  if (rc) return rc;
  rc = make_map_2d(&ta, d.in_tma, 2, A, K, M, BK, v.bn, CU_TENSOR_MAP_SWIZZLE_128B, lda);
  if (rc) return rc;
  rc = ensure_smem(dev, v.fn, v.smem);
  if (rc) return rc;

  SkinnyParams p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_n_tiles = static_cast<int>((N + BNT - 1) / BNT);
  p.num_k_tiles = static_cast<int>((K + kstep - 1) / kstep);
  const int64_t units = static_cast<int64_t>(p.num_n_tiles) * p.num_k_tiles;
  int grid = cfg.splits > 0 ? cfg.splits : di.sm_count;
  grid = static_cast<int>(std::min<int64_t>(grid, units));
  p.num_ctas = grid;
  p.total_units = units;
  // Largest number of CTAs that can share one n-tile: ceil(kt / per_cta) + 1.
  const int64_t per_cta_min = units / grid;
  int max_contrib = per_cta_min > 0 ? static_cast<int>((p.num_k_tiles + per_cta_min - 1) / per_cta_min) + 1
                                    : grid;
  max_contrib = std::min(max_contrib, grid);
  p.max_contrib = max_contrib;
  p.C = C;
  p.ldc = ldc;
  p.error_word = di.error_word;
  p.timeout_ns = static_cast<uint64_t>(cfg.timeout_ms > 0 ? cfg.timeout_ms : 2000) * 1000000ull;
  p.inject_stall = cfg.inject_stall;
  p.trace = static_cast<unsigned long long*>(cfg.trace);

  // Scratch: fp32 partial tiles [n_tile][contributor][MN x 128] then one
  // arrival counter per n-tile (zeroed here, and re-zeroed by the last arrival).
  // Partials are needed as soon as one CTA boundary falls inside an n-tile.
  bool split = false;
  for (int c = 1; c < grid && !split; ++c)
    split = ((static_cast<int64_t>(c) * units / grid) % p.num_k_tiles) != 0;
  size_t partial_bytes = 0, counter_bytes = 0;
  if (split) {
    partial_bytes = static_cast<size_t>(p.num_n_tiles) * max_contrib * v.bn * BNT * sizeof(float);
    counter_bytes = static_cast<size_t>(p.num_n_tiles) * sizeof(unsigned long long);
    if (fixed) {
      if (partial_bytes > fixed->partial_bytes || counter_bytes > fixed->counter_bytes) {
        char b[200];
        snprintf(b, sizeof(b),
                 "shape needs %zu bytes of split-K partials and %zu of counters; the fixed "
                 "scratch holds %zu and %zu",
                 partial_bytes, counter_bytes, fixed->partial_bytes, fixed->counter_bytes);
        t_last_error = b;
        return SPTG_ERR_CONFIG;
      }
      p.partials = static_cast<float*>(fixed->partials);
      p.counters = static_cast<unsigned long long*>(fixed->counters);
      p.generation = next_generation(fixed->generation);
    } else {
      if (counter_bytes > kCounterArea) {
        t_last_error = "too many column tiles for the split-K counter area";
        return SPTG_ERR_CONFIG;
      }
      ScratchView ws;
      rc = scratch_for(dev, stream, partial_bytes, &ws);
      if (rc) return rc;
      p.partials = static_cast<float*>(ws.data);
      p.counters = ws.counters;
      p.generation = ws.generation;
    }
  } else {
    p.partials = nullptr;
    p.counters = nullptr;
    p.generation = 0;
  }
  void* args[] = {&tb, &ta, &p};
  cudaError_t e = launch_variant(v, grid, stream, args, !cfg.no_overlap);
  ++t_launches;
  if (e != cudaSuccess) return cuda_fail(e, "skinny_gemm launch");
  set_config(
      "kernel=skinny dtype=%s mma_m=%lld mma_n=%lld bk=%lld stages=%lld grid=%lld n_tiles=%lld "
      "k_tiles=%lld units=%lld max_contrib=%lld smem=%lld",
      d.name, {BNT, v.bn, kstep, v.stages, grid, p.num_n_tiles, p.num_k_tiles, (long long)units,
               max_contrib, v.smem});
  return SPTG_OK;
}

// ------------------------------------------------- skinny kernel geometry
// Host-only decisions of the skinny kernels, shared by the launches below and
// by sptg_plan. Each returns SPTG_ERR_CONFIG when the shape does not suit the
// kernel (with t_last_error set when the kernel was forced).

// Output columns one SM would own: N / SMs rounded up to a multiple of 8.
int64_t columns_per_sm(int64_t N, int sm_count) {
  const int64_t c = ((N + sm_count - 1) / sm_count + 7) / 8 * 8;
  return c < 8 ? 8 : c;
}

// CTA pairs: output columns per CTA (forced bn, else columns_per_sm) and
// pairs. Unforced, at most 128 columns per CTA and one CTA per SM, and (with
// `fill`) at least three quarters of the SMs busy.
int pair_geometry(int64_t N, int sm_count, const sptg_config& cfg, bool forced, bool fill,
                  int64_t* nc_out, int64_t* pairs_out) {
  int64_t nc = cfg.bn;
  if (forced && nc > 0) {
    if (nc % 8 != 0 || nc < 8 || nc > 128) {
      t_last_error = "columns per CTA (bn) must be a multiple of 8 from 8 to 128";
      return SPTG_ERR_CONFIG;
    }
  } else {
    nc = columns_per_sm(N, sm_count);
  }
  const int64_t pairs = (N + 2 * nc - 1) / (2 * nc);
  if (!forced && (nc > 128 || 2 * pairs > sm_count ||
                  (fill && 8 * pairs < 3 * static_cast<int64_t>(sm_count))))
    return SPTG_ERR_CONFIG;
  if (nc > 128) {
    t_last_error = "N needs more than 128 columns per CTA on this GPU";
    return SPTG_ERR_CONFIG;
  }
  *nc_out = nc;
  *pairs_out = pairs;
  return SPTG_OK;
}

// Column strips: strip width (forced bn, else columns_per_sm) and strips.
// Unforced, 32 to 256 columns, at most one strip per SM and at least three
// quarters of the SMs busy.
int rows_geometry(int64_t N, int sm_count, const sptg_config& cfg, bool forced, int64_t* nt_out,
                  int64_t* strips_out) {
  int64_t nt = cfg.bn;
  if (forced && nt > 0) {
    if (nt % 8 != 0 || nt < 8 || nt > SKINNY_ROWS_MAX_NT) {
      t_last_error = "column-strip width (bn) must be a multiple of 8 from 8 to 256";
      return SPTG_ERR_CONFIG;
    }
  } else {
    nt = columns_per_sm(N, sm_count);
  }
  const int64_t strips = (N + nt - 1) / nt;
  if (!forced && (nt < 32 || nt > SKINNY_ROWS_MAX_NT || strips > sm_count ||
                  strips * 4 < 3 * static_cast<int64_t>(sm_count)))
    return SPTG_ERR_CONFIG;
  if (nt > SKINNY_ROWS_MAX_NT) {
    t_last_error = "N needs column strips wider than 256 on this GPU";
    return SPTG_ERR_CONFIG;
  }
  *nt_out = nt;
  *strips_out = strips;
  return SPTG_OK;
}

// Cluster split of variant v: 128-column tiles, K-steps of 64 * v.ksub and
// the cluster size -- forced (splits), else the largest of 4, 2, 1 whose CTAs
// (cluster size per column tile) fit the SMs, taken only if the grid fills at
// least three quarters of the SMs (unless `fill` is false). The receive
// buffer holds up to 3 x 32 columns (clusters of 4) for MMA N = 64 and 64
// columns (clusters of 2) for MMA N = 128.
int cluster_geometry(int64_t N, int64_t K, const KernelVariant& v, int sm_count,
                     const sptg_config& cfg, bool forced, bool fill, int* n_tiles_out,
                     int* k_tiles_out, int* cs_out) {
  const int n_tiles = static_cast<int>((N + 127) / 128);
  const int kstep = 64 * v.ksub;
  const int k_tiles = static_cast<int>((K + kstep - 1) / kstep);
  const int max_cs = v.bn <= 64 ? 4 : 2;
  int cs = 0;
  if (forced && cfg.splits > 0) {
    cs = cfg.splits;
    if ((cs != 1 && cs != 2 && cs != 4) || cs > max_cs) {
      t_last_error = max_cs == 4 ? "cluster size must be 1, 2 or 4"
                                 : "cluster size must be 1 or 2 for more than 64 rows";
      return SPTG_ERR_CONFIG;
    }
  } else {
    for (int c : {4, 2, 1}) {
      if (c > max_cs) continue;
      if (static_cast<int64_t>(n_tiles) * c <= sm_count && k_tiles >= 2 * c) {
        cs = c;
        break;
      }
    }
    if (cs == 0 && forced) {
      t_last_error = "no cluster size fits: the 128-column tiles outnumber the SMs";
      return SPTG_ERR_CONFIG;
    }
    if (cs == 0 || (!forced && fill && static_cast<int64_t>(n_tiles) * cs * 4 < 3 * sm_count))
      return SPTG_ERR_CONFIG;
  }
  *n_tiles_out = n_tiles;
  *k_tiles_out = k_tiles;
  *cs_out = cs;
  return SPTG_OK;
}

// The automatic choice for a memory-bound shape (float, M <= 256, N >= 1024):
// the kernels to try in order (5 CTA pairs, 4 column strips, 3 cluster split),
// each with whether its grid must fill three quarters of the SMs; if none
// takes the shape, stream-K (M <= 64) or the square kernel does. With c =
// columns_per_sm(N):
//  - up to 64 rows: CTA pairs over the whole of K for 32 <= c <= 64, one CTA
//    per column strip for 64 < c <= 256, the cluster split for c < 32 even
//    where its grid leaves SMs idle (its short K-ranges and the 4-CTA
//    exchange beat stream-K there) unless K is long, else the cluster split
//    when it fills the GPU, else stream-K;
//  - 65-128 rows: CTA pairs for c <= 128 (two 64-column blocks per CTA past
//    64) even where they leave SMs idle, else the cluster split when it
//    fills the GPU, else the square kernel;
//  - 129-256 rows: CTA pairs with MMA N = 256 for c <= 64, else the square
//    kernel.
// Measured on 152 SMs (bfloat16, K = 8192 unless given), us:
//   64 rows: N = 1024 cluster 12.9 (stream-K 24.1, pairs 15.1); 2048 13.3
//   (17.4, 15.3); 3072 14.8 (16.9, 15.7); 4096-9216 pairs (5120: 16.7
//   against cluster 19.6); 10240-38912 strips (32768 x 4096: 40.7
//   against stream-K 45.2); wider stream-K; K = 32768, N = 1024-2048:
//   stream-K 30-31, cluster 31-32, pairs 49;
//   128 rows: N = 1536 pairs 16.1 (square 66.1); 4096 17.3 (square
//   63.7); 8192 24.5-25.2 (cluster 27.7); 10240 34.9 (square 36.5);
//   96 x 14336: 40.3 (square 44.3); 16384-19456 K = 4096 level with the
//   cluster split. Up to 64 rows the strips beat pairs past c = 64
//   (10240: 29.2 against 31.9). 256 rows: N = 4096 (K = 4096) 16.4
//   (square 18.0), 8192 32.4-33.4 (square 34.4), 16384 (K = 4096) 31.5
//   (square 28.0: three stages fit); 160 rows x 8192: 31.4 (34.1).
struct SkinnyTry {
  int kernel;
  bool fill;
};
int skinny_order(int64_t M, int64_t N, int64_t K, int sm_count, SkinnyTry out[3]) {
  const int64_t c = columns_per_sm(N, sm_count);
  int n = 0;
  if ((M > 64 && M <= 128 && c <= 128) || (M > 128 && c <= 64) || (c >= 32 && c <= 64))
    out[n++] = {5, M <= 64};
  if (M <= 64 && c > 64) out[n++] = {4, true};
  out[n++] = {3, !(M <= 64 && c < 32 && K <= 16384)};
  return n;
}

// The skinny product with K split inside clusters: one cluster of `cs` CTAs
// per 128-column tile. Returns SPTG_ERR_CONFIG (and launches nothing) when
// the shape does not suit it, so that the caller can use the stream-K kernel.
int run_skinny_cluster(int dev, const DeviceInfo& di, const DtypeInfo& d, int64_t M, int64_t N,
                       int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                       void* C, int64_t ldc, cudaStream_t stream, const sptg_config& cfg,
                       bool forced, bool fill = true) {
  KernelVariant v;
  if (d.is_int8 || !skinny_cluster_variant(d.in_bf16, d.out_kind, cfg.stages, static_cast<int>(M),
                                           &v) ||
      M > v.bn) {
    if (forced) t_last_error = "no cluster-split skinny variant for the requested dtype/stages/M";
    return SPTG_ERR_CONFIG;
  }
  const int BNT = 128, BK = 64;
  const int kstep = BK * v.ksub;  // K per ring stage
  int n_tiles = 0, k_tiles = 0, cs = 0;
  int rc = cluster_geometry(N, K, v, di.sm_count, cfg, forced, fill, &n_tiles, &k_tiles, &cs);
  if (rc) return rc;
  rc = ensure_smem(dev, v.fn, v.smem);
  if (rc) return rc;
  if (cs > 1 && !forced && cluster_slots(dev, v, cs, di.sm_count) < n_tiles) return SPTG_ERR_CONFIG;
  CUtensorMap tb, ta, tc;
  // With several K-chunks per stage and K a multiple of 64, one 3-D copy per
  // operand moves a whole stage; otherwise one 2-D copy per chunk.
  int load3d = 0;
  if (v.ksub > 1 && K % 64 == 0 &&
      make_map_kchunks(&tb, d.in_tma, B, K, N, ldb, BNT, v.ksub) == SPTG_OK &&
      make_map_kchunks(&ta, d.in_tma, A, K, M, lda, v.bn, v.ksub) == SPTG_OK)
    load3d = 1;
  if (!load3d) {
    rc = make_map_2d(&tb, d.in_tma, 2, B, K, N, BK, BNT, CU_TENSOR_MAP_SWIZZLE_128B, ldb);
    if (rc) return rc;
    rc = make_map_2d(&ta, d.in_tma, 2, A, K, M, BK, v.bn, CU_TENSOR_MAP_SWIZZLE_128B, lda);
    if (rc) return rc;
  }
  // the output block a rank stores: v.bn rows of 128 / cs consecutive
  // outputs, unswizzled
  rc = make_map_2d(&tc, d.out_tma, d.out_bytes, C, N, M, BNT / cs, v.bn,
                   CU_TENSOR_MAP_SWIZZLE_NONE, ldc);
  if (rc) return rc;
  SkinnyClusterParams p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_n_tiles = n_tiles;
  p.num_k_tiles = k_tiles;
  p.load3d = load3d;
  p.error_word = di.error_word;
  p.timeout_ns = static_cast<uint64_t>(cfg.timeout_ms > 0 ? cfg.timeout_ms : 2000) * 1000000ull;
  p.inject_stall = cfg.inject_stall;
  p.trace = static_cast<unsigned long long*>(cfg.trace);
  const int grid = n_tiles * cs;
  void* args[] = {&tb, &ta, &tc, &p};
  cudaError_t e = launch_variant(v, grid, stream, args, !cfg.no_overlap, cs);
  ++t_launches;
  if (e != cudaSuccess) return cuda_fail(e, "skinny_cluster_gemm launch");
  set_config(
      "kernel=skinny-cluster dtype=%s mma_m=%lld mma_n=%lld bk=%lld stages=%lld grid=%lld "
      "cluster=%lld n_tiles=%lld k_tiles=%lld copies_3d=%lld smem=%lld",
      d.name, {BNT, v.bn, kstep, v.stages, grid, cs, n_tiles, k_tiles, load3d, v.smem});
  return SPTG_OK;
}

// The skinny product (M <= 64) with one CTA per strip of n_tile output
// columns over the whole of K: no split, nothing exchanged. The strip width is
// forced (bn) or the multiple of 8 that covers N with at most one strip per
// SM (up to 256); the ring is as deep as shared memory allows (or forced by
// stages). Returns SPTG_ERR_CONFIG (and launches nothing) when the shape does
// not suit it -- strips narrower than 32 columns, more strips than SMs, or
// fewer than three quarters of the SMs busy -- so that the caller can try the
// others.
int run_skinny_rows(int dev, const DeviceInfo& di, const DtypeInfo& d, int64_t M, int64_t N,
                    int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                    int64_t ldc, cudaStream_t stream, const sptg_config& cfg, bool forced) {
  if (d.is_int8 || M > 64) {
    if (forced) t_last_error = "the column-strip skinny kernel takes float products with M <= 64";
    return SPTG_ERR_CONFIG;
  }
  int64_t nt = 0, strips = 0;
  int rc = rows_geometry(N, di.sm_count, cfg, forced, &nt, &strips);
  if (rc) return rc;
  KernelVariant v;
  if (!skinny_rows_variant(d.in_bf16, d.out_kind, static_cast<int>(nt), &v)) {
    if (forced) t_last_error = "no column-strip skinny variant for the requested dtype";
    return SPTG_ERR_CONFIG;
  }
  const int ksub = v.ksub;
  const int stage_bytes = static_cast<int>(ksub * (64 + nt) * 128);
  int stages = cfg.stages ? cfg.stages : SKINNY_ROWS_RING_BUDGET / stage_bytes;
  if (stages > SKINNY_ROWS_MAX_STAGES) stages = SKINNY_ROWS_MAX_STAGES;
  if (stages < 1 || stages * stage_bytes > SKINNY_ROWS_RING_BUDGET) {
    t_last_error = "ring depth out of range for the column-strip skinny kernel";
    return SPTG_ERR_CONFIG;
  }
  const int smem = stages * stage_bytes + SKINNY_ROWS_BAR_BYTES + 1024;
  rc = ensure_smem(dev, v.fn, 232448);
  if (rc) return rc;
  CUtensorMap ta, tb;
  const int kstep = 64 * ksub;
  int load3d = 0;
  if (K % 64 == 0 &&
      make_map_kchunks(&ta, d.in_tma, A, K, M, lda, 64, ksub) == SPTG_OK &&
      make_map_kchunks(&tb, d.in_tma, B, K, N, ldb, static_cast<uint32_t>(nt), ksub) == SPTG_OK)
    load3d = 1;
  if (!load3d) {
    rc = make_map_2d(&ta, d.in_tma, 2, A, K, M, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, lda);
    if (rc) return rc;
    rc = make_map_2d(&tb, d.in_tma, 2, B, K, N, 64, static_cast<uint32_t>(nt),
                     CU_TENSOR_MAP_SWIZZLE_128B, ldb);
    if (rc) return rc;
  }
  SkinnyRowsParams p;
  p.C = C;
  p.ldc = ldc;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.n_tile = static_cast<int>(nt);
  p.num_k_tiles = static_cast<int>((K + kstep - 1) / kstep);
  p.stages = stages;
  p.stage_bytes = stage_bytes;
  p.load3d = load3d;
  // Staggered K-loops (see the kernel) for K >= 8192 over 64 stages or more
  // (same box, us, without / with: 64 x 16384 x 8192 41.3 / 40.1, 64 x 12288
  // x 16384 67.4 / 65.6, 64 x 24576 x 8192 60.5 / 59.6; 64 x 16384 x 4096
  // 21.6 / 21.4; at K = 4096 over 64 one-chunk stages 0.35 % slower: 64 x
  // 32768 x 4096 40.15 / 40.3, 32 x 32000 x 4096 39.0 / 39.1).
  p.k_rotate = (K >= 8192 && p.num_k_tiles >= 64) ? 1 : 0;
  p.error_word = di.error_word;
  p.timeout_ns = static_cast<uint64_t>(cfg.timeout_ms > 0 ? cfg.timeout_ms : 2000) * 1000000ull;
  p.inject_stall = cfg.inject_stall;
  p.trace = static_cast<unsigned long long*>(cfg.trace);
  v.stages = stages;
  v.smem = smem;
  const int grid = static_cast<int>(strips);
  void* args[] = {&ta, &tb, &p};
  cudaError_t e = launch_variant(v, grid, stream, args, !cfg.no_overlap);
  ++t_launches;
  if (e != cudaSuccess) return cuda_fail(e, "skinny_rows_gemm launch");
  set_config(
      "kernel=skinny-rows dtype=%s mma_m=%lld mma_n=%lld bk=%lld stages=%lld grid=%lld "
      "k_tiles=%lld copies_3d=%lld k_rotate=%lld smem=%lld",
      d.name, {64, nt, kstep, stages, grid, p.num_k_tiles, load3d, p.k_rotate, smem});
  return SPTG_OK;
}

// The skinny product (M <= 256) on CTA pairs with the 2-SM MMA, K never split:
// each pair owns 2 * n_cta output columns. n_cta is forced (bn) or the
// multiple of 8 that covers N with at most one CTA per SM; the ring is as
// deep as shared memory allows (or forced by stages). Returns SPTG_ERR_CONFIG
// (and launches nothing) when the shape does not suit it -- more than 128
// columns per CTA, more CTAs than SMs, or (with `fill`) fewer than three
// quarters of the SMs busy -- so that the caller can try the others.
int run_skinny_pair(int dev, const DeviceInfo& di, const DtypeInfo& d, int64_t M, int64_t N,
                    int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                    int64_t ldc, cudaStream_t stream, const sptg_config& cfg, bool forced,
                    bool fill = true) {
  if (d.is_int8 || M > 256) {
    if (forced) t_last_error = "the CTA-pair skinny kernel takes float products with M <= 256";
    return SPTG_ERR_CONFIG;
  }
  int64_t nc = 0, pairs = 0;
  int rc = pair_geometry(N, di.sm_count, cfg, forced, fill, &nc, &pairs);
  if (rc) return rc;
  KernelVariant v;
  if (!skinny_pair_variant(d.in_bf16, d.out_kind, static_cast<int>(M), static_cast<int>(nc), &v)) {
    if (forced) t_last_error = "no CTA-pair skinny variant for the requested dtype";
    return SPTG_ERR_CONFIG;
  }
  const int mn = v.bn;  // rows of A on the MMA's N side: 64 or 128
  const int ksub = v.ksub;
  const int stage_bytes = skinny_pair_stage_bytes(ksub, static_cast<int>(nc), mn);
  const int max_stages = std::min(SKINNY_PAIR_MAX_STAGES, SKINNY_PAIR_RING_BUDGET / stage_bytes);
  const int stages = cfg.stages ? cfg.stages : max_stages;
  if (stages < 1 || stages > max_stages) {
    t_last_error = "ring depth out of range for the CTA-pair skinny kernel";
    return SPTG_ERR_CONFIG;
  }
  // the epilogue stages the CTA's mn x nc block of C in the ring
  if (static_cast<int64_t>(mn) * nc * d.out_bytes > static_cast<int64_t>(stages) * stage_bytes) {
    t_last_error = "the CTA-pair skinny kernel's output block does not fit this ring depth";
    return SPTG_ERR_CONFIG;
  }
  const int smem = stages * stage_bytes + SKINNY_PAIR_BAR_BYTES + 1024;
  rc = ensure_smem(dev, v.fn, 232448);
  if (rc) return rc;
  CUtensorMap tb, ta, tc;
  const int kstep = 64 * ksub;
  int load3d = 0;
  if (K % 64 == 0 &&
      make_map_kchunks(&tb, d.in_tma, B, K, N, ldb, static_cast<uint32_t>(nc), ksub) == SPTG_OK &&
      make_map_kchunks(&ta, d.in_tma, A, K, M, lda, mn / 2, ksub) == SPTG_OK)
    load3d = 1;
  if (!load3d) {
    rc = make_map_2d(&tb, d.in_tma, 2, B, K, N, 64, static_cast<uint32_t>(nc),
                     CU_TENSOR_MAP_SWIZZLE_128B, ldb);
    if (rc) return rc;
    rc = make_map_2d(&ta, d.in_tma, 2, A, K, M, 64, mn / 2, CU_TENSOR_MAP_SWIZZLE_128B, lda);
    if (rc) return rc;
  }
  // the block a CTA stores: mn rows of n_cta consecutive outputs, unswizzled
  rc = make_map_2d(&tc, d.out_tma, d.out_bytes, C, N, M, static_cast<uint32_t>(nc),
                   static_cast<uint32_t>(mn), CU_TENSOR_MAP_SWIZZLE_NONE, ldc);
  if (rc) return rc;
  SkinnyPairParams p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.n_cta = static_cast<int>(nc);
  p.num_k_tiles = static_cast<int>((K + kstep - 1) / kstep);
  p.stages = stages;
  p.stage_bytes = stage_bytes;
  p.load3d = load3d;
  // Staggered K-loops (see the kernel) for loops of 64 stages or more, as
  // for the strip kernel (same box, us, without / with: 64 x 8192 x 16384 43.7 / 42.2, 128 x 8192
  // x 8192 25.15 / 24.65, 96 x 14336 x 8192 38.9 / 38.2, 256 x 8192 x 8192
  // 32.2 / 31.8); at 32 stages it measured level or 0.5 % slower (64 x 8192 x
  // 8192 22.06 / 22.13, 64 x 4096 x 8192 15.7 / 15.7).
  p.k_rotate = (K >= 8192 && p.num_k_tiles >= 64) ? 1 : 0;
  p.error_word = di.error_word;
  p.timeout_ns = static_cast<uint64_t>(cfg.timeout_ms > 0 ? cfg.timeout_ms : 2000) * 1000000ull;
  p.inject_stall = cfg.inject_stall;
  p.trace = static_cast<unsigned long long*>(cfg.trace);
  v.stages = stages;
  v.smem = smem;
  const int grid = static_cast<int>(2 * pairs);
  void* args[] = {&tb, &ta, &tc, &p};
  cudaError_t e = launch_variant(v, grid, stream, args, !cfg.no_overlap);
  ++t_launches;
  if (e != cudaSuccess) return cuda_fail(e, "skinny_pair_gemm launch");
  set_config(
      "kernel=skinny-pair dtype=%s mma_m=128 mma_n=%lld cols_per_cta=%lld bk=%lld stages=%lld "
      "grid=%lld pairs=%lld k_tiles=%lld copies_3d=%lld k_rotate=%lld smem=%lld",
      d.name, {mn, nc, kstep, stages, grid, pairs, p.num_k_tiles, load3d, p.k_rotate, smem});
  return SPTG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------ allocation-free entry
// Fixed device scratch of sptg_gemm_skinny_noalloc: split-K partial tiles
// followed by the per-n-tile arrival counters. Every device that loads the
// library holds it until the process exits.
constexpr size_t kNoAllocPartialBytes = SPTG_NOALLOC_PARTIAL_BYTES;
constexpr size_t kNoAllocCounterBytes = SPTG_NOALLOC_COUNTER_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocPartialBytes +
                                                                 kNoAllocCounterBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current. In host code the array's name is only a host-side stand-in.
std::map<int, unsigned char*> g_noalloc_addr;
std::atomic<unsigned int> g_noalloc_generation{0};

int noalloc_scratch(int dev, unsigned char** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_noalloc_addr.find(dev);
  if (it != g_noalloc_addr.end()) {
    *out = it->second;
    return SPTG_OK;
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    t_last_error = std::string("cudaGetSymbolAddress(noalloc scratch): ") + cudaGetErrorString(e);
    return SPTG_ERR_LAUNCH;
  }
  g_noalloc_addr[dev] = static_cast<unsigned char*>(p);
  *out = static_cast<unsigned char*>(p);
  return SPTG_OK;
}

}  // namespace

// ================================================================ C ABI
extern "C" {

int sptg_version(void) { return 101; }  // 1.01: sptg_plan, skinny kernels 4 and 5

int sptg_plan_square(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, int sm_count,
                     const sptg_config* cfg_in, int* out) {
  DtypeInfo d;
  if (!out || sm_count < 2 || !dtype_info(dtype, d) || M <= 0 || N <= 0 || K <= 0 ||
      M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) {
    t_last_error = "invalid argument";
    return SPTG_ERR_ARG;
  }
  sptg_config cfg;
  memset(&cfg, 0, sizeof(cfg));
  if (cfg_in) cfg = *cfg_in;
  if (cfg.stream_k < 0 || cfg.stream_k > 2 || cfg.cta_pair < 0 || cfg.cta_pair > 2 ||
      cfg.bn < 0 || cfg.splits < 0) {
    t_last_error = "invalid configuration field";
    return SPTG_ERR_ARG;
  }
  int bn = 0;
  bool pair = false, sk = false;
  choose_square_shape(M, N, K, sm_count, cfg, d.is_int8, &bn, &pair, &sk);
  if (cfg.bn && bn != cfg.bn) {
    t_last_error = "no square-kernel tile for the requested dtype, width and pairing";
    return SPTG_ERR_CONFIG;
  }
  const int64_t rows = pair ? 256 : 128;  // tile rows
  const int64_t T64 = ((M + rows - 1) / rows) * ((N + bn - 1) / bn);
  const int tiles = static_cast<int>(std::min<int64_t>(T64, INT32_MAX));
  const int kch = square_kch(d, bn, pair, K, cfg);  // as the launch: stages of kch K-chunks
  const int k_tiles = static_cast<int>((K + 64 * kch - 1) / (64 * kch));
  int workers = pair ? sm_count / 2 : sm_count;
  if (cfg.splits > 0) workers = std::min(workers, cfg.splits);
  int skt = 0, skw = 0, mc = 1;
  plan_stream_k(tiles, workers, k_tiles, cfg.stream_k == 2 ? 2 : (sk ? 0 : 1), &skt, &skw, &mc);
  if (skt == 0)
    workers = std::min(workers, tiles);
  else if (skt == tiles)
    workers = skw;
  out[0] = bn;
  out[1] = pair ? 1 : 0;
  out[2] = tiles;
  out[3] = workers;
  out[4] = skt;
  out[5] = skw;
  out[6] = mc;
  return SPTG_OK;
}

int sptg_plan(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, int sm_count,
              const sptg_config* cfg_in, int* out) {
  DtypeInfo d;
  if (!out || sm_count < 2 || !dtype_info(dtype, d) || M <= 0 || N <= 0 || K <= 0 ||
      M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) {
    t_last_error = "invalid argument";
    return SPTG_ERR_ARG;
  }
  sptg_config cfg;
  memset(&cfg, 0, sizeof(cfg));
  if (cfg_in) cfg = *cfg_in;
  if (cfg.kernel < 0 || cfg.kernel > 5 || cfg.stream_k < 0 || cfg.stream_k > 2 ||
      cfg.cta_pair < 0 || cfg.cta_pair > 2 || cfg.bn < 0 || cfg.splits < 0 || cfg.stages < 0) {
    t_last_error = "invalid configuration field";
    return SPTG_ERR_ARG;
  }
  for (int i = 0; i < 6; ++i) out[i] = 0;
  auto set = [&](int kernel, int64_t width, int64_t grid, int cluster, int mma_n, int cut) -> int {
    out[0] = kernel;
    out[1] = static_cast<int>(width);
    out[2] = static_cast<int>(std::min<int64_t>(grid, INT32_MAX));
    out[3] = cluster;
    out[4] = mma_n;
    out[5] = cut;
    return SPTG_OK;
  };
  auto pair = [&](bool forced, bool fill) -> int {
    if (d.is_int8 || M > 256) {
      if (forced) t_last_error = "the CTA-pair skinny kernel takes float products with M <= 256";
      return SPTG_ERR_CONFIG;
    }
    int64_t nc = 0, pairs = 0;
    int rc = pair_geometry(N, sm_count, cfg, forced, fill, &nc, &pairs);
    if (rc) return rc;
    KernelVariant v;
    if (!skinny_pair_variant(d.in_bf16, d.out_kind, static_cast<int>(M), static_cast<int>(nc), &v))
      return SPTG_ERR_CONFIG;
    return set(5, nc, 2 * pairs, 2, v.bn, 0);
  };
  auto rows = [&](bool forced) -> int {
    if (d.is_int8 || M > 64) {
      if (forced) t_last_error = "the column-strip skinny kernel takes float products with M <= 64";
      return SPTG_ERR_CONFIG;
    }
    int64_t nt = 0, strips = 0;
    int rc = rows_geometry(N, sm_count, cfg, forced, &nt, &strips);
    if (rc) return rc;
    return set(4, nt, strips, 1, 64, 0);
  };
  auto cluster = [&](bool forced, bool fill) -> int {
    KernelVariant v;
    if (d.is_int8 ||
        !skinny_cluster_variant(d.in_bf16, d.out_kind, cfg.stages, static_cast<int>(M), &v) ||
        M > v.bn) {
      if (forced) t_last_error = "no cluster-split skinny variant for the requested dtype/stages/M";
      return SPTG_ERR_CONFIG;
    }
    int n_tiles = 0, k_tiles = 0, cs = 0;
    int rc = cluster_geometry(N, K, v, sm_count, cfg, forced, fill, &n_tiles, &k_tiles, &cs);
    if (rc) return rc;
    return set(3, 128, static_cast<int64_t>(n_tiles) * cs, cs, v.bn, 0);
  };
  int kernel = cfg.kernel;
  if (kernel == 0 && !d.is_int8 && M <= 256 && N >= 1024) {
    SkinnyTry order[3];
    const int n_try = skinny_order(M, N, K, sm_count, order);
    for (int t = 0; t < n_try; ++t) {
      const int rc = order[t].kernel == 5   ? pair(false, order[t].fill)
                     : order[t].kernel == 4 ? rows(false)
                                            : cluster(false, order[t].fill);
      if (rc != SPTG_ERR_CONFIG) return rc;
    }
    kernel = M <= 64 ? 2 : 1;
  }
  if (kernel == 0) kernel = 1;
  if (kernel == 3) return cluster(true, true);
  if (kernel == 4) return rows(true);
  if (kernel == 5) return pair(true, true);
  if (kernel == 2) {
    KernelVariant v;
    if (d.is_int8 || !skinny_variant(d.in_bf16, d.out_kind, cfg.stages, &v) || M > v.bn) {
      t_last_error = "no skinny-kernel variant for the requested dtype/stages/M";
      return SPTG_ERR_CONFIG;
    }
    const int64_t n_tiles = (N + 127) / 128, kstep = 64 * v.ksub;
    const int64_t units = n_tiles * ((K + kstep - 1) / kstep);
    const int64_t grid = std::min<int64_t>(cfg.splits > 0 ? cfg.splits : sm_count, units);
    return set(2, 128, grid, 1, v.bn, 0);
  }
  int sq[7];
  const int rc = sptg_plan_square(M, N, K, dtype, sm_count, &cfg, sq);
  if (rc) return rc;
  return set(1, sq[0], static_cast<int64_t>(sq[3]) * (sq[1] ? 2 : 1), sq[1] ? 2 : 1, 0, sq[4]);
}

const char* sptg_status_string(int status) {
  switch (status) {
    case SPTG_OK: return "ok";
    case SPTG_ERR_ARG: return "invalid argument";
    case SPTG_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case SPTG_ERR_UNSUPPORTED: return "no sm_103 (compute capability 10.3) device";
    case SPTG_ERR_LAUNCH: return "CUDA runtime error";
    case SPTG_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case SPTG_ERR_NOMEM: return "scratch memory allocation failed";
    case SPTG_ERR_CONFIG: return "requested configuration not available";
    default: return "unknown status";
  }
}

const char* sptg_last_error(void) { return t_last_error.c_str(); }

int sptg_last_config(char* buf, size_t len) {
  const std::string text = config_text();
  if (buf && len) {
    size_t n = std::min(len - 1, text.size());
    memcpy(buf, text.data(), n);
    buf[n] = '\0';
  }
  return static_cast<int>(text.size());
}

int sptg_device_error(void* stream) {
  int dev = 0;
  DeviceInfo di;
  int rc = device_info(di, dev);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0, zero = 0;
  e = cudaMemcpy(&word, di.error_word, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
  e = cudaMemcpy(di.error_word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word reset)");
  if (word) {
    char b[96];
    snprintf(b, sizeof(b), "bounded wait ran out (site mask 0x%x)", word);
    t_last_error = b;
    return SPTG_ERR_TIMEOUT;
  }
  return SPTG_OK;
}

int sptg_gemm_strided(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, const void* A, int64_t lda,
                      const void* B, int64_t ldb, void* C, int64_t ldc, void* stream,
                      const sptg_config* cfg_in) {
  t_launches = 0;
  sptg_config cfg;
  memset(&cfg, 0, sizeof(cfg));
  if (cfg_in) cfg = *cfg_in;
  DtypeInfo d;
  if (!dtype_info(dtype, d)) {
    t_last_error = "unknown dtype";
    return SPTG_ERR_ARG;
  }
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) {
    t_last_error = "dimensions must be in [0, 2^31)";
    return SPTG_ERR_ARG;
  }
  if (cfg.kernel < 0 || cfg.kernel > 5 || cfg.stages < 0 || cfg.bn < 0 || cfg.splits < 0 ||
      cfg.timeout_ms < 0 || (cfg.inject_stall != 0 && cfg.inject_stall != 1) ||
      cfg.cta_pair < 0 || cfg.cta_pair > 2 || (cfg.no_overlap != 0 && cfg.no_overlap != 1) ||
      cfg.stream_k < 0 || cfg.stream_k > 2 ||
      (cfg.trace && (reinterpret_cast<uintptr_t>(cfg.trace) & 7u))) {
    t_last_error = "invalid configuration field";
    return SPTG_ERR_ARG;
  }
  if (M == 0 || N == 0) {
    set_config("kernel=none dtype=%s (empty output)", d.name, {});
    return SPTG_OK;
  }
  if (!C || (K > 0 && (!A || !B))) {
    t_last_error = "null pointer";
    return SPTG_ERR_ARG;
  }
  if (ldc < N || (K > 0 && (lda < K || ldb < K)) || ldc > INT32_MAX || lda > INT32_MAX ||
      ldb > INT32_MAX) {
    t_last_error = "leading dimensions must satisfy lda >= K, ldb >= K, ldc >= N (< 2^31)";
    return SPTG_ERR_ARG;
  }
  if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B))) ||
      (K * d.in_bytes) % 16 != 0 || (N * d.out_bytes) % 16 != 0 ||
      (ldc * d.out_bytes) % 16 != 0 || (K > 0 && ((lda * d.in_bytes) % 16 != 0 ||
                                                  (ldb * d.in_bytes) % 16 != 0))) {
    t_last_error = "TMA needs 16-byte aligned bases and row pitches";
    return SPTG_ERR_ALIGN;
  }
  int dev = 0;
  DeviceInfo di;
  int rc = device_info(di, dev);
  if (rc) return rc;
  cudaStream_t stream_h = static_cast<cudaStream_t>(stream);

  if (K == 0) {  // the empty sum
    cudaError_t e = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * d.out_bytes, 0,
                                      static_cast<size_t>(N) * d.out_bytes, M, stream_h);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset2DAsync");
    set_config("kernel=zero-fill dtype=%s", d.name, {});
    return SPTG_OK;
  }

  // Shape class: few output rows and a float type -> the memory-bound
  // swap-AB kernel; everything else -> the square tile kernel.
  int kernel = cfg.kernel;
  if (kernel == 0 && !d.is_int8 && M <= 256 && N >= 1024) {
    // memory-bound: the kernels skinny_order lists, in turn
    SkinnyTry order[3];
    const int n_try = skinny_order(M, N, K, di.sm_count, order);
    for (int t = 0; t < n_try; ++t) {
      if (order[t].kernel == 5)
        rc = run_skinny_pair(dev, di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg, false,
                             order[t].fill);
      else if (order[t].kernel == 4)
        rc = run_skinny_rows(dev, di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg, false);
      else
        rc = run_skinny_cluster(dev, di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg, false,
                                order[t].fill);
      if (rc != SPTG_ERR_CONFIG) return rc;
    }
    kernel = M <= 64 ? 2 : 1;
  }
  if (kernel == 0) kernel = 1;
  if (kernel == 4)
    return run_skinny_rows(dev, di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg, true);
  if (kernel == 5)
    return run_skinny_pair(dev, di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg, true);
  if (kernel == 3)
    return run_skinny_cluster(dev, di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg, true);
  if (kernel == 2) return run_skinny(dev, di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg);

  SquarePlan pl;
  rc = plan_square(dev, di, d, M, N, K, cfg, &pl);
  if (rc) return rc;
  if (d.is_int8) {
    // Widen both operands to dense binary16 copies in scratch, followed by
    // any stream-K partials (one request: the scratch cannot move within the
    // call), then run the exact path.
    const size_t a_bytes = static_cast<size_t>(M) * K * 2, b_bytes = static_cast<size_t>(N) * K * 2;
    const size_t a_pad = (a_bytes + 255) & ~static_cast<size_t>(255);
    const size_t b_pad = (b_bytes + 255) & ~static_cast<size_t>(255);
    ScratchView ws;
    rc = scratch_for(dev, stream_h, a_pad + b_pad + pl.partial_bytes, &ws);
    if (rc) return rc;
    void* A16 = ws.data;
    void* B16 = static_cast<char*>(ws.data) + a_pad;
    const int64_t na = M * (K / 8), nb = N * (K / 8);
    // four 256-thread blocks per SM, each thread with eight loads in flight
    const int blocks = static_cast<int>(std::min<int64_t>((na + nb + 255) / 256, 4 * di.sm_count));
    // A plain launch: under programmatic overlap its blocks would sit on the
    // SMs beside the previous GEMM's CTAs, which measured 14 us slower per
    // call on 4096^3. The GEMM that follows still overlaps this kernel's tail.
    cudaError_t e =
        launch_s8_to_f16(A, lda, M, B, ldb, N, K, A16, B16, blocks, stream_h, false);
    t_launches += 1;
    if (e != cudaSuccess) return cuda_fail(e, "s8_to_f16 launch");
    return launch_square(di, d, M, N, K, A16, K, B16, K, C, ldc, stream_h, cfg, pl,
                         static_cast<char*>(ws.data) + a_pad + b_pad, ws.counters, ws.generation);
  }
  if (pl.partial_bytes) {
    ScratchView ws;
    rc = scratch_for(dev, stream_h, pl.partial_bytes, &ws);
    if (rc) return rc;
    return launch_square(di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg, pl, ws.data,
                         ws.counters, ws.generation);
  }
  return launch_square(di, d, M, N, K, A, lda, B, ldb, C, ldc, stream_h, cfg, pl, nullptr, nullptr,
                       0);
}

int sptg_gemm_ex(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, const void* A, const void* B,
                 void* C, void* stream, const sptg_config* cfg) {
  return sptg_gemm_strided(M, N, K, dtype, A, K, B, K, C, N, stream, cfg);
}

int sptg_gemm_host(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, const void* A, const void* B,
                   void* C, void* stream, const sptg_config* cfg) {
  t_launches = 0;
  DtypeInfo d;
  if (!dtype_info(dtype, d)) {
    t_last_error = "unknown dtype";
    return SPTG_ERR_ARG;
  }
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) {
    t_last_error = "dimensions must be in [0, 2^31)";
    return SPTG_ERR_ARG;
  }
  if (M == 0 || N == 0) {
    set_config("kernel=none dtype=%s (empty output)", d.name, {});
    return SPTG_OK;
  }
  if (!C || (K > 0 && (!A || !B))) {
    t_last_error = "null pointer";
    return SPTG_ERR_ARG;
  }
  if ((K * d.in_bytes) % 16 != 0 || (N * d.out_bytes) % 16 != 0) {
    t_last_error = "TMA needs 16-byte row pitches";
    return SPTG_ERR_ALIGN;
  }
  int dev = 0;
  DeviceInfo di;
  int rc = device_info(di, dev);
  if (rc) return rc;
  cudaStream_t stream_h = static_cast<cudaStream_t>(stream);
  auto pad = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  const size_t a_bytes = static_cast<size_t>(M) * K * d.in_bytes;
  const size_t b_bytes = static_cast<size_t>(N) * K * d.in_bytes;
  const size_t c_bytes = static_cast<size_t>(M) * N * d.out_bytes;
  void* base = nullptr;
  rc = io_for(dev, stream_h, pad(a_bytes) + pad(b_bytes) + pad(c_bytes), &base);
  if (rc) return rc;
  char* dA = static_cast<char*>(base);
  char* dB = dA + pad(a_bytes);
  char* dC = dB + pad(b_bytes);
  cudaError_t e = cudaSuccess;
  if (a_bytes) e = cudaMemcpyAsync(dA, A, a_bytes, cudaMemcpyHostToDevice, stream_h);
  if (e == cudaSuccess && b_bytes)
    e = cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, stream_h);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (operands to the device)");
  rc = sptg_gemm_strided(M, N, K, dtype, dA, K, dB, K, dC, N, stream, cfg);
  if (rc) return rc;
  e = cudaMemcpyAsync(C, dC, c_bytes, cudaMemcpyDeviceToHost, stream_h);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (result to the host)");
  return SPTG_OK;
}

int sptg_gemm(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, const void* A, const void* B, void* C,
              void* stream) {
  return sptg_gemm_ex(M, N, K, dtype, A, B, C, stream, nullptr);
}

int sptg_stream_scale_ex(int64_t n, float alpha, const float* in, float* out, void* stream,
                         const sptg_config* cfg_in) {
  t_launches = 0;
  sptg_config cfg;
  memset(&cfg, 0, sizeof(cfg));
  if (cfg_in) cfg = *cfg_in;
  if (n < 0 || cfg.timeout_ms < 0 || (cfg.inject_stall != 0 && cfg.inject_stall != 1) ||
      (cfg.no_overlap != 0 && cfg.no_overlap != 1) ||
      (cfg.trace && (reinterpret_cast<uintptr_t>(cfg.trace) & 7u))) {
    t_last_error = "invalid argument";
    return SPTG_ERR_ARG;
  }
  if (n == 0) {
    set_config("kernel=none (empty)", "f32", {});
    return SPTG_OK;
  }
  if (!in || !out) {
    t_last_error = "null pointer";
    return SPTG_ERR_ARG;
  }
  if (!aligned16(in) || !aligned16(out)) {
    t_last_error = "bulk copies need 16-byte aligned buffers";
    return SPTG_ERR_ALIGN;
  }
  int dev = 0;
  DeviceInfo di;
  int rc = device_info(di, dev);
  if (rc) return rc;
  const KernelVariant v = stream_variant();
  rc = ensure_smem(dev, v.fn, v.smem);
  if (rc) return rc;
  StreamParams p;
  p.in = in;
  p.out = out;
  p.alpha = alpha;
  p.n = n;
  p.n_vec = n & ~static_cast<int64_t>(3);
  p.num_tiles = (p.n_vec * 4 + v.bn - 1) / v.bn;
  p.error_word = di.error_word;
  p.timeout_ns = static_cast<uint64_t>(cfg.timeout_ms > 0 ? cfg.timeout_ms : 2000) * 1000000ull;
  p.inject_stall = cfg.inject_stall;
  p.trace = static_cast<unsigned long long*>(cfg.trace);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(p.num_tiles, di.sm_count)));
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(grid, 1, 1);
  lc.blockDim = dim3(160, 1, 1);
  lc.dynamicSmemBytes = v.smem;
  lc.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  if (!cfg.no_overlap) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
  }
  void* args[] = {&p};
  cudaError_t e = cudaLaunchKernelExC(&lc, v.fn, args);
  ++t_launches;
  if (e != cudaSuccess) return cuda_fail(e, "stream_scale launch");
  set_config("kernel=stream dtype=%s tile_bytes=%lld stages=%lld grid=%lld tiles=%lld smem=%lld",
             "f32", {v.bn, v.stages, grid, p.num_tiles, v.smem});
  return SPTG_OK;
}

int sptg_stream_scale(int64_t n, float alpha, const float* in, float* out, void* stream) {
  return sptg_stream_scale_ex(n, alpha, in, out, stream, nullptr);
}

int sptg_gemm_skinny_noalloc(int64_t M, int64_t N, int64_t K, sptg_dtype dtype, const void* A,
                             const void* B, void* C, void* stream) {
  t_launches = 0;
  DtypeInfo d;
  if (!dtype_info(dtype, d)) {
    t_last_error = "unknown dtype";
    return SPTG_ERR_ARG;
  }
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) {
    t_last_error = "dimensions must be in [0, 2^31)";
    return SPTG_ERR_ARG;
  }
  if (d.is_int8 || M > 64) {
    t_last_error = "the allocation-free entry covers float dtypes with M <= 64 only";
    return SPTG_ERR_CONFIG;
  }
  if (M == 0 || N == 0) {
    set_config("kernel=none dtype=%s (empty output)", d.name, {});
    return SPTG_OK;
  }
  if (!C || (K > 0 && (!A || !B))) {
    t_last_error = "null pointer";
    return SPTG_ERR_ARG;
  }
  if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B))) ||
      (K * d.in_bytes) % 16 != 0 || (N * d.out_bytes) % 16 != 0) {
    t_last_error = "TMA needs 16-byte aligned bases and row pitches";
    return SPTG_ERR_ALIGN;
  }
  int dev = 0;
  DeviceInfo di;
  int rc = device_info(di, dev);
  if (rc) return rc;
  cudaStream_t stream_h = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    cudaError_t e = cudaMemsetAsync(C, 0, static_cast<size_t>(M) * N * d.out_bytes, stream_h);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    set_config("kernel=zero-fill dtype=%s", d.name, {});
    return SPTG_OK;
  }
  unsigned char* base = nullptr;
  rc = noalloc_scratch(dev, &base);
  if (rc) return rc;
  const FixedScratch fixed{base, kNoAllocPartialBytes, base + kNoAllocPartialBytes,
                           kNoAllocCounterBytes, &g_noalloc_generation};
  sptg_config cfg;
  memset(&cfg, 0, sizeof(cfg));
  return run_skinny(dev, di, d, M, N, K, A, K, B, K, C, N, stream_h, cfg, &fixed);
}

}  // extern "C"
