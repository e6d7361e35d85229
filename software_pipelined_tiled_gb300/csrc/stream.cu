// stream.cu -- instantiation of the streaming ring (out = alpha * in).
#include "stream_scale.cuh"
#include "variants.h"

namespace sptg {

// 32 KB tiles, 6 stages (192 KB of copies in flight per SM).
KernelVariant stream_variant() {
  constexpr int TILE = 32768, ST = 6;
  return {reinterpret_cast<const void*>(&stream_scale_kernel<TILE, ST>), TILE, ST,
          StreamLayout<TILE, ST>::SMEM_BYTES, false};
}

}  // namespace sptg
