// vla_tma.cuh -- 3-D tensor maps of the [BH][T][64] bf16 inputs of the
// tensor-core passes (d = 64) and the tiled tensor copy that lands a box of 64
// tokens in their operand-tile layout (128-byte swizzle).
#pragma once

#include <cuda.h>

#include "vla_tc_common.cuh"

namespace vla {

// Map of a [BH][T][d] bf16 tensor at `base` (d = 64 or 128): boxes of 64
// tokens x 64 features of one (b, h) (feature offset x a multiple of 64),
// 128-byte swizzle, zeros past T.  False when the driver's encoder is
// unavailable or rejects the arguments.
bool make_tile_map(CUtensorMap *m, const void *base, int BH, int T, int d = 64);
// Whether the driver's tensor-map encoder could be found.
bool tile_maps_available();

namespace tc {

// One box (features x, tokens y, unit z) into dst (1024-byte aligned), its
// bytes counted on the mbarrier `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace tc
}  // namespace vla
