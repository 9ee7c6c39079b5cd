// tma.cuh -- tiled TMA loads of expert code tiles (cp.async.bulk.tensor).
//
// One tensor map per code matrix: a 3-D byte tensor over the records,
// x = bytes along the input dimension (two codes per byte), y = rows of the
// matrix, z = expert (record stride).  Built once per layer on the host
// with cuTensorMapEncodeTiled, passed to kernels as __grid_constant__.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace moe {

struct alignas(128) PfMaps {
  CUtensorMap routed[2];  // gate|up kernel: gate, up codes;  down kernel: down codes, unused
  CUtensorMap shared[2];  // the same for the shared expert's record
};

struct LayerMaps {
  PfMaps gateup, down;
  int valid;
};

// 3-D tile load of box (bx bytes, by rows, 1 record) at (x, y, z) into
// shared memory, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
      "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "l"(policy)
      : "memory");
}

}  // namespace moe
