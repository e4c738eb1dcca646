// One cache block per TMA box, for the tensor-core kernels (decode and
// prefill) of bf16 caches [N][Hkv][B][D].
//
// The host views a cache as a 4D tensor (64 dims, 8 rows, D / 64 halves,
// N * Hkv * B / 8 groups of 8 rows; byte strides 2D, 128 and 16D), so that
// a box of (64, 8, D / 64, B / 8) is one block of one KV head, and it lands
// in shared memory with 128-byte swizzle as 8-row groups that each hold
// both 64-dim halves, 1 KB apart: row t (of a stage), half h at byte
// kv_row_offset(t, h), its 16-byte pieces swizzled by t & 7.  Read as a
// K-major tensor-core operand (keys) this is leading-dimension stride
// unused, 8-row group stride D / 64 KB; as an MN-major one (values), half
// stride 1 KB and the same group stride.
#pragma once

#include <cstdint>

#include "device_common.cuh"

namespace pa {

// 4D tiled TMA load of one box; x is the innermost (element) coordinate.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int w, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Byte offset in a stage of keys or values of row t (token of the stage)
// and 64-dim half h: 8-row groups kHalves KB apart, halves 1 KB apart.
template <int kHalves>
__device__ __forceinline__ int kv_row_offset(int t, int h) {
  return (t >> 3) * (kHalves * 1024) + h * 1024 + (t & 7) * 128;
}

}  // namespace pa
