// TMA tensor maps: host-side encoding (cached) and the device load helpers.
#pragma once
#include <cuda.h>
#include <cstdint>

namespace lmoe {

// Encodes (or returns a cached copy of) a tiled tensor map.  rank 2 or 3;
// dims/strides/box as for cuTensorMapEncodeTiled (strides: rank-1 entries, bytes).
// Returns LMOE_OK or LMOE_ECUDA.
int get_tmap(CUtensorMap* out, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
             const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swz);

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int c0, int c1, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1),
      "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int c0, int c1, int c2, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2),
      "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Byte offset inside a 128B-swizzled TMA box laid out [plane][row][128 B]
// (plane = outer box dim, row = middle box dim of `rows` rows): 16-byte chunk
// `c` of line (plane*rows + row) sits at chunk c ^ (row & 7).  rows must be a
// multiple of 8 and the box base 1024-byte aligned.
__device__ __forceinline__ uint32_t swz128(int plane, int rows, int row, int c) {
  return static_cast<uint32_t>(((plane * rows + row) << 7) + ((c ^ (row & 7)) << 4));
}

}  // namespace lmoe
