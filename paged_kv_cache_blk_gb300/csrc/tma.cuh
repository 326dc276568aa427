// Tensor-memory-accelerator (TMA) helpers shared by the kernels that stage
// tiles with cp.async.bulk.tensor: the device-side copy instructions and the
// host-side tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace pkv {

// Tiled tensor copies global -> shared, completion counted on an mbarrier.
// The innermost coordinate x times the element size must be a multiple of
// 16 bytes; the other coordinates may be anything (out-of-range elements
// read as zero).
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* m, int x, int y,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"((uint64_t)m), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* m, int x, int y, int z,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"((uint64_t)m), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap* m, int x, int y, int z,
                                       int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"((uint64_t)m), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// Encode a tiled tensor map (element strides 1, no interleave, 256-byte L2
// promotion, zero fill out of range).  strides[i] is the byte stride of
// dimension i + 1.  False when the driver entry point is missing or refuses
// the geometry.
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  CUtensorMapSwizzle swizzle);

}  // namespace pkv
