// Device helpers shared by the grouped-GEMM kernels: the clamped SwiGLU of
// the gate/up epilogues and the tile-table reader.  One definition, so that
// every kernel applies the same clamp.
#pragma once

#include <stdint.h>

#include "moe_kernels.h"

namespace moe {

// The expert activation between gate/up and down: the gate is clamped to
// (-inf, 10] before the SiLU and the up projection to [-10, 10]
// ("Add GLM-5.3-Flash (glm5next) support with ROCmFP mix qtypes (105/106)",
// section "Architecture").  silu(g) = g / (1 + exp(-g)), in fp32.
__device__ __forceinline__ float clamped_swiglu(float g, float u) {
  const float gc = fminf(g, 10.0f);
  const float uc = fminf(fmaxf(u, -10.0f), 10.0f);
  return gc / (1.0f + expf(-gc)) * uc;
}

// Entry i of a tile table (16-byte entries after the table's header).
__device__ __forceinline__ TileEntry table_entry(const int32_t* table, int i) {
  const int4 v =
      reinterpret_cast<const int4*>(reinterpret_cast<const char*>(table) + kTableHeaderBytes)[i];
  return TileEntry{v.x, v.y, v.z, v.w};
}

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

}  // namespace moe
