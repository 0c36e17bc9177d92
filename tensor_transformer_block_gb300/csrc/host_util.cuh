// Host-side helpers shared by the launchers: TMA tensor-map encoding through the
// driver entry point (no link-time dependency on libcuda), device properties.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tpb {

// Encodes a tiled TMA map over a row-major tensor of rank 2..5 with bf16 or fp32
// elements.  dims[0] is the contiguous dimension; box[i] <= 256; the
// innermost box extent times the element size must be <= 128 bytes for the
// 128-byte swizzle.  Returns true on success.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint32_t* box, CUtensorMapSwizzle swizzle);

// Streaming-multiprocessor count of the current device (cached per device).
int device_sm_count();

// Current device's compute capability as major*10+minor, or -1.
int device_cc();

}  // namespace tpb
