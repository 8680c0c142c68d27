// tmap.h -- host-side construction of TMA tensor maps (bf16, 128-byte swizzle)
// for the tensor-core kernels. The driver's encoder is looked up once through
// the runtime (no link against the driver library).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gqa {

// A bf16 tensor of up to 4 dimensions: dims[0] elements per row (innermost),
// byte strides of dimensions 1..3 (multiples of 16), box sizes (box[0] = 64: one
// 128-byte swizzle row). Elements outside the tensor read as zeros. Returns
// false if the encoder is unavailable or rejects the arguments.
bool make_tmap_bf16(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides[3],
                    const uint32_t box[4]);

}  // namespace gqa
