// Helpers shared by the two tensor-core tree-attention kernels
// (k_attn_tc.cu, k_attn_pipe.cu). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "tc_ptx.cuh"

namespace eagle {

constexpr int kPipeMaxSeqs = 256;  // sequences the persistent kernel orders in shared memory

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Three-input maximum (NaN operands are dropped, like fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Largest of 32 values: a tree of three-input maxima (depth 4).
__device__ __forceinline__ float max32(const float (&v)[32]) {
    float t[11];
#pragma unroll
    for (int q = 0; q < 10; ++q) t[q] = fmax3(v[3 * q], v[3 * q + 1], v[3 * q + 2]);
    t[10] = fmaxf(v[30], v[31]);
    return fmaxf(fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmax3(t[6], t[7], t[8])), fmaxf(t[9], t[10]));
}

// A 4-D bf16 tensor map with 128-byte swizzle (no out-of-bounds fill value).
inline bool make_map_bf16_4d(CUtensorMap* m, const void* base, const cuuint64_t dims[4],
                             const cuuint64_t strides_bytes[3], const cuuint32_t box[4]) {
    auto fn = tensor_map_encode_fn();
    if (!fn) return false;
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides_bytes, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace eagle
