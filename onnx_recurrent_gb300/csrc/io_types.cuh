// Element types of the activation tensors a plan reads and writes (X,
// initial_h, initial_c, Y, Y_h, Y_c): fp32, fp16 or bf16.  The arithmetic
// stays fp32: an fp16 or bf16 input is widened exactly, an output is rounded
// to nearest even once, and a NaN output is the type's canonical quiet NaN
// (0x7FC00000, 0x7E00, 0x7FC0).
#pragma once

#include <cstddef>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace rnngb {

enum IoType { kIoF32 = 0, kIoF16 = 1, kIoBF16 = 2 };

__device__ __forceinline__ float io_load(const float* base, size_t i, int io)
{
    if (io == kIoF16) return __half2float(reinterpret_cast<const __half*>(base)[i]);
    if (io == kIoBF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
    return base[i];
}

__device__ __forceinline__ void io_store(float* base, size_t i, float v, int io)
{
    if (io == kIoF16) {
        reinterpret_cast<__half*>(base)[i] = v != v ? __ushort_as_half((unsigned short)0x7E00u) : __float2half_rn(v);
    } else if (io == kIoBF16) {
        reinterpret_cast<__nv_bfloat16*>(base)[i] =
            v != v ? __ushort_as_bfloat16((unsigned short)0x7FC0u) : __float2bfloat16_rn(v);
    } else {
        base[i] = v;
    }
}

}  // namespace rnngb
