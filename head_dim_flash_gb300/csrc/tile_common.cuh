// Small device helpers shared by the forward and backward kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace ffpa {

// Rounds two fp32 values to the element type (RNE) and packs them.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w)
{
    if constexpr (BF16) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&w);
        return __bfloat1622float2(h);
    } else {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        return __half22float2(h);
    }
}

// Position in a shared-memory ring of `stages` slots, with the parity of the
// slot's current use (flips each time the ring wraps).
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance(int stages)
    {
        if (++slot == stages) {
            slot = 0;
            phase ^= 1u;
        }
    }
    __device__ __forceinline__ void retreat(int stages)
    {
        if (slot == 0) {
            slot = stages - 1;
            phase ^= 1u;
        } else {
            --slot;
        }
    }
};

// Byte offset of 16-byte unit `u` (0..7) of row `r` inside a 128-byte-swizzled
// tile whose rows are 128 bytes apart (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and the tcgen05 descriptors read).
__device__ __forceinline__ uint32_t sw128_offset(int r, int u)
{
    return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}

}  // namespace ffpa
