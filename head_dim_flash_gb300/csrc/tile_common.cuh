// Small device helpers shared by the forward and backward kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace ffpa {

// Sites of the status word for a packed sequence that breaks its contract.
enum : uint32_t { VS_PAIR = 0x70, VS_SINGLE = 0x71, VS_GEMM = 0x72 };

// Sequence b of a packed batch, as read from the device cu_seqlens: its first
// query / key token and its lengths. The FFPA varlen API refuses a batch it
// cannot process instead of silently unpacking part of it ("CuTe-DSL Backend"
// page, "Varlen (packed THD) API"); here a sequence whose offsets are
// negative or decreasing, run past total_q / total_k, or whose length exceeds
// the max_seqlen bound that sized the launch grid records
// DEV_INVALID | site | b in the status word (ffpa_get_status reports it) and
// returns false: the caller then returns before touching memory. Every CTA of
// a cluster reads the same entries, so the decision is uniform over it.
__device__ __forceinline__ bool varlen_seq(const Problem& pb, int b, uint32_t* status, uint32_t site, int& tq0,
                                           int& lq, int& tk0, int& lk)
{
    const long long q0 = pb.cu_q[b], q1 = pb.cu_q[b + 1], k0 = pb.cu_k[b], k1 = pb.cu_k[b + 1];
    const bool ok = q0 >= 0 && k0 >= 0 && q1 >= q0 && k1 >= k0 && q1 <= pb.total_q && k1 <= pb.total_k &&
                    q1 - q0 <= pb.Nq && k1 - k0 <= pb.Nkv;
    if (!ok) {
        if (threadIdx.x == 0)
            atomicCAS(status, 0u, DEV_INVALID | (site << 8) | ((static_cast<uint32_t>(b) & 0xffffu) << 16));
        return false;
    }
    tq0 = static_cast<int>(q0);
    lq = static_cast<int>(q1 - q0);
    tk0 = static_cast<int>(k0);
    lk = static_cast<int>(k1 - k0);
    return true;
}

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

// Index of this CTA's work unit in a grid laid out by unit_grid(): the units
// are numbered blockIdx.y + gridDim.y * blockIdx.z, in the order the hardware
// starts them (every CTA of a cluster along x shares the unit).
__device__ __forceinline__ long long unit_id()
{
    return static_cast<long long>(blockIdx.y) + static_cast<long long>(gridDim.y) * blockIdx.z;
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
