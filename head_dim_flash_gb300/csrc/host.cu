// Host-side helpers: driver entry point for TMA descriptor encoding, tensor
// maps over the dense and packed layouts, device queries.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"

namespace ffpa {

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Dense tensors [B, H, N, D] are described as 3-D (D, N, B*H) so that a box
// never crosses from one head into the next (rows past N read as zero).
// Packed tensors [T, H, D] are described as (D, H, T); a box of rows then
// walks along tokens of one head.
bool make_row_map(CUtensorMap* m, const void* base, const Problem& pb, bool kv_side, bool bf16, int box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const uint64_t D = static_cast<uint64_t>(pb.D);
    const uint64_t H = static_cast<uint64_t>(kv_side ? pb.Hkv : pb.Hq);
    cuuint64_t dims[3];
    cuuint64_t strides[2];
    cuuint32_t box[3];
    const cuuint32_t es[3] = {1, 1, 1};
    if (!pb.varlen) {
        const uint64_t N = static_cast<uint64_t>(kv_side ? pb.Nkv : pb.Nq);
        dims[0] = D;
        dims[1] = N;
        dims[2] = static_cast<uint64_t>(pb.B) * H;
        strides[0] = D * 2;
        strides[1] = N * D * 2;
        box[0] = kChunk;
        box[1] = static_cast<cuuint32_t>(box_rows);
        box[2] = 1;
    } else {
        const uint64_t T = static_cast<uint64_t>(kv_side ? pb.total_k : pb.total_q);
        dims[0] = D;
        dims[1] = H;
        dims[2] = T;
        strides[0] = D * 2;
        strides[1] = H * D * 2;
        box[0] = kChunk;
        box[1] = 1;
        box[2] = static_cast<cuuint32_t>(box_rows);
    }
    const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                           const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map that reads a D-slab of `rows` consecutive rows in ONE box: the
// head dim is split into (64 elements, D/64 chunks) and the box is
// 64 x rows x chunks, so shared memory receives [chunk][row][64] (128-byte
// swizzled rows), i.e. `chunks` row-blocks of rows x 128 bytes back to back.
// Dense: dims (64, N, D/64, B*H); packed: dims (64, T, D/64, H).
bool make_slab_map(CUtensorMap* m, const void* base, const Problem& pb, bool kv_side, bool bf16, int rows, int chunks)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const uint64_t D = static_cast<uint64_t>(pb.D);
    const uint64_t H = static_cast<uint64_t>(kv_side ? pb.Hkv : pb.Hq);
    cuuint64_t dims[4];
    cuuint64_t strides[3];
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(chunks), 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    dims[0] = 64;
    dims[2] = D / 64;
    strides[1] = 128;  // next 64-element chunk of the same row
    if (!pb.varlen) {
        const uint64_t N = static_cast<uint64_t>(kv_side ? pb.Nkv : pb.Nq);
        dims[1] = N;
        dims[3] = static_cast<uint64_t>(pb.B) * H;
        strides[0] = D * 2;
        strides[2] = N * D * 2;
    } else {
        const uint64_t T = static_cast<uint64_t>(kv_side ? pb.total_k : pb.total_q);
        dims[1] = T;
        dims[3] = H;
        strides[0] = H * D * 2;
        strides[2] = D * 2;
    }
    const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                           const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace ffpa
