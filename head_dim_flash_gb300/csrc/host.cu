// Host-side helpers: driver entry point for TMA descriptor encoding, tensor
// maps over strided dense views and the packed varlen layout, device queries.
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

namespace {

// Extents and byte strides of a tensor seen as (rows, heads, batch).
struct Geometry {
    uint64_t rows, heads, batch;
    uint64_t s_row, s_head, s_batch;  // bytes
};

Geometry geometry(const Problem& pb, bool kv_side, const View& v)
{
    Geometry g;
    g.heads = static_cast<uint64_t>(kv_side ? pb.Hkv : pb.Hq);
    if (pb.varlen) {
        g.rows = static_cast<uint64_t>(kv_side ? pb.total_k : pb.total_q);
        g.batch = 1;
    } else {
        g.rows = static_cast<uint64_t>(kv_side ? pb.Nkv : pb.Nq);
        g.batch = static_cast<uint64_t>(pb.B);
    }
    g.s_row = static_cast<uint64_t>(v.sn) * 2;
    g.s_head = static_cast<uint64_t>(v.sh) * 2;
    g.s_batch = static_cast<uint64_t>(v.sb) * 2;
    // A dimension with a single entry is never stepped over; give it a valid
    // stride (a positive multiple of 16 bytes) whatever the caller passed.
    const uint64_t any = static_cast<uint64_t>(pb.D) * 2;
    if (g.rows <= 1 && g.s_row == 0) g.s_row = any;
    if (g.heads <= 1 && g.s_head == 0) g.s_head = any;
    if (g.batch <= 1 && g.s_batch == 0) g.s_batch = any;
    if (g.rows == 0) g.rows = 1;
    if (g.heads == 0) g.heads = 1;
    if (g.batch == 0) g.batch = 1;
    return g;
}

}  // namespace

bool make_row_map(CUtensorMap* m, const void* base, const Problem& pb, bool kv_side, bool bf16, int box_rows,
                  const View& v)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const Geometry g = geometry(pb, kv_side, v);
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(pb.D), g.rows, g.heads, g.batch};
    const cuuint64_t strides[3] = {g.s_row, g.s_head, g.s_batch};
    const cuuint32_t box[4] = {kChunk, static_cast<cuuint32_t>(box_rows), 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                           const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The head dim is split into (64 elements, D/64 chunks) with a 128-byte chunk
// stride, so one box of rows x chunks lands in shared memory as `chunks`
// row-blocks of rows x 128 bytes back to back.
bool make_slab_map(CUtensorMap* m, const void* base, const Problem& pb, bool kv_side, bool bf16, int rows, int chunks,
                   const View& v)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const Geometry g = geometry(pb, kv_side, v);
    const cuuint64_t dims[5] = {64, g.rows, static_cast<cuuint64_t>(pb.D / 64), g.heads, g.batch};
    const cuuint64_t strides[4] = {g.s_row, 128, g.s_head, g.s_batch};
    const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(chunks), 1, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
                           const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// e4m3 codes of a contiguous [B, H, N, D] tensor as (128 bytes, N, D/128
// chunks, H, B): one box of rows x chunks lands as `chunks` row-blocks of
// rows x 128 bytes, as for the 16-bit maps.
bool make_u8_slab_map(CUtensorMap* m, const void* base, int B, int H, int N, int D, int rows, int chunks)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc || N <= 0 || D % 128 != 0) return false;
    const cuuint64_t dims[5] = {128, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(D / 128),
                                static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[4] = {static_cast<cuuint64_t>(D), 128, static_cast<cuuint64_t>(N) * D,
                                   static_cast<cuuint64_t>(H) * N * D};
    const cuuint32_t box[5] = {128, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(chunks), 1, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 V^T [B, Hkv, D, ldv] as (keys, D, Hkv, B) with boxes of 128 keys x
// box_rows head-dim rows (keys past N read as zero).
bool make_vt_map(CUtensorMap* m, const void* base, int B, int Hkv, int D, int N, int ldv, int box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc || N <= 0 || ldv % 16 != 0) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(D),
                                static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(ldv), static_cast<cuuint64_t>(D) * ldv,
                                   static_cast<cuuint64_t>(Hkv) * D * ldv};
    const cuuint32_t box[4] = {128, static_cast<cuuint32_t>(box_rows), 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool unit_grid(unsigned x, long long n_units, dim3* grid)
{
    constexpr long long kMaxDim = 65535;
    if (n_units < 1 || n_units > kMaxDim * kMaxDim) return false;
    const long long y = n_units < kMaxDim ? n_units : kMaxDim;
    *grid = dim3(x, static_cast<unsigned>(y), static_cast<unsigned>((n_units + y - 1) / y));
    return true;
}

int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace ffpa
