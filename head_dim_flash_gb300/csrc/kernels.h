// Internal interface between the C-ABI host layer (api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace ffpa {

constexpr int kChunk = 64;     // head-dim elements per 128-byte swizzled row
constexpr int kMaxSmem = 232448;

// Element strides of a tensor seen as [B, H, N, D] (head-dim stride 1).
// Dense tensors may be strided views; packed varlen tensors [T, H, D] are
// described with sn = H*D (one token), sh = D and sb unused (one batch).
struct View {
    long long sb, sh, sn;
};

// Problem description shared by every kernel. Dense problems use B/Nq/Nkv;
// varlen problems use cu_q/cu_k with Nq/Nkv holding the max sequence lengths.
struct Problem {
    int varlen;
    int B, Hq, Hkv, Nq, Nkv, D;
    int total_q, total_k;
    const int* cu_q;
    const int* cu_k;
    int causal;
    float scale;        // softmax scale
    float scale_log2;   // scale * log2(e)
    View vq, vk, vv, vo, vdo, vdq, vdk, vdv;  // layouts of the eight tensors
};

struct DeviceCtl {
    uint32_t* status;   // device status word
    uint64_t limit_ns;  // bound of any single device wait
};

struct FwdArgs {
    Problem pb;
    int bf16;
    const void *q, *k, *v;
    void* o;
    float* lse;
    DeviceCtl ctl;
};

struct BwdArgs {
    Problem pb;
    int bf16;
    const void *q, *k, *v, *o, *dO;
    const float* lse;
    void *dq, *dk, *dv;
    float* delta;      // workspace [rows] fp32: rowsum(dO * O)
    float* lse_log2;   // workspace [rows] fp32: LSE * log2(e), +inf for empty rows
    unsigned stages;   // bit 0 preprocess, bit 1 dV, bit 2 dQ, bit 3 dK, bit 4 dQ from the stored dS,
                       // bit 5 stored P (dK stores it, dV is the GEMM over it)
    void* ds;          // dS^T buffer of dsq_ds_bytes() bytes, or null (dQ recomputes S and dP)
    void* p;           // P^T buffer of the same size, or null (dV recomputes S)
    // > 0: the stored-tile backward runs in chunks of this many kv groups (a kv
    // head and its query heads), each chunk dK (storing its tiles), then the dV
    // and dQ GEMMs over them; ds and p then hold one chunk's tiles
    // (dsq_group_bytes() per group each). 0: all groups at once.
    int chunk_groups;
    DeviceCtl ctl;
};

// The four GEMM kernels of the cluster-exchange design.
enum XOp { XOP_FWD = 0, XOP_DQ = 1, XOP_DV = 2, XOP_DK = 3 };

struct XArgs {
    Problem pb;
    int bf16;
    const void *q, *k, *v, *dO;
    void* o;
    float* lse;                        // forward output
    const float* delta;                // backward: rowsum(dO * O)
    const float* lse_log2;             // backward: LSE * log2(e), +inf for empty rows
    void *dq, *dk, *dv;
    DeviceCtl ctl;
    // launch as a programmatic dependent of the previous kernel of the stream
    // (which must be one of these GEMM kernels that reads nothing this one writes)
    int pdl;
    // FP8 forward: e4m3 q8 / k8 (q, k above point at them), V transposed
    // [B, Hkv, D, ldv], and the fp32 dequantization scales per (batch, head)
    int f8;
    const void* v8t;
    int ldv;
    const float *f8_sq, *f8_sk, *f8_sv;
    // dK: also store every dS^T tile to ds ([B, Hq, Nkv, ldq], ldq = Nq rounded up to 8)
    int store_ds;
    void* ds;
    // dK: also store every P^T tile (input dtype) to p, the same layout
    int store_p;
    void* p;
    // output columns the epilogue stores (0: pb.D); the FP8 forward runs its
    // tiles over the head dim padded to 128 and stores the real ones
    int d_out;
    // dV / dK (rows = keys): only the kv heads [g0, g0 + ng) of every batch
    // entry (ng = 0: all of them); the stored tile buffers then hold the query
    // heads of those groups only, [B, ng * G, Nkv, ldq] (packed: [1, ng * G, ...])
    int g0, ng;
};

// The GEMMs over the tiles the dK kernel stored (dense, D a multiple of 64 up to 1024;
// dsq_ds_bytes is the size of one [B, Hq, Nkv, ldq] tile buffer):
//   dv = 0: dQ = scale * dS K from the stored dS^T;
//   dv = 1: dV = P^T dO from the stored P^T, over the query heads of the group.
struct DsqArgs {
    Problem pb;
    int bf16;
    int dv;
    const void* tiles;  // dS^T (dv = 0) or P^T (dv = 1)
    const void* rhs;    // K (dv = 0) or dO (dv = 1)
    void* out;          // dQ (dv = 0) or dV (dv = 1), in its view
    // only the kv groups [g0, g0 + ng) (ng = 0: all): dV rows of those kv heads,
    // dQ rows of their query heads; `tiles` holds those groups' heads only
    int g0, ng;
    DeviceCtl ctl;
};
bool dsq_supported(const Problem& pb);
size_t dsq_ds_bytes(const Problem& pb);     // one tile buffer, every head
size_t dsq_group_bytes(const Problem& pb);  // one tile buffer, the G query heads of one kv group
// map over a tile buffer of `heads` query heads (box: 64 queries x box_rows key rows)
bool make_ds_map(CUtensorMap* m, const void* ds, const Problem& pb, bool bf16, int box_rows, int heads);
cudaError_t launch_dsq(const DsqArgs& a, cudaStream_t s);

// Workspace of the FP8 forward (byte offsets, 256-byte aligned regions).
struct Fp8Layout {
    size_t q8, k8, v8t, sq, sk, sv, part, total;
    int ldv;
    int dp;  // code rows: the head dim rounded up to 128 (zero codes past D)
};
Fp8Layout fp8_layout(int B, int Hq, int Hkv, int Nq, int Nkv, int D);
// packed batches of `batch` sequences (codes of all tokens, per-(sequence, head) scales)
Fp8Layout fp8_varlen_layout(int batch, int Hq, int Hkv, int total_q, int total_k, int max_q, int max_k, int D);
Fp8Layout fp8_layout_of(const Problem& pb);
cudaError_t launch_fp8_quantize(const FwdArgs& a, void* workspace, cudaStream_t s);
// (quantization pass, then) the CTA-pair forward on the e4m3 operands in `workspace`
cudaError_t launch_fwd_fp8(const FwdArgs& a, void* workspace, cudaStream_t s, bool quantize);

// Runs one of the four GEMM kernels, in the CTA-pair form (2-SM MMAs,
// clusters of 2C CTAs, head dims that are multiples of 128 up to 768) or the
// one-CTA-per-slab form (clusters of C CTAs, every other head dim);
// FFPA_KERNEL=pair|single in the environment forces one of them.
cudaError_t launch_xchg(int op, const XArgs& a, cudaStream_t s);
bool xchg_uses_pair(const Problem& pb);  // the family launch_xchg picks for this problem
cudaError_t launch_pair(int op, const XArgs& a, cudaStream_t s);
cudaError_t launch_single(int op, const XArgs& a, cudaStream_t s);

// Function pointer to the driver's cuTensorMapEncodeTiled (resolved once).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// Tensor map over rows of head-dim vectors of a tensor with layout `v`,
// 4-D (D, rows, heads, batch): rows are N (dense) or tokens (packed), batch
// is B (dense) or 1 (packed). Box = 64 head-dim elements x `box_rows` rows,
// 128-byte swizzle; coordinates (d, row or token, head, b or 0).
bool make_row_map(CUtensorMap* m, const void* base, const Problem& pb, bool kv_side, bool bf16, int box_rows,
                  const View& v);

// Tensor map reading `rows` rows x `chunks` 64-wide head-dim chunks in one box
// (shared-memory layout [chunk][row][64], 128-byte swizzle), 5-D
// (64, rows, D/64, heads, batch); coordinates (0, row or token, chunk, head, b or 0).
bool make_slab_map(CUtensorMap* m, const void* base, const Problem& pb, bool kv_side, bool bf16, int rows, int chunks,
                   const View& v);

// True when the query side / key side of a problem has no rows at all. Such a
// side has no storage; tensor maps for it are built over the other side's
// tensor (never loaded from, because every tile loop is empty).
inline bool q_side_empty(const Problem& pb) { return pb.varlen ? pb.total_q == 0 : (pb.Nq == 0 || pb.B == 0); }
inline bool kv_side_empty(const Problem& pb) { return pb.varlen ? pb.total_k == 0 : (pb.Nkv == 0 || pb.B == 0); }

bool make_u8_slab_map(CUtensorMap* m, const void* base, int B, int H, int N, int D, int rows, int chunks);
bool make_vt_map(CUtensorMap* m, const void* base, int B, int Hkv, int D, int N, int ldv, int box_rows);
int num_sms();

// Grid for n_units work units of x CTAs each (x along the grid's x, one
// cluster per unit): the units are spread over y and z (unit_id() in device
// code), so that their number is not bounded by the 65535 of one dimension.
// Units past n_units (in the last z row) must return at once. False when
// n_units exceeds 65535 * 65535.
bool unit_grid(unsigned x, long long n_units, dim3* grid);

// Records `fmt` as the thread's last-error message (ffpa_last_error) and
// returns `status` (an ffpa_status value).
int set_error(int status, const char* fmt, ...);

// Decode / short-query forward (split over the keys), D % 64 == 0: a CTA
// takes kDecodeRows query rows of one kv head's group (G * Nq rows in all)
// and one split of its keys.
constexpr int kDecodeRows = 16;
constexpr int kDecodeMaxSplits = 64;
struct DecodePlan {
    int splits, rblocks, tiles_per, kt, chunks;
    size_t workspace_bytes;  // partial outputs and LSE of every split
};
DecodePlan decode_plan(const Problem& pb);
cudaError_t launch_decode(const FwdArgs& a, void* workspace, cudaStream_t s);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s);

}  // namespace ffpa
