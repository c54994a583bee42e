/*
 * ffpa.h — C ABI of the GB300 (sm_103a) large-head-dim exact attention library.
 *
 * Operation (FFPA docs, "Backends Overview" page, "Automatic SDPA fallback":
 * the SDPA-aligned result; "CuTe-DSL Backend" page, "Hard constraints" and
 * "Varlen (packed THD) API"):
 *
 *   S = scale * Q K^T, restricted to legal keys;  O = softmax(S) V;
 *   LSE_i = ln sum_j exp(S_ij)  (fp32, natural log, of the scaled scores);
 *   key j is legal for query i iff j < Lk and, when causal, j <= i + (Lk - Lq)
 *   (bottom-right / tail-aligned mask; per sequence for varlen);
 *   a row with no legal key gives O_i = 0, LSE_i = -inf and zero gradients.
 *   GQA/MQA: query head h reads kv head h / (Hq / Hkv).
 *   Backward for L = sum(dO * O) gives dQ, dK, dV (dK/dV summed over the
 *   query heads of each kv group).
 *
 * Element types: bf16 or fp16 for q, k, v, o, dO, dq, dk, dv (one type per
 * call); lse is fp32. Head dim D: a multiple of 32 in [64, 1024] (the FFPA
 * tuned range 320..1024 included; head dims that are not a multiple of 64 read
 * their last 64-wide chunk half from zero fill). The arithmetic runs on tcgen05 tensor cores
 * with fp32 accumulation; P is rounded to the input type before P*V.
 *
 * Memory and ownership: every pointer argument is DEVICE memory owned by the
 * caller, 16-byte aligned, contiguous in the layout stated per call (the
 * *_strided calls take strided views instead, see ffpa_view). The
 * library allocates nothing; backward scratch lives in a caller-provided
 * workspace of at least *_bwd_workspace_bytes(...) bytes.
 *
 * Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and does no host synchronisation. Outputs are fully
 * overwritten, never accumulated into.
 *
 * Errors: calls validate arguments before any launch and return
 *   FFPA_ERR_INVALID_VALUE  null pointer with a non-empty problem, misaligned
 *                           pointer, negative size, Hq not a multiple of Hkv,
 *                           non-finite scale, too small a workspace, bad
 *                           cu_seqlens sizes;
 *   FFPA_ERR_NOT_SUPPORTED  dtype other than bf16/fp16, D outside the range
 *                           above or not a multiple of 32, a device that is
 *                           not compute capability 10.3;
 *   FFPA_ERR_CUDA           a CUDA runtime/driver call failed (launch error);
 * and nothing is launched. A problem with no work (B, H or N zero) returns
 * FFPA_OK without a launch. Every device-side wait in the kernels is bounded;
 * a wait that runs out records FFPA_ERR_TIMEOUT in a device status word that
 * ffpa_get_status() reports. ffpa_last_error() gives a thread-local message
 * for the last failing call.
 */
#ifndef FFPA_H_
#define FFPA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FFPA_API __attribute__((visibility("default")))
#else
#define FFPA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FFPA_OK = 0,
    FFPA_ERR_INVALID_VALUE = 1,
    FFPA_ERR_NOT_SUPPORTED = 2,
    FFPA_ERR_CUDA = 3,
    FFPA_ERR_TIMEOUT = 4
} ffpa_status;

typedef enum { FFPA_BF16 = 0, FFPA_FP16 = 1 } ffpa_dtype;

/* Same object as cudaStream_t. */
typedef struct CUstream_st* ffpa_stream_t;

/*
 * Dense forward (FFPA docs, CuTe-DSL Backend page, "Hard constraints": dense
 * SDPA layout, causal bottom-right, MHA/GQA/MQA via zero-stride broadcast).
 *   q, o : [B, Hq, Nq, D]  contiguous, dtype dt        (o written)
 *   k, v : [B, Hkv, Nkv, D] contiguous, dtype dt
 *   lse  : [B, Hq, Nq] fp32 (written)
 *   causal: 0 or 1 (bottom-right aligned); scale: finite (usually 1/sqrt(D)).
 */
FFPA_API ffpa_status ffpa_fwd(ffpa_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale,
                     ffpa_stream_t stream);

/*
 * A strided view of a dense [B, H, N, D] tensor for the *_strided calls:
 * element (b, h, n, d) lives at data + (b*stride_b + h*stride_h + n*stride_n + d)
 * elements (the head-dim stride is 1). Covers the contiguous [B, H, N, D]
 * layout (stride_n = D, stride_h = N*D, stride_b = H*N*D), the [B, N, H, D]
 * layout that QKV projections produce (stride_n = H*D, stride_h = D,
 * stride_b = N*H*D) and views into fused QKV buffers, with no copy (FFPA
 * docs, "CuTe-DSL Backend" page: the dense SDPA layout; zero-copy strided and
 * fused-QKV inputs are the extension the FFPA pages list for later backends).
 * Requirements: data 16-byte aligned; every stride a multiple of 8 elements
 * (16 bytes) and positive when its dimension has more than one entry. Output
 * views must not overlap themselves or any input; overlapping inputs (for
 * example k and v in one fused buffer) are fine.
 */
typedef struct ffpa_view {
    void* data;
    int64_t stride_b, stride_h, stride_n;
} ffpa_view;

/*
 * Dense forward on strided views (otherwise as ffpa_fwd). q, o: [B, Hq, Nq, D]
 * views; k, v: [B, Hkv, Nkv, D] views; lse stays a contiguous fp32
 * [B, Hq, Nq] array. Strides that break the requirements above return
 * FFPA_ERR_INVALID_VALUE before any launch.
 */
FFPA_API ffpa_status ffpa_fwd_strided(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, ffpa_view o, float* lse,
                                      int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale,
                                      ffpa_stream_t stream);

/*
 * Decode / short-query forward (the pages' split-KV two-stage decode path,
 * FFPA docs "Backends Overview", feature support and fallback table; the
 * operation is exactly ffpa_fwd_strided's). The keys are split over CTAs;
 * a CTA takes 16 query rows of one kv head's group (G = Hq / Hkv heads x Nq
 * rows) and reads each K/V byte of its split once for all of them; a second
 * kernel combines the splits' partial outputs (O, LSE) from `workspace`.
 * Meant for few query rows per kv head (G * Nq <= 16 reads K/V exactly once;
 * larger groups re-read them once per 16 rows).
 *   q, o : [B, Hq, Nq, D] views; k, v : [B, Hkv, Nkv, D] views; lse: contiguous
 *   fp32 [B, Hq, Nq]. D must be a multiple of 64.
 *   workspace: device scratch of at least ffpa_decode_workspace_bytes()
 *   bytes, 256-byte aligned, sized on the current device (the split count
 *   follows its SM count); one call at a time per workspace.
 * Returns FFPA_ERR_NOT_SUPPORTED for D % 64 != 0 (use ffpa_fwd_strided) or
 * B * Hkv * ceil(G * Nq / 16) > 65535^2 (the launch grid), otherwise as
 * ffpa_fwd_strided.
 */
FFPA_API size_t ffpa_decode_workspace_bytes(ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D);
FFPA_API ffpa_status ffpa_decode_fwd(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, ffpa_view o, float* lse,
                                     void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv,
                                     int D, int causal, float scale, ffpa_stream_t stream);

/*
 * FP8 forward (FFPA docs, "Backends Overview" page: the FP8 forward takes
 * fp16/bf16 Q/K/V and quantizes them for the kernel). The inputs are
 * quantized to e4m3 with one fp32 scale per (batch, head) and tensor
 * (amax / 448; codes = round-to-nearest-even, saturating, of x * 448 / amax),
 * then O = softmax(scale * S) V runs on the e4m3 operands with fp32
 * accumulation; P is rounded to e4m3 for the P V product. O (bf16/fp16 as
 * the inputs) and LSE (fp32 [B, Hq, Nq]) as in ffpa_fwd_strided.
 *   D: any multiple of 32 in [64, 1024] (the pages' FP8 range, "Backends
 *   Overview", capability matrix), and Nkv >= 1 (else FFPA_ERR_NOT_SUPPORTED).
 *   Packed (THD) batches: ffpa_varlen_fwd_fp8 below.
 *   workspace: device scratch of at least ffpa_fp8_workspace_bytes() bytes,
 *   256-byte aligned; it holds the codes and scales afterwards, at the
 *   offsets ffpa_fp8_workspace_layout() gives, with the head dim of the codes
 *   padded to Dp = D rounded up to 128 (zero codes past D):
 *   offsets[0] q8 [B, Hq, Nq, Dp], [1] k8 [B, Hkv, Nkv, Dp], [2] V^T codes
 *   [B, Hkv, Dp, ldv], [3] sq fp32 [B*Hq], [4] sk fp32 [B*Hkv], [5] sv fp32
 *   [B*Hkv], [6] ldv (Nkv rounded up to 16), [7] total bytes.
 * ffpa_fp8_quantize runs only the quantization into the workspace.
 */
FFPA_API size_t ffpa_fp8_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nkv, int D);
FFPA_API size_t ffpa_fp8_workspace_layout(int B, int Hq, int Hkv, int Nq, int Nkv, int D, size_t* offsets);
FFPA_API ffpa_status ffpa_fp8_quantize(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, void* workspace,
                                       size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                                       ffpa_stream_t stream);
FFPA_API ffpa_status ffpa_fwd_fp8(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, ffpa_view o, float* lse,
                                  void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv,
                                  int D, int causal, float scale, ffpa_stream_t stream);
/* The attention of ffpa_fwd_fp8 alone, on a workspace that ffpa_fp8_quantize
 * (or ffpa_fwd_fp8) filled for the same sizes: for inputs quantized once and
 * attended many times (a cached e4m3 K/V). No q/k/v pointers are read. */
FFPA_API ffpa_status ffpa_fwd_fp8_quantized(ffpa_dtype dt, ffpa_view o, float* lse, const void* workspace,
                                            size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                                            int causal, float scale, ffpa_stream_t stream);
/* FP8 forward of a packed (THD) batch: the layout, cu_seqlens contract and
 * device-side checks of ffpa_varlen_fwd ("CuTe-DSL Backend", "Varlen (packed
 * THD) API"; a sequence that breaks them sets FFPA_ERR_INVALID_VALUE in the
 * status word), with the quantization of ffpa_fwd_fp8 applied per
 * (sequence, head) and tensor. The pages' FP8 rows ("Backends Overview",
 * capability matrix) offer no packed layout; this is the plain extension:
 * each sequence is quantized and attended as the dense FP8 forward would one
 * batch entry.
 *   total_k >= 1 when total_q >= 1 (else FFPA_ERR_NOT_SUPPORTED); D as for
 *   ffpa_fwd_fp8.
 *   workspace: device scratch of at least ffpa_varlen_fp8_workspace_bytes()
 *   bytes, 256-byte aligned (codes of every token, head dim padded to a
 *   multiple of 128; V transposed with sequence b's keys from column
 *   16 ceil(cu_k[b] / 16) + 16 b; per-(sequence, head) scales). Its contents
 *   afterwards are not part of the interface.
 *   Returns before any launch on invalid arguments; asynchronous on `stream`. */
FFPA_API size_t ffpa_varlen_fp8_workspace_bytes(int batch, int total_q, int total_k, int max_seqlen_q,
                                                int max_seqlen_k, int Hq, int Hkv, int D);
FFPA_API ffpa_status ffpa_varlen_fwd_fp8(ffpa_dtype dt, const void* q, const void* k, const void* v, void* o,
                                         float* lse, const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                                         int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int Hq,
                                         int Hkv, int D, int causal, float scale, void* workspace,
                                         size_t workspace_bytes, ffpa_stream_t stream);

/* Workspace bytes ffpa_bwd needs for this problem (fp32 row statistics). */
FFPA_API size_t ffpa_bwd_workspace_bytes(ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D);
/*
 * Workspace bytes that also hold dS^T and P^T for the stored-tile backward:
 * on a dense problem whose head dim is a multiple of 64 up to 1024,
 * ffpa_bwd / ffpa_bwd_strided given a
 * workspace at least this large
 *   - have the dK launch also store every P^T tile (in the input dtype) and
 *     form dV = P^T dO with one GEMM after it, instead of a dV launch that
 *     computes S^T = K Q^T again (2 GEMM units become 1);
 *   - have the dK launch also store every dS tile (bf16/fp16, the same
 *     rounded values it multiplies) and form dQ = scale dS K with one GEMM,
 *     instead of recomputing S and dP in a dQ launch (3 GEMM units become 1).
 * Each buffer is B * Hq * Nkv * round_up(Nq, 8) * 2 bytes. A workspace with
 * room for the dS buffer only (ffpa_bwd_workspace_bytes() plus one buffer)
 * keeps the stored dS and the dV launch that recomputes S^T. Returns
 * ffpa_bwd_workspace_bytes() where the path does not apply.
 */
FFPA_API size_t ffpa_bwd_workspace_bytes_ds(ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                                            int causal);

/*
 * The stored-tile backward within a memory budget (the FFPA pages' training
 * path is FlashAttention-style, "Backends Overview", "Choosing a backend":
 * its scratch stays bounded however long the sequences are). A workspace
 * smaller than ffpa_bwd_workspace_bytes_ds() but with room for both tile sets
 * (dS^T and P^T) of at least one kv group (a kv head and its Hq / Hkv query
 * heads: 2 * B * (Hq / Hkv) * Nkv * round_up(Nq, 8) * 2 bytes, plus 256) runs
 * the same kernels in chunks of kv groups: per chunk, dK over the chunk's kv
 * heads storing their tiles, then the dV and dQ GEMMs over them. Each group's
 * gradients are complete within its chunk (no cross-chunk accumulation, the
 * same results as the one-chunk path). The chunks hold as many groups as fit,
 * evened out over the kv heads. Chunks apply to calls that run the dV, dK and
 * dQ stages together (ffpa_bwd, ffpa_bwd_strided, ffpa_varlen_bwd, or
 * ffpa_bwd_stages with bits 1..3 and neither bit 4 nor 5).
 * This query returns the workspace size to pass for at most `budget` bytes:
 * ffpa_bwd_workspace_bytes_ds() when it fits, else the bytes of the largest
 * evened-out chunk that fits, else ffpa_bwd_workspace_bytes() (the
 * recomputing backward). Its result depends only on the problem and the
 * budget, not on the device's free memory.
 */
FFPA_API size_t ffpa_bwd_workspace_bytes_budget(ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                                                int causal, size_t budget);

/*
 * Dense backward (FFPA docs, CuTe-DSL Backend page, "Blackwell status": a
 * preprocess launch followed by gradient launches; gradients are returned in
 * the input dtype, "Configuration"). Runs four kernels in stream order:
 * delta = rowsum(dO * O), then dV, dK and dQ.
 *   q, o, dO, dq : [B, Hq, Nq, D];  k, v, dk, dv : [B, Hkv, Nkv, D]
 *   lse : [B, Hq, Nq] fp32 as written by ffpa_fwd for the same inputs.
 *   workspace : device scratch of >= ffpa_bwd_workspace_bytes() bytes,
 *               256-byte aligned; its contents on entry do not matter.
 */
FFPA_API ffpa_status ffpa_bwd(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes,
                     int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale,
                     ffpa_stream_t stream);

/*
 * Dense backward on strided views (otherwise as ffpa_bwd; the workspace is
 * sized by ffpa_bwd_workspace_bytes). q, o, dO, dq: [B, Hq, Nq, D] views;
 * k, v, dk, dv: [B, Hkv, Nkv, D] views; lse: contiguous fp32 [B, Hq, Nq].
 */
FFPA_API ffpa_status ffpa_bwd_strided(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, ffpa_view o,
                                      const float* lse, ffpa_view dO, ffpa_view dq, ffpa_view dk, ffpa_view dv,
                                      void* workspace, size_t workspace_bytes,
                                      int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale,
                                      ffpa_stream_t stream);

/*
 * The launches of ffpa_bwd, selectable: bit 0 = preprocess (delta and scaled
 * LSE into the workspace), bit 1 = dV, bit 2 = dQ, bit 3 = dK. Stages run in
 * the order preprocess, dV, dK, dQ on `stream`; the gradient stages read the
 * workspace the preprocess stage wrote, so a caller that splits them issues
 * bit 0 first (the FFPA docs' CuTe-DSL page, "Blackwell status", describes the
 * same four launches). ffpa_bwd(...) == ffpa_bwd_stages(..., 15).
 * With the workspace of ffpa_bwd_workspace_bytes_ds (dense, D % 64 == 0, D <= 1024),
 * a dK stage also stores dS and a dQ stage in the same call is the
 * dS K GEMM; bit 4 runs that GEMM alone on the dS an earlier dK stage stored
 * in this workspace for the same inputs (bit 2 alone recomputes S and dP).
 * With dV and dK in one call, the dK stage also stores P^T and the dV stage
 * is the P^T dO GEMM, run after dK; bit 5 selects that mode for a dK or dV
 * stage on its own (a dV stage with bit 5 reads the P an earlier dK stage
 * with bit 5 stored in this workspace for the same inputs). Bits 4 and 5
 * without the workspace room they use are FFPA_ERR_INVALID_VALUE. Arguments
 * otherwise as ffpa_bwd.
 */
FFPA_API ffpa_status ffpa_bwd_stages(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes,
                                     int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale,
                                     unsigned stages, ffpa_stream_t stream);

/*
 * Dense backward that allocates nothing and takes no workspace. The FFPA
 * pages have no counterpart of this call; it exists for callers that cannot
 * allocate device memory at all (a fixed, pre-planned memory pool with no
 * spare buffer, a plugin host that owns every allocation, or a latency path
 * where cudaMalloc would synchronise the device).
 *   Arguments, layouts and results are those of ffpa_bwd without the
 *   workspace pair. The scratch comes from a 4 MiB array inside the library's
 *   device image, which holds B*Hq*Nq <= 524288 query rows; larger problems
 *   return FFPA_ERR_INVALID_VALUE (use ffpa_bwd). Every GPU that loads the
 *   library keeps that array until the process exits.
 *   It always runs the four launches of ffpa_bwd with the small workspace
 *   (preprocess, then dV, dK and dQ, each recomputing its scores), never the
 *   stored-tile path.
 *   The first call on a device looks up the array's device address (once per
 *   device); make that first call before any stream capture. The address is
 *   not looked up again: the call is not valid after a cudaDeviceReset of its
 *   device in the same process.
 *   All calls on a device share the array: calls whose kernels overlap on the
 *   GPU (unordered streams) race on it. Calls ordered on one stream do not;
 *   nothing in the array needs to start at zero.
 */
FFPA_API ffpa_status ffpa_bwd_noalloc(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                      int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale,
                                      ffpa_stream_t stream);

/*
 * Packed varlen forward (FFPA docs, CuTe-DSL Backend page, "Varlen (packed
 * THD) API"): sequences are packed along T; sequence b owns query rows
 * [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key rows
 * [cu_seqlens_k[b], cu_seqlens_k[b+1]). Causal is bottom-right per sequence.
 *   q, o : [total_q, Hq, D];  k, v : [total_k, Hkv, D]
 *   lse  : [Hq, total_q] fp32
 *   cu_seqlens_q, cu_seqlens_k : int32 [batch+1] DEVICE arrays, start at 0,
 *     nondecreasing, last entries equal total_q / total_k (both required; pass
 *     the same pointer twice for self-attention). Read on the device only.
 *   max_seqlen_q / max_seqlen_k : upper bounds of the per-sequence lengths
 *     (they size the launch grid).
 * cu_seqlens live on the device, so their contract is checked there: a
 * sequence whose offsets are negative or decreasing, run past total_q /
 * total_k, or whose length exceeds max_seqlen_q / max_seqlen_k is not
 * processed, and the kernels record the error in the device status word;
 * the next ffpa_get_status() returns FFPA_ERR_INVALID_VALUE naming the
 * sequence (the FFPA varlen API raises instead of silently unpacking a batch
 * it cannot process). Outputs of such a call are undefined; nothing is read
 * or written outside the caller's tensors.
 */
FFPA_API ffpa_status ffpa_varlen_fwd(ffpa_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int total_q,
                            int total_k, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                            int causal, float scale, ffpa_stream_t stream);

FFPA_API size_t ffpa_varlen_bwd_workspace_bytes(ffpa_dtype dt, int batch, int total_q, int total_k, int max_seqlen_q,
                                       int max_seqlen_k, int Hq, int Hkv, int D);
/*
 * Workspace bytes of the stored-tile varlen backward (as
 * ffpa_bwd_workspace_bytes_ds, for packed batches with D a multiple of 64 up
 * to 1024). The two tile buffers are Hq x (total_k + 256 * batch) x
 * round_up(max_seqlen_q, 8) 16-bit values each: sequence b's key rows start
 * at row cu_seqlens_k[b] + 256 b, and its queries are the columns from 0.
 * Returns ffpa_varlen_bwd_workspace_bytes() where the path does not apply.
 */
FFPA_API size_t ffpa_varlen_bwd_workspace_bytes_ds(ffpa_dtype dt, int batch, int total_q, int total_k,
                                                   int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                                   int causal);

/* As ffpa_bwd_workspace_bytes_budget, for packed batches (one group's tiles are
 * 2 * (Hq / Hkv) * (total_k + 256 * batch) * round_up(max_seqlen_q, 8) * 2 bytes). */
FFPA_API size_t ffpa_varlen_bwd_workspace_bytes_budget(ffpa_dtype dt, int batch, int total_q, int total_k,
                                                       int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                                       int causal, size_t budget);

/* Packed varlen backward; layouts as in ffpa_varlen_fwd, dq like q, dk/dv like k.
 * cu_seqlens and max_seqlen_* are checked on the device as in ffpa_varlen_fwd. */
FFPA_API ffpa_status ffpa_varlen_bwd(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv,
                            const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int total_q,
                            int total_k, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                            int causal, float scale, void* workspace, size_t workspace_bytes,
                            ffpa_stream_t stream);

/*
 * Synchronises `stream`, then reports and clears the device status word:
 * FFPA_OK, FFPA_ERR_TIMEOUT (a bounded device wait ran out; the kernel
 * returned early and its outputs are undefined), FFPA_ERR_INVALID_VALUE (a
 * packed varlen sequence broke the cu_seqlens / max_seqlen contract; see
 * ffpa_varlen_fwd) or FFPA_ERR_CUDA (the stream reported an error).
 */
FFPA_API ffpa_status ffpa_get_status(ffpa_stream_t stream);

/* Message for the last failing call on this host thread ("" if none). */
FFPA_API const char* ffpa_last_error(void);

/*
 * Upper bound, in nanoseconds, of any single device-side wait in later
 * launches (default 2e9). 0 restores the default.
 */
FFPA_API void ffpa_set_wait_limit_ns(uint64_t ns);

/*
 * Self-test of the bounded-wait path: launches one block whose single thread
 * waits on a barrier that nothing completes, with a limit of `limit_ns`, and
 * returns what ffpa_get_status() then reports (FFPA_ERR_TIMEOUT when the
 * mechanism works). Touches no user memory.
 */
FFPA_API ffpa_status ffpa_selftest_wait_timeout(uint64_t limit_ns, ffpa_stream_t stream);

/* Number of streaming multiprocessors of the current device (0 on error). */
FFPA_API int ffpa_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* FFPA_H_ */
