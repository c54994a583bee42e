// FP8 (e4m3) quantization of the forward's inputs.
//
// The FFPA docs ("Backends Overview" page, capability matrix notes) list FP8
// forward kernels that take fp16/bf16 Q/K/V and quantize them in the kernel.
// Here the quantization is one pass ahead of the attention kernel (every
// K/V tile is read by many row tiles, so it is quantized once, not once per
// use) and writes the operands in the layouts the tensor cores read:
//   q8  [B, Hq,  Nq,  Dp] e4m3, rows of Dp bytes (K-major for S = Q K^T)
//   k8  [B, Hkv, Nkv, Dp] e4m3
//   v8t [B, Hkv, Dp, ldv] e4m3, V transposed (keys contiguous, ldv = Nkv
//       rounded up to 16) so that O += P V reads it K-major
// with the head dim padded to Dp = D rounded up to 128 (whole 128-byte code
// chunks for the tensor maps and the MMAs): the pad holds zero codes, which
// add nothing to the scores, and the output columns past D are not stored.
//   sq [B*Hq], sk [B*Hkv], sv [B*Hkv] fp32 dequantization scales
// Packed (varlen) batches of B sequences are laid out as one batch entry of
// all tokens: q8 [1, Hq, total_q, Dp], k8 [1, Hkv, total_k, Dp], and v8t
// [1, Hkv, Dp, ldv] with sequence b's keys from column
//   vt_col0(b) = 16 ceil(cu_k[b] / 16) + 16 b
// (tensor-map loads of 8-bit codes start at multiples of 16 columns) and zero
// codes in the gaps between sequences; the scales are per (sequence, head).
// One scale per (batch, head) and tensor: amax = max |x| over the head,
// scale = amax / 448, inv = 448 / amax (fp32, correctly rounded; 1 and 1 for
// an all-zero head), code = e4m3(fp32(x * inv)) rounded to nearest even with
// saturation to +-448 (cvt.rn.satfinite).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr int kQRows = 64;     // rows per block of the amax and q/k passes
constexpr int kVKeys = 64;     // keys per block of the V transpose
constexpr float kE4M3Max = 448.f;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct QArgs {
    const void *q, *k, *v;
    View vq, vk, vv;
    int B, Hq, Hkv, Nq, Nkv, D, ldv;  // packed batches: B sequences, Nq / Nkv their bound
    const int *cu_q, *cu_k;           // packed batches: sequence offsets (device), else null
    int total_q, total_k;
    int Dp;                 // code row length: D rounded up to 128 (zero codes past D)
    int nsq, nsk;           // row blocks per q head / per k or v head
    uint8_t *q8, *k8, *v8t;
    float *sq, *sk, *sv;
    float* part;            // [B*Hq*nsq | B*Hkv*nsk (k) | B*Hkv*nsk (v)] partial amax
};

__device__ __forceinline__ float to_f(uint16_t u, bool bf16)
{
    return bf16 ? __uint_as_float(static_cast<uint32_t>(u) << 16) : __half2float(__ushort_as_half(u));
}

// tensor t (0 q, 1 k, 2 v) and head index of grid row y
__device__ __forceinline__ void tensor_of(const QArgs& a, int y, int& t, int& hi)
{
    const int nq = a.B * a.Hq, nk = a.B * a.Hkv;
    if (y < nq) { t = 0; hi = y; }
    else if (y < nq + nk) { t = 1; hi = y - nq; }
    else { t = 2; hi = y - nq - nk; }
}

// Rows of head hi (b * H + h) of tensor t: the n-th has token tok0 + n, n < len.
// A packed sequence that breaks its bounds counts as empty here and returns
// false (the attention kernel reports it).
__device__ __forceinline__ bool seq_rows(const QArgs& a, int t, int hi, int& tok0, int& len)
{
    const int H = t == 0 ? a.Hq : a.Hkv;
    const int N = t == 0 ? a.Nq : a.Nkv;
    tok0 = 0;
    len = N;
    if (a.cu_q) {
        const int* cu = t == 0 ? a.cu_q : a.cu_k;
        const int total = t == 0 ? a.total_q : a.total_k;
        const int b = hi / H;
        const int c0 = cu[b], c1 = cu[b + 1];
        const bool good = c0 >= 0 && c1 >= c0 && c1 <= total && c1 - c0 <= N;
        tok0 = good ? c0 : 0;
        len = good ? c1 - c0 : 0;
        return good;
    }
    return true;
}

__device__ __forceinline__ const uint16_t* row_ptr(const QArgs& a, int t, int hi, int n)
{
    const int H = t == 0 ? a.Hq : a.Hkv;
    const View& v = t == 0 ? a.vq : (t == 1 ? a.vk : a.vv);
    const void* base = t == 0 ? a.q : (t == 1 ? a.k : a.v);
    const long b = hi / H, h = hi % H;
    return reinterpret_cast<const uint16_t*>(base) + b * v.sb + h * v.sh + static_cast<long>(n) * v.sn;
}

__device__ __forceinline__ float block_max(float m, float* red)
{
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    }
    return m;  // valid in thread 0
}

// Pass 1: partial amax of kQRows rows of one head of q, k or v.
__global__ void __launch_bounds__(256) amax_kernel(const QArgs a, bool bf16)
{
    __shared__ float red[8];
    const long long y = unit_id();  // head of q, k or v
    if (y >= static_cast<long long>(a.B) * (a.Hq + 2 * a.Hkv)) return;
    int t, hi;
    tensor_of(a, static_cast<int>(y), t, hi);
    int tok0, N;
    seq_rows(a, t, hi, tok0, N);
    const int ns = t == 0 ? a.nsq : a.nsk;
    if (static_cast<int>(blockIdx.x) >= ns) return;
    const int n0 = blockIdx.x * kQRows, n1 = min(N, n0 + kQRows);
    const int units = a.D / 8;  // 16-byte units per row
    float m = 0.f;
    for (int e = threadIdx.x; e < (n1 - n0) * units; e += blockDim.x) {
        const uint4 w = *reinterpret_cast<const uint4*>(row_ptr(a, t, hi, tok0 + n0 + e / units) + (e % units) * 8);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m = fmaxf(m, fabsf(to_f(static_cast<uint16_t>(u[i] & 0xffffu), bf16)));
            m = fmaxf(m, fabsf(to_f(static_cast<uint16_t>(u[i] >> 16), bf16)));
        }
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) {
        const size_t base = t == 0 ? 0 : (t == 1 ? static_cast<size_t>(a.B) * a.Hq * a.nsq
                                                 : static_cast<size_t>(a.B) * a.Hq * a.nsq +
                                                       static_cast<size_t>(a.B) * a.Hkv * a.nsk);
        a.part[base + static_cast<size_t>(hi) * ns + blockIdx.x] = m;
    }
}

// amax of a head from its partials -> (scale, inv); block-wide, result in shared memory
__device__ __forceinline__ void head_scale(const QArgs& a, int t, int hi, float* sm)
{
    __shared__ float red[8];
    const int ns = t == 0 ? a.nsq : a.nsk;
    const size_t base = t == 0 ? 0 : (t == 1 ? static_cast<size_t>(a.B) * a.Hq * a.nsq
                                             : static_cast<size_t>(a.B) * a.Hq * a.nsq +
                                                   static_cast<size_t>(a.B) * a.Hkv * a.nsk);
    float m = 0.f;
    for (int i = threadIdx.x; i < ns; i += blockDim.x) m = fmaxf(m, a.part[base + static_cast<size_t>(hi) * ns + i]);
    m = block_max(m, red);
    if (threadIdx.x == 0) {
        sm[0] = m > 0.f ? m / kE4M3Max : 1.f;   // IEEE division (no fast-math): correctly rounded
        sm[1] = m > 0.f ? kE4M3Max / m : 1.f;
    }
    __syncthreads();
}

// Pass 2a: q and k rows -> e4m3 codes (row-major), and the scales.
__global__ void __launch_bounds__(256) quant_rows_kernel(const QArgs a, bool bf16)
{
    __shared__ float sm[2];
    const long long y = unit_id();  // head of q or k
    if (y >= static_cast<long long>(a.B) * (a.Hq + a.Hkv)) return;
    int t, hi;
    tensor_of(a, static_cast<int>(y), t, hi);
    int tok0, N;
    seq_rows(a, t, hi, tok0, N);
    const int ns = t == 0 ? a.nsq : a.nsk;
    if (static_cast<int>(blockIdx.x) >= ns) return;
    head_scale(a, t, hi, sm);
    const float inv = sm[1];
    if (blockIdx.x == 0 && threadIdx.x == 0) (t == 0 ? a.sq : a.sk)[hi] = sm[0];
    // codes of row n at out + n * Dp (packed: the head's token rows, from token tok0)
    const int H = t == 0 ? a.Hq : a.Hkv;
    const size_t head_rows = a.cu_q ? static_cast<size_t>(hi % H) * (t == 0 ? a.total_q : a.total_k) + tok0
                                    : static_cast<size_t>(hi) * N;
    uint8_t* out = (t == 0 ? a.q8 : a.k8) + head_rows * a.Dp;
    const int n0 = blockIdx.x * kQRows, n1 = min(N, n0 + kQRows);
    const int units = a.Dp / 8, in_units = a.D / 8;  // 8 codes per unit; units past D write zero codes
    for (int e = threadIdx.x; e < (n1 - n0) * units; e += blockDim.x) {
        const int n = n0 + e / units, u8 = e % units;
        const uint4 w = u8 < in_units ? *reinterpret_cast<const uint4*>(row_ptr(a, t, hi, tok0 + n) + u8 * 8)
                                      : make_uint4(0, 0, 0, 0);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float x0 = to_f(static_cast<uint16_t>(u[2 * i] & 0xffffu), bf16) * inv;
            const float x1 = to_f(static_cast<uint16_t>(u[2 * i] >> 16), bf16) * inv;
            const float x2 = to_f(static_cast<uint16_t>(u[2 * i + 1] & 0xffffu), bf16) * inv;
            const float x3 = to_f(static_cast<uint16_t>(u[2 * i + 1] >> 16), bf16) * inv;
            o[i] = static_cast<uint32_t>(cvt_e4m3x2(x0, x1)) | (static_cast<uint32_t>(cvt_e4m3x2(x2, x3)) << 16);
        }
        *reinterpret_cast<uint2*>(out + static_cast<size_t>(n) * a.Dp + u8 * 8) = make_uint2(o[0], o[1]);
    }
}

// Pass 2b: v -> transposed e4m3 codes. Block (key tile, b * Hkv): kVKeys keys
// x all of D, through shared memory in 64-column slices.
__global__ void __launch_bounds__(256) quant_vt_kernel(const QArgs a, bool bf16)
{
    __shared__ float sm[2];
    __shared__ float tile[kVKeys][64 + 1];
    const long long y = unit_id();
    if (y >= static_cast<long long>(a.B) * a.Hkv) return;
    const int hi = static_cast<int>(y);  // b * Hkv + hk
    head_scale(a, 2, hi, sm);
    const float inv = sm[1];
    if (blockIdx.x == 0 && threadIdx.x == 0) a.sv[hi] = sm[0];
    int tok0, Nk;
    if (!seq_rows(a, 2, hi, tok0, Nk)) return;  // nothing of a malformed sequence is written
    const int k0 = blockIdx.x * kVKeys;
    const int nk = min(kVKeys, Nk - k0);
    // the head's code rows; packed: the sequence's first column vt_col0(b)
    int col0 = 0;
    uint8_t* out = a.v8t + static_cast<size_t>(hi) * a.Dp * a.ldv;
    if (a.cu_q) {
        const int b = hi / a.Hkv;
        col0 = 16 * ((tok0 + 15) / 16) + 16 * b;
        out = a.v8t + static_cast<size_t>(hi % a.Hkv) * a.Dp * a.ldv + col0;
        if (blockIdx.x == 0) {
            // zero codes from the sequence's last 16-key group to the next sequence
            const int b1 = 16 * ((tok0 + Nk + 15) / 16) + 16 * (b + 1);  // cu_k[b + 1] = tok0 + Nk
            const int z0 = col0 + (Nk + 15) / 16 * 16;
            const int zn = min(b1, a.ldv) - z0;  // columns
            for (int e = threadIdx.x; zn > 0 && e < a.Dp * zn; e += blockDim.x)
                out[static_cast<size_t>(e / zn) * a.ldv + (z0 - col0) + e % zn] = 0;
        }
    }
    for (int d0 = 0; d0 < a.Dp; d0 += 64) {
        // load kVKeys x 64 (16-byte units: 8 per row; zeros past the keys and past D)
        for (int e = threadIdx.x; e < kVKeys * 8; e += blockDim.x) {
            const int r = e / 8, u = e % 8;
            uint4 w = make_uint4(0, 0, 0, 0);
            if (r < nk && d0 + u * 8 < a.D)
                w = *reinterpret_cast<const uint4*>(row_ptr(a, 2, hi, tok0 + k0 + r) + d0 + u * 8);
            const uint32_t uu[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                tile[r][u * 8 + 2 * i] = to_f(static_cast<uint16_t>(uu[i] & 0xffffu), bf16) * inv;
                tile[r][u * 8 + 2 * i + 1] = to_f(static_cast<uint16_t>(uu[i] >> 16), bf16) * inv;
            }
        }
        __syncthreads();
        // store 64 d-rows x kVKeys keys: each thread 16 keys of one d-row
        {
            const int dr = threadIdx.x / (kVKeys / 16), kq = threadIdx.x % (kVKeys / 16);
            if (dr < 64 && k0 + kq * 16 < Nk) {
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kk = kq * 16 + 4 * i;
                    o[i] = static_cast<uint32_t>(cvt_e4m3x2(tile[kk][dr], tile[kk + 1][dr])) |
                           (static_cast<uint32_t>(cvt_e4m3x2(tile[kk + 2][dr], tile[kk + 3][dr])) << 16);
                }
                *reinterpret_cast<uint4*>(out + static_cast<size_t>(d0 + dr) * a.ldv + k0 + kq * 16) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        __syncthreads();
    }
}

}  // namespace

Fp8Layout fp8_layout(int B, int Hq, int Hkv, int Nq, int Nkv, int D)
{
    Fp8Layout L{};
    L.ldv = (Nkv + 15) & ~15;
    L.dp = (D + 127) & ~127;
    const size_t Dp = static_cast<size_t>(L.dp);
    size_t off = 0;
    L.q8 = off;
    off = align256(off + static_cast<size_t>(B) * Hq * Nq * Dp);
    L.k8 = off;
    off = align256(off + static_cast<size_t>(B) * Hkv * Nkv * Dp);
    L.v8t = off;
    off = align256(off + static_cast<size_t>(B) * Hkv * Dp * L.ldv);
    L.sq = off;
    off = align256(off + static_cast<size_t>(B) * Hq * sizeof(float));
    L.sk = off;
    off = align256(off + static_cast<size_t>(B) * Hkv * sizeof(float));
    L.sv = off;
    off = align256(off + static_cast<size_t>(B) * Hkv * sizeof(float));
    L.part = off;
    const size_t nsq = (Nq + kQRows - 1) / kQRows, nsk = (Nkv + kQRows - 1) / kQRows;
    off = align256(off + (static_cast<size_t>(B) * Hq * nsq + 2 * static_cast<size_t>(B) * Hkv * nsk) * sizeof(float));
    L.total = off;
    return L;
}

Fp8Layout fp8_varlen_layout(int batch, int Hq, int Hkv, int total_q, int total_k, int max_q, int max_k, int D)
{
    Fp8Layout L{};
    // sequence b's keys from column 16 ceil(cu_k[b] / 16) + 16 b: the last one ends
    // by 16 ceil(total_k / 16) + 16 (batch - 1) + 16
    L.ldv = 16 * ((total_k + 15) / 16) + 16 * batch;
    L.dp = (D + 127) & ~127;
    const size_t Dp = static_cast<size_t>(L.dp);
    size_t off = 0;
    L.q8 = off;
    off = align256(off + static_cast<size_t>(Hq) * total_q * Dp);
    L.k8 = off;
    off = align256(off + static_cast<size_t>(Hkv) * total_k * Dp);
    L.v8t = off;
    off = align256(off + static_cast<size_t>(Hkv) * Dp * L.ldv);
    L.sq = off;
    off = align256(off + static_cast<size_t>(batch) * Hq * sizeof(float));
    L.sk = off;
    off = align256(off + static_cast<size_t>(batch) * Hkv * sizeof(float));
    L.sv = off;
    off = align256(off + static_cast<size_t>(batch) * Hkv * sizeof(float));
    L.part = off;
    const size_t nsq = (max_q + kQRows - 1) / kQRows, nsk = (max_k + kQRows - 1) / kQRows;
    off = align256(off + (static_cast<size_t>(batch) * Hq * nsq + 2 * static_cast<size_t>(batch) * Hkv * nsk) *
                             sizeof(float));
    L.total = off;
    return L;
}

Fp8Layout fp8_layout_of(const Problem& pb)
{
    return pb.varlen ? fp8_varlen_layout(pb.B, pb.Hq, pb.Hkv, pb.total_q, pb.total_k, pb.Nq, pb.Nkv, pb.D)
                     : fp8_layout(pb.B, pb.Hq, pb.Hkv, pb.Nq, pb.Nkv, pb.D);
}

cudaError_t launch_fp8_quantize(const FwdArgs& f, void* workspace, cudaStream_t s)
{
    const Problem& pb = f.pb;
    const Fp8Layout L = fp8_layout_of(pb);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    QArgs a{};
    a.q = f.q;
    a.k = f.k;
    a.v = f.v;
    a.vq = pb.vq;
    a.vk = pb.vk;
    a.vv = pb.vv;
    a.B = pb.B;
    a.Hq = pb.Hq;
    a.Hkv = pb.Hkv;
    a.Nq = pb.Nq;
    a.Nkv = pb.Nkv;
    a.cu_q = pb.varlen ? pb.cu_q : nullptr;
    a.cu_k = pb.varlen ? pb.cu_k : nullptr;
    a.total_q = pb.total_q;
    a.total_k = pb.total_k;
    a.D = pb.D;
    a.Dp = L.dp;
    a.ldv = L.ldv;
    a.nsq = (pb.Nq + kQRows - 1) / kQRows;
    a.nsk = (pb.Nkv + kQRows - 1) / kQRows;
    a.q8 = ws + L.q8;
    a.k8 = ws + L.k8;
    a.v8t = ws + L.v8t;
    a.sq = reinterpret_cast<float*>(ws + L.sq);
    a.sk = reinterpret_cast<float*>(ws + L.sk);
    a.sv = reinterpret_cast<float*>(ws + L.sv);
    a.part = reinterpret_cast<float*>(ws + L.part);
    const long long heads = static_cast<long long>(pb.B) * (pb.Hq + 2 * pb.Hkv);
    const int splits = max(a.nsq, a.nsk);
    // grids of (row block, head) over x and the heads spread by unit_grid
    dim3 g_amax, g_rows, g_vt;
    if (!unit_grid(splits, heads, &g_amax) || !unit_grid(splits, static_cast<long long>(pb.B) * (pb.Hq + pb.Hkv), &g_rows) ||
        !unit_grid((pb.Nkv + kVKeys - 1) / kVKeys > 0 ? (pb.Nkv + kVKeys - 1) / kVKeys : 1,
                   static_cast<long long>(pb.B) * pb.Hkv, &g_vt))
        return cudaErrorInvalidConfiguration;
    amax_kernel<<<g_amax, 256, 0, s>>>(a, f.bf16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    quant_rows_kernel<<<g_rows, 256, 0, s>>>(a, f.bf16);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (pb.Nkv > 0) {
        quant_vt_kernel<<<g_vt, 256, 0, s>>>(a, f.bf16);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_fwd_fp8(const FwdArgs& f, void* workspace, cudaStream_t s, bool quantize)
{
    const Problem& pb = f.pb;
    if (quantize) {
        const cudaError_t e = launch_fp8_quantize(f, workspace, s);
        if (e != cudaSuccess) return e;
    }
    const Fp8Layout L = fp8_layout_of(pb);
    const uint8_t* ws = static_cast<const uint8_t*>(workspace);
    XArgs x{};
    x.pb = pb;
    x.pb.D = L.dp;     // the tiles run over the padded head dim (zero codes past D) ...
    x.d_out = pb.D;    // ... and the epilogue stores the D real columns
    x.bf16 = f.bf16;
    x.q = ws + L.q8;
    x.k = ws + L.k8;
    x.v = nullptr;
    x.o = f.o;
    x.lse = f.lse;
    x.ctl = f.ctl;
    x.f8 = 1;
    x.v8t = ws + L.v8t;
    x.ldv = L.ldv;
    x.f8_sq = reinterpret_cast<const float*>(ws + L.sq);
    x.f8_sk = reinterpret_cast<const float*>(ws + L.sk);
    x.f8_sv = reinterpret_cast<const float*>(ws + L.sv);
    return launch_pair(XOP_FWD, x, s);
}

}  // namespace ffpa
