// Decode / short-query forward: exact attention for a few query rows per head
// against a long key sequence, split over the keys (flash-decoding).
//
// The operation is the forward of the FFPA docs ("CuTe-DSL Backend" page,
// "Hard constraints": bottom-right causal mask, GQA/MQA head broadcast, empty
// rows give O = 0 and LSE = -inf). With Nq small the work is reading K and V
// once from HBM, so the layout differs from the tile kernels:
//   - a CTA owns one (batch, kv head, key split) and 16 of the R = G * Nq
//     query rows of that kv head's group (one m16 MMA tile; R > 16 takes
//     ceil(R / 16) row blocks), so every K/V byte is read once per split and
//     row block and serves all rows of the block;
//   - a producer warp streams K and V tiles of KT keys into a ring of shared
//     memory stages with TMA (5-D chunked maps over the strided views);
//   - eight compute warps each own 64-wide head-dim chunks: partial scores
//     S = Q K^T over their chunks (mma.sync m16n8k16, fp32 accumulate), a sum
//     of the eight partials through shared memory, the online softmax (row
//     maximum and sum, per key tile), and O += P V on their chunks;
//   - each split writes its normalised partial O (fp32) and its LSE to a
//     workspace; a second kernel combines the splits:
//       LSE = ln sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
// Every wait is bounded (mbarrier waits with the time limit of the device
// control block); the compute warps never leave the tile loop early, so the
// shared-memory reductions always see all eight warps.
#include <cstring>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr int kDecThreads = 288;   // warps 0..7 compute, warp 8 TMA producer
constexpr int kDecRows = kDecodeRows;  // query rows per CTA (one m16 tile)
constexpr int kDecStages = 3;
// reduction buffers (18 KiB), also the Q staging area (16 rows x 1024 x 2 B at most)
constexpr int kDecRedBytes = 32768;
static_assert((8 * 8 * 32 + 8 * 32) * 8 <= kDecRedBytes && kDecRows * 1024 * 2 <= kDecRedBytes, "reduction area");
constexpr float kLn2 = 0.693147180559945309f;

enum DecSite : uint32_t { DS_PROD = 96, DS_FULL, DS_DRAIN };

// Barriers in one static block of exactly 1 KiB, so that the dynamic shared
// memory after it (the TMA stages, 128-byte swizzled) starts 1024-byte aligned.
struct __align__(1024) DecStatic {
    uint64_t full[kDecStages], empty[kDecStages];
    int abort_flag;
};
static_assert(sizeof(DecStatic) == 1024, "static shared block must be exactly 1 KiB");

struct DecGeo {
    int splits;       // key splits per (batch, kv head, row block)
    int rblocks;      // blocks of kDecRows query rows per kv head's group
    int tiles_per;    // key tiles per split
    int kt;           // keys per tile (32, or 16 when D > 512)
    int chunks;       // 64-wide head-dim chunks (ceil(D / 64))
    int stage_bytes;  // K + V bytes of one stage
    float* o_part;    // [splits][B*Hq*Nq][D] normalised partial outputs
    float* lse_part;  // [splits][B*Hq*Nq] natural-log partial LSE
};

// ---- warp-level tensor-core and shared-memory matrix helpers
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                               bool bf16)
{
    if (bf16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Shared address of 16-byte unit u (0..7) of row r in a 128-byte-swizzled
// block of rows (the layout TMA writes with SWIZZLE_128B; the block is 1 KiB aligned).
__device__ __forceinline__ uint32_t swz(uint32_t block, int r, int u)
{
    return block + static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
}

template <bool BF16>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tK, const __grid_constant__ CUtensorMap tV, const FwdArgs a,
                  const DecGeo gm)
{
    const Problem& pb = a.pb;
    const int G = pb.Hq / pb.Hkv;
    const int R = G * pb.Nq;            // query rows of the group
    // (batch, kv head, row block) in linear order, row block fastest
    const long long u = unit_id();
    if (u >= static_cast<long long>(pb.B) * pb.Hkv * gm.rblocks) return;  // past the last unit
    const int rb = static_cast<int>(u % gm.rblocks);  // this CTA's block of kDecRows of them
    const int unit = static_cast<int>(u / gm.rblocks);
    const int r0 = rb * kDecRows;        // group row of the CTA's row 0
    const int split = blockIdx.x;
    const int b = unit / pb.Hkv;
    const int hk = unit % pb.Hkv;
    const int KT = gm.kt;
    const int nch = gm.chunks;
    const int off = pb.Nkv - pb.Nq;      // causal: key j legal for query i iff j <= i + off
    const int key_begin = split * gm.tiles_per * KT;
    const int key_end = min(pb.Nkv, key_begin + gm.tiles_per * KT);
    const int n_tiles = key_end > key_begin ? (key_end - key_begin + KT - 1) / KT : 0;

    __shared__ DecStatic sh;
    uint64_t* const full = sh.full;
    uint64_t* const empty = sh.empty;
    extern __shared__ __align__(1024) uint8_t smem[];
    // stages: [K: chunks x KT rows x 128 B][V: same]; then kDecRedBytes for
    // the score reduction, part[8 warps][8 slots][32 lanes] and fin[8][32]
    // (float2), which holds Q (16 rows x D, 16-bit) before the first tile
    float* red_s = reinterpret_cast<float*>(smem + kDecStages * gm.stage_bytes);
    float2* const part = reinterpret_cast<float2*>(red_s);
    float2* const fin = part + 8 * 8 * 32;
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) atomicCAS(a.ctl.status, 0u, 5u | (0xffu << 8));
        return;
    }
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 8);  // one arrival per compute warp
        }
        sh.abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    volatile int* abort_p = &sh.abort_flag;
    uint32_t* status = a.ctl.status;
    const uint64_t lim = a.ctl.limit_ns;
    const uint32_t half_bytes = static_cast<uint32_t>(gm.stage_bytes / 2);

    if (warp == 8) {
        // ------------------------------------------------------ producer
        // lane 0 loads K, lane 1 loads V (one issuing thread serialises its
        // boxes; two keep the SM's share of HBM bandwidth in flight)
        if (lane < 2 && n_tiles > 0) {
            prefetch_tmap(lane == 0 ? &tK : &tV);
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % kDecStages;
                const uint32_t ph = static_cast<uint32_t>((t / kDecStages) & 1);
                if (!__all_sync(0x3u, mbar_wait(&empty[st], ph ^ 1u, abort_p, status, lim, DS_PROD))) break;
                uint8_t* dst = smem + st * gm.stage_bytes;
                if (lane == 0) mbar_arrive_expect_tx(&full[st], gm.stage_bytes);
                __syncwarp(0x3u);
                const int k0 = key_begin + t * KT;
                if (lane == 0)
                    tma_load_5d(dst, &tK, &full[st], 0, k0, 0, hk, b);
                else
                    tma_load_5d(dst + half_bytes, &tV, &full[st], 0, k0, 0, hk, b);
                ++issued;
            }
            // no loads in flight when the CTA leaves: wait for the last ones to be consumed
            if (lane == 0)
                for (int t = max(0, issued - kDecStages); t < issued; ++t) {
                    int dummy = 0;
                    if (!mbar_wait(&empty[t % kDecStages], static_cast<uint32_t>((t / kDecStages) & 1), &dummy, status,
                                   lim, DS_DRAIN, false))
                        break;
                }
        }
        return;
    }

    // ---------------------------------------------------------- compute warps
    // my head-dim chunks: warp, warp + 8 (D <= 1024 gives at most two)
    const int my_chunks = (warp < nch) + (warp + 8 < nch);
    const int r_lo = lane >> 2, r_hi = r_lo + 8;   // fragment rows of this thread
    const int cpair = (lane & 3) * 2;              // fragment column pair
    // Q rows of the group -> A fragments in registers, through shared memory
    // (red_s is free until the first tile)
    uint32_t qa[2][4][4];  // [chunk][k16 step][reg]
    {
        uint16_t* qs = reinterpret_cast<uint16_t*>(red_s);  // [16][nch*64] bf16/fp16, plain row-major
        const int width = nch * 64;
        for (int e = threadIdx.x; e < kDecRows * width / 8; e += 256) {
            const int r = e / (width / 8), u = e % (width / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r0 + r < R && u * 8 < pb.D) {
                const int g = (r0 + r) / pb.Nq, i = (r0 + r) % pb.Nq;
                const size_t o = static_cast<size_t>(b) * pb.vq.sb + static_cast<size_t>(hk * G + g) * pb.vq.sh +
                                 static_cast<size_t>(i) * pb.vq.sn + static_cast<size_t>(u) * 8;
                v = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + o);
            }
            *reinterpret_cast<uint4*>(qs + r * width + u * 8) = v;
        }
        // all 256 compute threads wrote their share; named barrier 1 covers the compute warps only
        asm volatile("bar.sync 1, 256;" ::: "memory");
        for (int cc = 0; cc < my_chunks; ++cc) {
            const int ch = warp + 8 * cc;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                // matrices: rows 0-7 / 8-15 x k 0-7 / 8-15 of this k16 step
                const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int mcol = ch * 64 + ks * 16 + (lane >> 4) * 8;
                ldsm_x4(smem_u32(qs + mrow * width + mcol), qa[cc][ks]);
            }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
    }

    float o_acc[2][8][4];  // [chunk][n8 tile of 64 columns][C fragment]
#pragma unroll
    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) o_acc[cc][n][e] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;  // log2-domain running max, sums
    // legal keys of a fragment row: j < jlim (rows past R have none; causal
    // rows stop at i + Nkv - Nq, bottom-right aligned)
    auto key_limit = [&](int r) {
        if (r0 + r >= R) return key_begin;
        return pb.causal ? min(key_end, (r0 + r) % pb.Nq + off + 1) : key_end;
    };
    const int jlim_lo = key_limit(r_lo), jlim_hi = key_limit(r_hi);
    const float c2 = pb.scale_log2;
    const int nkt8 = KT / 8;  // n8 tiles of keys per tile (4 or 2)
    bool ok = true;

    // Three steps per key tile, software-pipelined so that the score MMAs of
    // tile t + 1 are issued before the P V MMAs of tile t (independent work
    // for the tensor pipe while either waits):
    //   scores(t): wait for the stage, partial S over my head-dim chunks;
    //   softmax(t): reduce the partials across the eight warps, mask, online
    //               softmax -> P (A fragments) and the rescale factors;
    //   pv(t): rescale O, O += P V over my chunks, release the stage.
    float s[4][4];
    uint32_t pa[2][4];  // P of the current tile as A fragments: [k16 step][reg]
    float al_lo = 1.f, al_hi = 1.f;

    auto scores = [&](int t) {
        const int st = t % kDecStages;
        const uint32_t ph = static_cast<uint32_t>((t / kDecStages) & 1);
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[st], ph, abort_p, status, lim, DS_FULL));
        const uint32_t kbase = smem_u32(smem + st * gm.stage_bytes);
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
        if (!ok) return;
        for (int cc = 0; cc < my_chunks; ++cc) {
            const uint32_t blk = kbase + (warp + 8 * cc) * KT * 128;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    if (np * 2 >= nkt8) break;
                    // keys 16 np .. 16 np + 15, head-dim units 2 ks, 2 ks + 1 of the chunk
                    uint32_t kb[4];
                    const int krow = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    const int kunit = ks * 2 + ((lane >> 3) & 1);
                    ldsm_x4(swz(blk, krow, kunit), kb);
                    mma_bf16_16816(s[np * 2], qa[cc][ks], kb[0], kb[1], BF16);
                    mma_bf16_16816(s[np * 2 + 1], qa[cc][ks], kb[2], kb[3], BF16);
                }
            }
        }
    };

    auto softmax = [&](int t) {
        // sum the eight partials through shared memory as a reduce-scatter:
        // warp w stores its fragment as part[w][slot][lane] (slot j = 2 n + hi
        // holds the float2 of n-tile n, row r_lo or r_hi), thread (w', l) sums
        // slot w' of lane l over the eight warps into fin[w'][l], and every
        // warp then reads fin back in its own fragment layout. All accesses
        // are 256 contiguous bytes per warp (no bank conflicts); named barrier
        // 1 spans the 256 compute threads, which all pass it on every tile.
        const int nslots = nkt8 * 2;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            if (n >= nkt8) break;
            part[(warp * 8 + 2 * n) * 32 + lane] = make_float2(s[n][0], s[n][1]);
            part[(warp * 8 + 2 * n + 1) * 32 + lane] = make_float2(s[n][2], s[n][3]);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (warp < nslots) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const float2 p = part[(w * 8 + warp) * 32 + lane];
                acc.x += p.x;
                acc.y += p.y;
            }
            fin[warp * 32 + lane] = acc;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        float x[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            if (n >= nkt8) break;
            const float2 lo = fin[(2 * n) * 32 + lane], hi = fin[(2 * n + 1) * 32 + lane];
            const float acc[4] = {lo.x, lo.y, hi.x, hi.y};
            // scale to log2 units and mask (keys at or past the row's limit)
            const int j = key_begin + t * KT + n * 8 + cpair;
#pragma unroll
            for (int e = 0; e < 4; ++e) x[n][e] = j + (e & 1) < (e < 2 ? jlim_lo : jlim_hi) ? acc[e] * c2 : -INFINITY;
        }
        // online softmax over this tile (the four lanes of a row hold its columns)
        float tmax_lo = -INFINITY, tmax_hi = -INFINITY;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            if (n >= nkt8) break;
            tmax_lo = fmaxf(tmax_lo, fmaxf(x[n][0], x[n][1]));
            tmax_hi = fmaxf(tmax_hi, fmaxf(x[n][2], x[n][3]));
        }
        tmax_lo = fmaxf(tmax_lo, __shfl_xor_sync(0xffffffffu, tmax_lo, 1));
        tmax_lo = fmaxf(tmax_lo, __shfl_xor_sync(0xffffffffu, tmax_lo, 2));
        tmax_hi = fmaxf(tmax_hi, __shfl_xor_sync(0xffffffffu, tmax_hi, 1));
        tmax_hi = fmaxf(tmax_hi, __shfl_xor_sync(0xffffffffu, tmax_hi, 2));
        const float mn_lo = fmaxf(m_lo, tmax_lo), mn_hi = fmaxf(m_hi, tmax_hi);
        al_lo = (mn_lo == -INFINITY) ? 1.f : ex2_approx(m_lo - mn_lo);
        al_hi = (mn_hi == -INFINITY) ? 1.f : ex2_approx(m_hi - mn_hi);
        const float mu_lo = (mn_lo == -INFINITY) ? 0.f : mn_lo, mu_hi = (mn_hi == -INFINITY) ? 0.f : mn_hi;
        m_lo = mn_lo;
        m_hi = mn_hi;
        float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            if (n >= nkt8) break;
            const float p0 = ex2_approx(x[n][0] - mu_lo), p1 = ex2_approx(x[n][1] - mu_lo);
            const float p2 = ex2_approx(x[n][2] - mu_hi), p3 = ex2_approx(x[n][3] - mu_hi);
            ps_lo += p0 + p1;
            ps_hi += p2 + p3;
            // C fragment of n-tile n -> A fragment of k16 step n / 2 (regs 0,1 or 2,3)
            pa[n >> 1][(n & 1) * 2] = pack2<BF16>(p0, p1);
            pa[n >> 1][(n & 1) * 2 + 1] = pack2<BF16>(p2, p3);
        }
        l_lo = l_lo * al_lo + ps_lo;
        l_hi = l_hi * al_hi + ps_hi;
    };

    auto pv = [&](int t) {
        const int st = t % kDecStages;
        const uint32_t vbase = smem_u32(smem + st * gm.stage_bytes) + half_bytes;
        for (int cc = 0; cc < my_chunks; ++cc) {
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                o_acc[cc][n][0] *= al_lo;
                o_acc[cc][n][1] *= al_lo;
                o_acc[cc][n][2] *= al_hi;
                o_acc[cc][n][3] *= al_hi;
            }
            if (!ok) continue;
            const uint32_t blk = vbase + (warp + 8 * cc) * KT * 128;
#pragma unroll
            for (int kp = 0; kp < 2; ++kp) {
                if (kp * 16 >= KT) break;
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    // keys 16 kp .. 16 kp + 15 (rows of V), head-dim units 2 np, 2 np + 1
                    uint32_t vb[4];
                    const int vrow = kp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int vunit = np * 2 + (lane >> 4);
                    ldsm_x4_trans(swz(blk, vrow, vunit), vb);
                    mma_bf16_16816(o_acc[cc][np * 2], pa[kp], vb[0], vb[1], BF16);
                    mma_bf16_16816(o_acc[cc][np * 2 + 1], pa[kp], vb[2], vb[3], BF16);
                }
            }
        }
        // K and V of this stage are read
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    };

    // the trip counts are the same in every compute warp, so all of them pass
    // the named barriers inside softmax() equally often
    if (n_tiles > 0) {
        scores(0);
        softmax(0);
    }
    for (int t = 0; t < n_tiles; ++t) {
        const bool more = t + 1 < n_tiles;
        if (more) scores(t + 1);
        pv(t);
        if (more) softmax(t + 1);
    }

    // ------------------------------------------------------------ partial outputs
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    const size_t rows_total = static_cast<size_t>(pb.B) * pb.Hq * pb.Nq;
    for (int hi = 0; hi < 2; ++hi) {
        const int r = hi ? r_hi : r_lo;
        if (r0 + r >= R) continue;
        const float l = hi ? l_hi : l_lo, m = hi ? m_hi : m_lo;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int g = (r0 + r) / pb.Nq, i = (r0 + r) % pb.Nq;
        const size_t row = (static_cast<size_t>(b) * pb.Hq + hk * G + g) * pb.Nq + i;  // LSE layout [B, Hq, Nq]
        float* dst = gm.o_part + (static_cast<size_t>(split) * rows_total + row) * pb.D;
        for (int cc = 0; cc < my_chunks; ++cc) {
            const int c0 = (warp + 8 * cc) * 64;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int col = c0 + n * 8 + cpair;
                if (col < pb.D) {
                    const float2 v = make_float2(o_acc[cc][n][hi * 2] * inv, o_acc[cc][n][hi * 2 + 1] * inv);
                    *reinterpret_cast<float2*>(dst + col) = v;
                }
            }
        }
        if (warp == 0 && (lane & 3) == 0)
            gm.lse_part[static_cast<size_t>(split) * rows_total + row] = l > 0.f ? (m + lg2_approx(l)) * kLn2 : -INFINITY;
    }
}

// One CTA per query row, two head-dim columns per thread: combine the
// splits' partial outputs and LSE (every thread reads the row's split LSEs,
// which the CTA shares through L1; the partial O rows are read coalesced).
template <bool BF16>
__global__ void __launch_bounds__(512) decode_combine_kernel(const FwdArgs a, const DecGeo gm)
{
    const Problem& pb = a.pb;
    const long rows_total = static_cast<long>(pb.B) * pb.Hq * pb.Nq;
    const long row = blockIdx.x;
    const int c = 2 * threadIdx.x;
    float mx = -INFINITY;
    for (int s = 0; s < gm.splits; ++s) mx = fmaxf(mx, gm.lse_part[static_cast<size_t>(s) * rows_total + row]);
    float wsum = 0.f, v0 = 0.f, v1 = 0.f;
    if (mx > -INFINITY)
        for (int s = 0; s < gm.splits; ++s) {
            const float l = gm.lse_part[static_cast<size_t>(s) * rows_total + row];
            if (l == -INFINITY) continue;
            const float w = __expf(l - mx);
            const float2 p = *reinterpret_cast<const float2*>(gm.o_part + (static_cast<size_t>(s) * rows_total + row) * pb.D + c);
            wsum += w;
            v0 = fmaf(w, p.x, v0);
            v1 = fmaf(w, p.y, v1);
        }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const long b = row / (static_cast<long>(pb.Hq) * pb.Nq), h = (row / pb.Nq) % pb.Hq, i = row % pb.Nq;
    uint16_t* out = reinterpret_cast<uint16_t*>(a.o) + b * pb.vo.sb + h * pb.vo.sh + i * pb.vo.sn;
    *reinterpret_cast<uint32_t*>(out + c) = pack2<BF16>(v0 * inv, v1 * inv);
    if (threadIdx.x == 0) a.lse[row] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}

}  // namespace

// Split plan. One CTA fits per SM (its registers and shared memory), so with
// U = B * Hkv units split s ways into splits of t key tiles the run takes
// ceil(U * s / SMs) waves of t tiles each, plus a fixed start-up per CTA
// (Q load, first loads in flight) worth about two tiles. Take the split count
// with the least modelled time (fewest splits among equals).
DecodePlan decode_plan(const Problem& pb)
{
    DecodePlan p{};
    p.chunks = (pb.D + 63) / 64;
    p.kt = p.chunks > 8 ? 16 : 32;
    const long long rb = (static_cast<long long>(pb.Hq / max(1, pb.Hkv)) * pb.Nq + kDecodeRows - 1) / kDecodeRows;
    p.rblocks = static_cast<int>(rb < 1 ? 1 : (rb > 0x7fffffffLL ? 0x7fffffffLL : rb));
    const long units = max(1L, static_cast<long>(pb.B) * pb.Hkv * p.rblocks);
    const int tiles = max(1, (pb.Nkv + p.kt - 1) / p.kt);
    const long sms = num_sms() > 0 ? num_sms() : 148;
    long best = -1;
    p.tiles_per = tiles;
    p.splits = 1;
    for (int s = 1; s <= min(tiles, kDecodeMaxSplits); ++s) {
        const int per = (tiles + s - 1) / s;
        const int used = (tiles + per - 1) / per;
        if (used != s) continue;  // same split as a smaller s
        const long cost = (units * used + sms - 1) / sms * (per + 2);
        if (best < 0 || cost < best) {
            best = cost;
            p.tiles_per = per;
            p.splits = used;
        }
    }
    const size_t rows_total = static_cast<size_t>(pb.B) * pb.Hq * pb.Nq;
    p.workspace_bytes = static_cast<size_t>(p.splits) * rows_total * (static_cast<size_t>(pb.D) + 1) * sizeof(float);
    return p;
}

namespace {

DecGeo plan(const Problem& pb, float* ws)
{
    const DecodePlan p = decode_plan(pb);
    DecGeo gm{};
    gm.chunks = p.chunks;
    gm.kt = p.kt;
    gm.stage_bytes = 2 * gm.kt * gm.chunks * 128;
    gm.tiles_per = p.tiles_per;
    gm.splits = p.splits;
    gm.rblocks = p.rblocks;
    const size_t rows_total = static_cast<size_t>(pb.B) * pb.Hq * pb.Nq;
    gm.o_part = ws;
    gm.lse_part = ws + static_cast<size_t>(gm.splits) * rows_total * pb.D;
    return gm;
}

template <bool BF16>
cudaError_t launch_variant(const FwdArgs& a, const DecGeo& gm, const CUtensorMap& tk, const CUtensorMap& tv,
                           cudaStream_t s)
{
    const int smem = kDecStages * gm.stage_bytes + kDecRedBytes;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid;
    if (!unit_grid(gm.splits, static_cast<long long>(a.pb.B) * a.pb.Hkv * gm.rblocks, &grid))
        return cudaErrorInvalidConfiguration;
    decode_kernel<BF16><<<grid, kDecThreads, smem, s>>>(tk, tv, a, gm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long rows = static_cast<long>(a.pb.B) * a.pb.Hq * a.pb.Nq;
    if (rows > 0x7fffffffL) return cudaErrorInvalidValue;
    decode_combine_kernel<BF16><<<static_cast<unsigned>(rows), a.pb.D / 2, 0, s>>>(a, gm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const FwdArgs& a, void* workspace, cudaStream_t s)
{
    const Problem& pb = a.pb;
    DecGeo gm = plan(pb, static_cast<float*>(workspace));
    CUtensorMap tk, tv;
    std::memset(&tk, 0, sizeof(tk));
    std::memset(&tv, 0, sizeof(tv));
    // with no keys the producer issues nothing and the maps are never read
    if (pb.Nkv > 0 && (!make_slab_map(&tk, a.k, pb, true, a.bf16, gm.kt, gm.chunks, pb.vk) ||
                       !make_slab_map(&tv, a.v, pb, true, a.bf16, gm.kt, gm.chunks, pb.vv)))
        return cudaErrorInvalidValue;
    return a.bf16 ? launch_variant<true>(a, gm, tk, tv, s) : launch_variant<false>(a, gm, tk, tv, s);
}

}  // namespace ffpa
