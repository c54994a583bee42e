// dQ and dV from the tiles the dK kernel stored: plain GEMMs for problems
// whose dS^T and P^T the dK kernel wrote to the backward workspace (FFPA
// docs, "CuTe-DSL Backend" page, "Blackwell status": the backward as a
// preprocess plus separate gradient launches; here the dQ and dV launches
// reuse the dK launch's tiles instead of recomputing S (and dP), which turns
// 3 + 2 GEMM units into 1 + 1).
//
// The dK kernel stores dS^T and P^T, each [B, Hq, Nkv, ldq] (keys x queries,
// queries contiguous; packed batches: [1, Hq, total_k + 256 B, ldq], sequence
// b's key rows from cu_k[b] + 256 b, its queries from column 0), tile by
// tile; masked entries are stored zeros, and under the bottom-right causal
// mask every tile that holds a legal entry is stored. A CTA pair owns 256 output rows (128 per CTA, in its TMEM lanes)
// and one slab of at most 512 head-dim columns (fp32 in TMEM; D > 512 takes
// two pairs, each reading the stored tiles); a ring of 4 stages feeds M=256,
// N=256 pair MMAs (the last one N=128 when the slab ends 64 or 128 columns
// past a multiple of 256), acc[:, 256 j ..] += A B_j:
//   dQ = scale dS K (rows = queries of one head; causal grids take the
//       longest tiles, the last ones, first). K runs over keys in blocks of
//       64, up to the last key any row of the pair may see.
//       A = dS for my 128 queries x 64 keys, read from dS^T as an MN-major
//       operand (two 64-query boxes of 64 key rows x 128 bytes);
//       B = K for 64 keys x my 128 columns of each 256-column half of D,
//       also MN-major (the forward's value-operand form).
//   dV = P^T dO (rows = keys of one KV head; the first tiles are the
//       longest). K runs over the query heads of the group and, per head,
//       over queries in blocks of 64 from the first that any row of the pair
//       may see.
//       A = P^T for my 128 keys x 64 queries, K-major (one box);
//       B = dO for 64 queries x my 128 columns of each half, MN-major.
// Warp 0 lanes 0 / 1 load A / B with TMA, warp 1 of the even rank issues the
// MMAs, warps 2..5 scale and store the output rows.
#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr int kQThreads = 192;
constexpr int kQStages = 4;

enum QSite : uint32_t { QS_PROD = 112, QS_RING, QS_ACC, QS_DRAIN };

struct __align__(1024) QStatic {
    uint64_t full[kQStages], empty[kQStages], acc;
    uint64_t ostage;  // every epilogue thread staged its output row
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(QStatic) == 1024, "static shared block must be exactly 1 KiB");

struct QGeo {
    int nj_max;       // pair MMAs (N = 256, the last one of a slab N = 128 if it is narrower) of the widest slab
    int stage_bytes;  // ring slot per CTA: A (16 KiB) + B (nj_max x 16 KiB)
    int n_rt;         // row tiles of 256 per (batch, head) in the grid (of the longest sequence)
    int n_bz;         // (batch, head) entries in the grid
    int ostore;       // the output map is valid: whole 128-row tiles leave through shared memory and TMA
};

template <bool BF16, bool DV>
__global__ void __launch_bounds__(kQThreads, 1)
    dsq_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
               const __grid_constant__ CUtensorMap tO, const DsqArgs a, const QGeo gm)
{
    const Problem& pb = a.pb;
    const int rank = static_cast<int>(cluster_ctarank());
    const int rh = rank & 1;
    const bool leader = rh == 0;
    const int G = pb.Hq / pb.Hkv;
    // dQ: (b, query head h); dV: (b, KV head hk), the group's query heads hk*G ..
    // units in linear pair order: row tile fastest, then (b, head)
    const long long unit = unit_id();
    if (unit >= static_cast<long long>(gm.n_rt) * gm.n_bz) return;  // past the last unit: uniform over the pair
    const int rtile = static_cast<int>(unit % gm.n_rt), bz = static_cast<int>(unit / gm.n_rt);
    // (b, head) over the kv groups [g0, g0 + ng) of the launch: dV takes their
    // kv heads, dQ their query heads; the tile buffer holds those query heads
    // only, the first at index 0
    const int ng = a.ng > 0 ? a.ng : pb.Hkv;
    const int hb = DV ? ng : ng * G;
    const int b = bz / hb, h = (DV ? a.g0 : a.g0 * G) + bz % hb, hk = DV ? h : h / G;
    const int th0 = a.g0 * G;  // query head of tile buffer head 0
    // the sequence: lengths, and (packed batches) its first query / key token
    // and the first row of its key rows in the tile buffers (one 256-row pad
    // per sequence, so that no row tile reaches the next sequence's rows)
    int lq = pb.Nq, lk = pb.Nkv, tq0 = 0, tk0 = 0, tr0 = 0, bco = b;
    if (pb.varlen) {
        if (!varlen_seq(pb, b, a.ctl.status, VS_GEMM, tq0, lq, tk0, lk)) return;  // uniform over the pair
        tr0 = tk0 + 256 * b;
        bco = 0;
    }
    const int off = lk - lq;  // causal: key j legal for query i iff j <= i + off
    const int n_rows = DV ? lk : lq;
    const int n_rt_seq = (n_rows + 255) / 256;
    if (rtile >= n_rt_seq) return;  // uniform over the pair, before any barrier
    // causal: the longest tiles first (dQ: the last query tiles, dV: the first key tiles)
    const int tile = (pb.causal && !DV) ? n_rt_seq - 1 - rtile : rtile;
    const int row0 = tile * 256;
    const int rc = row0 + 128 * rh;  // my first row (query for dQ, key for dV)
    // K blocks of 64 (both CTAs of the pair alike): dQ keys [0, key_end);
    // dV per query head: queries [64 qb_lo, lq)
    int kb_lo = 0, n_kb;
    if constexpr (DV) {
        const int i_lo = pb.causal ? max(0, row0 - off) : 0;
        kb_lo = i_lo / 64;
        n_kb = i_lo < lq ? (lq + 63) / 64 - kb_lo : 0;
    } else {
        const int key_end = pb.causal ? min(lk, row0 + 255 + off + 1) : lk;
        n_kb = key_end > 0 ? (key_end + 63) / 64 : 0;
    }
    const int n_it = DV ? G * n_kb : n_kb;  // K iterations
    // the pair's head-dim slab: columns [c0, c0 + w), w <= 512, as nj MMAs of N = 256;
    // the last one N = last_n, the rest of the slab rounded up to 128 (columns past
    // D are loaded as zeros and not stored)
    const int c0 = static_cast<int>(blockIdx.x >> 1) * 512;
    const int w = min(512, pb.D - c0);
    const int nj = (w + 255) / 256;
    const int last_n = (w - (nj - 1) * 256 + 127) / 128 * 128;
    const int tx_bytes = 16384 * (1 + nj);  // bytes one CTA loads per K block
    auto n_of = [&](int j) { return j == nj - 1 ? last_n : 256; };
    const int tcols = gm.nj_max * 256;

    __shared__ QStatic sh;
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {  // uniform over the cluster: report, do not run misaligned
        if (threadIdx.x == 0) atomicCAS(a.ctl.status, 0u, 5u | (0xffu << 8));
        return;
    }
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        mbar_init(&sh.acc, 1);
        mbar_init(&sh.ostage, 128);
        sh.abort_flag = 0;
        // the even rank's full barriers count both CTAs' bytes
        if (leader)
            for (int i = 0; i < kQStages; ++i) mbar_arrive_expect_tx(&sh.full[i], 2 * tx_bytes);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&sh.tmem_base, tcols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    volatile int* abort_flag = &sh.abort_flag;
    uint32_t* status = a.ctl.status;
    const uint64_t lim = a.ctl.limit_ns;
    const int lead_rank = rank & ~1;
    const uint16_t pair_mask = static_cast<uint16_t>(3u << lead_rank);

    if (warp == 0) {
        // ------------------------------------------------------ TMA producers
        const int lane = static_cast<int>(lane_id());
        if (lane < 2) {
            if (lane == 0) {
                prefetch_tmap(&tA);
                prefetch_tmap(&tB);
            }
            RingPos rp;
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const bool got = mbar_wait(&sh.empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, QS_PROD);
                if (!__all_sync(0x3u, got)) break;
                uint8_t* st = smem + rp.slot * gm.stage_bytes;
                const uint32_t fb = mapa_shared(smem_u32(&sh.full[rp.slot]), lead_rank);
                if constexpr (DV) {
                    const int hq = hk * G + it / n_kb;    // query head of the group
                    const int i0 = (kb_lo + it % n_kb) * 64;  // first query of the block
                    if (lane == 0) {
                        // A: P^T rows = my 128 keys, queries [i0, +64)
                        tma_load_4d_pair(st, &tA, fb, i0, tr0 + rc, hq - th0, bco);
                    } else {
                        // B: dO rows = queries [i0, +64), my half of each MMA's N columns
                        // (a 128-column box; an N = 128 MMA reads its first 64)
                        for (int j = 0; j < nj; ++j)
                            tma_load_5d_pair(st + 16384 * (1 + j), &tB, fb, 0, tq0 + i0,
                                             (c0 + j * 256 + rh * n_of(j) / 2) / 64, hq, bco);
                    }
                } else {
                    const int kb = it;
                    if (lane == 0) {
                        // A: dS^T rows = keys [64 kb, +64), my 128 queries as two 64-query boxes
                        tma_load_4d_pair(st, &tA, fb, rc, tr0 + kb * 64, h - th0, bco);
                        tma_load_4d_pair(st + 8192, &tA, fb, rc + 64, tr0 + kb * 64, h - th0, bco);
                    } else {
                        // B: K rows = keys [64 kb, +64), my half of each MMA's N columns
                        for (int j = 0; j < nj; ++j)
                            tma_load_5d_pair(st + 16384 * (1 + j), &tB, fb, 0, tk0 + kb * 64,
                                             (c0 + j * 256 + rh * n_of(j) / 2) / 64, hk, bco);
                    }
                }
                rp.advance(kQStages);
                ++issued;
            }
            // no loads in flight when the CTA leaves
            if (lane == 0) {
                RingPos dp = rp;
                for (int i = 0; i < min(issued, kQStages); ++i) {
                    dp.retreat(kQStages);
                    int dummy = 0;
                    if (!mbar_wait(&sh.empty[dp.slot], dp.phase, &dummy, status, lim, QS_DRAIN, false)) break;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer (pair)
        if (leader && elect_one()) {
            // A: MN-major dS (dQ) or K-major P^T (dV); B: MN-major
            const uint32_t idesc = idesc_f16(256, 256, BF16, !DV, true);
            const uint32_t idesc_n128 = idesc_f16(256, 128, BF16, !DV, true);
            RingPos rp;
            for (int it = 0; it < n_it; ++it) {
                if (!mbar_wait_cluster(&sh.full[rp.slot], rp.phase, abort_flag, status, lim, QS_RING)) break;
                mbar_arrive_expect_tx(&sh.full[rp.slot], 2 * tx_bytes);  // arm the slot's next fill
                tc_fence_after();
                const uint8_t* st = smem + rp.slot * gm.stage_bytes;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    // 16 K values per MMA. MN-major operands: 16 rows x 128 bytes, with
                    // 64-element chunks along M (A) and N (B) 64 rows x 128 bytes apart;
                    // K-major A (dV): 32 bytes into each of the 128 rows of the box
                    const uint64_t ad = DV ? sdesc_sw128(smem_u32(st + kk * 32), 16, 1024)
                                           : sdesc_sw128(smem_u32(st + kk * 2048), 8192, 1024);
                    for (int j = 0; j < nj; ++j) {
                        const uint64_t bd = sdesc_sw128(smem_u32(st + 16384 * (1 + j) + kk * 2048), 8192, 1024);
                        umma_f16_pair(tmem + j * 256, ad, bd, n_of(j) == 256 ? idesc : idesc_n128, (it | kk) != 0);
                    }
                }
                umma_commit_pair_multicast(&sh.empty[rp.slot], pair_mask);
                rp.advance(kQStages);
            }
            umma_commit_pair_multicast(&sh.acc, pair_mask);
        }
    } else {
        // ------------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;
        const int r = quarter * 32 + static_cast<int>(lane_id());
        const int q = rc + r;  // my output row
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&sh.acc, 0, abort_flag, status, lim, QS_ACC));
        tc_fence_after();
        if (ok) {
            // no K block for any row of the pair: zero rows (the accumulator was never written)
            const float mul = n_it > 0 ? (DV ? 1.f : pb.scale) : 0.f;
            const View& vo = DV ? pb.vdv : pb.vdq;
            const size_t tok = static_cast<size_t>((DV ? tk0 : tq0) + q);  // row (packed: token)
            uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) + static_cast<size_t>(bco) * vo.sb +
                            static_cast<size_t>(h) * vo.sh + tok * vo.sn + c0;
            // Whole 128-row tiles leave through the idle ring and TMA stores of 128
            // rows x 128 columns (columns past D fall outside the map): one row per
            // thread would make every warp store touch 32 rows.
            const bool via_tma = gm.ostore && n_it > 0 && rc + 128 <= n_rows;
            if (via_tma) {
                for (int cc = 0; cc < w; cc += 64) {
                    uint32_t va[32], vb[32];
                    tmem_ld32(tmem + lane_off + cc, va);
                    tmem_ld32(tmem + lane_off + cc + 32, vb);
                    tmem_ld_wait(va, vb);
                    // box cc / 128 holds 64-column chunks 2 q, 2 q + 1 of the slab, 16 KiB each
                    uint8_t* blk = smem + (cc >> 7) * 32768 + ((cc >> 6) & 1) * 16384;
#pragma unroll
                    for (int p2 = 0; p2 < 2; ++p2) {
                        const uint32_t (&v)[32] = p2 ? vb : va;
                        uint32_t wp[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            wp[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<uint4*>(blk + sw128_offset(r, 4 * p2 + e)) =
                                make_uint4(wp[4 * e], wp[4 * e + 1], wp[4 * e + 2], wp[4 * e + 3]);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&sh.ostage);
                if (threadIdx.x == 64) {
                    if (mbar_wait(&sh.ostage, 0, abort_flag, status, lim, QS_ACC)) {
                        const int row_first = (DV ? tk0 : tq0) + rc;
                        for (int qb = 0; qb < (w + 127) / 128; ++qb)
                            tma_store_5d(&tO, smem + qb * 32768, 0, row_first, c0 / 64 + 2 * qb, h, bco);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                }
            }
            for (int cc = 0; cc < (via_tma ? 0 : w); cc += 32) {
                uint32_t v[32];
                if (n_it > 0) {
                    tmem_ld32(tmem + lane_off + cc, v);
                    tmem_ld_wait(v);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
                if (q < n_rows) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
                    uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
                    for (int e = 0; e < 4; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
            }
        }
    }

    // -------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, tcols);
    }
}

}  // namespace

bool dsq_supported(const Problem& pb)
{
    // whole 64-column chunks (the 5-D operand maps), at most two 512-column slabs
    if (pb.varlen) return pb.D % 64 == 0 && pb.D <= 1024 && pb.total_q > 0 && pb.total_k > 0 && pb.Nq > 0;
    return pb.D % 64 == 0 && pb.D <= 1024 && pb.Nq > 0 && pb.Nkv > 0;
}

// Tile buffer rows per (batch, head): the keys (dense), or every sequence's
// keys plus a 256-row pad each (packed: sequence b starts at row cu_k[b] + 256 b)
static size_t tile_rows(const Problem& pb)
{
    return pb.varlen ? static_cast<size_t>(pb.total_k) + 256 * static_cast<size_t>(pb.B) : static_cast<size_t>(pb.Nkv);
}

size_t dsq_ds_bytes(const Problem& pb)
{
    const size_t ldq = (static_cast<size_t>(pb.Nq) + 7) & ~static_cast<size_t>(7);
    return static_cast<size_t>(pb.varlen ? 1 : pb.B) * pb.Hq * tile_rows(pb) * ldq * 2;
}

size_t dsq_group_bytes(const Problem& pb)
{
    return pb.Hkv > 0 ? dsq_ds_bytes(pb) / pb.Hkv : 0;  // G query heads of every batch entry
}

bool make_ds_map(CUtensorMap* m, const void* ds, const Problem& pb, bool bf16, int box_rows, int heads)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    // (packed batches: Nq is the longest sequence, and one batch of tile_rows rows)
    const cuuint64_t ldq = (static_cast<cuuint64_t>(pb.Nq) + 7) & ~static_cast<cuuint64_t>(7);
    const cuuint64_t rows = tile_rows(pb);
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(pb.Nq), rows, static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(pb.varlen ? 1 : pb.B)};
    const cuuint64_t strides[3] = {ldq * 2, rows * ldq * 2, static_cast<cuuint64_t>(heads) * rows * ldq * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(ds),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_dsq(const DsqArgs& a, cudaStream_t s)
{
    const Problem& pb = a.pb;
    if (!dsq_supported(pb)) return cudaErrorInvalidConfiguration;
    CUtensorMap tA, tB;
    // dQ: dS^T as 64 queries x 64 key rows boxes, K rows; dV: P^T as 64 queries x
    // 128 key rows boxes, dO rows (the query side)
    const int G = pb.Hq / pb.Hkv;
    const int ng = a.ng > 0 ? a.ng : pb.Hkv;  // kv groups of this launch (their query heads in the tiles)
    if (a.g0 < 0 || a.g0 + ng > pb.Hkv) return cudaErrorInvalidValue;
    CUtensorMap tO;
    const bool okm = a.dv ? make_ds_map(&tA, a.tiles, pb, a.bf16, 128, ng * G) &&
                                make_slab_map(&tB, a.rhs, pb, false, a.bf16, 64, 2, pb.vdo)
                          : make_ds_map(&tA, a.tiles, pb, a.bf16, 64, ng * G) &&
                                make_slab_map(&tB, a.rhs, pb, true, a.bf16, 64, 2, pb.vk);
    if (!okm) return cudaErrorInvalidValue;
    QGeo gm{};
    // the output as 128-row x 2-chunk boxes (a view the map cannot describe keeps the row stores)
    gm.ostore = make_slab_map(&tO, a.out, pb, a.dv != 0, a.bf16, 128, 2, a.dv ? pb.vdv : pb.vdq) ? 1 : 0;
    if (!gm.ostore) tO = tA;
    gm.nj_max = (min(pb.D, 512) + 255) / 256;
    gm.stage_bytes = 16384 * (1 + gm.nj_max);
    const int n_slab = (pb.D + 511) / 512;
    const int smem = kQStages * gm.stage_bytes;
    gm.n_rt = a.dv ? (pb.Nkv + 255) / 256 : (pb.Nq + 255) / 256;
    gm.n_bz = a.dv ? pb.B * ng : pb.B * ng * G;
    if (gm.n_rt == 0 || gm.n_bz == 0) return cudaSuccess;
    dim3 grid;
    if (!unit_grid(2 * n_slab, static_cast<long long>(gm.n_rt) * gm.n_bz, &grid)) return cudaErrorInvalidConfiguration;
    auto kern = a.dv ? (a.bf16 ? dsq_kernel<true, true> : dsq_kernel<false, true>)
                     : (a.bf16 ? dsq_kernel<true, false> : dsq_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kQThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tA, tB, tO, a, gm);
}

}  // namespace ffpa
