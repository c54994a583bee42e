// CTA-pair exchange kernels: the forward and the three backward GEMM kernels
// (dV, dK, dQ) of exact attention at large head dim, with every tensor-core
// product issued as a 2-SM (cta_group::2) MMA of M = 256 rows.
//
// A cluster holds C pairs of CTAs (2C CTAs; ranks 2c and 2c+1 form pair c,
// the even rank issues the pair's MMAs). The cluster owns one 256-row tile of
// "rows" (queries for the forward and dQ, keys for dV and dK); CTA 2c+h holds
// rows [128h, 128h + 128) of it in its TMEM lanes. The cluster walks over
// 128-wide tiles of "columns" (keys, resp. queries) in super-steps of C
// tiles. In super-step s, pair c
//   1. computes the score tile(s) of column tile C*s + c for all 256 rows with
//      M=256, N=128 pair MMAs over the full head dim: X = S (and Y = dP for
//      dQ / dK); each CTA supplies its own 128 rows of the row operand and
//      64 of the 128 column-tile rows,
//   2. turns them, row by row, into one 16-bit operand tile Z (P, P^T, dS or
//      dS^T; the forward first agrees on a per-row softmax reference with the
//      CTAs of the other pairs that hold the same rows),
//   3. writes its 128-row half of Z into its own shared memory and copies it
//      into the CTA of every other pair that holds the same rows, and
//   4. accumulates its own head-dim slab (<= 256 columns) of the output over
//      all C tiles of the super-step, acc += Z_{c'} W_{tile C*s+c'}[:, slab],
//      as M=256, N=slab pair MMAs (each CTA supplies half of the slab's
//      columns of W).
// Each score product is therefore computed once, the fp32 accumulator of a
// 256-row tile is split over C pairs by head-dim slabs, and each pair MMA
// keeps both SMs' tensor cores busy on one instruction stream.
//
// The pages this implements: FFPA docs, "CuTe-DSL Backend" page, "Hard
// constraints" (bottom-right causal, GQA/MQA broadcast, empty rows give
// O = 0, LSE = -inf and zero gradients), "Varlen (packed THD) API" (packed
// layout, LSE [H, T]), "Blackwell status" (preprocess plus separate
// gradient launches, split because one SM cannot hold a whole dK/dV tile).
//
// Warp roles in every CTA: warp 0 TMA producer, warp 1 MMA issuer (even rank)
// or barrier forwarder (odd rank), warps 2..9 elementwise (two threads per
// TMEM row) and epilogue.
#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 320;
constexpr int kStages = 16;      // upper bound of the TMA ring depth
constexpr int kMaxC = 4;         // pairs per cluster (D <= 1024 in 256-column slabs; <= 8 CTAs)
constexpr int kSlot = 16384;     // bytes of one ring slot in each CTA
constexpr float kTau = 8.0f;     // forward: rescale O only when the row max grows by more than 2^8
constexpr float kLn2 = 0.693147180559945309f;

enum Site : uint32_t {
    PS_PROD = 64, PS_A1, PS_XFREE, PS_RING, PS_ZFULL, PS_ZPEER, PS_ZPAIR, PS_XFULL, PS_RMAX, PS_ACC, PS_SLOT,
    PS_STAT, PS_LSUM, PS_EPI, PS_DRAIN, PS_FWDR
};

struct PGeo {
    int C;       // pairs per cluster (= head-dim slabs of <= 256 columns)
    int stages;  // TMA ring depth
    int res;     // leading 64-wide chunks of the first row operand kept resident in shared memory
};

template <int OP>
struct Traits {
    static constexpr bool kTwo = (OP == XOP_DQ || OP == XOP_DK);     // X and Y score tiles
    static constexpr bool kRowsQ = (OP == XOP_FWD || OP == XOP_DQ);  // rows are queries
    static constexpr bool kXdb = !kTwo;                              // X double-buffered
};

// Barriers and flags: one static block of exactly 1 KiB so that the dynamic
// shared memory after it starts 1024-byte aligned (checked at run time).
struct __align__(1024) StaticSmem {
    uint64_t full[kStages], empty[kStages];
    uint64_t a1, x_full[2], x_free[2], z_full, zpair, acc;
    uint64_t zpeer[kMaxC], slot_free[kMaxC], stat[2], rmax[2], lsum, drain, half;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(StaticSmem) == 1024, "static shared block must be exactly 1 KiB");

// Bytes of the per-kernel statistics area (rounded to 1 KiB):
//   forward: rmax[2][C-1][128] and lsum[C-1][128] (values of the other pairs)
//   dV / dK: lse2[2][128] and delta[2][128] (column statistics, double-buffered)
__host__ __device__ inline int pair_stats_bytes(int op, int C)
{
    int b = 0;
    if (op == XOP_FWD) b = 3 * (C > 1 ? C - 1 : 0) * 128 * 4;
    else if (op == XOP_DV || op == XOP_DK) b = 4 * 128 * 4;
    return (b + 1023) & ~1023;
}

template <int OP, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    pair_kernel(const __grid_constant__ CUtensorMap tA1, const __grid_constant__ CUtensorMap tA2,
                const __grid_constant__ CUtensorMap tB1, const __grid_constant__ CUtensorMap tB2,
                const __grid_constant__ CUtensorMap tW, const XArgs a, const PGeo gm)
{
    using T = Traits<OP>;
    const Problem& pb = a.pb;
    const int C = gm.C;
    const int rank = static_cast<int>(cluster_ctarank());
    const int c = rank >> 1;      // pair = head-dim slab
    const int rh = rank & 1;      // row half of the 256-row tile
    const bool leader = rh == 0;  // issues the pair's MMAs
    const int G = pb.Hq / pb.Hkv;

    // ------------------------------------------------------------ work unit
    const int n_rt = gridDim.y;  // 256-row tiles
    const int bz = blockIdx.z;
    int b, h = 0, hk;
    if (T::kRowsQ) {
        b = bz / pb.Hq;
        h = bz % pb.Hq;
        hk = h / G;
    } else {
        b = bz / pb.Hkv;
        hk = bz % pb.Hkv;
    }
    int lq, lk, tq0 = 0, tk0 = 0;
    if constexpr (VARLEN) {
        tq0 = pb.cu_q[b];
        lq = pb.cu_q[b + 1] - tq0;
        tk0 = pb.cu_k[b];
        lk = pb.cu_k[b + 1] - tk0;
    } else {
        lq = pb.Nq;
        lk = pb.Nkv;
    }
    const int off = lk - lq;  // causal: key j legal for query i iff j <= i + off
    const int rt = (T::kRowsQ && pb.causal) ? (n_rt - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
    const int R0 = rt * 256;            // first row of the cluster's tile
    const int r0 = R0 + 128 * rh;       // first row of this CTA
    const int row_len = T::kRowsQ ? lq : lk;
    if (R0 >= row_len) return;  // uniform over the cluster, before any cluster barrier

    // Column tiles of the unit, for all 256 rows (both CTAs of a pair run the
    // same MMAs; rows that a tile does not reach are masked element-wise).
    int n_ct;
    int m_start = 0, n_mt = 0;
    if (T::kRowsQ) {
        n_ct = (lk + 127) / 128;
        if (pb.causal) {
            const int kmax = min(R0 + 255, lq - 1) + off;
            n_ct = kmax < 0 ? 0 : min(n_ct, kmax / 128 + 1);
        }
    } else {
        if (pb.causal) m_start = max(0, R0 - off) / 128;
        n_mt = max(0, (lq + 127) / 128 - m_start);
        n_ct = G * n_mt;
    }
    const int n_steps = (n_ct + C - 1) / C;

    const int nd = pb.D / 64;          // 64-wide head-dim chunks
    const int nb2 = (nd + 1) / 2;      // chunk pairs (one column-operand box each)
    const int d0 = c * 256;            // first column of my pair's slab
    const int d_pad = (pb.D + 127) & ~127;
    const int sw = min(256, d_pad - d0);  // slab width: 256 or 128 (N of the value MMA)
    // first 64-wide chunk of my half of the slab's W columns; clamped so that a
    // box never starts past the head dim (columns past D are computed, never stored)
    const int w_chunk = min(d0 / 64 + rh * (sw / 128), nd - 1);

    // ------------------------------------------------------------ shared memory
    __shared__ StaticSmem sh;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sA1 = smem;                     // resident row-operand chunks: res x 16 KiB
    uint8_t* sZ = sA1 + gm.res * kSlot;      // C-1 slots of the other pairs + own slot, 32 KiB each
    uint8_t* sZown = sZ + (C - 1) * 32768;
    float* stats = reinterpret_cast<float*>(sZ + C * 32768);
    uint8_t* sRing = reinterpret_cast<uint8_t*>(stats) + pair_stats_bytes(OP, C);
    if (smem_u32(smem) & 1023u) {  // uniform over the cluster: report, do not run misaligned
        if (threadIdx.x == 0) atomicCAS(a.ctl.status, 0u, 5u | (0xffu << 8));
        return;
    }

    const int warp = threadIdx.x / 32;
    const int zpair_count = 8 + (C > 1 ? 1 : 0);  // follower: 8 elementwise warps + forwarder
    if (threadIdx.x == 0) {
        for (int i = 0; i < gm.stages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        mbar_init(&sh.a1, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.x_full[i], 1);
            mbar_init(&sh.x_free[i], 16);  // 8 elementwise warps of each CTA of the pair
            mbar_init(&sh.stat[i], 256);
            mbar_init(&sh.rmax[i], 1);
        }
        mbar_init(&sh.z_full, 256);
        mbar_init(&sh.zpair, zpair_count);
        mbar_init(&sh.half, 256);
        mbar_init(&sh.acc, 1);
        for (int i = 0; i < kMaxC; ++i) {
            mbar_init(&sh.zpeer[i], 1);
            mbar_init(&sh.slot_free[i], 1);
        }
        mbar_init(&sh.lsum, 1);
        mbar_init(&sh.drain, 1);
        sh.abort_flag = 0;
        // Byte-counting barriers are armed by their receiver before any writer
        // can deliver the phase they guard: here the first phase (the first two
        // for the double-buffered row maxima), later right after each completed
        // wait. The ring's full barriers count the bytes of both CTAs of the pair
        // and live in the even rank.
        if (leader) {
            for (int i = 0; i < gm.stages; ++i) mbar_arrive_expect_tx(&sh.full[i], 2 * kSlot);
            if (gm.res > 0 && n_steps > 0) mbar_arrive_expect_tx(&sh.a1, 2 * gm.res * kSlot);
        }
        if (C > 1) {
            for (int i = 0; i < C - 1; ++i) mbar_arrive_expect_tx(&sh.zpeer[i], 32768);
            if (OP == XOP_FWD) {
                mbar_arrive_expect_tx(&sh.rmax[0], 512 * (C - 1));
                mbar_arrive_expect_tx(&sh.rmax[1], 512 * (C - 1));
                mbar_arrive_expect_tx(&sh.lsum, 512 * (C - 1));
            }
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&sh.tmem_base, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // every CTA's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const uint32_t t_acc = tmem;        // [0, 256): accumulator slab (128 lanes = my rows)
    const uint32_t t_x0 = tmem + 256;   // X buffers (and Y for the two-product kernels)
    volatile int* abort_flag = &sh.abort_flag;
    uint32_t* status = a.ctl.status;
    const uint64_t lim = a.ctl.limit_ns;
    const int lead_rank = rank & ~1;
    const uint16_t pair_mask = static_cast<uint16_t>(3u << lead_rank);

    // Pairs: slot index of writer pair w inside consumer pair p's slot array;
    // the CTA of pair p that holds my rows has rank 2p + rh.
    auto slot_of = [&](int writer, int consumer) { return writer < consumer ? writer : writer - 1; };
    auto xrank = [&](int p) { return 2 * p + rh; };

    // Column tile t -> (head, first row) on the column side; t past the end is
    // clamped for loading (its results are masked to zero).
    auto col_head = [&](int t) { return T::kRowsQ ? hk : hk * G + min(t, n_ct - 1) / max(n_mt, 1); };
    auto col_row0 = [&](int t) {
        const int tc = min(t, n_ct - 1);
        return T::kRowsQ ? tc * 128 : (m_start + tc % max(n_mt, 1)) * 128;
    };
    // TMA coordinates. Dense maps: (d, row, b*H + head) / (64, row, chunk, b*H + head);
    // packed maps: (d, head, token) / (64, token, chunk, head).
    auto q_c1 = [&](int head, int row) { return VARLEN ? head : row; };
    auto q_c2 = [&](int head, int row) { return VARLEN ? tq0 + row : b * pb.Hq + head; };
    auto k_c1 = [&](int head, int row) { return VARLEN ? head : row; };
    auto k_c2 = [&](int head, int row) { return VARLEN ? tk0 + row : b * pb.Hkv + head; };
    auto row_c1 = [&](int row) { return T::kRowsQ ? q_c1(h, row) : k_c1(hk, row); };
    auto row_c2 = [&](int row) { return T::kRowsQ ? q_c2(h, row) : k_c2(hk, row); };
    // 4-D slab boxes on the column side: (row coordinate, head coordinate)
    auto col_slab_row = [&](int head, int row) {
        return VARLEN ? (T::kRowsQ ? tk0 + row : tq0 + row) : row;
    };
    auto col_slab_head = [&](int head) {
        return VARLEN ? head : (T::kRowsQ ? b * pb.Hkv + head : b * pb.Hq + head);
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // Both CTAs of the pair load the same sequence of slots (each its own
        // part of every operand); every load completes on the even rank's
        // full barrier, which its MMA thread arms with both CTAs' bytes.
        if (elect_one()) {
            prefetch_tmap(&tA1);
            prefetch_tmap(&tB1);
            prefetch_tmap(&tW);
            if (T::kTwo) {
                prefetch_tmap(&tA2);
                prefetch_tmap(&tB2);
            }
            RingPos rp;
            int issued = 0;
            bool ok = true;
            auto slot_wait = [&]() -> bool {
                return mbar_wait(&sh.empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, PS_PROD);
            };
            auto lead_full = [&](int slot) { return mapa_shared(smem_u32(&sh.full[slot]), lead_rank); };
            auto put_row = [&](const CUtensorMap* m, int chunk) -> bool {
                if (!slot_wait()) return false;
                tma_load_3d_pair(sRing + rp.slot * kSlot, m, lead_full(rp.slot), chunk * 64, row_c1(r0), row_c2(r0));
                rp.advance(gm.stages);
                ++issued;
                return true;
            };
            auto put_slab = [&](const CUtensorMap* m, int chunk, int head, int row) -> bool {
                if (!slot_wait()) return false;
                tma_load_4d_pair(sRing + rp.slot * kSlot, m, lead_full(rp.slot), 0, col_slab_row(head, row), chunk,
                                 col_slab_head(head));
                rp.advance(gm.stages);
                ++issued;
                return true;
            };
            if (gm.res > 0 && n_steps > 0) {
                const uint32_t a1 = mapa_shared(smem_u32(&sh.a1), lead_rank);
                for (int d = 0; d < gm.res; ++d)
                    tma_load_3d_pair(sA1 + d * kSlot, &tA1, a1, d * 64, row_c1(r0), row_c2(r0));
            }
            // score operands of step s: per product, per chunk pair j: A(2j), B(j), A(2j+1)
            auto load_score = [&](int s) -> bool {
                const int t = s * C + c;
                const int hh = col_head(t), cr = col_row0(t) + 64 * rh;
                for (int prod = 0; prod < (T::kTwo ? 2 : 1); ++prod) {
                    const CUtensorMap* mA = prod ? &tA2 : &tA1;
                    const CUtensorMap* mB = prod ? &tB2 : &tB1;
                    for (int j = 0; j < nb2; ++j) {
                        if (!(prod == 0 && 2 * j < gm.res) && !put_row(mA, 2 * j)) return false;
                        if (!put_slab(mB, 2 * j, hh, cr)) return false;
                        if (2 * j + 1 < nd && !(prod == 0 && 2 * j + 1 < gm.res) && !put_row(mA, 2 * j + 1))
                            return false;
                    }
                }
                return true;
            };
            // value operand of step s: per column tile, two boxes of 64 keys x my
            // two 64-wide chunks of the slab
            auto load_value = [&](int s) -> bool {
                for (int cc = 0; cc < C; ++cc) {
                    const int t = s * C + cc;
                    const int hh = col_head(t), cr = col_row0(t);
                    for (int i = 0; i < 2; ++i)
                        if (!put_slab(&tW, w_chunk, hh, cr + 64 * i)) return false;
                }
                return true;
            };
            if (n_steps > 0) ok = load_score(0);
            for (int s = 0; ok && s < n_steps; ++s) {
                if (s + 1 < n_steps) ok = load_score(s + 1);
                if (ok) ok = load_value(s);
            }
            // No CTA leaves with loads in flight: the MMA thread releases a slot only
            // after its data landed in both CTAs and was consumed.
            const int last = min(issued, gm.stages);
            RingPos dp = rp;
            for (int i = 0; i < last; ++i) {
                dp.retreat(gm.stages);
                int dummy = 0;
                if (!mbar_wait(&sh.empty[dp.slot], dp.phase, &dummy, status, lim, PS_DRAIN, false)) break;
            }
        }
    } else if (warp == 1) {
        if (leader) {
            // -------------------------------------------------- MMA issuer (pair)
            if (elect_one()) {
                const uint32_t idesc_s = idesc_f16(256, 128, BF16, false, false);
                const uint32_t idesc_v = idesc_f16(256, sw, BF16, false, true);
                uint16_t others = 0;  // every CTA outside my pair
                for (int p = 0; p < 2 * C; ++p)
                    if ((p >> 1) != c) others |= static_cast<uint16_t>(1u << p);
                RingPos rp;
                bool ok = true;
                if (gm.res > 0 && n_steps > 0) {
                    ok = mbar_wait_cluster(&sh.a1, 0, abort_flag, status, lim, PS_A1);
                    tc_fence_after();
                }
                auto take = [&]() -> const uint8_t* {
                    if (!mbar_wait_cluster(&sh.full[rp.slot], rp.phase, abort_flag, status, lim, PS_RING)) return nullptr;
                    // arm the slot's next phase before releasing it to the producers
                    mbar_arrive_expect_tx(&sh.full[rp.slot], 2 * kSlot);
                    tc_fence_after();
                    return sRing + rp.slot * kSlot;
                };
                auto give = [&](int slot) { umma_commit_pair_multicast(&sh.empty[slot], pair_mask); };
                auto issue_score = [&](int s) -> bool {
                    const int sb = T::kXdb ? (s & 1) : 0;
                    // XDB: buffer sb last held X of step s-2 (read by then);
                    // two-product kernels: X/Y of step s-1 released by the elementwise warps
                    if (T::kXdb ? s >= 2 : s >= 1) {
                        const uint32_t par = T::kXdb ? (((s - 2) >> 1) & 1) : ((s - 1) & 1);
                        if (!mbar_wait_cluster(&sh.x_free[sb], par, abort_flag, status, lim, PS_XFREE)) return false;
                        tc_fence_after();
                    }
                    for (int prod = 0; prod < (T::kTwo ? 2 : 1); ++prod) {
                        const uint32_t dst = t_x0 + (T::kXdb ? sb * 128 : prod * 128);
                        for (int j = 0; j < nb2; ++j) {
                            const uint8_t* B = nullptr;
                            int b_slot = -1;
                            for (int u = 0; u < 2; ++u) {
                                const int d = 2 * j + u;
                                if (d >= nd) break;
                                const uint8_t* A;
                                int a_slot = -1;
                                if (prod == 0 && d < gm.res) {
                                    A = sA1 + d * kSlot;
                                } else {
                                    A = take();
                                    if (!A) return false;
                                    a_slot = rp.slot;
                                    rp.advance(gm.stages);
                                }
                                if (u == 0) {
                                    B = take();
                                    if (!B) return false;
                                    b_slot = rp.slot;
                                    rp.advance(gm.stages);
                                }
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    umma_f16_pair(dst, sdesc_sw128(smem_u32(A + kk * 32), 16, 1024),
                                                  sdesc_sw128(smem_u32(B + u * 8192 + kk * 32), 16, 1024), idesc_s,
                                                  (d | kk) != 0);
                                if (a_slot >= 0) give(a_slot);
                            }
                            give(b_slot);
                        }
                    }
                    umma_commit_pair_multicast(&sh.x_full[sb], pair_mask);
                    return true;
                };
                auto issue_value = [&](int s) -> bool {
                    if (!mbar_wait(&sh.z_full, s & 1, abort_flag, status, lim, PS_ZFULL)) return false;
                    for (int p = 0; p < C; ++p)
                        if (p != c) {
                            if (!mbar_wait_cluster(&sh.zpeer[slot_of(p, c)], s & 1, abort_flag, status, lim, PS_ZPEER))
                                return false;
                            // arm the next phase before this step's slot_free lets the writer in
                            mbar_arrive_expect_tx(&sh.zpeer[slot_of(p, c)], 32768);
                        }
                    if (!mbar_wait_cluster(&sh.zpair, s & 1, abort_flag, status, lim, PS_ZPAIR)) return false;
                    tc_fence_after();
                    for (int cc = 0; cc < C; ++cc) {
                        const uint8_t* zs = (cc == c) ? sZown : sZ + slot_of(cc, c) * 32768;
                        for (int i = 0; i < 2; ++i) {
                            const uint8_t* W = take();
                            if (!W) return false;
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                // keys 64 i + 16 t of the tile: Z chunk i, W rows 16 t (MN-major,
                                // 64-column blocks 64 keys x 128 bytes apart)
                                const uint64_t bd = sdesc_sw128(smem_u32(W + t * 2048), 64 * 128, 1024);
                                const uint32_t acc = (s | cc | i | t) != 0;
                                umma_f16_pair(t_acc, sdesc_sw128(smem_u32(zs + i * 16384 + t * 32), 16, 1024), bd,
                                              idesc_v, acc);
                            }
                            give(rp.slot);
                            rp.advance(gm.stages);
                        }
                    }
                    umma_commit_pair_multicast(&sh.acc, pair_mask);
                    if (C > 1) umma_commit_pair_multicast(&sh.slot_free[c], others);
                    return true;
                };
                if (ok && n_steps > 0) ok = issue_score(0);
                for (int s = 0; ok && s < n_steps; ++s) {
                    if (s + 1 < n_steps) ok = issue_score(s + 1);
                    if (ok) ok = issue_value(s);
                }
                umma_commit_pair_multicast(&sh.drain, static_cast<uint16_t>(1u << rank));
                int dummy = 0;
                mbar_wait(&sh.drain, 0, &dummy, status, lim, PS_DRAIN, false);
            }
        } else if (C > 1) {
            // -------------------------------------------------- forwarder (odd rank)
            // The other pairs' Z tiles land in this CTA's shared memory and complete
            // on this CTA's barriers; the MMA thread of the even rank learns of them
            // through one arrival per step.
            if (elect_one()) {
                const uint32_t lead_zpair = mapa_shared(smem_u32(&sh.zpair), lead_rank);
                for (int s = 0; s < n_steps; ++s) {
                    bool ok = true;
                    for (int p = 0; p < C && ok; ++p)
                        if (p != c) {
                            ok = mbar_wait_cluster(&sh.zpeer[slot_of(p, c)], s & 1, abort_flag, status, lim, PS_FWDR);
                            if (ok) mbar_arrive_expect_tx(&sh.zpeer[slot_of(p, c)], 32768);
                        }
                    if (!ok) break;
                    mbar_arrive_remote(lead_zpair);
                }
            }
        }
    } else {
        // ------------------------------------------------------ elementwise
        // Two threads per tile row: warps 2..5 take columns [0, 64), warps 6..9
        // columns [64, 128) of the same TMEM lanes.
        const int quarter = warp & 3;
        const int lane = static_cast<int>(lane_id());
        const int r = quarter * 32 + lane;         // tile row = TMEM lane
        const int ew = threadIdx.x - 64;           // 0..255
        const int half = ew >> 7;
        const int col0 = half * 64;                // my columns [col0, col0 + 64)
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float c2 = pb.scale_log2;
        const int row = r0 + r;  // query (rows = queries) or key (rows = keys)
        // rows = queries: legal keys [0, key_end); rows = keys: legal queries [i_min, lq)
        const int key_end = pb.causal ? min(lk, row + off + 1) : lk;
        const int i_min = pb.causal ? max(0, row - off) : 0;
        const bool row_ok = row < row_len;
        const uint32_t lead_xfree0 = mapa_shared(smem_u32(&sh.x_free[0]), lead_rank);
        const uint32_t lead_xfree1 = mapa_shared(smem_u32(&sh.x_free[1]), lead_rank);
        const uint32_t lead_zpair = mapa_shared(smem_u32(&sh.zpair), lead_rank);
        float l2_row = INFINITY, dl_row = 0.f;  // dQ: own row statistics
        if (OP == XOP_DQ && row_ok) {
            const size_t si = VARLEN ? static_cast<size_t>(h) * pb.total_q + tq0 + row
                                     : (static_cast<size_t>(b) * pb.Hq + h) * pb.Nq + row;
            l2_row = a.lse_log2[si];
            dl_row = a.delta[si];
        }
        float m_ref = -INFINITY, l_part = 0.f;  // forward softmax state (l over my columns of own tiles)
        bool ok = true;
        auto warp_ok = [&](bool v) { return __all_sync(0xffffffffu, v); };
        for (int s = 0; s < n_steps; ++s) {
            const int t = s * C + c;
            const int sb = T::kXdb ? (s & 1) : 0;
            const uint32_t tx = t_x0 + sb * 128 + lane_off;
            const uint32_t ty = t_x0 + 128 + lane_off;  // Y (two-product kernels)
            const int sbuf = s & 1;
            if (!T::kRowsQ) {
                // stage the column statistics of tile t (threads of half 0): +inf
                // lse2 masks queries past the sequence and tiles past the end
                if (half == 0) {
                    const int qi = col_row0(t) + r;
                    const int hh = col_head(t);
                    float l2 = INFINITY, dl = 0.f;
                    if (t < n_ct && qi < lq) {
                        const size_t si = VARLEN ? static_cast<size_t>(hh) * pb.total_q + tq0 + qi
                                                 : (static_cast<size_t>(b) * pb.Hq + hh) * pb.Nq + qi;
                        l2 = a.lse_log2[si];
                        dl = a.delta[si];
                    }
                    stats[sbuf * 128 + r] = l2;
                    stats[256 + sbuf * 128 + r] = dl;
                }
                mbar_arrive(&sh.stat[sbuf]);
            }
            const uint32_t xpar = T::kXdb ? ((s >> 1) & 1) : (s & 1);
            if (!warp_ok(mbar_wait(&sh.x_full[sb], xpar, abort_flag, status, lim, PS_XFULL))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (!T::kRowsQ && !warp_ok(mbar_wait(&sh.stat[sbuf], (s >> 1) & 1, abort_flag, status, lim, PS_STAT))) {
                ok = false;
                break;
            }
            uint32_t z[32];  // my 64 columns of Z as packed pairs
            if constexpr (OP == XOP_FWD) {
                const int limit = key_end - t * 128;  // legal columns [0, limit)
                float mx = -INFINITY;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t x[32];
                    tmem_ld32(tx + q4 * 32, x);
                    tmem_ld_wait(x);
                    if (limit >= 128) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(x[j]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (q4 * 32 + j < limit) mx = fmaxf(mx, __uint_as_float(x[j]));
                    }
                }
                float m_tile = mx * c2;
                if (C > 1) {
                    // agree on the row maximum with the CTAs of the other pairs holding
                    // the same rows: rmax[sbuf][slot][r] at stats + (sbuf*(C-1) + slot)*128 + r
                    if (half == 0)
                        for (int p = 0; p < C; ++p) {
                            if (p == c) continue;
                            float* dst = stats + (sbuf * (C - 1) + slot_of(c, p)) * 128 + r;
                            st_async_f32(mapa_shared(smem_u32(dst), xrank(p)), m_tile,
                                         mapa_shared(smem_u32(&sh.rmax[sbuf]), xrank(p)));
                        }
                    if (!warp_ok(mbar_wait_cluster(&sh.rmax[sbuf], (s >> 1) & 1, abort_flag, status, lim, PS_RMAX))) {
                        ok = false;
                        break;
                    }
                    for (int q = 0; q < C - 1; ++q) m_tile = fmaxf(m_tile, stats[(sbuf * (C - 1) + q) * 128 + r]);
                    // re-arm this buffer for step s+2: no writer reaches it before every
                    // thread here has passed this wait and sent its step s+1 maximum
                    if (ew == 0) mbar_arrive_expect_tx(&sh.rmax[sbuf], 512 * (C - 1));
                }
                float new_ref = m_ref;
                bool need = false;
                if (m_tile > -INFINITY) {
                    if (m_ref == -INFINITY) {
                        new_ref = m_tile;
                    } else if (m_tile > m_ref + kTau) {
                        new_ref = m_tile;
                        need = true;
                    }
                }
                const float alpha = need ? ex2_approx(m_ref - new_ref) : 1.f;
                if (__any_sync(0xffffffffu, need)) {
                    // O must be stable: wait for the previous super-step's value MMAs;
                    // each half rescales half of the row's accumulator columns
                    if (s > 0 && !warp_ok(mbar_wait(&sh.acc, (s - 1) & 1, abort_flag, status, lim, PS_ACC))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int half_w = sw / 2;
                    for (int cc = half * half_w; cc < (half + 1) * half_w; cc += 32) {
                        uint32_t o[32];
                        tmem_ld32(t_acc + lane_off + cc, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(t_acc + lane_off + cc, o);
                    }
                    tmem_st_wait();
                }
                l_part *= alpha;
                m_ref = new_ref;
                const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
                float sum = 0.f;
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    uint32_t x[32];
                    tmem_ld32(tx + col0 + q2 * 32, x);
                    tmem_ld_wait(x);
                    const int lim2 = limit - col0 - q2 * 32;
                    if (lim2 >= 32) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float p0 = ex2_approx(fmaf(__uint_as_float(x[2 * e]), c2, -mu));
                            const float p1 = ex2_approx(fmaf(__uint_as_float(x[2 * e + 1]), c2, -mu));
                            sum += p0 + p1;
                            z[q2 * 16 + e] = pack2<BF16>(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float p0 = (2 * e < lim2) ? ex2_approx(fmaf(__uint_as_float(x[2 * e]), c2, -mu)) : 0.f;
                            const float p1 = (2 * e + 1 < lim2) ? ex2_approx(fmaf(__uint_as_float(x[2 * e + 1]), c2, -mu)) : 0.f;
                            sum += p0 + p1;
                            z[q2 * 16 + e] = pack2<BF16>(p0, p1);
                        }
                    }
                }
                l_part += sum;
            } else {
                // legal columns of this tile: [j_lo, j_hi)
                int j_lo, j_hi;
                if (T::kRowsQ) {  // dQ: keys below key_end
                    j_lo = 0;
                    j_hi = key_end - t * 128;
                } else {          // dV / dK: queries at or after i_min (sequence end folded into lse2 = +inf)
                    j_lo = row_ok ? i_min - col_row0(t) : 128;
                    j_hi = 128;
                }
                const bool full = j_lo <= col0 && j_hi >= col0 + 64;
                const float* s_l2 = stats + sbuf * 128;
                const float* s_dl = stats + 256 + sbuf * 128;
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    uint32_t x[32], y[32];
                    tmem_ld32(tx + col0 + q2 * 32, x);
                    if (T::kTwo) tmem_ld32(ty + col0 + q2 * 32, y);
                    tmem_ld_wait(x);
                    if (T::kTwo) tmem_ld_wait(y);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float zz[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int j = col0 + q2 * 32 + 2 * e + u;
                            const bool legal = full || (j >= j_lo && j < j_hi);
                            const float sv = __uint_as_float(x[2 * e + u]);
                            float v;
                            if (T::kRowsQ) {  // dQ: dS = P (dP - delta) with the row's statistics
                                const float p = legal ? ex2_approx(fmaf(sv, c2, -l2_row)) : 0.f;
                                v = p * (__uint_as_float(y[2 * e + u]) - dl_row);
                            } else {          // dV: P^T; dK: dS^T = P^T (dP^T - delta)
                                const float p = legal ? ex2_approx(fmaf(sv, c2, -s_l2[j])) : 0.f;
                                v = (OP == XOP_DK) ? p * (__uint_as_float(y[2 * e + u]) - s_dl[j]) : p;
                            }
                            zz[u] = v;
                        }
                        z[q2 * 16 + e] = pack2<BF16>(zz[0], zz[1]);
                    }
                }
            }
            // X (and Y) are read: the pair's next score products into this buffer may start
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(sb ? lead_xfree1 : lead_xfree0);
            // The own slot may be rewritten once the previous step's value MMAs of my
            // pair (acc) and of every other pair (slot_free: it consumed my copy, so
            // the copy has read the slot) are done with it.
            if (s > 0 && !warp_ok(mbar_wait(&sh.acc, (s - 1) & 1, abort_flag, status, lim, PS_ACC))) {
                ok = false;
                break;
            }
            if (C > 1 && s > 0) {
                bool got = true;
                for (int p = 0; p < C && got; ++p)
                    if (p != c) got = mbar_wait_cluster(&sh.slot_free[p], (s - 1) & 1, abort_flag, status, lim, PS_SLOT);
                if (!warp_ok(got)) {
                    ok = false;
                    break;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<uint4*>(sZown + half * 16384 + sw128_offset(r, u)) =
                    make_uint4(z[4 * u], z[4 * u + 1], z[4 * u + 2], z[4 * u + 3]);
            fence_proxy_async_smem();
            mbar_arrive(&sh.z_full);
            if (!leader) {
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(lead_zpair);
            }
            if (C > 1 && ew == 0) {
                // one bulk copy of the whole slot into the CTA of every other pair that
                // holds my rows, once all 256 threads have written it (on a time-out
                // the copies are skipped; the abort flag then ends every wait)
                if (mbar_wait(&sh.z_full, s & 1, abort_flag, status, lim, PS_ZFULL)) {
                    for (int p = 0; p < C; ++p) {
                        if (p == c) continue;
                        bulk_copy_s2cluster(mapa_shared(smem_u32(sZ + slot_of(c, p) * 32768), xrank(p)), sZown, 32768,
                                            mapa_shared(smem_u32(&sh.zpeer[slot_of(c, p)]), xrank(p)));
                    }
                }
            }
        }
        // ------------------------------------------------------ epilogue
        if (ok && n_steps > 0) {
            ok = warp_ok(mbar_wait(&sh.acc, (n_steps - 1) & 1, abort_flag, status, lim, PS_EPI));
            tc_fence_after();
        }
        float l_tot = 0.f;
        if (OP == XOP_FWD && ok && n_steps > 0) {
            // Row sum: both halves' parts (the ring is idle now and serves as
            // scratch), then the sums of the other pairs' CTAs holding my rows.
            float* lsum_local = reinterpret_cast<float*>(sRing);
            lsum_local[half * 128 + r] = l_part;
            mbar_arrive(&sh.half);
            ok = warp_ok(mbar_wait(&sh.half, 0, abort_flag, status, lim, PS_LSUM));
            const float l_cta = lsum_local[r] + lsum_local[128 + r];
            l_tot = l_cta;
            if (ok && C > 1) {
                if (half == 0)
                    for (int p = 0; p < C; ++p)
                        if (p != c) {
                            float* dst = stats + (2 * (C - 1) + slot_of(c, p)) * 128 + r;
                            st_async_f32(mapa_shared(smem_u32(dst), xrank(p)), l_cta,
                                         mapa_shared(smem_u32(&sh.lsum), xrank(p)));
                        }
                ok = warp_ok(mbar_wait_cluster(&sh.lsum, 0, abort_flag, status, lim, PS_LSUM));
                for (int q = 0; q < C - 1; ++q) l_tot += stats[(2 * (C - 1) + q) * 128 + r];
            }
        }
        if (ok) {
            float mul;
            void* out;
            int out_heads, out_n, t0, head;
            if (OP == XOP_FWD) {
                mul = l_tot > 0.f ? 1.f / l_tot : 0.f;
                out = a.o;
            } else if (OP == XOP_DQ) {
                mul = pb.scale;
                out = a.dq;
            } else if (OP == XOP_DV) {
                mul = 1.f;
                out = a.dv;
            } else {
                mul = pb.scale;
                out = a.dk;
            }
            if (T::kRowsQ) {
                out_heads = pb.Hq;
                out_n = pb.Nq;
                t0 = tq0;
                head = h;
            } else {
                out_heads = pb.Hkv;
                out_n = pb.Nkv;
                t0 = tk0;
                head = hk;
            }
            const size_t orow = VARLEN ? (static_cast<size_t>(t0 + row) * out_heads + head) * pb.D
                                       : ((static_cast<size_t>(b) * out_heads + head) * out_n + row) * pb.D;
            uint16_t* dst = reinterpret_cast<uint16_t*>(out) + orow + d0;
            const int c_end = min((half + 1) * (sw / 2), pb.D - d0);  // columns past D are not stored
            for (int cc = half * (sw / 2); cc < c_end; cc += 32) {
                uint32_t v[32];
                if (n_steps > 0) {
                    tmem_ld32(t_acc + lane_off + cc, v);
                    tmem_ld_wait(v);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
                if (row_ok) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
                    for (int e = 0; e < 4; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
            }
            if (OP == XOP_FWD && c == 0 && half == 0 && row_ok) {
                const float lse = l_tot > 0.f ? (m_ref + log2f(l_tot)) * kLn2 : -INFINITY;
                const size_t li = VARLEN ? static_cast<size_t>(h) * pb.total_q + tq0 + row
                                         : (static_cast<size_t>(b) * pb.Hq + h) * pb.Nq + row;
                a.lse[li] = lse;
            }
        }
    }

    // -------------------------------------------------------------- teardown
    // No CTA leaves while another may still write into its shared memory or
    // (the even rank's MMAs) into its TMEM.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

template <int OP, bool BF16, bool VARLEN>
cudaError_t launch_op(const XArgs& a, const CUtensorMap* maps, const PGeo& gm, int n_rt, int bz, int smem,
                      cudaStream_t s)
{
    auto kern = pair_kernel<OP, BF16, VARLEN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * gm.C, n_rt, bz);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * gm.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], a, gm);
}

template <int OP>
cudaError_t dispatch(const XArgs& a, const CUtensorMap* maps, const PGeo& gm, int n_rt, int bz, int smem,
                     cudaStream_t s)
{
    if (a.bf16) return a.pb.varlen ? launch_op<OP, true, true>(a, maps, gm, n_rt, bz, smem, s)
                                   : launch_op<OP, true, false>(a, maps, gm, n_rt, bz, smem, s);
    return a.pb.varlen ? launch_op<OP, false, true>(a, maps, gm, n_rt, bz, smem, s)
                       : launch_op<OP, false, false>(a, maps, gm, n_rt, bz, smem, s);
}

}  // namespace

cudaError_t launch_pair(int op, const XArgs& a, cudaStream_t s)
{
    const Problem& pb = a.pb;
    const bool q_empty = q_side_empty(pb), kv_empty = kv_side_empty(pb);
    const bool rows_q = (op == XOP_FWD || op == XOP_DQ);
    if (rows_q ? q_empty : kv_empty) return cudaSuccess;  // no output rows
    const int nd = pb.D / 64;
    const int d_pad = (pb.D + 127) & ~127;
    PGeo gm;
    gm.C = (d_pad + 255) / 256;
    if (gm.C > kMaxC) return cudaErrorInvalidConfiguration;
    const int slots_bytes = gm.C * 32768;  // own slot + C-1 slots of the other pairs
    const int budget = kMaxSmem - static_cast<int>(sizeof(StaticSmem));
    // keep as many leading chunks of the first row operand resident as leave a
    // ring of >= 10 stages
    {
        const int spare = budget - slots_bytes - pair_stats_bytes(op, gm.C) - 10 * kSlot;
        gm.res = spare > 0 ? spare / kSlot : 0;
        if (gm.res > nd) gm.res = nd;
    }
    const int fixed = gm.res * kSlot + slots_bytes + pair_stats_bytes(op, gm.C);
    gm.stages = (budget - fixed) / kSlot;
    if (gm.stages > kStages) gm.stages = kStages;
    if (gm.stages < 2) return cudaErrorInvalidConfiguration;
    const int smem = fixed + gm.stages * kSlot;

    // maps: A1, A2 (row side, 128-row boxes of one chunk), B1, B2 (column side,
    // 64 rows x 2 chunks), W (column side, 64 rows x 2 chunks)
    const void* qp = q_empty ? a.k : a.q;
    const void* dop = q_empty ? a.k : (a.dO ? a.dO : a.q);
    const void* kp = kv_empty ? a.q : a.k;
    const void* vp = kv_empty ? a.q : a.v;
    const bool qs = q_empty;   // side flag of the q-side maps (kv side when q is empty)
    const bool ks = !kv_empty; // side flag of the kv-side maps
    CUtensorMap m[5];
    bool okm = true;
    auto row = [&](int i, const void* p, bool kv_side) { okm = okm && make_row_map(&m[i], p, pb, kv_side, a.bf16, 128); };
    auto slab = [&](int i, const void* p, bool kv_side) { okm = okm && make_slab_map(&m[i], p, pb, kv_side, a.bf16, 64, 2); };
    int n_rows;
    int bz;
    switch (op) {
    case XOP_FWD:
        row(0, qp, qs); row(1, qp, qs); slab(2, kp, ks); slab(3, kp, ks); slab(4, vp, ks);
        n_rows = pb.Nq; bz = pb.B * pb.Hq;
        break;
    case XOP_DQ:
        row(0, qp, qs); row(1, dop, qs); slab(2, kp, ks); slab(3, vp, ks); slab(4, kp, ks);
        n_rows = pb.Nq; bz = pb.B * pb.Hq;
        break;
    case XOP_DV:
        row(0, kp, ks); row(1, kp, ks); slab(2, qp, qs); slab(3, qp, qs); slab(4, dop, qs);
        n_rows = pb.Nkv; bz = pb.B * pb.Hkv;
        break;
    default:  // XOP_DK
        row(0, kp, ks); row(1, vp, ks); slab(2, qp, qs); slab(3, dop, qs); slab(4, qp, qs);
        n_rows = pb.Nkv; bz = pb.B * pb.Hkv;
        break;
    }
    if (!okm) return cudaErrorInvalidValue;
    const int n_rt = (n_rows + 255) / 256;
    if (n_rt == 0 || bz == 0) return cudaSuccess;
    switch (op) {
    case XOP_FWD: return dispatch<XOP_FWD>(a, m, gm, n_rt, bz, smem, s);
    case XOP_DQ: return dispatch<XOP_DQ>(a, m, gm, n_rt, bz, smem, s);
    case XOP_DV: return dispatch<XOP_DV>(a, m, gm, n_rt, bz, smem, s);
    default: return dispatch<XOP_DK>(a, m, gm, n_rt, bz, smem, s);
    }
}

}  // namespace ffpa
