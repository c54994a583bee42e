// Cluster-exchange kernels: the forward and the three backward GEMM kernels
// (dV, dK, dQ) of exact attention at large head dim on sm_103a.
//
// Every kernel here has the same shape. A cluster of C CTAs owns one 128-row
// tile of "rows" (queries for the forward and dQ, keys for dV and dK) and
// walks over 128-wide tiles of "columns" (keys, resp. queries) in
// super-steps of C tiles. In super-step s, CTA c
//   1. computes the score tile(s) of column tile C*s + c with tcgen05 MMAs
//      over the full head dim: X = S (and Y = dP for dQ / dK),
//   2. turns them into one bf16/fp16 operand tile Z (P, P^T, dS or dS^T;
//      the forward first exchanges row maxima with its peers so every CTA
//      uses the same softmax reference),
//   3. keeps Z in TMEM for itself and writes it into every peer's shared
//      memory (DSMEM), and
//   4. accumulates its own D-slab of the output over all C tiles of the
//      super-step: acc += Z_{c'} W_{tile C*s+c'}[:, slab] for c' = 0..C-1
//      (W = V, K, dO or Q), own Z read from TMEM, peers' Z from shared memory.
// So each score product is computed once, while the fp32 accumulator of a
// 128-row tile is split over C CTAs by head-dim slabs of <= 256 columns (a
// 128 x 512 fp32 tile would fill all 512 TMEM columns of one SM).
//
// The pages this implements: FFPA docs, "CuTe-DSL Backend" page, "Hard
// constraints" (bottom-right causal, GQA/MQA broadcast, empty rows give
// O = 0, LSE = -inf and zero gradients), "Varlen (packed THD) API" (packed
// layout, LSE [H, T]), "Blackwell status" (preprocess plus separate
// gradient launches, split because one SM cannot hold a whole dK/dV tile).
//
// Warp roles: warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner),
// warps 2..5 elementwise (one tile row per thread) and epilogue.
#include <cstdlib>
#include <cstring>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 elementwise (two per TMEM row)
constexpr int kStages = 16;      // upper bound of the TMA ring depth
constexpr int kMaxC = 4;         // cluster size bound (D <= 1024 in 256-column slabs)
constexpr float kTau = 8.0f;     // forward: rescale O only when the row max grows by more than 2^8
constexpr float kLn2 = 0.693147180559945309f;

enum Site : uint32_t {
    XS_PROD = 32, XS_A1, XS_XFREE, XS_RING, XS_ZFULL, XS_ZPEER, XS_XFULL, XS_RMAX, XS_ACC, XS_SLOT, XS_STAT,
    XS_LSUM, XS_EPI, XS_DRAIN
};

struct Geo {
    int C;            // CTAs per cluster (= D-slabs)
    int slab_chunks;  // 64-wide head-dim chunks per slab (the last slab may be smaller)
    int stages;       // TMA ring depth
    int res;          // leading 64-wide chunks of the first row operand kept resident in shared memory
    int n_rt;         // row tiles of 128 per (batch, head) in the grid (of the longest sequence)
    int n_bz;         // (batch, head) entries in the grid
    int ostore;       // the output map is valid: whole 128-row tiles leave through shared memory and TMA
};

template <int OP>
struct Traits {
    static constexpr bool kTwo = (OP == XOP_DQ || OP == XOP_DK);      // X and Y score tiles
    static constexpr bool kRowsQ = (OP == XOP_FWD || OP == XOP_DQ);   // rows are queries
    static constexpr bool kXdb = !kTwo;                               // X double-buffered
};

// Barriers and flags live in one static block of exactly 1 KiB, so that the
// dynamic shared memory right after it starts 1024-byte aligned (the 128-byte
// swizzle of TMA tiles and MMA descriptors needs that); the kernel checks the
// alignment at run time and reports an error instead of running misaligned.
struct __align__(1024) StaticSmem {
    uint64_t full[kStages], empty[kStages];
    uint64_t a1, x_full[2], x_free[2], z_full, acc;
    uint64_t zpeer[kMaxC], slot_free[kMaxC], stat[2], rmax[2], lsum, drain, half;
    uint32_t tmem_base;
    int abort_flag;
    // dK storing tiles: the own slot holds P^T / its store read it; the dS store read it
    uint64_t p_full, p_read, stored;
    uint64_t ostage;  // every elementwise thread staged its part of the output tile
};
static_assert(sizeof(StaticSmem) == 1024, "static shared block must be exactly 1 KiB");

// Bytes of the per-kernel statistics area (rounded to 1 KiB):
//   forward: rmax[2][C-1][128] and lsum[C-1][128] (peer values, by slot)
//   dV / dK: lse2[2][128] and delta[2][128] (column statistics, double-buffered)
__host__ __device__ inline int stats_bytes(int op, int C)
{
    int b = 0;
    if (op == XOP_FWD) b = 3 * (C > 1 ? C - 1 : 0) * 128 * 4;
    else if (op == XOP_DV || op == XOP_DK) b = 4 * 128 * 4;
    return (b + 1023) & ~1023;
}

template <int OP, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    xchg_kernel(const __grid_constant__ CUtensorMap tA1, const __grid_constant__ CUtensorMap tA2,
                const __grid_constant__ CUtensorMap tB1, const __grid_constant__ CUtensorMap tB2,
                const __grid_constant__ CUtensorMap tW, const __grid_constant__ CUtensorMap tS,
                const __grid_constant__ CUtensorMap tP, const __grid_constant__ CUtensorMap tO, const XArgs a,
                const Geo gm)
{
    // the next GEMM kernel of a backward may take SMs as this grid's last CTAs start
    pdl_trigger();
    using T = Traits<OP>;
    const Problem& pb = a.pb;
    const int C = gm.C;
    const int c = static_cast<int>(cluster_ctarank());
    const int G = pb.Hq / pb.Hkv;

    // ------------------------------------------------------------ work unit
    // All CTAs of a cluster share blockIdx.y / blockIdx.z, hence the same unit.
    // Units in linear cluster order: row tile fastest, then b*H, or (causal)
    // b*H fastest, then row tile. The hardware starts clusters in that order:
    // the first keeps the clusters that run together on few heads (their K/V
    // tiles stay in L2); the second starts every head's longest tile before any
    // head's next one, which balances the unequal causal tiles.
    const long long unit = unit_id();
    if (unit >= static_cast<long long>(gm.n_rt) * gm.n_bz) return;  // past the last unit: uniform over the cluster
    const int bz = static_cast<int>(pb.causal ? unit % gm.n_bz : unit / gm.n_rt);
    const int tile = static_cast<int>(pb.causal ? unit / gm.n_bz : unit % gm.n_rt);
    int b, h = 0, hk;
    if (T::kRowsQ) {
        b = bz / pb.Hq;
        h = bz % pb.Hq;
        hk = h / G;
    } else {
        // the kv heads [g0, g0 + ng) of the launch (all of them unless the
        // stored-tile backward runs in chunks of kv groups)
        const int ng = a.ng > 0 ? a.ng : pb.Hkv;
        b = bz / ng;
        hk = a.g0 + bz % ng;
    }
    int lq, lk, tq0 = 0, tk0 = 0;
    if constexpr (VARLEN) {
        if (!varlen_seq(pb, b, a.ctl.status, VS_SINGLE, tq0, lq, tk0, lk)) return;  // uniform over the cluster
    } else {
        lq = pb.Nq;
        lk = pb.Nkv;
    }
    const int off = lk - lq;  // causal: key j legal for query i iff j <= i + off
    const int row_len = T::kRowsQ ? lq : lk;
    // causal, rows = queries: the last row tiles of a sequence see the most keys
    // and go first; rows = keys: the first key tiles see the most queries
    const int n_rt_seq = (row_len + 127) / 128;
    const int rt = (T::kRowsQ && pb.causal) ? (n_rt_seq - 1 - tile) : tile;
    const int r0 = rt * 128;
    if (rt < 0 || r0 >= row_len) return;  // uniform over the cluster, before any cluster barrier

    int n_ct;            // column tiles of the unit
    int m_start = 0, n_mt = 0;
    if (T::kRowsQ) {
        n_ct = (lk + 127) / 128;
        if (pb.causal) {
            const int kmax = min(r0 + 127, lq - 1) + off;
            n_ct = kmax < 0 ? 0 : min(n_ct, kmax / 128 + 1);
        }
    } else {
        if (pb.causal) {
            // dK storing tiles starts where the 256-key tile that holds my rows
            // starts, at an even query tile: every tile a GEMM tile of the stored-tile
            // GEMMs reads is then written (the extra tiles are fully masked: zeros)
            const bool st = OP == XOP_DK && (a.store_ds || a.store_p);
            m_start = max(0, (st ? (r0 & ~255) : r0) - off) / 128;
            if (st) m_start &= ~1;
        }
        n_mt = max(0, (lq + 127) / 128 - m_start);
        n_ct = G * n_mt;
    }
    const int n_steps = (n_ct + C - 1) / C;

    const int nd = (pb.D + 63) / 64;  // 64-wide head-dim chunks (the last one half-filled when D % 64 = 32)
    const int c_begin = c * gm.slab_chunks;
    const int nb = min(gm.slab_chunks, nd - c_begin);  // 64-wide blocks in my slab
    const int sw = nb * 64;
    const int d0 = c_begin * 64;

    // ------------------------------------------------------------ shared memory
    __shared__ StaticSmem sh;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* sA1 = smem;                                    // resident row-operand chunks: res x 16 KiB
    uint8_t* sZ = sA1 + gm.res * 16384;                     // C-1 peer slots + own slot, 32 KiB each
    uint8_t* sZown = sZ + (C - 1) * 32768;                  // own slot
    float* stats = reinterpret_cast<float*>(sZ + C * 32768);
    uint8_t* sRing = reinterpret_cast<uint8_t*>(stats) + stats_bytes(OP, C);
    uint64_t* const bar_full = sh.full;
    uint64_t* const bar_empty = sh.empty;
    uint64_t& bar_a1 = sh.a1;
    uint64_t* const bar_x_full = sh.x_full;
    uint64_t* const bar_x_free = sh.x_free;
    uint64_t& bar_z_full = sh.z_full;
    uint64_t& bar_acc = sh.acc;
    uint64_t* const bar_zpeer = sh.zpeer;
    uint64_t* const bar_slot_free = sh.slot_free;
    uint64_t* const bar_stat = sh.stat;
    uint64_t* const bar_rmax = sh.rmax;
    uint64_t& bar_lsum = sh.lsum;
    uint64_t& bar_drain = sh.drain;
    uint64_t& bar_half = sh.half;      // forward epilogue: both halves' row sums written
    if (smem_u32(smem) & 1023u) {  // uniform over the block: report, do not run misaligned
        if (threadIdx.x == 0) atomicCAS(a.ctl.status, 0u, 5u | (0xffu << 8));
        return;
    }

    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < gm.stages; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_a1, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_x_full[i], 1);
            mbar_init(&bar_x_free[i], 256);
            mbar_init(&bar_stat[i], 256);
            mbar_init(&bar_rmax[i], 1);
        }
        mbar_init(&bar_z_full, 256);
        mbar_init(&bar_half, 256);
        mbar_init(&sh.ostage, 256);
        mbar_init(&bar_acc, 1);
        for (int i = 0; i < kMaxC; ++i) {
            mbar_init(&bar_zpeer[i], 1);
            mbar_init(&bar_slot_free[i], 1);
        }
        mbar_init(&bar_lsum, 1);
        mbar_init(&bar_drain, 1);
        mbar_init(&sh.p_full, 256);
        mbar_init(&sh.p_read, 1);
        mbar_init(&sh.stored, 1);
        sh.abort_flag = 0;
        // Peers deliver with st.async, completing bytes on these barriers; each is
        // armed (one arrival + expected bytes) by its receiver before any peer can
        // write the phase it guards: here for the first phase (the first two for
        // the double-buffered row maxima), later right after each completed wait.
        if (C > 1) {
            for (int i = 0; i < C - 1; ++i) mbar_arrive_expect_tx(&bar_zpeer[i], 32768);
            if (OP == XOP_FWD) {
                mbar_arrive_expect_tx(&bar_rmax[0], 512 * (C - 1));
                mbar_arrive_expect_tx(&bar_rmax[1], 512 * (C - 1));
                mbar_arrive_expect_tx(&bar_lsum, 512 * (C - 1));
            }
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync_all();  // every CTA's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const uint32_t t_acc = tmem;        // [0, 256): accumulator slab
    const uint32_t t_x0 = tmem + 256;   // X buffers (and Y for the two-product kernels)
    volatile int* abort_flag = &sh.abort_flag;
    uint32_t* status = a.ctl.status;
    const uint64_t lim = a.ctl.limit_ns;

    // Peer bookkeeping: slot index of writer w inside consumer p's slot array.
    auto slot_of = [&](int writer, int consumer) { return writer < consumer ? writer : writer - 1; };
    uint16_t peer_mask = 0;
    for (int p = 0; p < C; ++p)
        if (p != c) peer_mask |= static_cast<uint16_t>(1u << p);

    // Column tile t -> (head, first row) on the column side; t past the end is
    // clamped for loading (its results are masked to zero).
    auto col_head = [&](int t) { return T::kRowsQ ? hk : hk * G + min(t, n_ct - 1) / max(n_mt, 1); };
    auto col_row0 = [&](int t) {
        const int tc = min(t, n_ct - 1);
        return T::kRowsQ ? tc * 128 : (m_start + tc % max(n_mt, 1)) * 128;
    };
    // TMA coordinates: row maps (d, row or token, head, b or 0), slab maps
    // (0, row or token, chunk, head, b or 0).
    const int bco = VARLEN ? 0 : b;
    const int row_head = T::kRowsQ ? h : hk;
    auto row_co = [&](int row) { return VARLEN ? (T::kRowsQ ? tq0 : tk0) + row : row; };
    auto col_co = [&](int row) { return VARLEN ? (T::kRowsQ ? tk0 : tq0) + row : row; };
    // key row -> row of the stored tile buffers (packed batches: sequence b's rows
    // start at cu_k[b] + 256 b, so that no tile reaches the next sequence's rows)
    auto tile_row = [&](int row) { return VARLEN ? tk0 + 256 * b + row : row; };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (elect_one()) {
            prefetch_tmap(&tA1);
            prefetch_tmap(&tB1);
            prefetch_tmap(&tW);
            RingPos rp;
            int issued = 0;
            bool ok = true;
            // one 64 x 128-row box of chunk d
            auto put = [&](const CUtensorMap* m, int d, int row, int head) -> bool {
                if (!mbar_wait(&bar_empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, XS_PROD)) return false;
                uint8_t* dst = sRing + rp.slot * 16384;
                mbar_arrive_expect_tx(&bar_full[rp.slot], 16384);
                tma_load_4d(dst, m, &bar_full[rp.slot], d * 64, row, head, bco);
                rp.advance(gm.stages);
                ++issued;
                return true;
            };
            if (gm.res > 0 && n_steps > 0) {
                mbar_arrive_expect_tx(&bar_a1, gm.res * 16384);
                for (int d = 0; d < gm.res; ++d) tma_load_4d(sA1 + d * 16384, &tA1, &bar_a1, d * 64, row_co(r0), row_head, bco);
            }
            auto load_score = [&](int s) -> bool {
                const int t = s * C + c;
                const int hh = col_head(t), cr = col_row0(t);
                for (int d = 0; d < nd; ++d) {
                    if (d >= gm.res && !put(&tA1, d, row_co(r0), row_head)) return false;
                    if (!put(&tB1, d, col_co(cr), hh)) return false;
                }
                if (T::kTwo)
                    for (int d = 0; d < nd; ++d) {
                        if (!put(&tA2, d, row_co(r0), row_head)) return false;
                        if (!put(&tB2, d, col_co(cr), hh)) return false;
                    }
                return true;
            };
            // value operand: one 4-D box = 32 rows x my slab's 64-wide chunks (chunks past
            // the head dim of a narrower last slab read as zero and are not used)
            const int wbytes = 32 * 128 * gm.slab_chunks;
            auto load_value = [&](int s) -> bool {
                for (int cc = 0; cc < C; ++cc) {
                    const int t = s * C + cc;
                    const int hh = col_head(t), cr = col_row0(t);
                    for (int vc = 0; vc < 4; ++vc) {
                        if (!mbar_wait(&bar_empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, XS_PROD)) return false;
                        uint8_t* dst = sRing + rp.slot * 16384;
                        if (pb.D % 64 == 0) {
                            mbar_arrive_expect_tx(&bar_full[rp.slot], wbytes);
                            tma_load_5d(dst, &tW, &bar_full[rp.slot], 0, col_co(cr + vc * 32), c_begin, hh, bco);
                        } else {
                            // head dim not a multiple of 64: one 64 x 32 box per chunk of my
                            // slab from a row map over the true D (the tail reads as zero)
                            mbar_arrive_expect_tx(&bar_full[rp.slot], nb * 32 * 128);
                            for (int i = 0; i < nb; ++i)
                                tma_load_4d(dst + i * 32 * 128, &tW, &bar_full[rp.slot], (c_begin + i) * 64,
                                            col_co(cr + vc * 32), hh, bco);
                        }
                        rp.advance(gm.stages);
                        ++issued;
                    }
                }
                return true;
            };
            if (n_steps > 0) ok = load_score(0);
            for (int s = 0; ok && s < n_steps; ++s) {
                if (s + 1 < n_steps) ok = load_score(s + 1);
                if (ok) ok = load_value(s);
            }
            const int last = min(issued, gm.stages);
            RingPos dp = rp;
            for (int i = 0; i < last; ++i) {
                dp.retreat(gm.stages);
                int dummy = 0;
                mbar_wait(&bar_full[dp.slot], dp.phase, &dummy, status, lim, XS_DRAIN, false);
            }
            if (gm.res > 0 && n_steps > 0) {
                int dummy = 0;
                mbar_wait(&bar_a1, 0, &dummy, status, lim, XS_DRAIN, false);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (elect_one()) {
            const uint32_t idesc_s = idesc_f16(128, 128, BF16, false, false);
            const uint32_t idesc_v = idesc_f16(128, sw, BF16, false, true);
            RingPos rp;
            bool ok = true;
            if (gm.res > 0 && n_steps > 0) {
                ok = mbar_wait(&bar_a1, 0, abort_flag, status, lim, XS_A1);
                tc_fence_after();
            }
            auto take = [&]() -> const uint8_t* {
                if (!mbar_wait(&bar_full[rp.slot], rp.phase, abort_flag, status, lim, XS_RING)) return nullptr;
                tc_fence_after();
                return sRing + rp.slot * 16384;
            };
            auto give = [&](int slot) { umma_commit(&bar_empty[slot]); };
            auto issue_score = [&](int s) -> bool {
                const int sb = T::kXdb ? (s & 1) : 0;
                // XDB: buffer sb last held Z of step s-2 (freed by value(s-2));
                // own-slot kernels: X/Y of step s-1 released by the elementwise warps
                if (T::kXdb ? s >= 2 : s >= 1) {
                    const uint32_t par = T::kXdb ? (((s - 2) >> 1) & 1) : ((s - 1) & 1);
                    if (!mbar_wait(&bar_x_free[sb], par, abort_flag, status, lim, XS_XFREE)) return false;
                    tc_fence_after();
                }
                for (int prod = 0; prod < (T::kTwo ? 2 : 1); ++prod) {
                    const uint32_t dst = t_x0 + (T::kXdb ? sb * 128 : prod * 128);
                    for (int d = 0; d < nd; ++d) {
                        const uint8_t* A;
                        int a_slot = -1;
                        if (prod == 0 && d < gm.res) {
                            A = sA1 + d * 16384;
                        } else {
                            A = take();
                            if (!A) return false;
                            a_slot = rp.slot;
                            rp.advance(gm.stages);
                        }
                        const uint8_t* B = take();
                        if (!B) return false;
                        // one descriptor per tile, stepped by 32 bytes per MMA (K-major)
                        const uint64_t da = sdesc_sw128(smem_u32(A), 16, 1024);
                        const uint64_t db = sdesc_sw128(smem_u32(B), 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f16(dst, sdesc_advance(da, kk * 32), sdesc_advance(db, kk * 32), idesc_s, (d | kk) != 0);
                        if (a_slot >= 0) give(a_slot);
                        give(rp.slot);
                        rp.advance(gm.stages);
                    }
                }
                umma_commit(&bar_x_full[sb]);
                return true;
            };
            auto issue_value = [&](int s) -> bool {
                if (!mbar_wait(&bar_z_full, s & 1, abort_flag, status, lim, XS_ZFULL)) return false;
                for (int p = 0; p < C; ++p)
                    if (p != c) {
                        if (!mbar_wait_cluster(&bar_zpeer[slot_of(p, c)], s & 1, abort_flag, status, lim, XS_ZPEER))
                            return false;
                        // arm the next phase before this step's slot_free lets the peer write it
                        mbar_arrive_expect_tx(&bar_zpeer[slot_of(p, c)], 32768);
                    }
                fence_proxy_async_smem();
                tc_fence_after();
                for (int cc = 0; cc < C; ++cc) {
                    const uint8_t* zs = (cc == c) ? sZown : sZ + slot_of(cc, c) * 32768;
                    const uint64_t dz = sdesc_sw128(smem_u32(zs), 16, 1024);
                    for (int vc = 0; vc < 4; ++vc) {
                        const uint8_t* W = take();
                        if (!W) return false;
                        const uint64_t dw = sdesc_sw128(smem_u32(W), 32 * 128, 1024);
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const int kt = vc * 32 + t * 16;
                            const uint32_t acc = (s | cc | vc | t) != 0;
                            umma_f16(t_acc, sdesc_advance(dz, (kt / 64) * 16384 + (kt % 64) * 2), sdesc_advance(dw, t * 2048),
                                     idesc_v, acc);
                        }
                        give(rp.slot);
                        rp.advance(gm.stages);
                    }
                }
                umma_commit(&bar_acc);
                if (C > 1) umma_commit_multicast(&bar_slot_free[c], peer_mask);
                return true;
            };
            if (ok && n_steps > 0) ok = issue_score(0);
            for (int s = 0; ok && s < n_steps; ++s) {
                if (s + 1 < n_steps) ok = issue_score(s + 1);
                if (ok) ok = issue_value(s);
            }
            umma_commit(&bar_drain);
            int dummy = 0;
            mbar_wait(&bar_drain, 0, &dummy, status, lim, XS_DRAIN, false);
        }
    } else {
        // ------------------------------------------------------ elementwise
        // Two threads per tile row: warps 2..5 take columns [0, 64), warps 6..9
        // columns [64, 128) of the same TMEM lanes.
        const int quarter = warp & 3;
        const int r = quarter * 32 + static_cast<int>(lane_id());  // tile row = TMEM lane
        const int ew = threadIdx.x - 64;                              // 0..255
        const int half = ew >> 7;
        const int col0 = half * 64;                                   // my columns [col0, col0 + 64)
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float c2 = pb.scale_log2;
        const int row = r0 + r;  // query (rows = queries) or key (rows = keys)
        // rows = queries: legal keys [0, key_end); rows = keys: legal queries [i_min, lq)
        const int key_end = pb.causal ? min(lk, row + off + 1) : lk;
        const int i_min = pb.causal ? max(0, row - off) : 0;
        const bool row_ok = row < row_len;
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
        // dK storing dS^T / P^T tiles ([B, Hq, Nkv, ldq]): thread ew == 0 stores the
        // own slot with two TMA stores (evict-first: later launches read them)
        const bool st_ds = OP == XOP_DK && a.store_ds != 0;
        const bool st_p = OP == XOP_DK && a.store_p != 0;
        const uint64_t pol = (ew == 0 && (st_ds || st_p)) ? l2_policy_evict_first() : 0;
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
                    stats[sbuf * 128 + r] = l2;          // lse2[sbuf][column]
                    stats[256 + sbuf * 128 + r] = dl;    // delta[sbuf][column]
                }
                mbar_arrive(&bar_stat[sbuf]);
            }
            const uint32_t xpar = T::kXdb ? ((s >> 1) & 1) : (s & 1);
            if (!warp_ok(mbar_wait(&bar_x_full[sb], xpar, abort_flag, status, lim, XS_XFULL))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (!T::kRowsQ && !warp_ok(mbar_wait(&bar_stat[sbuf], (s >> 1) & 1, abort_flag, status, lim, XS_STAT))) {
                ok = false;
                break;
            }
            // The own slot may be rewritten once the previous step's value MMAs here
            // (acc) and every peer (slot_free: it consumed our copy, so the copy has
            // read the slot) are done with it, and (dK storing dS) the store of the
            // previous step's dS^T has read it.
            auto own_free = [&]() -> bool {
                if (s == 0) return true;
                bool got = mbar_wait(&bar_acc, (s - 1) & 1, abort_flag, status, lim, XS_ACC);
                for (int p = 0; p < C && got; ++p)
                    if (p != c) got = mbar_wait_cluster(&bar_slot_free[p], (s - 1) & 1, abort_flag, status, lim, XS_SLOT);
                if (got && st_ds) got = mbar_wait(&sh.stored, (s - 1) & 1, abort_flag, status, lim, XS_ZFULL);
                return warp_ok(got);
            };
            uint32_t z[32];  // my 64 columns of Z as packed pairs
            if constexpr (OP == XOP_FWD) {
                const int limit = key_end - t * 128;  // legal columns [0, limit)
                // row maximum over all 128 columns (both threads of a row compute it)
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
                    // exchange row maxima so every CTA of the cluster uses one reference:
                    // rmax[sbuf][slot][r] at stats + (sbuf*(C-1) + slot)*128 + r
                    if (half == 0)
                        for (int p = 0; p < C; ++p) {
                            if (p == c) continue;
                            float* dst = stats + (sbuf * (C - 1) + slot_of(c, p)) * 128 + r;
                            st_async_f32(mapa_shared(smem_u32(dst), p), m_tile, mapa_shared(smem_u32(&bar_rmax[sbuf]), p));
                        }
                    if (!warp_ok(mbar_wait_cluster(&bar_rmax[sbuf], (s >> 1) & 1, abort_flag, status, lim, XS_RMAX))) {
                        ok = false;
                        break;
                    }
                    for (int q = 0; q < C - 1; ++q) m_tile = fmaxf(m_tile, stats[(sbuf * (C - 1) + q) * 128 + r]);
                    // re-arm this buffer for step s+2: no peer writes it before every
                    // thread here has passed this wait and sent its step s+1 maximum
                    if (ew == 0) mbar_arrive_expect_tx(&bar_rmax[sbuf], 512 * (C - 1));
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
                    if (s > 0 && !warp_ok(mbar_wait(&bar_acc, (s - 1) & 1, abort_flag, status, lim, XS_ACC))) {
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
                // column statistics of my columns col0 + 4 i .. + 3 in one 16-byte load
                // (the statistics area is 1 KiB aligned, col0 a multiple of 64)
                auto stat4 = [&](const float* base, int jj) { return *reinterpret_cast<const float4*>(base + jj); };
                if (OP == XOP_DK && st_p) {
                    // dK storing P: P^T (input dtype) goes through the own slot first;
                    // its store runs while dS^T is formed, then dS^T replaces it
                    uint32_t pp[32];  // P of my 64 columns as fp16 pairs
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        uint32_t x[32];
                        tmem_ld32(tx + col0 + q2 * 32, x);
                        tmem_ld_wait(x);
                        float4 l4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if ((e & 1) == 0) l4 = stat4(s_l2, col0 + q2 * 32 + 2 * e);
                            const float l2e[2] = {(e & 1) ? l4.z : l4.x, (e & 1) ? l4.w : l4.y};
                            float pv[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int j = col0 + q2 * 32 + 2 * e + u;
                                const bool legal = full || (j >= j_lo && j < j_hi);
                                pv[u] = legal ? ex2_approx(fmaf(__uint_as_float(x[2 * e + u]), c2, -l2e[u])) : 0.f;
                            }
                            pp[q2 * 16 + e] = pack2<false>(pv[0], pv[1]);
                        }
                    }
                    if (!own_free()) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 pv = unpack2<false>(pp[4 * u + e]);
                            w4[e] = pack2<BF16>(pv.x, pv.y);
                        }
                        *reinterpret_cast<uint4*>(sZown + half * 16384 + sw128_offset(r, u)) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&sh.p_full);
                    if (ew == 0) {
                        // all 256 threads wrote it: store it, and report once the store read it
                        if (mbar_wait(&sh.p_full, s & 1, abort_flag, status, lim, XS_ZFULL)) {
                            if (t < n_ct) {
                                tma_store_4d_hint(&tP, sZown, col_row0(t), tile_row(r0), col_head(t) - a.g0 * G, bco, pol);
                                tma_store_4d_hint(&tP, sZown + 16384, col_row0(t) + 64, tile_row(r0), col_head(t) - a.g0 * G, bco,
                                                  pol);
                                bulk_commit_group();
                                bulk_wait_read_all();
                            }
                            mbar_arrive(&sh.p_read);
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        uint32_t y[32];
                        tmem_ld32(ty + col0 + q2 * 32, y);
                        tmem_ld_wait(y);
                        float4 d4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if ((e & 1) == 0) d4 = stat4(s_dl, col0 + q2 * 32 + 2 * e);
                            const float2 pv = unpack2<false>(pp[q2 * 16 + e]);
                            z[q2 * 16 + e] = pack2<BF16>(pv.x * (__uint_as_float(y[2 * e]) - ((e & 1) ? d4.z : d4.x)),
                                                         pv.y * (__uint_as_float(y[2 * e + 1]) - ((e & 1) ? d4.w : d4.y)));
                        }
                    }
                } else {
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    uint32_t x[32], y[32];
                    tmem_ld32(tx + col0 + q2 * 32, x);
                    if (T::kTwo) tmem_ld32(ty + col0 + q2 * 32, y);
                    tmem_ld_wait(x);
                    if (T::kTwo) tmem_ld_wait(y);
                    float4 l4 = make_float4(0.f, 0.f, 0.f, 0.f), d4 = l4;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (!T::kRowsQ && (e & 1) == 0) {
                            l4 = stat4(s_l2, col0 + q2 * 32 + 2 * e);
                            if (OP == XOP_DK) d4 = stat4(s_dl, col0 + q2 * 32 + 2 * e);
                        }
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
                                const float l2c = u ? ((e & 1) ? l4.w : l4.y) : ((e & 1) ? l4.z : l4.x);
                                const float dlc = u ? ((e & 1) ? d4.w : d4.y) : ((e & 1) ? d4.z : d4.x);
                                const float p = legal ? ex2_approx(fmaf(sv, c2, -l2c)) : 0.f;
                                v = (OP == XOP_DK) ? p * (__uint_as_float(y[2 * e + u]) - dlc) : p;
                            }
                            zz[u] = v;
                        }
                        z[q2 * 16 + e] = pack2<BF16>(zz[0], zz[1]);
                    }
                }
                }
            }
            // X (and Y) are read: the next score products into this buffer may start
            tc_fence_before();
            mbar_arrive(&bar_x_free[sb]);
            if (OP == XOP_DK && st_p) {
                // the P^T written to the own slot has been read by its store
                if (!warp_ok(mbar_wait(&sh.p_read, s & 1, abort_flag, status, lim, XS_ZFULL))) {
                    ok = false;
                    break;
                }
            } else if (!own_free()) {
                ok = false;
                break;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<uint4*>(sZown + half * 16384 + sw128_offset(r, u)) =
                    make_uint4(z[4 * u], z[4 * u + 1], z[4 * u + 2], z[4 * u + 3]);
            fence_proxy_async_smem();
            mbar_arrive(&bar_z_full);
            if ((C > 1 || st_ds) && ew == 0) {
                // one bulk copy of the whole slot into every peer, once all 256 threads
                // have written it (on a time-out the copies are skipped; the abort flag
                // then ends every wait of this CTA and of its peers); dK storing dS then
                // also stores the slot and reports once the store read it
                if (mbar_wait(&bar_z_full, s & 1, abort_flag, status, lim, XS_ZFULL)) {
                    for (int p = 0; p < C; ++p) {
                        if (p == c) continue;
                        bulk_copy_s2cluster(mapa_shared(smem_u32(sZ + slot_of(c, p) * 32768), p), sZown, 32768,
                                            mapa_shared(smem_u32(&bar_zpeer[slot_of(c, p)]), p));
                    }
                    if (st_ds) {
                        if (t < n_ct) {
                            tma_store_4d_hint(&tS, sZown, col_row0(t), tile_row(r0), col_head(t) - a.g0 * G, bco, pol);
                            tma_store_4d_hint(&tS, sZown + 16384, col_row0(t) + 64, tile_row(r0), col_head(t) - a.g0 * G, bco, pol);
                            bulk_commit_group();
                            bulk_wait_read_all();
                        }
                        mbar_arrive(&sh.stored);
                    }
                }
            }
        }
        // the tile stores are complete before the CTA leaves
        if ((st_ds || st_p) && ew == 0) bulk_wait_all();
        // ------------------------------------------------------ epilogue
        if (ok && n_steps > 0) {
            ok = warp_ok(mbar_wait(&bar_acc, (n_steps - 1) & 1, abort_flag, status, lim, XS_EPI));
            tc_fence_after();
        }
        float l_tot = 0.f;
        if (OP == XOP_FWD && ok && n_steps > 0) {
            // Row sum: both halves' parts (the TMA ring is idle now and serves as
            // scratch), then the CTA sums of the peers.
            float* lsum_local = reinterpret_cast<float*>(sRing);
            lsum_local[half * 128 + r] = l_part;
            mbar_arrive(&bar_half);
            ok = warp_ok(mbar_wait(&bar_half, 0, abort_flag, status, lim, XS_LSUM));
            const float l_cta = lsum_local[r] + lsum_local[128 + r];
            l_tot = l_cta;
            if (ok && C > 1) {
                if (half == 0)
                    for (int p = 0; p < C; ++p)
                        if (p != c) {
                            float* dst = stats + (2 * (C - 1) + slot_of(c, p)) * 128 + r;
                            st_async_f32(mapa_shared(smem_u32(dst), p), l_cta, mapa_shared(smem_u32(&bar_lsum), p));
                        }
                ok = warp_ok(mbar_wait_cluster(&bar_lsum, 0, abort_flag, status, lim, XS_LSUM));
                for (int q = 0; q < C - 1; ++q) l_tot += stats[(2 * (C - 1) + q) * 128 + r];
            }
        }
        if (ok) {
            float mul;
            void* out;
            View ov;
            if (OP == XOP_FWD) {
                mul = l_tot > 0.f ? 1.f / l_tot : 0.f;
                out = a.o;
                ov = pb.vo;
            } else if (OP == XOP_DQ) {
                mul = pb.scale;
                out = a.dq;
                ov = pb.vdq;
            } else if (OP == XOP_DV) {
                mul = 1.f;
                out = a.dv;
                ov = pb.vdv;
            } else {
                mul = pb.scale;
                out = a.dk;
                ov = pb.vdk;
            }
            // element offset of the output row in its (strided or packed) layout
            const size_t orow = static_cast<size_t>(bco) * ov.sb + static_cast<size_t>(row_head) * ov.sh +
                                static_cast<size_t>(row_co(row)) * ov.sn;
            uint16_t* dst = reinterpret_cast<uint16_t*>(out) + orow + d0;
            // Whole 128-row tiles leave through the idle ring (after its first KiB,
            // the forward's row-sum scratch) and one TMA store per 64-column chunk of
            // the slab: one row per thread would make every warp store touch 32 rows.
            uint8_t* ostage = sRing + 1024;
            const bool via_tma = gm.ostore && n_steps > 0 && r0 + 128 <= row_len &&
                                 1024 + nb * 16384 <= gm.stages * 16384;
            if (via_tma) {
                for (int cc = half * (sw / 2); cc < (half + 1) * (sw / 2); cc += 32) {
                    uint32_t v[32];
                    tmem_ld32(t_acc + lane_off + cc, v);
                    tmem_ld_wait(v);
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
                    uint8_t* blk = ostage + (cc >> 6) * 16384;  // chunk cc / 64: 128 rows x 128 bytes
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        *reinterpret_cast<uint4*>(blk + sw128_offset(r, ((cc & 63) >> 3) + e)) =
                            make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
                fence_proxy_async_smem();
                mbar_arrive(&sh.ostage);
                if (ew == 0) {
                    if (mbar_wait(&sh.ostage, 0, abort_flag, status, lim, XS_EPI)) {
                        for (int j = 0; j < nb; ++j)
                            tma_store_5d(&tO, ostage + j * 16384, 0, row_co(r0), c_begin + j, row_head, bco);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                }
            }
            // columns past D are not stored
            const int c_end = via_tma ? 0 : min((half + 1) * (sw / 2), pb.D - d0);
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
    // No CTA leaves while a peer may still write into its shared memory.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // launched as a dependent: do not complete before the previous grid, so
    // that work after this kernel in the stream also follows that grid
    if (threadIdx.x == 0) pdl_wait();
}

template <int OP, bool BF16, bool VARLEN>
cudaError_t launch_op(const XArgs& a, const CUtensorMap* maps, Geo gm, int n_rt, int bz, int smem, cudaStream_t s)
{
    auto kern = xchg_kernel<OP, BF16, VARLEN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gm.n_rt = n_rt;
    gm.n_bz = bz;
    cudaLaunchConfig_t cfg = {};
    if (!unit_grid(gm.C, static_cast<long long>(n_rt) * bz, &cfg.gridDim)) return cudaErrorInvalidConfiguration;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = gm.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], a,
                              gm);
}

template <int OP>
cudaError_t dispatch(const XArgs& a, const CUtensorMap* maps, const Geo& gm, int n_rt, int bz, int smem,
                     cudaStream_t s)
{
    if (a.bf16) return a.pb.varlen ? launch_op<OP, true, true>(a, maps, gm, n_rt, bz, smem, s)
                                   : launch_op<OP, true, false>(a, maps, gm, n_rt, bz, smem, s);
    return a.pb.varlen ? launch_op<OP, false, true>(a, maps, gm, n_rt, bz, smem, s)
                       : launch_op<OP, false, false>(a, maps, gm, n_rt, bz, smem, s);
}

}  // namespace

cudaError_t launch_single(int op, const XArgs& a, cudaStream_t s)
{
    const Problem& pb = a.pb;
    const bool q_empty = q_side_empty(pb), kv_empty = kv_side_empty(pb);
    const bool rows_q = (op == XOP_FWD || op == XOP_DQ);
    if (rows_q ? q_empty : kv_empty) return cudaSuccess;  // no output rows
    const int nd = (pb.D + 63) / 64;
    Geo gm;
    gm.C = (nd + 3) / 4;
    gm.slab_chunks = (nd + gm.C - 1) / gm.C;
    const int slots_bytes = gm.C * 32768;  // own slot + C-1 peer slots
    const int budget = kMaxSmem - static_cast<int>(sizeof(StaticSmem));
    // keep as many leading chunks of the first row operand resident as leave a
    // ring of >= 10 stages (they are reused by every step of the work unit; the
    // ring depth matters more than the bytes they save)
    {
        const int spare = budget - slots_bytes - stats_bytes(op, gm.C) - 10 * 16384;
        gm.res = spare > 0 ? spare / 16384 : 0;
        if (gm.res > nd) gm.res = nd;
    }
    const int fixed = gm.res * 16384 + slots_bytes + stats_bytes(op, gm.C);
    gm.stages = (kMaxSmem - static_cast<int>(sizeof(StaticSmem)) - fixed) / 16384;
    if (gm.stages > kStages) gm.stages = kStages;
    if (gm.stages < 2) return cudaErrorInvalidConfiguration;
    const int smem = fixed + gm.stages * 16384;

    // maps: A1, A2 (row side, 128-row boxes), B1, B2 (column side, 128-row boxes), W (32-row boxes)
    // An empty side has no storage: its maps are built over the other side's
    // tensor (and layout) and are never loaded from.
    struct Src {
        const void* p;
        View v;
        bool kv_side;
    };
    const Src sq = q_empty ? Src{a.k, pb.vk, true} : Src{a.q, pb.vq, false};
    const Src sdo = q_empty ? Src{a.k, pb.vk, true} : (a.dO ? Src{a.dO, pb.vdo, false} : sq);
    const Src sk = kv_empty ? Src{a.q, pb.vq, false} : Src{a.k, pb.vk, true};
    const Src sv = kv_empty ? Src{a.q, pb.vq, false} : Src{a.v, pb.vv, true};
    CUtensorMap m[8];
    bool okm = true;
    auto mk = [&](int i, const Src& x, int rows) {
        // value operand: one box of 32 rows x the slab's chunks, or (D % 64 != 0) a
        // row map read chunk by chunk
        okm = okm && (rows == 32 && pb.D % 64 == 0 ? make_slab_map(&m[i], x.p, pb, x.kv_side, a.bf16, 32, gm.slab_chunks, x.v)
                                                   : make_row_map(&m[i], x.p, pb, x.kv_side, a.bf16, rows, x.v));
    };
    int n_rt, bz;
    // dV / dK: the kv groups [g0, g0 + ng) (all unless the stored-tile backward runs in chunks)
    const int ng = a.ng > 0 ? a.ng : pb.Hkv;
    if (a.g0 < 0 || a.g0 + ng > pb.Hkv) return cudaErrorInvalidValue;
    switch (op) {
    case XOP_FWD:
        mk(0, sq, 128); mk(1, sq, 128); mk(2, sk, 128); mk(3, sk, 128); mk(4, sv, 32);
        n_rt = (pb.Nq + 127) / 128; bz = pb.B * pb.Hq;
        break;
    case XOP_DQ:
        mk(0, sq, 128); mk(1, sdo, 128); mk(2, sk, 128); mk(3, sv, 128); mk(4, sk, 32);
        n_rt = (pb.Nq + 127) / 128; bz = pb.B * pb.Hq;
        break;
    case XOP_DV:
        mk(0, sk, 128); mk(1, sk, 128); mk(2, sq, 128); mk(3, sq, 128); mk(4, sdo, 32);
        n_rt = (pb.Nkv + 127) / 128; bz = pb.B * ng;
        break;
    default:  // XOP_DK
        mk(0, sk, 128); mk(1, sv, 128); mk(2, sq, 128); mk(3, sdo, 128); mk(4, sq, 32);
        n_rt = (pb.Nkv + 127) / 128; bz = pb.B * ng;
        break;
    }
    // dK storing dS^T / P^T: those buffers as stored tiles (64 queries x 128 key rows)
    if (op == XOP_DK && a.store_ds) okm = okm && make_ds_map(&m[5], a.ds, pb, a.bf16, 128, ng * (pb.Hq / pb.Hkv));
    else m[5] = m[0];
    if (op == XOP_DK && a.store_p) okm = okm && make_ds_map(&m[6], a.p, pb, a.bf16, 128, ng * (pb.Hq / pb.Hkv));
    else m[6] = m[0];
    if (!okm) return cudaErrorInvalidValue;
    // the output as 128-row x 1-chunk boxes (whole row tiles leave through it;
    // head dims that are not whole 64-column chunks, and views the map cannot
    // describe, keep the per-row stores)
    {
        const void* out = op == XOP_FWD ? a.o : op == XOP_DQ ? a.dq : op == XOP_DV ? a.dv : a.dk;
        const View ov = op == XOP_FWD ? pb.vo : op == XOP_DQ ? pb.vdq : op == XOP_DV ? pb.vdv : pb.vdk;
        gm.ostore = (pb.D % 64 == 0 && make_slab_map(&m[7], out, pb, !rows_q, a.bf16, 128, 1, ov)) ? 1 : 0;
        if (!gm.ostore) m[7] = m[0];
    }
    if (n_rt == 0 || bz == 0) return cudaSuccess;
    switch (op) {
    case XOP_FWD: return dispatch<XOP_FWD>(a, m, gm, n_rt, bz, smem, s);
    case XOP_DQ: return dispatch<XOP_DQ>(a, m, gm, n_rt, bz, smem, s);
    case XOP_DV: return dispatch<XOP_DV>(a, m, gm, n_rt, bz, smem, s);
    default: return dispatch<XOP_DK>(a, m, gm, n_rt, bz, smem, s);
    }
}

bool xchg_uses_pair(const Problem& pb)
{
    // CTA pairs where the head dim splits into 256-column slabs without padding
    // waste and the cluster stays within 6 CTAs (measured faster there on
    // GB300); one CTA per slab otherwise. FFPA_KERNEL=pair|single overrides.
    const char* e = std::getenv("FFPA_KERNEL");
    const int forced = e == nullptr ? 0 : std::strcmp(e, "single") == 0 ? 1 : (std::strcmp(e, "pair") == 0 ? 2 : 0);
    // (head dims that are not a multiple of 64 only run in the one-CTA form)
    return pb.D % 64 == 0 && (forced ? forced == 2 : (pb.D % 128 == 0 && pb.D <= 768));
}

cudaError_t launch_xchg(int op, const XArgs& a, cudaStream_t s)
{
    return xchg_uses_pair(a.pb) ? launch_pair(op, a, s) : launch_single(op, a, s);
}

}  // namespace ffpa
