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
// When shared memory allows, the Z tiles are double-buffered (own tile and
// the copies received from the other pairs), so that producing and shipping
// Z of step s overlaps the value products of step s-1; the value products
// take the pair's own tile first, which needs no copy.
//
// Warp roles in every CTA: warp 0 TMA producer, warp 1 MMA issuer (even rank)
// or barrier forwarder (odd rank), warps 2..9 elementwise (two threads per
// TMEM row) and epilogue, warp 10 ships the own Z tile to the other pairs.
//
// Every per-step barrier is indexed by buffer and every waiter observes each
// of its phases in order, at most one phase away from the barrier's state,
// so that the parity waits are exact.
#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 352;
constexpr int kStages = 8;       // upper bound of the TMA ring depth
constexpr int kMaxC = 4;         // pairs per cluster (D <= 1024 in 256-column slabs; <= 8 CTAs)
constexpr int kSlot = 32768;     // bytes of one ring slot (one TMA box) in each CTA
constexpr float kTau = 8.0f;     // forward: rescale O only when the row max grows by more than 2^8
constexpr float kLn2 = 0.693147180559945309f;

enum Site : uint32_t {
    PS_PROD = 64, PS_A1, PS_XFREE, PS_RING, PS_ZFULL, PS_ZPEER, PS_ZPAIR, PS_XFULL, PS_RMAX, PS_ACC, PS_SLOT,
    PS_STAT, PS_LSUM, PS_EPI, PS_DRAIN, PS_FWDR, PS_COPY
};

struct PGeo {
    int C;       // pairs per cluster (= head-dim slabs of <= 256 columns)
    int stages;  // TMA ring depth
    int res;     // leading 64-wide chunks of the first row operand kept resident in shared memory
    int nbuf;    // Z buffers per slot (1 or 2)
    int nprod;   // producer lanes (ring positions are dealt round-robin)
    int n_rt;    // row tiles of 256 per (batch, head) in the grid (of the longest sequence)
    int n_bz;    // (batch, head) entries in the grid
    int ostore;  // the output map is valid: whole 128-row tiles leave through shared memory and TMA
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
    uint64_t a1, x_full[2], x_free[2], z_full[2], zpair_own[2], zpair_peer[2], acc[2];
    uint64_t zpeer[kMaxC][2], slot_free[kMaxC][2], stat[2], rmax[2], lsum, drain, half;
    uint32_t tmem_base;
    int abort_flag;
    uint32_t relay_sink[4];  // (even rank) target of the odd rank's 4-byte relay stores
    uint64_t stored[2];      // (dK storing dS) the store of the own Z buffer has read it
    uint64_t p_full[2];      // (dK storing P) the own Z buffer holds the step's P^T
    uint64_t p_read[2];      // (dK storing P) the store of that P^T has read the buffer
    uint64_t ostage;         // every elementwise thread staged its part of the output tile
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

// F8 (forward only): Q, K and P are e4m3 and the value operand is the e4m3
// transpose of V (K-major); 128-byte chunks hold 128 elements, the Z tile is
// 16 KiB, the MMAs are kind::f8f6f4 (the same 32 bytes per instruction), and
// the per-head dequantization scales enter the softmax exponent (Q, K) and
// the epilogue (V). BF16 is then the output type.
template <int OP, bool BF16, bool VARLEN, bool F8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    pair_kernel(const __grid_constant__ CUtensorMap tA1, const __grid_constant__ CUtensorMap tA2,
                const __grid_constant__ CUtensorMap tB1, const __grid_constant__ CUtensorMap tB2,
                const __grid_constant__ CUtensorMap tW, const __grid_constant__ CUtensorMap tS,
                const __grid_constant__ CUtensorMap tP, const __grid_constant__ CUtensorMap tO, const XArgs a,
                const PGeo gm)
{
    // the next GEMM kernel of a backward may take SMs as this grid's last CTAs start
    pdl_trigger();
    using T = Traits<OP>;
    const Problem& pb = a.pb;
    const int C = gm.C;
    const int rank = static_cast<int>(cluster_ctarank());
    const int c = rank >> 1;      // pair = head-dim slab
    const int rh = rank & 1;      // row half of the 256-row tile
    const bool leader = rh == 0;  // issues the pair's MMAs
    const int G = pb.Hq / pb.Hkv;

    // ------------------------------------------------------------ work unit
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
        if (!varlen_seq(pb, b, a.ctl.status, VS_PAIR, tq0, lq, tk0, lk)) return;  // uniform over the cluster
    } else {
        lq = pb.Nq;
        lk = pb.Nkv;
    }
    const int off = lk - lq;  // causal: key j legal for query i iff j <= i + off
    const int row_len = T::kRowsQ ? lq : lk;
    // causal, rows = queries: the last row tiles of a sequence see the most keys
    // and go first; rows = keys: the first key tiles see the most queries
    const int n_rt_seq = (row_len + 255) / 256;
    const int rt = (T::kRowsQ && pb.causal) ? (n_rt_seq - 1 - tile) : tile;
    const int R0 = rt * 256;            // first row of the cluster's tile
    const int r0 = R0 + 128 * rh;       // first row of this CTA
    if (rt < 0 || R0 >= row_len) return;  // uniform over the cluster, before any cluster barrier

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
        if (pb.causal) {
            m_start = max(0, R0 - off) / 128;
            // dK storing dS: start at an even query tile, so that every 256-query
            // tile of the dQ GEMM finds all of its dS blocks written (the extra
            // tile is fully masked: stored zeros)
            if (OP == XOP_DK && a.store_ds) m_start &= ~1;
        }
        n_mt = max(0, (lq + 127) / 128 - m_start);
        n_ct = G * n_mt;
    }
    const int n_steps = (n_ct + C - 1) / C;

    constexpr int kZ = F8 ? 16384 : 32768;  // bytes of one Z tile half (128 rows x 128 columns)
    const int nd = F8 ? pb.D / 128 : pb.D / 64;  // 128-byte head-dim chunks (64 or 128 elements)
    const int nb4 = (nd + 3) / 4;      // groups of four chunks (one column-operand box each)
    const int d0 = c * 256;            // first column of my pair's slab
    const int d_pad = (pb.D + 127) & ~127;
    const int sw = min(256, d_pad - d0);  // slab width: 256 or 128 (N of the value MMA)
    // first 64-wide chunk of my half of the slab's W columns; clamped so that a
    // box never starts past the head dim (columns past D are computed, never stored)
    const int w_chunk = min(d0 / 64 + rh * (sw / 128), nd - 1);

    // ------------------------------------------------------------ shared memory
    __shared__ StaticSmem sh;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int nbuf = gm.nbuf;
    uint8_t* sA1 = smem;                          // resident row-operand chunks, two per 32 KiB
    uint8_t* sZ = sA1 + (gm.res / 2) * kSlot;     // Z slots, kZ bytes each: [C-1 other pairs + own][nbuf]
    float* stats = reinterpret_cast<float*>(sZ + C * nbuf * kZ);
    uint8_t* sRing = reinterpret_cast<uint8_t*>(stats) + pair_stats_bytes(OP, C);
    if (smem_u32(smem) & 1023u) {  // uniform over the cluster: report, do not run misaligned
        if (threadIdx.x == 0) atomicCAS(a.ctl.status, 0u, 5u | (0xffu << 8));
        return;
    }

    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < gm.stages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        mbar_init(&sh.a1, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.x_full[i], 1);
            // X / Y read: the CTA's 8 elementwise warps (even rank: + the MMA thread's arming
            // arrival, whose 4 transaction bytes the odd rank's relay store completes)
            mbar_init(&sh.x_free[i], leader ? 9 : 8);
            mbar_init(&sh.stat[i], 256);
            mbar_init(&sh.rmax[i], 1);
            mbar_init(&sh.z_full[i], 256);    // own elementwise threads wrote the own Z buffer
            // (even rank) the odd rank's own Z buffer is written / it received the other
            // pairs' Z: the MMA thread's arming arrival + 4 bytes of a relay store
            mbar_init(&sh.zpair_own[i], 1);
            mbar_init(&sh.zpair_peer[i], 1);
            mbar_init(&sh.acc[i], 1);
            for (int j = 0; j < kMaxC; ++j) {
                mbar_init(&sh.zpeer[j][i], 1);
                mbar_init(&sh.slot_free[j][i], 1);
            }
        }
        mbar_init(&sh.half, 256);
        mbar_init(&sh.ostage, 256);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.stored[i], 1);
            mbar_init(&sh.p_full[i], 256);
            mbar_init(&sh.p_read[i], 1);
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
            // the relayed events of the odd rank complete 4 transaction bytes each
            for (int i = 0; i < 2; ++i) {
                mbar_arrive_expect_tx(&sh.x_free[i], 4);
                mbar_arrive_expect_tx(&sh.zpair_own[i], 4);
                mbar_arrive_expect_tx(&sh.zpair_peer[i], 4);
            }
            if (gm.res > 0 && n_steps > 0) mbar_arrive_expect_tx(&sh.a1, 2 * (gm.res / 2) * kSlot);
        }
        if (C > 1) {
            for (int i = 0; i < C - 1; ++i)
                for (int bb = 0; bb < nbuf; ++bb) mbar_arrive_expect_tx(&sh.zpeer[i][bb], kZ);
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
    auto zslot = [&](int slot, int bb) { return sZ + (slot * nbuf + bb) * kZ; };  // slot C-1 = own
    // Step s uses Z buffer s % nbuf for the (s / nbuf)-th time.
    auto zbuf = [&](int s) { return s % nbuf; };
    auto zpar = [&](int s) { return static_cast<uint32_t>((s / nbuf) & 1); };
    auto accpar = [&](int s) { return static_cast<uint32_t>((s >> 1) & 1); };  // acc[s & 1]

    // Column tile t -> (head, first row) on the column side; t past the end is
    // clamped for loading (its results are masked to zero).
    auto col_head = [&](int t) { return T::kRowsQ ? hk : hk * G + min(t, n_ct - 1) / max(n_mt, 1); };
    auto col_row0 = [&](int t) {
        const int tc = min(t, n_ct - 1);
        return T::kRowsQ ? tc * 128 : (m_start + tc % max(n_mt, 1)) * 128;
    };
    // TMA coordinates of the 5-D maps: (0, row or token, chunk, head, b or 0).
    const int bco = VARLEN ? 0 : b;
    const int row_head = T::kRowsQ ? h : hk;
    auto row_co = [&](int row) { return VARLEN ? (T::kRowsQ ? tq0 : tk0) + row : row; };
    auto col_co = [&](int row) { return VARLEN ? (T::kRowsQ ? tk0 : tq0) + row : row; };
    // key row -> row of the stored tile buffers (packed batches: sequence b's rows
    // start at cu_k[b] + 256 b, so that no tile reaches the next sequence's rows)
    auto tile_row = [&](int row) { return VARLEN ? tk0 + 256 * b + row : row; };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producers
        // Both CTAs of the pair load the same sequence of slots (each its own
        // part of every operand); every load completes on the even rank's full
        // barrier, which its MMA thread arms with both CTAs' bytes. Lanes
        // 0 .. nprod-1 issue the ring positions round-robin: the loads one thread
        // issues are served one after another, several threads keep several
        // boxes in flight at a time.
        const int me = static_cast<int>(lane_id());
        const int nprod = gm.nprod;
        if (me < nprod) {
            if (me == 0) {
                prefetch_tmap(&tA1);
                prefetch_tmap(&tB1);
                prefetch_tmap(&tW);
                if (T::kTwo) {
                    prefetch_tmap(&tA2);
                    prefetch_tmap(&tB2);
                }
            }
            RingPos rp;
            int pos = 0;  // ring positions handed out so far (both lanes)
            bool ok = true;
            auto lead_full = [&](int slot) { return mapa_shared(smem_u32(&sh.full[slot]), lead_rank); };
            // one 4-D box into the next ring position, if that position is mine
            auto put = [&](const CUtensorMap* m, int row_coord, int chunk, int head) -> bool {
                bool got = true;
                if (pos % nprod == me) {
                    got = mbar_wait(&sh.empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, PS_PROD);
                    if (got)
                        tma_load_5d_pair(sRing + rp.slot * kSlot, m, lead_full(rp.slot), 0, row_coord, chunk, head, bco);
                }
                rp.advance(gm.stages);
                ++pos;
                return got;
            };
            if (me == 0 && gm.res > 0 && n_steps > 0) {
                const uint32_t a1 = mapa_shared(smem_u32(&sh.a1), lead_rank);
                for (int j = 0; 2 * j < gm.res; ++j)
                    tma_load_5d_pair(sA1 + j * kSlot, &tA1, a1, 0, row_co(r0), 2 * j, row_head, bco);
            }
            // score operands of step s, per product and per group of four chunks q:
            // A(4q, 4q+1), B(4q .. 4q+3), A(4q+2, 4q+3)
            auto load_score = [&](int s) -> bool {
                const int t = s * C + c;
                const int hh = col_head(t), cr = col_row0(t) + 64 * rh;
                for (int prod = 0; prod < (T::kTwo ? 2 : 1); ++prod) {
                    const CUtensorMap* mA = prod ? &tA2 : &tA1;
                    const CUtensorMap* mB = prod ? &tB2 : &tB1;
                    for (int q = 0; q < nb4; ++q) {
                        if (!(prod == 0 && 4 * q < gm.res) && !put(mA, row_co(r0), 4 * q, row_head)) return false;
                        if (!put(mB, col_co(cr), 4 * q, hh)) return false;
                        if (4 * q + 2 < nd && !(prod == 0 && 4 * q + 2 < gm.res) && !put(mA, row_co(r0), 4 * q + 2, row_head))
                            return false;
                    }
                }
                return true;
            };
            // value operand of step s: per column tile (own pair's tile first), one
            // box of the tile's 128 keys x my two 64-wide chunks of the slab
            // (F8: one 16 KiB box of my 128 head-dim rows of V^T x the tile's 128
            // keys, two tiles per slot, the second repeated when C is odd)
            auto load_value = [&](int s) -> bool {
                if constexpr (F8) {
                    const int vt_row = d0 + rh * (sw / 2);  // my half of the slab's V^T rows
                    // V^T column of a key row of the sequence (packed: sequence b's keys
                    // start at column 16 ceil(cu_k[b] / 16) + 16 b)
                    const int vt0 = VARLEN ? 16 * ((tk0 + 15) / 16) + 16 * b : 0;
                    for (int k = 0; k < C; k += 2) {
                        const int ta = s * C + (c + k) % C;
                        const int tb = s * C + (c + min(k + 1, C - 1)) % C;
                        bool got = true;
                        if (pos % nprod == me) {
                            got = mbar_wait(&sh.empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, PS_PROD);
                            if (got) {
                                uint8_t* dst = sRing + rp.slot * kSlot;
                                tma_load_4d_pair(dst, &tW, lead_full(rp.slot), vt0 + col_row0(ta), vt_row,
                                                 col_head(ta), bco);
                                tma_load_4d_pair(dst + 16384, &tW, lead_full(rp.slot), vt0 + col_row0(tb), vt_row,
                                                 col_head(tb), bco);
                            }
                        }
                        rp.advance(gm.stages);
                        ++pos;
                        if (!got) return false;
                    }
                    return true;
                } else {
                    for (int k = 0; k < C; ++k) {
                        const int t = s * C + (c + k) % C;
                        const int hh = col_head(t);
                        if (!put(&tW, col_co(col_row0(t)), w_chunk, hh)) return false;
                    }
                    return true;
                }
            };
            if (n_steps > 0) ok = load_score(0);
            for (int s = 0; ok && s < n_steps; ++s) {
                if (s + 1 < n_steps) ok = load_score(s + 1);
                if (ok) ok = load_value(s);
            }
            // No CTA leaves with loads in flight: the MMA thread releases a slot only
            // after its data landed in both CTAs and was consumed.
            const int last = min(pos, gm.stages);
            RingPos dp = rp;
            for (int i = 0; i < last; ++i) {
                dp.retreat(gm.stages);
                if ((pos - 1 - i) % nprod != me) continue;
                int dummy = 0;
                if (!mbar_wait(&sh.empty[dp.slot], dp.phase, &dummy, status, lim, PS_DRAIN, false)) break;
            }
        }
    } else if (warp == 1) {
        if (leader) {
            // -------------------------------------------------- MMA issuer (pair)
            if (elect_one()) {
                // (F8: format code 0 = e4m3 in both operand fields; V^T is K-major)
                const uint32_t idesc_s = idesc_f16(256, 128, F8 ? false : BF16, false, false);
                const uint32_t idesc_v = idesc_f16(256, sw, F8 ? false : BF16, false, !F8);
                auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t id, uint32_t acc) {
                    if constexpr (F8)
                        umma_f8_pair(d, ad, bd, id, acc);
                    else
                        umma_f16_pair(d, ad, bd, id, acc);
                };
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
                    for (int prod = 0; prod < (T::kTwo ? 2 : 1); ++prod) {
                        // XDB: buffer sb last held X of step s-2 (read by then); two-product
                        // kernels: X (prod 0) and Y (prod 1) of step s-1, released separately
                        const int fb = T::kTwo ? prod : sb;
                        if (T::kXdb ? s >= 2 : s >= 1) {
                            const uint32_t par = T::kXdb ? (((s - 2) >> 1) & 1) : ((s - 1) & 1);
                            if (!mbar_wait_cluster(&sh.x_free[fb], par, abort_flag, status, lim, PS_XFREE)) return false;
                            mbar_arrive_expect_tx(&sh.x_free[fb], 4);  // arm the next phase's relay
                            tc_fence_after();
                        }
                        const uint32_t dst = t_x0 + (T::kXdb ? sb * 128 : prod * 128);
                        for (int q = 0; q < nb4; ++q) {
                            // A slots hold chunks (4q, 4q+1) and (4q+2, 4q+3), 128 rows each;
                            // the B slot holds chunks 4q .. 4q+3, 64 rows each
                            const uint8_t* B = nullptr;
                            int b_slot = -1;
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const int d_first = 4 * q + 2 * h2;
                                if (d_first >= nd) break;
                                const uint8_t* A;
                                int a_slot = -1;
                                if (prod == 0 && d_first < gm.res) {
                                    A = sA1 + (d_first / 2) * kSlot;
                                } else {
                                    A = take();
                                    if (!A) return false;
                                    a_slot = rp.slot;
                                    rp.advance(gm.stages);
                                }
                                if (h2 == 0) {
                                    B = take();
                                    if (!B) return false;
                                    b_slot = rp.slot;
                                    rp.advance(gm.stages);
                                }
                                // one descriptor per tile, stepped by offsets (K-major, 32 bytes per MMA)
                                const uint64_t da = sdesc_sw128(smem_u32(A), 16, 1024);
                                const uint64_t db = sdesc_sw128(smem_u32(B), 16, 1024);
                                for (int u2 = 0; u2 < 2; ++u2) {
                                    const int d = d_first + u2;
                                    if (d >= nd) break;
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        mma(dst, sdesc_advance(da, u2 * 16384 + kk * 32),
                                            sdesc_advance(db, (2 * h2 + u2) * 8192 + kk * 32), idesc_s, (d | kk) != 0);
                                }
                                if (a_slot >= 0) give(a_slot);
                            }
                            give(b_slot);
                        }
                        // two-product kernels: X and Y are announced separately
                        if (T::kTwo) umma_commit_pair_multicast(&sh.x_full[prod], pair_mask);
                    }
                    if (!T::kTwo) umma_commit_pair_multicast(&sh.x_full[sb], pair_mask);
                    return true;
                };
                auto issue_value = [&](int s) -> bool {
                    const int bb = zbuf(s);
                    const uint8_t* w8 = nullptr;  // F8: the slot holding V^T of two tiles
                    const uint32_t par = zpar(s);
                    // own tile: written by both CTAs' elementwise threads
                    if (!mbar_wait(&sh.z_full[bb], par, abort_flag, status, lim, PS_ZFULL)) return false;
                    if (!mbar_wait_cluster(&sh.zpair_own[bb], par, abort_flag, status, lim, PS_ZPAIR)) return false;
                    mbar_arrive_expect_tx(&sh.zpair_own[bb], 4);  // arm the next phase's relay
                    tc_fence_after();
                    for (int k = 0; k < C; ++k) {
                        const int cc = (c + k) % C;
                        const uint8_t* zs = zslot(k == 0 ? C - 1 : slot_of(cc, c), bb);
                        if (k > 0) {
                            // another pair's tile: landed here and (forwarded) in the odd rank
                            if (!mbar_wait_cluster(&sh.zpeer[slot_of(cc, c)][bb], par, abort_flag, status, lim, PS_ZPEER))
                                return false;
                            // arm the buffer's next use before this step's slot_free lets the writer in
                            mbar_arrive_expect_tx(&sh.zpeer[slot_of(cc, c)][bb], kZ);
                            if (k == 1) {
                                if (!mbar_wait_cluster(&sh.zpair_peer[bb], par, abort_flag, status, lim, PS_ZPAIR))
                                    return false;
                                mbar_arrive_expect_tx(&sh.zpair_peer[bb], 4);  // arm the next phase's relay
                            }
                            tc_fence_after();
                        }
                        if constexpr (F8) {
                            // two tiles per slot: V^T of tile k at byte (k & 1) * 16 KiB
                            if ((k & 1) == 0) {
                                w8 = take();
                                if (!w8) return false;
                            }
                            const uint8_t* W = w8 + (k & 1) * 16384;
                            const uint64_t dz = sdesc_sw128(smem_u32(zs), 16, 1024);
                            const uint64_t dw = sdesc_sw128(smem_u32(W), 16, 1024);
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                // keys 32 t of the tile: 32 bytes into Z's and V^T's 128-byte rows
                                const uint32_t acc = (s | k | t) != 0;
                                mma(t_acc, sdesc_advance(dz, t * 32), sdesc_advance(dw, t * 32), idesc_v, acc);
                            }
                            if ((k & 1) == 1 || k == C - 1) {
                                give(rp.slot);
                                rp.advance(gm.stages);
                            }
                        } else {
                            const uint8_t* W = take();
                            if (!W) return false;
                            const uint64_t dz = sdesc_sw128(smem_u32(zs), 16, 1024);
                            const uint64_t dw = sdesc_sw128(smem_u32(W), 128 * 128, 1024);
#pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                // keys 16 t of the tile: Z chunk t / 4, W rows 16 t (MN-major,
                                // 64-column blocks 128 keys x 128 bytes apart)
                                const uint32_t acc = (s | k | t) != 0;
                                umma_f16_pair(t_acc, sdesc_advance(dz, (t >> 2) * 16384 + (t & 3) * 32),
                                              sdesc_advance(dw, t * 2048), idesc_v, acc);
                            }
                            give(rp.slot);
                            rp.advance(gm.stages);
                        }
                        // pair cc may overwrite its copy in this buffer once these MMAs are done
                        if (k > 0) umma_commit_pair_multicast(&sh.slot_free[c][bb], static_cast<uint16_t>(3u << (2 * cc)));
                    }
                    umma_commit_pair_multicast(&sh.acc[s & 1], pair_mask);
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
        } else {
            // -------------------------------------------------- forwarder (odd rank)
            // Relays this CTA's events to the even rank's MMA thread, so that the
            // elementwise warps only ever arrive on barriers of their own CTA: X
            // (and Y) read, own Z buffer written, and (C > 1) the other pairs' Z
            // tiles landed here. Each kind of event is forwarded in step order; the
            // kinds are polled together so that a late one does not hold back the
            // others. A relay is a 4-byte st.async into the even rank, whose
            // complete-tx (release at cluster scope, after this thread's acquire of
            // the local event) finishes the phase that the MMA thread armed; unlike
            // a remote arrive it does not hold this thread until it lands.
            if (elect_one()) {
                const uint32_t sink = mapa_shared(smem_u32(&sh.relay_sink[0]), lead_rank);
                auto relay = [&](uint64_t* bar) { st_async_f32(sink, 0.f, mapa_shared(smem_u32(bar), lead_rank)); };
                const int n_x = T::kTwo ? 2 * n_steps : n_steps;
                int nx = 0, nz = 0, np = 0, kp = 1;
                uint64_t t_last = global_timer_ns();
                for (uint32_t it = 1; nx < n_x || nz < n_steps || (C > 1 && np < n_steps); ++it) {
                    bool progress = false;
                    if (nx < n_x) {
                        // event nx: X buffer nx & 1 of step nx (forward, dV), or X (even nx) /
                        // Y (odd nx) of step nx / 2 (dK, dQ); both reach phase (nx / 2) & 1
                        const int idx = nx & 1;
                        const uint32_t par = static_cast<uint32_t>((nx >> 1) & 1);
                        if (mbar_test(&sh.x_free[idx], par)) {
                            relay(&sh.x_free[idx]);
                            ++nx;
                            progress = true;
                        }
                    }
                    if (nz < n_steps && mbar_test(&sh.z_full[zbuf(nz)], zpar(nz))) {
                        relay(&sh.zpair_own[zbuf(nz)]);
                        ++nz;
                        progress = true;
                    }
                    if (C > 1 && np < n_steps) {
                        // the other pairs' tiles of step np, in pair order c+1, c+2, ...
                        const int bb = zbuf(np);
                        const int p = (c + kp) % C;
                        uint64_t* zb = &sh.zpeer[slot_of(p, c)][bb];
                        if (mbar_test_cluster(zb, zpar(np))) {
                            mbar_arrive_expect_tx(zb, kZ);  // arm the buffer's next use
                            progress = true;
                            if (++kp == C) {
                                relay(&sh.zpair_peer[bb]);
                                kp = 1;
                                ++np;
                            }
                        }
                    }
                    if (progress) {
                        t_last = global_timer_ns();
                    } else if ((it & 63u) == 0) {
                        if (*abort_flag || *reinterpret_cast<volatile uint32_t*>(status) != 0u) {
                            *abort_flag = 1;
                            break;
                        }
                        if (global_timer_ns() - t_last > lim) {
                            *abort_flag = 1;
                            const uint32_t blk = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
                            atomicCAS(status, 0u, DEV_TIMEOUT | (PS_FWDR << 8) | (blk << 16));
                            break;
                        }
                    }
                }
            }
        }
    } else if (warp == 10) {
        // ------------------------------------------------------ Z copier
        // Ships the own Z tile of every step, once all 256 elementwise threads
        // wrote it, into the CTA of every other pair that holds my rows, as one
        // bulk copy each, once that pair's value products consumed the previous
        // copy in the target buffer. The dK kernel that stores dS then also writes
        // the tile (dS^T: my 128 key rows x the tile's 128 queries) to that buffer
        // with two TMA stores and reports when they have read it; the dK kernel
        // that stores P does the same, earlier in the step, with the P^T tile the
        // elementwise threads put in the buffer before dS.
        const bool store_ds = OP == XOP_DK && a.store_ds != 0;
        const bool store_p = OP == XOP_DK && a.store_p != 0;
        if ((C > 1 || store_ds || store_p) && elect_one()) {
            if (store_ds) prefetch_tmap(&tS);
            if (store_p) prefetch_tmap(&tP);
            // the stored tiles are read by later launches, after many more were
            // written: they leave L2 before the operand tiles this kernel reuses
            const uint64_t pol = l2_policy_evict_first();
            for (int s = 0; s < n_steps; ++s) {
                const int bb = zbuf(s);
                const int t = s * C + c;
                const uint8_t* zown_base = zslot(C - 1, bb);
                bool ok = true;
                if (store_p) {
                    ok = mbar_wait(&sh.p_full[bb], zpar(s), abort_flag, status, lim, PS_COPY);
                    if (ok) {
                        if (t < n_ct) {
                            tma_store_4d_hint(&tP, zown_base, col_row0(t), tile_row(r0), col_head(t) - a.g0 * G, bco, pol);
                            tma_store_4d_hint(&tP, zown_base + 16384, col_row0(t) + 64, tile_row(r0), col_head(t) - a.g0 * G, bco,
                                              pol);
                            bulk_commit_group();
                            bulk_wait_read_all();
                        }
                        mbar_arrive(&sh.p_read[bb]);
                    }
                }
                if (ok) ok = mbar_wait(&sh.z_full[bb], zpar(s), abort_flag, status, lim, PS_COPY);
                // the exchange first (the other pairs' value products wait for it)
                for (int k = 1; k < C && ok; ++k) {
                    const int p = (c + k) % C;
                    if (s >= nbuf)
                        ok = mbar_wait_cluster(&sh.slot_free[p][bb], zpar(s) ^ 1u, abort_flag, status, lim, PS_SLOT);
                    if (ok)
                        bulk_copy_s2cluster(mapa_shared(smem_u32(zslot(slot_of(c, p), bb)), xrank(p)), zown_base,
                                            kZ, mapa_shared(smem_u32(&sh.zpeer[slot_of(c, p)][bb]), xrank(p)));
                }
                if (ok && store_ds) {
                    if (t < n_ct) {
                        tma_store_4d_hint(&tS, zown_base, col_row0(t), tile_row(r0), col_head(t) - a.g0 * G, bco, pol);
                        tma_store_4d_hint(&tS, zown_base + 16384, col_row0(t) + 64, tile_row(r0), col_head(t) - a.g0 * G, bco, pol);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                    mbar_arrive(&sh.stored[bb]);
                }
                if (!ok) break;
            }
            if (store_ds || store_p) bulk_wait_all();  // the stores are complete before the CTA leaves
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
        // F8: S = sq * sk * (Q8 K8^T), so the dequantization scales join the exponent
        const float c2 = F8 ? pb.scale_log2 * a.f8_sq[static_cast<size_t>(b) * pb.Hq + h] *
                                  a.f8_sk[static_cast<size_t>(b) * pb.Hkv + hk]
                            : pb.scale_log2;
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
        // dV / dK: column statistic of tile t for column r, fetched one step ahead
        // (half 0: lse2, +inf past the sequence or the last tile; half 1: delta)
        auto fetch_stat = [&](int t) -> float {
            const int qi = col_row0(t) + r;
            const int hh = col_head(t);
            if (t < n_ct && qi < lq) {
                const size_t si = VARLEN ? static_cast<size_t>(hh) * pb.total_q + tq0 + qi
                                         : (static_cast<size_t>(b) * pb.Hq + hh) * pb.Nq + qi;
                return half == 0 ? a.lse_log2[si] : a.delta[si];
            }
            return half == 0 ? INFINITY : 0.f;
        };
        float stat_next = (!T::kRowsQ && n_steps > 0) ? fetch_stat(c) : 0.f;
        // Own buffer zbuf(s) was last used at step s - nbuf: it may be rewritten once
        // the value MMAs of that step (acc, observed here at every step, in order)
        // and the copies of it (slot_free of every other pair: it consumed the copy,
        // so the copy has read the buffer) are done, and (dK storing dS) the store
        // of that step's dS has read it.
        auto own_free = [&](int s) -> bool {
            if (s < nbuf) return true;
            const int sp = s - nbuf, bb = zbuf(s);
            bool got = mbar_wait(&sh.acc[sp & 1], accpar(sp), abort_flag, status, lim, PS_ACC);
            for (int p = 0; p < C && got; ++p)
                if (p != c) got = mbar_wait_cluster(&sh.slot_free[p][bb], zpar(sp), abort_flag, status, lim, PS_SLOT);
            if (got && OP == XOP_DK && a.store_ds) got = mbar_wait(&sh.stored[bb], zpar(sp), abort_flag, status, lim, PS_COPY);
            return warp_ok(got);
        };
        for (int s = 0; s < n_steps; ++s) {
            const int t = s * C + c;
            const int sb = T::kXdb ? (s & 1) : 0;
            const uint32_t tx = t_x0 + sb * 128 + lane_off;
            const uint32_t ty = t_x0 + 128 + lane_off;  // Y (two-product kernels)
            const int sbuf = s & 1;
            if (!T::kRowsQ) {
                // stage the column statistics of tile t: lse2[sbuf][r] (half 0, +inf
                // masks queries past the sequence and tiles past the end) and
                // delta[sbuf][r] (half 1); then fetch those of the next step
                stats[half * 256 + sbuf * 128 + r] = stat_next;
                mbar_arrive(&sh.stat[sbuf]);
                if (s + 1 < n_steps) stat_next = fetch_stat(t + C);
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
                // row maximum over the other half's 64 columns, then over mine, which
                // stay in registers for P (two batched loads, two waits)
                uint32_t xa[32], xb[32];
                const int colp = 64 - col0;
                tmem_ld32(tx + colp, xa);
                tmem_ld32(tx + colp + 32, xb);
                tmem_ld_wait(xa, xb);
                float mx = -INFINITY;
                auto max32 = [&](const uint32_t (&x)[32], int c_first) {
                    if (limit >= c_first + 32) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(x[j]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c_first + j < limit) mx = fmaxf(mx, __uint_as_float(x[j]));
                    }
                };
                max32(xa, colp);
                max32(xb, colp + 32);
                tmem_ld32(tx + col0, xa);
                tmem_ld32(tx + col0 + 32, xb);
                tmem_ld_wait(xa, xb);
                max32(xa, col0);
                max32(xb, col0 + 32);
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
                    if (s > 0 && !warp_ok(mbar_wait(&sh.acc[(s - 1) & 1], accpar(s - 1), abort_flag, status, lim, PS_ACC))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int half_w = sw / 2;
                    for (int cc = half * half_w; cc < (half + 1) * half_w; cc += 16) {
                        uint32_t o[16];
                        tmem_ld16(t_acc + lane_off + cc, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st16(t_acc + lane_off + cc, o);
                    }
                    tmem_st_wait();
                }
                l_part *= alpha;
                m_ref = new_ref;
                const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
                float sum = 0.f;
                // 16-bit P: z[q2 * 16 + e] holds columns 2e, 2e+1 of my q2-th 32; e4m3 P
                // (F8): z[q2 * 8 + e / 2] holds columns 4(e/2) .. 4(e/2)+3, low byte first
                uint32_t pend = 0;  // F8: the low half of z[q2 * 8 + e / 2], written at odd e
                auto put_p = [&](int q2, int e, float p0, float p1) {
                    if constexpr (F8) {
                        const uint32_t v = cvt_e4m3x2(p0, p1);
                        if (e & 1)
                            z[q2 * 8 + (e >> 1)] = pend | (v << 16);
                        else
                            pend = v;
                    } else {
                        z[q2 * 16 + e] = pack2<BF16>(p0, p1);
                    }
                };
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    const uint32_t (&x)[32] = q2 ? xb : xa;
                    const int lim2 = limit - col0 - q2 * 32;
                    if (lim2 >= 32) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float p0 = ex2_approx(fmaf(__uint_as_float(x[2 * e]), c2, -mu));
                            const float p1 = ex2_approx(fmaf(__uint_as_float(x[2 * e + 1]), c2, -mu));
                            sum += p0 + p1;
                            put_p(q2, e, p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float p0 = (2 * e < lim2) ? ex2_approx(fmaf(__uint_as_float(x[2 * e]), c2, -mu)) : 0.f;
                            const float p1 = (2 * e + 1 < lim2) ? ex2_approx(fmaf(__uint_as_float(x[2 * e + 1]), c2, -mu)) : 0.f;
                            sum += p0 + p1;
                            put_p(q2, e, p0, p1);
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
                if constexpr (!T::kTwo) {
                    // dV: Z = P^T of my 64 columns
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
                            float zz[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int j = col0 + q2 * 32 + 2 * e + u;
                                const bool legal = full || (j >= j_lo && j < j_hi);
                                zz[u] = legal ? ex2_approx(fmaf(__uint_as_float(x[2 * e + u]), c2, -l2e[u])) : 0.f;
                            }
                            z[q2 * 16 + e] = pack2<BF16>(zz[0], zz[1]);
                        }
                    }
                } else {
                    // dK / dQ: P of my 64 columns from X, kept as fp16 pairs until dP is read
                    uint32_t pp[32];
                    {
                    uint32_t xa[32], xb[32];
                    tmem_ld32(tx + col0, xa);
                    tmem_ld32(tx + col0 + 32, xb);
                    tmem_ld_wait(xa, xb);
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const uint32_t (&x)[32] = q2 ? xb : xa;
                        float4 l4 = make_float4(l2_row, l2_row, l2_row, l2_row);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if (!T::kRowsQ && (e & 1) == 0) l4 = stat4(s_l2, col0 + q2 * 32 + 2 * e);
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
                    }
                    // X is read: the pair's next S product may start while dP is processed
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.x_free[0]);
                    if (OP == XOP_DK && a.store_p) {
                        // dK storing P: P^T (input dtype) goes through the own buffer first;
                        // the copier stores it while dP^T is computed, then dS^T replaces it
                        if (!own_free(s)) {
                            ok = false;
                            break;
                        }
                        uint8_t* zp = zslot(C - 1, zbuf(s)) + half * 16384;
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 pv = unpack2<false>(pp[4 * u + e]);
                                w[e] = pack2<BF16>(pv.x, pv.y);
                            }
                            *reinterpret_cast<uint4*>(zp + sw128_offset(r, u)) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(&sh.p_full[zbuf(s)]);
                    }
                    if (!warp_ok(mbar_wait(&sh.x_full[1], s & 1, abort_flag, status, lim, PS_XFULL))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // dQ: dS = P (dP - delta) with the row's statistics;
                    // dK: dS^T = P^T (dP^T - delta) with the columns' statistics
                    uint32_t ya[32], yb[32];
                    tmem_ld32(ty + col0, ya);
                    tmem_ld32(ty + col0 + 32, yb);
                    tmem_ld_wait(ya, yb);
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const uint32_t (&y)[32] = q2 ? yb : ya;
                        float4 d4 = make_float4(dl_row, dl_row, dl_row, dl_row);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float2 pv = unpack2<false>(pp[q2 * 16 + e]);
                            if (!T::kRowsQ && (e & 1) == 0) d4 = stat4(s_dl, col0 + q2 * 32 + 2 * e);
                            const float d0v = (e & 1) ? d4.z : d4.x;
                            const float d1v = (e & 1) ? d4.w : d4.y;
                            z[q2 * 16 + e] = pack2<BF16>(pv.x * (__uint_as_float(y[2 * e]) - d0v),
                                                         pv.y * (__uint_as_float(y[2 * e + 1]) - d1v));
                        }
                    }
                }
            }
            // X (dK / dQ: Y) is read: the pair's next score product into this buffer may start
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.x_free[(T::kTwo || sb) ? 1 : 0]);
            const int bb = zbuf(s);
            uint8_t* zown = zslot(C - 1, bb);
            if (OP == XOP_DK && a.store_p) {
                // the P^T of this step, written to the buffer earlier, has been read by its store
                if (!warp_ok(mbar_wait(&sh.p_read[bb], zpar(s), abort_flag, status, lim, PS_COPY))) {
                    ok = false;
                    break;
                }
            } else if (!own_free(s)) {
                ok = false;
                break;
            }
            if constexpr (F8) {
                // one 128-byte row of 128 e4m3 values: my 64 columns are 16-byte units 4 half .. 4 half + 3
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4*>(zown + sw128_offset(r, 4 * half + u)) =
                        make_uint4(z[4 * u], z[4 * u + 1], z[4 * u + 2], z[4 * u + 3]);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<uint4*>(zown + half * 16384 + sw128_offset(r, u)) =
                        make_uint4(z[4 * u], z[4 * u + 1], z[4 * u + 2], z[4 * u + 3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&sh.z_full[bb]);
        }
        // ------------------------------------------------------ epilogue
        if (ok && n_steps > 0) {
            // the last two steps' value MMAs, in order (earlier ones were observed above)
            if (n_steps >= 2) ok = warp_ok(mbar_wait(&sh.acc[n_steps & 1], accpar(n_steps - 2), abort_flag, status, lim, PS_EPI));
            if (ok) ok = warp_ok(mbar_wait(&sh.acc[(n_steps - 1) & 1], accpar(n_steps - 1), abort_flag, status, lim, PS_EPI));
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
            View ov;
            if (OP == XOP_FWD) {
                mul = l_tot > 0.f ? 1.f / l_tot : 0.f;
                if constexpr (F8) mul *= a.f8_sv[static_cast<size_t>(b) * pb.Hkv + hk];  // O = sv * (P V8) / l
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
            // the forward's row-sum scratch) and TMA stores of 128 rows x 128
            // columns: one row per thread would make every warp store touch 32 rows.
            // Columns past the (real) head dim fall outside the map.
            uint8_t* ostage = sRing + 1024;
            const bool via_tma = gm.ostore && n_steps > 0 && r0 + 128 <= row_len &&
                                 1024 + 128 * sw * 2 <= gm.stages * kSlot;
            if (via_tma) {
                // one 64-column chunk per round: two TMEM loads, one wait
                for (int cc = half * (sw / 2); cc < (half + 1) * (sw / 2); cc += 64) {
                    uint32_t va[32], vb[32];
                    tmem_ld32(t_acc + lane_off + cc, va);
                    tmem_ld32(t_acc + lane_off + cc + 32, vb);
                    tmem_ld_wait(va, vb);
                    // box cc / 128 holds 64-column chunks 2 q, 2 q + 1 of the slab, 16 KiB each
                    uint8_t* blk = ostage + (cc >> 7) * 32768 + ((cc >> 6) & 1) * 16384;
#pragma unroll
                    for (int p2 = 0; p2 < 2; ++p2) {
                        const uint32_t (&v)[32] = p2 ? vb : va;
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<uint4*>(blk + sw128_offset(r, 4 * p2 + e)) =
                                make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&sh.ostage);
                if (ew == 0) {
                    if (mbar_wait(&sh.ostage, 0, abort_flag, status, lim, PS_EPI)) {
                        for (int q = 0; q < sw / 128; ++q)
                            tma_store_5d(&tO, ostage + q * 32768, 0, row_co(r0), d0 / 64 + 2 * q, row_head, bco);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                }
            }
            // columns past the output's head dim are not stored
            const int c_end = via_tma ? 0 : min((half + 1) * (sw / 2), (a.d_out > 0 ? a.d_out : pb.D) - d0);
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
    // launched as a dependent: do not complete before the previous grid, so
    // that work after this kernel in the stream also follows that grid
    if (threadIdx.x == 0) pdl_wait();
}

template <int OP, bool BF16, bool VARLEN, bool F8 = false>
cudaError_t launch_op(const XArgs& a, const CUtensorMap* maps, PGeo gm, int n_rt, int bz, int smem, cudaStream_t s)
{
    auto kern = pair_kernel<OP, BF16, VARLEN, F8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gm.n_rt = n_rt;
    gm.n_bz = bz;
    cudaLaunchConfig_t cfg = {};
    if (!unit_grid(2 * gm.C, static_cast<long long>(n_rt) * bz, &cfg.gridDim)) return cudaErrorInvalidConfiguration;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * gm.C;
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
    if (pb.D % 64 != 0) return cudaErrorInvalidConfiguration;  // chunked 5-D maps need D % 64 == 0
    // FP8 forward: the head dim padded to whole 128-column chunks (1 to 4 pairs)
    const bool f8 = a.f8 != 0;
    if (f8 && (op != XOP_FWD || pb.D % 128 != 0 || pb.D > 1024)) return cudaErrorInvalidConfiguration;
    const int nd = f8 ? pb.D / 128 : pb.D / 64;  // 128-byte chunks
    const int zb = f8 ? 16384 : 32768;           // bytes of one Z tile half
    const int d_pad = (pb.D + 127) & ~127;
    PGeo gm;
    gm.C = (d_pad + 255) / 256;
    if (gm.C > kMaxC) return cudaErrorInvalidConfiguration;
    const int budget = kMaxSmem - static_cast<int>(sizeof(StaticSmem));
    // double-buffer the Z slots when that leaves a ring of >= 4 stages
    gm.nbuf = (budget - 2 * gm.C * zb - pair_stats_bytes(op, gm.C) >= 4 * kSlot) ? 2 : 1;
    const int slots_bytes = gm.nbuf * gm.C * zb;
    gm.nprod = 2;  // measured on GB300: 2 lanes beat 1, 3 and 4 with 32 KiB boxes
    // keep as many leading chunk pairs of the first row operand resident as leave
    // a ring of >= 5 stages (they are reused by every step of the work unit)
    {
        const int spare = budget - slots_bytes - pair_stats_bytes(op, gm.C) - 5 * kSlot;
        gm.res = spare > 0 ? 2 * (spare / kSlot) : 0;
        if (gm.res > ((nd + 1) & ~1)) gm.res = (nd + 1) & ~1;
    }
    const int fixed = (gm.res / 2) * kSlot + slots_bytes + pair_stats_bytes(op, gm.C);
    gm.stages = (budget - fixed) / kSlot;
    if (gm.stages > kStages) gm.stages = kStages;
    if (gm.stages < 2) return cudaErrorInvalidConfiguration;
    const int smem = fixed + gm.stages * kSlot;

    // maps (one 32 KiB box each): A1, A2 (row side, 128 rows x 2 chunks), B1, B2
    // (column side, 64 rows x 4 chunks), W (column side, 128 rows x 2 chunks)
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
    auto row = [&](int i, const Src& x) { okm = okm && make_slab_map(&m[i], x.p, pb, x.kv_side, a.bf16, 128, 2, x.v); };
    auto col = [&](int i, const Src& x) { okm = okm && make_slab_map(&m[i], x.p, pb, x.kv_side, a.bf16, 64, 4, x.v); };
    auto val = [&](int i, const Src& x) { okm = okm && make_slab_map(&m[i], x.p, pb, x.kv_side, a.bf16, 128, 2, x.v); };
    int n_rows;
    int bz;
    // dV / dK: the kv groups [g0, g0 + ng) (all unless the stored-tile backward runs in chunks)
    const int ng = a.ng > 0 ? a.ng : pb.Hkv;
    if (a.g0 < 0 || a.g0 + ng > pb.Hkv) return cudaErrorInvalidValue;
    if (f8) {
        // e4m3 codes: q8 (rows), k8 (columns), V^T (value operand, 128 head-dim rows per CTA);
        // packed batches: one batch entry of all tokens, V^T over all ldv columns
        // (the gaps between sequences hold zero codes)
        const int b8 = pb.varlen ? 1 : pb.B;
        okm = make_u8_slab_map(&m[0], a.q, b8, pb.Hq, pb.varlen ? pb.total_q : pb.Nq, pb.D, 128, 2) &&
              make_u8_slab_map(&m[2], a.k, b8, pb.Hkv, pb.varlen ? pb.total_k : pb.Nkv, pb.D, 64, 4) &&
              make_vt_map(&m[4], a.v8t, b8, pb.Hkv, pb.D, pb.varlen ? a.ldv : pb.Nkv, a.ldv, 128);
        m[1] = m[0];
        m[3] = m[2];
        m[5] = m[0];
        m[6] = m[0];
        if (!okm) return cudaErrorInvalidValue;
        // O (the input dtype, the real head dim) as 128-row x 2-chunk boxes
        {
            Problem po = pb;
            po.D = a.d_out > 0 ? a.d_out : pb.D;
            gm.ostore = (po.D % 64 == 0 && make_slab_map(&m[7], a.o, po, false, a.bf16, 128, 2, pb.vo)) ? 1 : 0;
            if (!gm.ostore) m[7] = m[0];
        }
        const int n_rt8 = (pb.Nq + 255) / 256;
        const int bz8 = pb.B * pb.Hq;
        if (n_rt8 == 0 || bz8 == 0) return cudaSuccess;
        if (pb.varlen)
            return a.bf16 ? launch_op<XOP_FWD, true, true, true>(a, m, gm, n_rt8, bz8, smem, s)
                          : launch_op<XOP_FWD, false, true, true>(a, m, gm, n_rt8, bz8, smem, s);
        return a.bf16 ? launch_op<XOP_FWD, true, false, true>(a, m, gm, n_rt8, bz8, smem, s)
                      : launch_op<XOP_FWD, false, false, true>(a, m, gm, n_rt8, bz8, smem, s);
    }
    switch (op) {
    case XOP_FWD:
        row(0, sq); row(1, sq); col(2, sk); col(3, sk); val(4, sv);
        n_rows = pb.Nq; bz = pb.B * pb.Hq;
        break;
    case XOP_DQ:
        row(0, sq); row(1, sdo); col(2, sk); col(3, sv); val(4, sk);
        n_rows = pb.Nq; bz = pb.B * pb.Hq;
        break;
    case XOP_DV:
        row(0, sk); row(1, sk); col(2, sq); col(3, sq); val(4, sdo);
        n_rows = pb.Nkv; bz = pb.B * ng;
        break;
    default:  // XOP_DK
        row(0, sk); row(1, sv); col(2, sq); col(3, sdo); val(4, sq);
        n_rows = pb.Nkv; bz = pb.B * ng;
        break;
    }
    // dK storing dS: the dS^T buffer as stored tiles (64 queries x 128 key rows)
    if (op == XOP_DK && a.store_ds) okm = okm && make_ds_map(&m[5], a.ds, pb, a.bf16, 128, ng * (pb.Hq / pb.Hkv));
    else m[5] = m[0];
    // dK storing P: the P^T buffer, the same layout
    if (op == XOP_DK && a.store_p) okm = okm && make_ds_map(&m[6], a.p, pb, a.bf16, 128, ng * (pb.Hq / pb.Hkv));
    else m[6] = m[0];
    if (!okm) return cudaErrorInvalidValue;
    // the output as 128-row x 2-chunk boxes (the kernel stores whole row tiles
    // through it; a view the map cannot describe keeps the per-row stores)
    {
        const void* out = op == XOP_FWD ? a.o : op == XOP_DQ ? a.dq : op == XOP_DV ? a.dv : a.dk;
        const View ov = op == XOP_FWD ? pb.vo : op == XOP_DQ ? pb.vdq : op == XOP_DV ? pb.vdv : pb.vdk;
        gm.ostore = make_slab_map(&m[7], out, pb, !rows_q, a.bf16, 128, 2, ov) ? 1 : 0;
        if (!gm.ostore) m[7] = m[0];
    }
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
