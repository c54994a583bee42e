// Backward kernels for exact softmax attention on sm_103a.
//
// For L = sum(dO * O) (FFPA docs, "CuTe-DSL Backend" page, "Blackwell status":
// a preprocess launch and separate gradient launches; "Hard constraints":
// rows without a legal key get exactly zero gradient; "Configuration":
// gradients are returned in the input dtype):
//   preprocess : delta_i = sum_d dO_id O_id,  lse2_i = LSE_i * log2(e)
//   dK/dV      : per key tile, over the query heads of its GQA group and all
//                query tiles:  S^T = K Q^T, dP^T = V dO^T,
//                P = exp2(scale*log2e*S - lse2), dS = P (dP - delta),
//                dV += P^T dO,  dK += dS^T Q   (scale applied at the end)
//   dQ         : per query tile, over key tiles: S = Q K^T, dP = dO V^T,
//                dS as above, dQ += dS K      (scale applied at the end)
// Both gradient kernels keep their accumulators in TMEM (fp32) for a D-slab
// of the output and stream every operand through a TMA ring; the S/dP
// products are recomputed per slab.
#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr int kBwdThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 elementwise
constexpr int kMaxStages = 12;
constexpr float kLog2e = 1.4426950408889634f;

enum BwdSite : uint32_t {
    BSITE_PROD = 16, BSITE_MMA_FULL, BSITE_MMA_SEMPTY, BSITE_MMA_PFULL, BSITE_EW_SFULL, BSITE_EW_PDONE,
    BSITE_EPI, BSITE_DRAIN
};

// ----------------------------------------------------------------- preprocess
// One warp per query row: delta = dO . O (fp32) and lse2 = LSE*log2e
// (+inf for rows without a legal key, so that exp2(x - lse2) = 0 there).
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdArgs a, long rows)
{
    const Problem& pb = a.pb;
    const int lanes = 32;
    const long warp_global = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) / lanes;
    const long n_warps = static_cast<long>(gridDim.x) * blockDim.x / lanes;
    const int lane = threadIdx.x & 31;
    const int D = pb.D;
    for (long r = warp_global; r < rows; r += n_warps) {
        // r indexes the LSE layout: dense [B*Hq, Nq], packed [Hq, T]
        size_t off;
        if (pb.varlen) {
            const long h = r / pb.total_q, t = r % pb.total_q;
            off = (static_cast<size_t>(t) * pb.Hq + h) * D;
        } else {
            off = static_cast<size_t>(r) * D;
        }
        const uint4* o4 = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.o) + off);
        const uint4* d4 = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.dO) + off);
        float acc = 0.f;
        for (int i = lane; i < D / 8; i += lanes) {
            const uint4 x = o4[i], y = d4[i];
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 p = unpack2<BF16>(xs[e]), q = unpack2<BF16>(ys[e]);
                acc = fmaf(p.x, q.x, acc);
                acc = fmaf(p.y, q.y, acc);
            }
        }
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
        if (lane == 0) {
            a.delta[r] = acc;
            const float l = a.lse[r];
            a.lse_log2[r] = (l == -INFINITY) ? INFINITY : l * kLog2e;
        }
    }
}

// Per-sequence geometry of a work unit.
struct SeqGeom {
    int b, lq, lk, tq0, tk0;
};

template <bool VARLEN>
__device__ __forceinline__ SeqGeom seq_geom(const Problem& pb, int b)
{
    SeqGeom g;
    g.b = b;
    if constexpr (VARLEN) {
        g.tq0 = pb.cu_q[b];
        g.lq = pb.cu_q[b + 1] - g.tq0;
        g.tk0 = pb.cu_k[b];
        g.lk = pb.cu_k[b + 1] - g.tk0;
    } else {
        g.tq0 = g.tk0 = 0;
        g.lq = pb.Nq;
        g.lk = pb.Nkv;
    }
    return g;
}

// Index of a row statistic (lse2 / delta) of query i of head h.
template <bool VARLEN>
__device__ __forceinline__ size_t stat_index(const Problem& pb, const SeqGeom& g, int h, int i)
{
    if constexpr (VARLEN) return static_cast<size_t>(h) * pb.total_q + g.tq0 + i;
    else return (static_cast<size_t>(g.b) * pb.Hq + h) * pb.Nq + i;
}

// Element offset of row `i` (of head h with H heads) of a dense or packed tensor.
template <bool VARLEN>
__device__ __forceinline__ size_t row_offset(const Problem& pb, int b, int H, int N, int t0, int h, int i)
{
    if constexpr (VARLEN) return (static_cast<size_t>(t0 + i) * H + h) * pb.D;
    else return ((static_cast<size_t>(b) * H + h) * N + i) * pb.D;
}

// ------------------------------------------------------------------ dK / dV
// CTA = (d-slab of 128 columns, key tile, b*Hkv + hkv). TMEM columns:
// [0,128) S^T, [128,256) dP^T, [256,384) dV slab, [384,512) dK slab; TMEM lane
// = key row. P^T and dS^T go to shared memory (double-buffered) as the A
// operands of dV += P^T dO_slab and dK += dS^T Q_slab.
template <bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_q32, const __grid_constant__ CUtensorMap tm_do32,
                    const BwdArgs a, int stages)
{
    const Problem& pb = a.pb;
    const int slab = blockIdx.x;  // 128 columns (the last slab may be 64)
    const int nt = blockIdx.y;
    const int bhk = blockIdx.z;
    const int b = bhk / pb.Hkv, hk = bhk % pb.Hkv;
    const int G = pb.Hq / pb.Hkv;
    const SeqGeom g = seq_geom<VARLEN>(pb, b);
    const int n0 = nt * kBlockN;
    if (n0 >= g.lk) return;
    const int nd = pb.D / kChunk;
    const int d0 = slab * 128;
    const int sw = min(2, nd - 2 * slab) * kChunk;  // slab width
    const int off = g.lk - g.lq;  // causal: key j legal for query i iff j <= i + off
    int m_start = 0;
    if (pb.causal) m_start = max(0, n0 - off) / kBlockM;
    const int m_end = (g.lq + kBlockM - 1) / kBlockM;
    const int n_mt = max(0, m_end - m_start);
    const int n_steps = G * n_mt;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sPt = smem;           // 2 buffers x 32 KiB: P^T [128 keys x 128 queries]
    uint8_t* sdSt = smem + 65536;  // 2 buffers x 32 KiB: dS^T
    uint8_t* sRing = smem + 131072;

    __shared__ uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
    __shared__ uint64_t bar_s_full, bar_s_empty, bar_p_full[2], bar_pv_done[2], bar_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_s_full, 1);
        mbar_init(&bar_s_empty, 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_p_full[i], 128);
            mbar_init(&bar_pv_done[i], 1);
        }
        mbar_init(&bar_drain, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abort_flag = &abort_sh;
    uint32_t* status = a.ctl.status;
    const uint64_t lim = a.ctl.limit_ns;

    // step s -> (query head h, query tile m)
    auto step_h = [&](int s) { return hk * G + s / n_mt; };
    auto step_q0 = [&](int s) { return (m_start + s % n_mt) * kBlockM; };
    auto q_c1 = [&](int h, int row) { return VARLEN ? h : row; };
    auto q_c2 = [&](int h, int row) { return VARLEN ? g.tq0 + row : b * pb.Hq + h; };
    auto k_c1 = [&](int row) { return VARLEN ? hk : row; };
    auto k_c2 = [&](int row) { return VARLEN ? g.tk0 + row : bhk; };

    if (warp == 0) {
        if (elect_one()) {
            RingPos rp;
            int issued = 0;
            bool ok = true;
            auto put = [&](const CUtensorMap* m, int boxes, int bytes_per_box, int c0, int c1, int c2,
                           int c0_step) -> bool {
                if (!mbar_wait(&bar_empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, BSITE_PROD)) return false;
                uint8_t* dst = sRing + rp.slot * 16384;
                mbar_arrive_expect_tx(&bar_full[rp.slot], boxes * bytes_per_box);
                for (int i = 0; i < boxes; ++i)
                    tma_load_3d(dst + i * bytes_per_box, m, &bar_full[rp.slot], c0 + i * c0_step, c1, c2);
                rp.advance(stages);
                ++issued;
                return true;
            };
            auto load_sdp = [&](int s) -> bool {
                const int h = step_h(s), qr = step_q0(s);
                for (int c = 0; c < nd; ++c) {
                    if (!put(&tm_k, 1, 16384, c * kChunk, k_c1(n0), k_c2(n0), 0)) return false;
                    if (!put(&tm_q, 1, 16384, c * kChunk, q_c1(h, qr), q_c2(h, qr), 0)) return false;
                }
                for (int c = 0; c < nd; ++c) {
                    if (!put(&tm_v, 1, 16384, c * kChunk, k_c1(n0), k_c2(n0), 0)) return false;
                    if (!put(&tm_do, 1, 16384, c * kChunk, q_c1(h, qr), q_c2(h, qr), 0)) return false;
                }
                return true;
            };
            auto load_slab = [&](int s) -> bool {
                const int h = step_h(s), qr = step_q0(s);
                for (int vc = 0; vc < kBlockM / kVKeys; ++vc) {
                    const int row = qr + vc * kVKeys;
                    if (!put(&tm_do32, sw / kChunk, kVKeys * 128, d0, q_c1(h, row), q_c2(h, row), kChunk)) return false;
                    if (!put(&tm_q32, sw / kChunk, kVKeys * 128, d0, q_c1(h, row), q_c2(h, row), kChunk)) return false;
                }
                return true;
            };
            if (n_steps > 0) ok = load_sdp(0);
            for (int s = 0; ok && s < n_steps; ++s) {
                if (s + 1 < n_steps) ok = load_sdp(s + 1);
                if (ok) ok = load_slab(s);
            }
            const int last = min(issued, stages);
            RingPos dp = rp;
            for (int i = 0; i < last; ++i) {
                dp.retreat(stages);
                int dummy = 0;
                mbar_wait(&bar_full[dp.slot], dp.phase, &dummy, status, lim, BSITE_DRAIN, false);
            }
        }
    } else if (warp == 1) {
        if (elect_one()) {
            const uint32_t idesc_s = idesc_f16(kBlockN, kBlockM, BF16, false, false);
            const uint32_t idesc_g = idesc_f16(kBlockN, sw, BF16, false, true);
            const uint32_t t_st = tmem, t_dpt = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 384;
            RingPos rp;
            bool ok = true;
            auto take = [&]() -> const uint8_t* {
                if (!mbar_wait(&bar_full[rp.slot], rp.phase, abort_flag, status, lim, BSITE_MMA_FULL)) return nullptr;
                tc_fence_after();
                return sRing + rp.slot * 16384;
            };
            auto release = [&]() {
                umma_commit(&bar_empty[rp.slot]);
                rp.advance(stages);
            };
            auto issue_sdp = [&](int s) -> bool {
                if (s >= 1) {
                    if (!mbar_wait(&bar_s_empty, (s - 1) & 1, abort_flag, status, lim, BSITE_MMA_SEMPTY)) return false;
                    tc_fence_after();
                }
                for (int pass = 0; pass < 2; ++pass) {
                    const uint32_t dst = pass == 0 ? t_st : t_dpt;
                    for (int c = 0; c < nd; ++c) {
                        const uint8_t* A = take();
                        if (!A) return false;
                        const int a_slot = rp.slot;
                        rp.advance(stages);
                        const uint8_t* B = take();
                        if (!B) return false;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f16(dst, sdesc_sw128(smem_u32(A + kk * 32), 16, 1024),
                                     sdesc_sw128(smem_u32(B + kk * 32), 16, 1024), idesc_s, (c | kk) != 0);
                        umma_commit(&bar_empty[a_slot]);
                        release();
                    }
                }
                umma_commit(&bar_s_full);
                return true;
            };
            auto issue_grad = [&](int s) -> bool {
                const int pb_ = s & 1;
                if (!mbar_wait(&bar_p_full[pb_], (s >> 1) & 1, abort_flag, status, lim, BSITE_MMA_PFULL)) return false;
                tc_fence_after();
                const uint8_t* Pt = sPt + pb_ * 32768;
                const uint8_t* dSt = sdSt + pb_ * 32768;
                for (int vc = 0; vc < kBlockM / kVKeys; ++vc) {
                    for (int which = 0; which < 2; ++which) {  // 0: dV += P^T dO ; 1: dK += dS^T Q
                        const uint8_t* Bm = take();
                        if (!Bm) return false;
#pragma unroll
                        for (int t = 0; t < kVKeys / 16; ++t) {
                            const int kt = vc * kVKeys + t * 16;
                            const uint8_t* Am = (which == 0 ? Pt : dSt) + (kt / 64) * 16384 + (kt % 64) * 2;
                            umma_f16(which == 0 ? t_dv : t_dk, sdesc_sw128(smem_u32(Am), 16, 1024),
                                     sdesc_sw128(smem_u32(Bm + t * 2048), kVKeys * 128, 1024), idesc_g,
                                     (s | vc | t) != 0);
                        }
                        release();
                    }
                }
                umma_commit(&bar_pv_done[pb_]);
                return true;
            };
            if (n_steps > 0) ok = issue_sdp(0);
            for (int s = 0; ok && s < n_steps; ++s) {
                if (s + 1 < n_steps) ok = issue_sdp(s + 1);
                if (ok) ok = issue_grad(s);
            }
            umma_commit(&bar_drain);
            int dummy = 0;
            mbar_wait(&bar_drain, 0, &dummy, status, lim, BSITE_DRAIN, false);
        }
    } else {
        // ---------------------------------------------- elementwise (key rows)
        const int quarter = warp & 3;
        const int r = quarter * 32 + static_cast<int>(lane_id());  // key row in tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int key = n0 + r;
        const float c2 = pb.scale_log2;
        bool ok = true;
        for (int s = 0; s < n_steps; ++s) {
            const int h = step_h(s), qr = step_q0(s);
            const int pb_ = s & 1;
            // row statistics of this query tile: every thread reads the same
            // addresses (broadcast loads); rows past the sequence end are masked
            const float* L2 = a.lse_log2 + stat_index<VARLEN>(pb, g, h, 0);
            const float* DL = a.delta + stat_index<VARLEN>(pb, g, h, 0);
            const bool got = mbar_wait(&bar_s_full, s & 1, abort_flag, status, lim, BSITE_EW_SFULL);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (s >= 2) {
                const bool done = mbar_wait(&bar_pv_done[pb_], ((s - 2) >> 1) & 1, abort_flag, status, lim,
                                            BSITE_EW_PDONE);
                if (!__all_sync(0xffffffffu, done)) {
                    ok = false;
                    break;
                }
            }
            // legal queries for this key: i >= key - off (causal), i < lq
            const int i_min = pb.causal ? max(0, key - off) : 0;
            const int i_lim = key < g.lk ? g.lq : 0;  // legal queries: [i_min, i_lim)
            uint8_t* Pt = sPt + pb_ * 32768;
            uint8_t* dSt = sdSt + pb_ * 32768;
#pragma unroll 1
            for (int cc = 0; cc < kBlockM; cc += 32) {
                uint32_t sv[32], dpv[32];
                tmem_ld32(tmem + lane_off + cc, sv);
                tmem_ld32(tmem + 128 + lane_off + cc, dpv);
                tmem_ld_wait(sv);
                tmem_ld_wait(dpv);
                uint32_t wp[16], wd[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const int i = qr + cc + 2 * e + z;
                        const bool legal = i >= i_min && i < i_lim;
                        float p = 0.f, d = 0.f;
                        if (legal) {
                            p = ex2_approx(__uint_as_float(sv[2 * e + z]) * c2 - __ldg(L2 + i));
                            d = p * (__uint_as_float(dpv[2 * e + z]) - __ldg(DL + i));
                        }
                        pv[z] = p;
                        dv[z] = d;
                    }
                    wp[e] = pack2<BF16>(pv[0], pv[1]);
                    wd[e] = pack2<BF16>(dv[0], dv[1]);
                }
                // 32 queries = units 4*(cc/32) .. +3 of chunk cc/64
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int unit = (cc % 64) / 8 + u;
                    const uint32_t o = (cc / 64) * 16384 + sw128_offset(r, unit);
                    *reinterpret_cast<uint4*>(Pt + o) = make_uint4(wp[4 * u], wp[4 * u + 1], wp[4 * u + 2], wp[4 * u + 3]);
                    *reinterpret_cast<uint4*>(dSt + o) = make_uint4(wd[4 * u], wd[4 * u + 1], wd[4 * u + 2], wd[4 * u + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_s_empty);
            fence_proxy_async_smem();
            mbar_arrive(&bar_p_full[pb_]);
        }
        // ------------------------------------------------------- epilogue
        if (ok && n_steps > 0) {
            const int sl = n_steps - 1;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bar_pv_done[sl & 1], (sl >> 1) & 1, abort_flag, status, lim, BSITE_EPI));
            tc_fence_after();
        }
        if (ok) {
            const bool valid = key < g.lk;
            const size_t row = row_offset<VARLEN>(pb, b, pb.Hkv, pb.Nkv, g.tk0, hk, key);
            for (int which = 0; which < 2; ++which) {
                uint16_t* out = reinterpret_cast<uint16_t*>(which == 0 ? a.dv : a.dk) + row + d0;
                const float mul = which == 0 ? 1.f : pb.scale;
                for (int cc = 0; cc < sw; cc += 32) {
                    uint32_t v[32];
                    if (n_steps > 0) {
                        tmem_ld32(tmem + (which == 0 ? 256 : 384) + lane_off + cc, v);
                        tmem_ld_wait(v);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(out + cc);
#pragma unroll
                        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ----------------------------------------------------------------------- dQ
// CTA = (d-slab of <= 256 columns, query tile, b*Hq + h). TMEM columns:
// [0,256) dQ slab, [256,384) S, [384,512) dP; TMEM lane = query row. dS goes
// to shared memory (double-buffered) as the A operand of dQ += dS K_slab.
template <bool BF16, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k32, const BwdArgs a, int slab_chunks, int stages)
{
    const Problem& pb = a.pb;
    const int slab = blockIdx.x;
    const int n_mt = gridDim.y;
    const int mt = pb.causal ? (n_mt - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
    const int bh = blockIdx.z;
    const int b = bh / pb.Hq, h = bh % pb.Hq;
    const int hk = h / (pb.Hq / pb.Hkv);
    const SeqGeom g = seq_geom<VARLEN>(pb, b);
    const int q0 = mt * kBlockM;
    if (q0 >= g.lq) return;
    const int nd = pb.D / kChunk;
    const int c_begin = slab * slab_chunks;
    const int c_end = min(nd, c_begin + slab_chunks);
    const int sw = (c_end - c_begin) * kChunk;
    int n_kv = (g.lk + kBlockN - 1) / kBlockN;
    if (pb.causal) {
        const int i_max = min(q0 + kBlockM - 1, g.lq - 1);
        const int kmax = i_max + (g.lk - g.lq);
        n_kv = kmax < 0 ? 0 : min(n_kv, kmax / kBlockN + 1);
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sdS = smem;  // 2 x 32 KiB: dS [128 queries x 128 keys]
    uint8_t* sRing = smem + 65536;

    __shared__ uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
    __shared__ uint64_t bar_s_full, bar_s_empty, bar_p_full[2], bar_pv_done[2], bar_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_s_full, 1);
        mbar_init(&bar_s_empty, 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_p_full[i], 128);
            mbar_init(&bar_pv_done[i], 1);
        }
        mbar_init(&bar_drain, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abort_flag = &abort_sh;
    uint32_t* status = a.ctl.status;
    const uint64_t lim = a.ctl.limit_ns;

    auto q_c1 = [&]() { return VARLEN ? h : q0; };
    auto q_c2 = [&]() { return VARLEN ? g.tq0 + q0 : bh; };
    auto k_c1 = [&](int row) { return VARLEN ? hk : row; };
    auto k_c2 = [&](int row) { return VARLEN ? g.tk0 + row : b * pb.Hkv + hk; };

    if (warp == 0) {
        if (elect_one()) {
            RingPos rp;
            int issued = 0;
            bool ok = true;
            auto put = [&](const CUtensorMap* m, int boxes, int bytes_per_box, int c0, int c1, int c2,
                           int c0_step) -> bool {
                if (!mbar_wait(&bar_empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, BSITE_PROD)) return false;
                uint8_t* dst = sRing + rp.slot * 16384;
                mbar_arrive_expect_tx(&bar_full[rp.slot], boxes * bytes_per_box);
                for (int i = 0; i < boxes; ++i)
                    tma_load_3d(dst + i * bytes_per_box, m, &bar_full[rp.slot], c0 + i * c0_step, c1, c2);
                rp.advance(stages);
                ++issued;
                return true;
            };
            auto load_sdp = [&](int j) -> bool {
                const int k0 = j * kBlockN;
                for (int c = 0; c < nd; ++c) {
                    if (!put(&tm_q, 1, 16384, c * kChunk, q_c1(), q_c2(), 0)) return false;
                    if (!put(&tm_k, 1, 16384, c * kChunk, k_c1(k0), k_c2(k0), 0)) return false;
                }
                for (int c = 0; c < nd; ++c) {
                    if (!put(&tm_do, 1, 16384, c * kChunk, q_c1(), q_c2(), 0)) return false;
                    if (!put(&tm_v, 1, 16384, c * kChunk, k_c1(k0), k_c2(k0), 0)) return false;
                }
                return true;
            };
            auto load_slab = [&](int j) -> bool {
                const int k0 = j * kBlockN;
                const int nb = c_end - c_begin;
                for (int vc = 0; vc < kBlockN / kVKeys; ++vc) {
                    const int row = k0 + vc * kVKeys;
                    if (!put(&tm_k32, nb, kVKeys * 128, c_begin * kChunk, k_c1(row), k_c2(row), kChunk)) return false;
                }
                return true;
            };
            if (n_kv > 0) ok = load_sdp(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) ok = load_sdp(j + 1);
                if (ok) ok = load_slab(j);
            }
            const int last = min(issued, stages);
            RingPos dp = rp;
            for (int i = 0; i < last; ++i) {
                dp.retreat(stages);
                int dummy = 0;
                mbar_wait(&bar_full[dp.slot], dp.phase, &dummy, status, lim, BSITE_DRAIN, false);
            }
        }
    } else if (warp == 1) {
        if (elect_one()) {
            const uint32_t idesc_s = idesc_f16(kBlockM, kBlockN, BF16, false, false);
            const uint32_t idesc_g = idesc_f16(kBlockM, sw, BF16, false, true);
            const uint32_t t_dq = tmem, t_s = tmem + 256, t_dp = tmem + 384;
            RingPos rp;
            bool ok = true;
            auto take = [&]() -> const uint8_t* {
                if (!mbar_wait(&bar_full[rp.slot], rp.phase, abort_flag, status, lim, BSITE_MMA_FULL)) return nullptr;
                tc_fence_after();
                return sRing + rp.slot * 16384;
            };
            auto release = [&]() {
                umma_commit(&bar_empty[rp.slot]);
                rp.advance(stages);
            };
            auto issue_sdp = [&](int j) -> bool {
                if (j >= 1) {
                    if (!mbar_wait(&bar_s_empty, (j - 1) & 1, abort_flag, status, lim, BSITE_MMA_SEMPTY)) return false;
                    tc_fence_after();
                }
                for (int pass = 0; pass < 2; ++pass) {
                    const uint32_t dst = pass == 0 ? t_s : t_dp;
                    for (int c = 0; c < nd; ++c) {
                        const uint8_t* A = take();
                        if (!A) return false;
                        const int a_slot = rp.slot;
                        rp.advance(stages);
                        const uint8_t* B = take();
                        if (!B) return false;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f16(dst, sdesc_sw128(smem_u32(A + kk * 32), 16, 1024),
                                     sdesc_sw128(smem_u32(B + kk * 32), 16, 1024), idesc_s, (c | kk) != 0);
                        umma_commit(&bar_empty[a_slot]);
                        release();
                    }
                }
                umma_commit(&bar_s_full);
                return true;
            };
            auto issue_grad = [&](int j) -> bool {
                const int pb_ = j & 1;
                if (!mbar_wait(&bar_p_full[pb_], (j >> 1) & 1, abort_flag, status, lim, BSITE_MMA_PFULL)) return false;
                tc_fence_after();
                const uint8_t* dS = sdS + pb_ * 32768;
                for (int vc = 0; vc < kBlockN / kVKeys; ++vc) {
                    const uint8_t* Bm = take();
                    if (!Bm) return false;
#pragma unroll
                    for (int t = 0; t < kVKeys / 16; ++t) {
                        const int kt = vc * kVKeys + t * 16;
                        umma_f16(t_dq, sdesc_sw128(smem_u32(dS + (kt / 64) * 16384 + (kt % 64) * 2), 16, 1024),
                                 sdesc_sw128(smem_u32(Bm + t * 2048), kVKeys * 128, 1024), idesc_g, (j | vc | t) != 0);
                    }
                    release();
                }
                umma_commit(&bar_pv_done[pb_]);
                return true;
            };
            if (n_kv > 0) ok = issue_sdp(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) ok = issue_sdp(j + 1);
                if (ok) ok = issue_grad(j);
            }
            umma_commit(&bar_drain);
            int dummy = 0;
            mbar_wait(&bar_drain, 0, &dummy, status, lim, BSITE_DRAIN, false);
        }
    } else {
        // ------------------------------------------ elementwise (query rows)
        const int quarter = warp & 3;
        const int r = quarter * 32 + static_cast<int>(lane_id());
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int qi = q0 + r;
        const int key_end = pb.causal ? min(g.lk, qi + (g.lk - g.lq) + 1) : g.lk;
        float l2 = INFINITY, dl = 0.f;
        if (qi < g.lq) {
            const size_t si = stat_index<VARLEN>(pb, g, h, qi);
            l2 = a.lse_log2[si];
            dl = a.delta[si];
        }
        const float c2 = pb.scale_log2;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int pb_ = j & 1;
            const bool got = mbar_wait(&bar_s_full, j & 1, abort_flag, status, lim, BSITE_EW_SFULL);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (j >= 2) {
                const bool done = mbar_wait(&bar_pv_done[pb_], ((j - 2) >> 1) & 1, abort_flag, status, lim,
                                            BSITE_EW_PDONE);
                if (!__all_sync(0xffffffffu, done)) {
                    ok = false;
                    break;
                }
            }
            const int limit = key_end - j * kBlockN;
            uint8_t* dS = sdS + pb_ * 32768;
#pragma unroll 1
            for (int cc = 0; cc < kBlockN; cc += 32) {
                uint32_t sv[32], dpv[32];
                tmem_ld32(tmem + 256 + lane_off + cc, sv);
                tmem_ld32(tmem + 384 + lane_off + cc, dpv);
                tmem_ld_wait(sv);
                tmem_ld_wait(dpv);
                uint32_t wd[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float dv[2];
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const int col = cc + 2 * e + z;
                        const float p = col < limit ? ex2_approx(__uint_as_float(sv[2 * e + z]) * c2 - l2) : 0.f;
                        dv[z] = p * (__uint_as_float(dpv[2 * e + z]) - dl);
                    }
                    wd[e] = pack2<BF16>(dv[0], dv[1]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int unit = (cc % 64) / 8 + u;
                    const uint32_t o = (cc / 64) * 16384 + sw128_offset(r, unit);
                    *reinterpret_cast<uint4*>(dS + o) = make_uint4(wd[4 * u], wd[4 * u + 1], wd[4 * u + 2], wd[4 * u + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_s_empty);
            fence_proxy_async_smem();
            mbar_arrive(&bar_p_full[pb_]);
        }
        if (ok && n_kv > 0) {
            const int jl = n_kv - 1;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bar_pv_done[jl & 1], (jl >> 1) & 1, abort_flag, status, lim, BSITE_EPI));
            tc_fence_after();
        }
        if (ok) {
            const bool valid = qi < g.lq;
            const size_t row = row_offset<VARLEN>(pb, b, pb.Hq, pb.Nq, g.tq0, h, qi);
            uint16_t* out = reinterpret_cast<uint16_t*>(a.dq) + row + c_begin * kChunk;
            for (int cc = 0; cc < sw; cc += 32) {
                uint32_t v[32];
                if (n_kv > 0) {
                    tmem_ld32(tmem + lane_off + cc, v);
                    tmem_ld_wait(v);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack2<BF16>(__uint_as_float(v[2 * e]) * pb.scale, __uint_as_float(v[2 * e + 1]) * pb.scale);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(out + cc);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <typename K>
cudaError_t set_smem(K kern, int smem)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <bool BF16, bool VARLEN>
cudaError_t launch_bwd_variant(const BwdArgs& a, cudaStream_t st)
{
    const Problem& pb = a.pb;
    const long rows = pb.varlen ? static_cast<long>(pb.Hq) * pb.total_q : static_cast<long>(pb.B) * pb.Hq * pb.Nq;
    const bool q_empty = q_side_empty(pb), kv_empty = kv_side_empty(pb);
    cudaError_t e;
    if (!q_empty && (a.stages & 1u)) {
        const int sms = num_sms() > 0 ? num_sms() : 148;
        long blocks = (rows + 7) / 8;
        const long cap = static_cast<long>(sms) * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        bwd_preprocess_kernel<BF16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, rows);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // a side without rows is described over the other side's tensor (never loaded)
    const void* qp = q_empty ? a.k : a.q;
    const void* dop = q_empty ? a.k : a.dO;
    const void* kp = kv_empty ? a.q : a.k;
    const void* vp = kv_empty ? a.q : a.v;
    CUtensorMap tq, tk, tv, tdo, tq32, tdo32, tk32;
    if (!make_row_map(&tq, qp, pb, q_empty, BF16, kBlockM) || !make_row_map(&tdo, dop, pb, q_empty, BF16, kBlockM) ||
        !make_row_map(&tk, kp, pb, !kv_empty, BF16, kBlockN) || !make_row_map(&tv, vp, pb, !kv_empty, BF16, kBlockN) ||
        !make_row_map(&tq32, qp, pb, q_empty, BF16, kVKeys) || !make_row_map(&tdo32, dop, pb, q_empty, BF16, kVKeys) ||
        !make_row_map(&tk32, kp, pb, !kv_empty, BF16, kVKeys))
        return cudaErrorInvalidValue;
    const int nd = pb.D / kChunk;
    // dK/dV: 128-column slabs
    if (!kv_empty && (a.stages & 2u)) {
        const int fixed = 1024 + 1024 + 131072;
        int stages = (kMaxSmem - fixed) / 16384;
        if (stages > kMaxStages) stages = kMaxStages;
        const int smem = 1024 + 131072 + stages * 16384;
        const int n_nt = (pb.Nkv + kBlockN - 1) / kBlockN;
        if (n_nt == 0 || pb.B * pb.Hkv == 0) return cudaSuccess;
        dim3 grid((nd + 1) / 2, n_nt, pb.B * pb.Hkv);
        auto kern = bwd_dkdv_kernel<BF16, VARLEN>;
        if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
        kern<<<grid, kBwdThreads, smem, st>>>(tq, tk, tv, tdo, tq32, tdo32, a, stages);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // dQ: <= 256-column slabs
    if (!q_empty && (a.stages & 4u)) {
        const int n_slabs = (nd + 3) / 4;
        const int slab_chunks = (nd + n_slabs - 1) / n_slabs;
        const int fixed = 1024 + 1024 + 65536;
        int stages = (kMaxSmem - fixed) / 16384;
        if (stages > kMaxStages) stages = kMaxStages;
        const int smem = 1024 + 65536 + stages * 16384;
        const int n_mt = (pb.Nq + kBlockM - 1) / kBlockM;
        if (n_mt == 0 || pb.B * pb.Hq == 0) return cudaSuccess;
        dim3 grid(n_slabs, n_mt, pb.B * pb.Hq);
        auto kern = bwd_dq_kernel<BF16, VARLEN>;
        if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
        kern<<<grid, kBwdThreads, smem, st>>>(tq, tk, tv, tdo, tk32, a, slab_chunks, stages);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s)
{
    if (a.bf16) return a.pb.varlen ? launch_bwd_variant<true, true>(a, s) : launch_bwd_variant<true, false>(a, s);
    return a.pb.varlen ? launch_bwd_variant<false, true>(a, s) : launch_bwd_variant<false, false>(a, s);
}

}  // namespace ffpa
