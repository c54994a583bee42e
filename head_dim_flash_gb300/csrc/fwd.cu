// Forward kernel: exact softmax attention with a split-D schedule on sm_103a.
//
// Computes O = softmax(scale * Q K^T [bottom-right causal mask]) V and the
// natural-log LSE per query row (FFPA docs, "CuTe-DSL Backend" page, "Hard
// constraints"; "Varlen (packed THD) API" for the packed layout).
//
// One CTA owns a 128-row query tile of one (sequence, head) and one D-slab of
// the output (<= 256 head-dim columns, so the fp32 O slab takes <= 256 TMEM
// columns next to two 128-column S buffers). Per 128-key tile:
//   S = Q K^T      tcgen05.mma, K = D streamed in 64-wide chunks by TMA
//                  (Q stays resident in shared memory when D <= 512)
//   softmax        4 warps, one query row per thread, read S from TMEM,
//                  online max with lazy rescaling of O (only when the row max
//                  grows by more than 2^8), P rounded to the input type and
//                  written to shared memory in the MMA operand layout
//   O += P V_slab  tcgen05.mma into the TMEM O slab
// Warp roles: warp 0 issues TMA loads, warp 1 issues MMAs (one elected
// thread each), warps 2..5 run the softmax and the epilogue.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr int kFwdThreads = 192;
constexpr int kMaxStages = 12;
constexpr float kRescaleTau = 8.0f;  // log2 of the largest P value allowed before O is rescaled
constexpr float kLn2 = 0.693147180559945309f;

enum FwdSite : uint32_t {
    SITE_PROD_EMPTY = 1, SITE_MMA_Q, SITE_MMA_SEMPTY, SITE_MMA_FULL, SITE_MMA_PFULL,
    SITE_SM_SFULL, SITE_SM_ODONE, SITE_EPI_ODONE, SITE_DRAIN
};

template <bool BF16, bool QRES, bool VARLEN>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdArgs a, int slab_chunks, int stages)
{
    const Problem& pb = a.pb;
    // ---------------------------------------------------------- work unit
    const int slab = blockIdx.x;
    const int n_mt = gridDim.y;
    const int mt = pb.causal ? (n_mt - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
    const int bh = blockIdx.z;
    const int b = bh / pb.Hq, h = bh % pb.Hq;
    const int hk = h / (pb.Hq / pb.Hkv);
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
    const int q0 = mt * kBlockM;
    if (q0 >= lq) return;  // uniform across the block, before any barrier
    const int nd = pb.D / kChunk;
    const int c_begin = slab * slab_chunks;
    const int c_end = min(nd, c_begin + slab_chunks);
    const int sw = (c_end - c_begin) * kChunk;  // O slab width = PV MMA N
    int n_kv = (lk + kBlockN - 1) / kBlockN;
    if (pb.causal) {
        const int i_max = min(q0 + kBlockM - 1, lq - 1);
        const int kmax = i_max + (lk - lq);
        n_kv = kmax < 0 ? 0 : min(n_kv, kmax / kBlockN + 1);
    }

    // ---------------------------------------------------------- shared memory
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sP = smem + (QRES ? nd * 16384 : 0);
    uint8_t* sRing = sP + 32768;

    __shared__ uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
    __shared__ uint64_t bar_q, bar_s_full[2], bar_s_empty[2], bar_p_full, bar_o_done, bar_drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < stages; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_empty[i], 1);
        }
        mbar_init(&bar_q, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_s_full[i], 1);
            mbar_init(&bar_s_empty[i], 128);
        }
        mbar_init(&bar_p_full, 128);
        mbar_init(&bar_o_done, 1);
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
    const uint32_t t_o = tmem;
    volatile int* abort_flag = &abort_sh;
    uint32_t* status = a.ctl.status;
    const uint64_t lim = a.ctl.limit_ns;

    // TMA coordinates: dense maps are (d, row, b*H + h), packed maps (d, h, token).
    auto q_c1 = [&](int row) { return VARLEN ? h : q0 + row; };
    auto q_c2 = [&](int row) { return VARLEN ? tq0 + q0 + row : bh; };
    auto k_c1 = [&](int key) { return VARLEN ? hk : key; };
    auto k_c2 = [&](int key) { return VARLEN ? tk0 + key : b * pb.Hkv + hk; };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (elect_one()) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            RingPos rp;
            int issued = 0;
            bool ok = true;
            auto acquire = [&]() -> bool {
                return mbar_wait(&bar_empty[rp.slot], rp.phase ^ 1u, abort_flag, status, lim, SITE_PROD_EMPTY);
            };
            if (QRES && n_kv > 0) {
                mbar_arrive_expect_tx(&bar_q, nd * 16384);
                for (int c = 0; c < nd; ++c) tma_load_3d(sQ + c * 16384, &tm_q, &bar_q, c * kChunk, q_c1(0), q_c2(0));
            }
            auto load_s = [&](int j) -> bool {
                const int k0 = j * kBlockN;
                for (int c = 0; c < nd; ++c) {
                    if (!QRES) {
                        if (!acquire()) return false;
                        uint8_t* dst = sRing + rp.slot * 16384;
                        mbar_arrive_expect_tx(&bar_full[rp.slot], 16384);
                        tma_load_3d(dst, &tm_q, &bar_full[rp.slot], c * kChunk, q_c1(0), q_c2(0));
                        rp.advance(stages);
                        ++issued;
                    }
                    if (!acquire()) return false;
                    uint8_t* dst = sRing + rp.slot * 16384;
                    mbar_arrive_expect_tx(&bar_full[rp.slot], 16384);
                    tma_load_3d(dst, &tm_k, &bar_full[rp.slot], c * kChunk, k_c1(k0), k_c2(k0));
                    rp.advance(stages);
                    ++issued;
                }
                return true;
            };
            auto load_v = [&](int j) -> bool {
                const int k0 = j * kBlockN;
                const int nb = c_end - c_begin;
                for (int vc = 0; vc < kBlockN / kVKeys; ++vc) {
                    if (!acquire()) return false;
                    uint8_t* dst = sRing + rp.slot * 16384;
                    mbar_arrive_expect_tx(&bar_full[rp.slot], nb * kVKeys * 128);
                    const int key = k0 + vc * kVKeys;
                    for (int bb = 0; bb < nb; ++bb)
                        tma_load_3d(dst + bb * kVKeys * 128, &tm_v, &bar_full[rp.slot], (c_begin + bb) * kChunk,
                                    k_c1(key), k_c2(key));
                    rp.advance(stages);
                    ++issued;
                }
                return true;
            };
            if (n_kv > 0) ok = load_s(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) ok = load_s(j + 1);
                if (ok) ok = load_v(j);
            }
            // Drain: wait until the last copies into every slot have landed.
            const int last = min(issued, stages);
            RingPos dp = rp;
            for (int i = 0; i < last; ++i) {
                dp.retreat(stages);
                int dummy = 0;
                mbar_wait(&bar_full[dp.slot], dp.phase, &dummy, status, lim, SITE_DRAIN, false);
            }
            if (QRES && n_kv > 0) {
                int dummy = 0;
                mbar_wait(&bar_q, 0, &dummy, status, lim, SITE_DRAIN, false);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (elect_one()) {
            const uint32_t idesc_s = idesc_f16(kBlockM, kBlockN, BF16, false, false);
            const uint32_t idesc_pv = idesc_f16(kBlockM, sw, BF16, false, true);
            RingPos rp;
            bool ok = true;
            if (QRES && n_kv > 0) {
                ok = mbar_wait(&bar_q, 0, abort_flag, status, lim, SITE_MMA_Q);
                tc_fence_after();
            }
            auto issue_s = [&](int j) -> bool {
                const int sb = j & 1;
                const uint32_t t_s = tmem + 256 + sb * 128;
                if (j >= 2) {
                    if (!mbar_wait(&bar_s_empty[sb], ((j - 2) >> 1) & 1, abort_flag, status, lim, SITE_MMA_SEMPTY))
                        return false;
                    tc_fence_after();
                }
                for (int c = 0; c < nd; ++c) {
                    const uint8_t* qa;
                    int q_slot = -1;
                    if (QRES) {
                        qa = sQ + c * 16384;
                    } else {
                        if (!mbar_wait(&bar_full[rp.slot], rp.phase, abort_flag, status, lim, SITE_MMA_FULL)) return false;
                        q_slot = rp.slot;
                        qa = sRing + rp.slot * 16384;
                        rp.advance(stages);
                    }
                    if (!mbar_wait(&bar_full[rp.slot], rp.phase, abort_flag, status, lim, SITE_MMA_FULL)) return false;
                    tc_fence_after();
                    const uint8_t* kb = sRing + rp.slot * 16384;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_sw128(smem_u32(qa + kk * 32), 16, 1024);
                        const uint64_t bd = sdesc_sw128(smem_u32(kb + kk * 32), 16, 1024);
                        umma_f16(t_s, ad, bd, idesc_s, (c | kk) != 0);
                    }
                    umma_commit(&bar_empty[rp.slot]);
                    if (!QRES) umma_commit(&bar_empty[q_slot]);
                    rp.advance(stages);
                }
                umma_commit(&bar_s_full[sb]);
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                if (!mbar_wait(&bar_p_full, j & 1, abort_flag, status, lim, SITE_MMA_PFULL)) return false;
                tc_fence_after();
                for (int vc = 0; vc < kBlockN / kVKeys; ++vc) {
                    if (!mbar_wait(&bar_full[rp.slot], rp.phase, abort_flag, status, lim, SITE_MMA_FULL)) return false;
                    tc_fence_after();
                    const uint8_t* vb = sRing + rp.slot * 16384;
#pragma unroll
                    for (int t = 0; t < kVKeys / 16; ++t) {
                        const int kt = vc * kVKeys + t * 16;
                        const uint64_t ad = sdesc_sw128(smem_u32(sP + (kt / 64) * 16384 + (kt % 64) * 2), 16, 1024);
                        const uint64_t bd = sdesc_sw128(smem_u32(vb + t * 2048), kVKeys * 128, 1024);
                        umma_f16(t_o, ad, bd, idesc_pv, (j | vc | t) != 0);
                    }
                    umma_commit(&bar_empty[rp.slot]);
                    rp.advance(stages);
                }
                umma_commit(&bar_o_done);
                return true;
            };
            if (ok && n_kv > 0) ok = issue_s(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) ok = issue_s(j + 1);
                if (ok) ok = issue_pv(j);
            }
            // Drain: every MMA issued by this thread has completed.
            umma_commit(&bar_drain);
            int dummy = 0;
            mbar_wait(&bar_drain, 0, &dummy, status, lim, SITE_DRAIN, false);
        }
    } else {
        // ------------------------------------------------------ softmax + epilogue
        const int quarter = warp & 3;
        const int r = quarter * 32 + static_cast<int>(lane_id());
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int qi = q0 + r;
        const int diag = qi + (lk - lq);
        const int key_end = pb.causal ? min(lk, diag + 1) : lk;  // legal keys: [0, key_end)
        const float c2 = pb.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            const bool got_s = mbar_wait(&bar_s_full[sb], (j >> 1) & 1, abort_flag, status, lim, SITE_SM_SFULL);
            if (!__all_sync(0xffffffffu, got_s)) {  // keeps the warp converged for tcgen05.ld
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[128];
            const uint32_t t_s = tmem + 256 + sb * 128 + lane_off;
            tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
            tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
            tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
            tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
            tmem_ld_wait(s);
            tc_fence_before();
            mbar_arrive(&bar_s_empty[sb]);

            const int limit = key_end - j * kBlockN;  // keys [0, limit) of this tile are legal
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c)
                if (c < limit) mx = fmaxf(mx, __uint_as_float(s[c]));
            const float m_tile = mx * c2;
            float new_ref = m_ref;
            bool need = false;
            if (m_tile > -INFINITY) {
                if (m_ref == -INFINITY) {
                    new_ref = m_tile;
                } else if (m_tile > m_ref + kRescaleTau) {
                    new_ref = m_tile;
                    need = true;
                }
            }
            const float alpha = need ? ex2_approx(m_ref - new_ref) : 1.f;
            if (j > 0) {
                // P buffer is free and O is stable once PV(j-1) has completed.
                const bool got_o = mbar_wait(&bar_o_done, (j - 1) & 1, abort_flag, status, lim, SITE_SM_ODONE);
                if (!__all_sync(0xffffffffu, got_o)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, need)) {
                for (int cc = 0; cc < sw; cc += 32) {
                    uint32_t o[32];
                    tmem_ld32(t_o + lane_off + cc, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(t_o + lane_off + cc, o);
                }
                tmem_st_wait();
            }
            l *= alpha;
            m_ref = new_ref;
            const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
            float sum = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = u * 8 + e * 2;
                    const float p0 = (c < limit) ? ex2_approx(__uint_as_float(s[c]) * c2 - mu) : 0.f;
                    const float p1 = (c + 1 < limit) ? ex2_approx(__uint_as_float(s[c + 1]) * c2 - mu) : 0.f;
                    sum += p0 + p1;
                    w[e] = pack2<BF16>(p0, p1);
                }
                uint8_t* dst = sP + (u >> 3) * 16384 + sw128_offset(r, u & 7);
                *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            l += sum;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar_p_full);
        }
        // ---------------------------------------------------- epilogue
        if (ok) {
            if (n_kv > 0) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bar_o_done, (n_kv - 1) & 1, abort_flag, status, lim, SITE_EPI_ODONE));
                tc_fence_after();
            }
        }
        if (ok) {
            const bool valid = qi < lq;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            size_t row;
            if constexpr (VARLEN) row = (static_cast<size_t>(tq0 + qi) * pb.Hq + h) * pb.D;
            else row = (static_cast<size_t>(bh) * pb.Nq + qi) * pb.D;
            uint16_t* orow = reinterpret_cast<uint16_t*>(a.o) + row + c_begin * kChunk;
            for (int cc = 0; cc < sw; cc += 32) {
                uint32_t o[32];
                if (n_kv > 0) {
                    tmem_ld32(t_o + lane_off + cc, o);
                    tmem_ld_wait(o);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cc);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
            }
            if (valid && slab == 0) {
                const float lse = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
                if constexpr (VARLEN) a.lse[static_cast<size_t>(h) * pb.total_q + tq0 + qi] = lse;
                else a.lse[static_cast<size_t>(bh) * pb.Nq + qi] = lse;
            }
        }
    }

    // -------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <bool BF16, bool QRES, bool VARLEN>
cudaError_t launch_variant(const FwdArgs& a, cudaStream_t s, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, dim3 grid, int slab_chunks, int stages, int smem)
{
    auto kern = fwd_kernel<BF16, QRES, VARLEN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kFwdThreads, smem, s>>>(tq, tk, tv, a, slab_chunks, stages);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s)
{
    const Problem& pb = a.pb;
    const int nd = pb.D / kChunk;
    const int n_slabs = (nd + 3) / 4;
    const int slab_chunks = (nd + n_slabs - 1) / n_slabs;
    const bool qres = pb.D <= 512;
    const int fixed = 1024 + 1024 /* static smem margin */ + (qres ? nd * 16384 : 0) + 32768;
    int stages = (kMaxSmem - fixed) / 16384;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return cudaErrorInvalidConfiguration;
    const int smem = 1024 + (qres ? nd * 16384 : 0) + 32768 + stages * 16384;

    CUtensorMap tq, tk, tv;
    const bool kv_empty = kv_side_empty(pb);
    if (!make_row_map(&tq, a.q, pb, false, a.bf16, kBlockM) ||
        !make_row_map(&tk, kv_empty ? a.q : a.k, pb, !kv_empty, a.bf16, kBlockN) ||
        !make_row_map(&tv, kv_empty ? a.q : a.v, pb, !kv_empty, a.bf16, kVKeys))
        return cudaErrorInvalidValue;
    const int n_mt = (pb.Nq + kBlockM - 1) / kBlockM;
    if (n_mt == 0 || pb.B * pb.Hq == 0) return cudaSuccess;
    dim3 grid(n_slabs, n_mt, pb.B * pb.Hq);
    if (a.bf16) {
        if (pb.varlen) return qres ? launch_variant<true, true, true>(a, s, tq, tk, tv, grid, slab_chunks, stages, smem)
                                   : launch_variant<true, false, true>(a, s, tq, tk, tv, grid, slab_chunks, stages, smem);
        return qres ? launch_variant<true, true, false>(a, s, tq, tk, tv, grid, slab_chunks, stages, smem)
                    : launch_variant<true, false, false>(a, s, tq, tk, tv, grid, slab_chunks, stages, smem);
    }
    if (pb.varlen) return qres ? launch_variant<false, true, true>(a, s, tq, tk, tv, grid, slab_chunks, stages, smem)
                               : launch_variant<false, false, true>(a, s, tq, tk, tv, grid, slab_chunks, stages, smem);
    return qres ? launch_variant<false, true, false>(a, s, tq, tk, tv, grid, slab_chunks, stages, smem)
                : launch_variant<false, false, false>(a, s, tq, tk, tv, grid, slab_chunks, stages, smem);
}

}  // namespace ffpa
