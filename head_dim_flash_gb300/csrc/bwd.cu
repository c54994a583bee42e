// Backward of exact softmax attention on sm_103a.
//
// For L = sum(dO * O) (FFPA docs, "CuTe-DSL Backend" page, "Blackwell status":
// a preprocess launch and separate dV, dK and dQ launches, split because one
// SM cannot hold a whole dK/dV tile at D = 512; "Hard constraints": rows
// without a legal key get exactly zero gradient; "Configuration": gradients
// are returned in the input dtype):
//   preprocess : delta_i = sum_d dO_id O_id,  lse2_i = LSE_i * log2(e)
//   dV         : per key tile, over the query heads of its GQA group and all
//                query tiles: P^T = exp2(scale*log2e * K Q^T - lse2), dV += P^T dO
//   dK         : same tiles: dS^T = P^T (V dO^T - delta), dK += scale * dS^T Q
//   dQ         : per query tile, over key tiles: dS = P (dO V^T - delta),
//                dQ += scale * dS K
// The three gradient launches run the cluster-exchange kernel (xchg.cu). With
// room in the workspace (dense, D a multiple of 64 up to 1024), the dK launch
// also stores its P^T and dS^T tiles, and dV = P^T dO and dQ = scale dS K
// become plain GEMMs over them (dsq.cu): preprocess, dK, dV, dQ.
#include "kernels.h"
#include "ptx.cuh"
#include "tile_common.cuh"

namespace ffpa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

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
        // r indexes the LSE layout: dense [B, Hq, Nq] (row i of head h of batch b),
        // packed [Hq, T] (token t of head h); O and dO are read through their views
        long bb = 0, h, i;
        if (pb.varlen) {
            h = r / pb.total_q;
            i = r % pb.total_q;
        } else {
            bb = r / (static_cast<long>(pb.Hq) * pb.Nq);
            h = (r / pb.Nq) % pb.Hq;
            i = r % pb.Nq;
        }
        const size_t off_o = bb * pb.vo.sb + h * pb.vo.sh + i * pb.vo.sn;
        const size_t off_d = bb * pb.vdo.sb + h * pb.vdo.sh + i * pb.vdo.sn;
        const uint4* o4 = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.o) + off_o);
        const uint4* d4 = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.dO) + off_d);
        // every load of the row is issued before the first product (D <= 1024:
        // at most four 16-byte units of each tensor per lane)
        constexpr int kMaxUnits = 1024 / 8 / 32;
        uint4 xo[kMaxUnits], yd[kMaxUnits];
#pragma unroll
        for (int k = 0; k < kMaxUnits; ++k) {
            const int i = lane + lanes * k;
            if (i < D / 8) {
                xo[k] = o4[i];
                yd[k] = d4[i];
            }
        }
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxUnits; ++k) {
            if (lane + lanes * k >= D / 8) break;
            const uint32_t xs[4] = {xo[k].x, xo[k].y, xo[k].z, xo[k].w}, ys[4] = {yd[k].x, yd[k].y, yd[k].z, yd[k].w};
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

template <bool BF16, bool VARLEN>
cudaError_t launch_bwd_variant(const BwdArgs& a, cudaStream_t st)
{
    const Problem& pb = a.pb;
    const long rows = pb.varlen ? static_cast<long>(pb.Hq) * pb.total_q : static_cast<long>(pb.B) * pb.Hq * pb.Nq;
    const bool q_empty = q_side_empty(pb), kv_empty = kv_side_empty(pb);
    cudaError_t e;
    if (!q_empty && (a.stages & 1u)) {
        const int sms = num_sms() > 0 ? num_sms() : 148;
        // one wave of resident blocks (a grid-stride loop over the rows)
        static int per_sm = 0;
        if (per_sm == 0 &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bwd_preprocess_kernel<BF16>, 256, 0) != cudaSuccess)
            per_sm = 4;
        long blocks = (rows + 7) / 8;
        const long cap = static_cast<long>(sms) * (per_sm > 0 ? per_sm : 4);
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        bwd_preprocess_kernel<BF16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a, rows);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    XArgs x{};
    x.pb = pb;
    x.bf16 = BF16;
    x.q = a.q;
    x.k = a.k;
    x.v = a.v;
    x.dO = a.dO;
    x.delta = a.delta;
    x.lse_log2 = a.lse_log2;
    x.dq = a.dq;
    x.dk = a.dk;
    x.dv = a.dv;
    x.ctl = a.ctl;
    // dV, dK and dQ read only the inputs and the preprocess output and write
    // disjoint outputs: each after the first is a programmatic dependent of the
    // one before, so it fills the SMs that the previous one's last wave leaves
    // idle (the first waits for the preprocess as usual; the later ones start
    // only once all of its CTAs have started, hence after the preprocess).
    // Stored tiles (dense, D % 64 == 0 up to 1024, the buffers given; the dK
    // kernels of both families store them):
    //  - dS: the dK launch also writes dS^T into a.ds and dQ is a plain GEMM
    //    over it; stage bit 4 runs that GEMM alone on a buffer an earlier dK
    //    launch filled;
    //  - P: with dV and dK in one call, or stage bit 5, the dK launch also
    //    writes P^T into a.p and dV is a plain GEMM over it, after dK.
    const bool use_ds = a.ds != nullptr && !q_empty && !kv_empty && dsq_supported(pb);
    if ((a.stages & 16u) && !use_ds) return cudaErrorInvalidConfiguration;  // no stored dS to read
    const bool use_p = use_ds && a.p != nullptr;
    if ((a.stages & 32u) && !use_p) return cudaErrorInvalidConfiguration;  // no P buffer
    const bool p_mode = use_p && ((a.stages & 32u) || ((a.stages & 2u) && (a.stages & 8u)));
    auto tile_gemm = [&](bool dv, int g0 = 0, int ng = 0) {
        DsqArgs d{};
        d.pb = pb;
        d.bf16 = BF16;
        d.dv = dv ? 1 : 0;
        d.tiles = dv ? a.p : a.ds;
        d.rhs = dv ? a.dO : a.k;
        d.out = dv ? a.dv : a.dq;
        d.g0 = g0;
        d.ng = ng;
        d.ctl = a.ctl;
        // a plain launch: the GEMM reads what the dK launch wrote
        return launch_dsq(d, st);
    };
    x.pdl = 0;
    if (a.chunk_groups > 0) {
        // Stored tiles in chunks of kv groups (the workspace holds one chunk's
        // P^T and dS^T): per chunk, dK over its kv heads (storing the tiles of
        // their query heads), then dV = P^T dO for those kv heads and
        // dQ = scale dS K for those query heads. A group's gradients are
        // complete within its chunk, so nothing accumulates across chunks.
        // Every launch is a plain one: a chunk's dK rewrites the buffers the
        // previous chunk's GEMMs read.
        if (!use_p || (a.stages & 14u) != 14u || (a.stages & 48u)) return cudaErrorInvalidConfiguration;
        for (int g0 = 0; g0 < pb.Hkv; g0 += a.chunk_groups) {
            const int ng = min(a.chunk_groups, pb.Hkv - g0);
            XArgs xk = x;
            xk.store_ds = 1;
            xk.ds = a.ds;
            xk.store_p = 1;
            xk.p = a.p;
            xk.g0 = g0;
            xk.ng = ng;
            if ((e = launch_xchg(XOP_DK, xk, st)) != cudaSuccess) return e;
            if ((e = tile_gemm(true, g0, ng)) != cudaSuccess) return e;
            if ((e = tile_gemm(false, g0, ng)) != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (!kv_empty && (a.stages & 2u) && !p_mode) {
        if ((e = launch_xchg(XOP_DV, x, st)) != cudaSuccess) return e;
        x.pdl = 1;
    }
    if (!kv_empty && (a.stages & 8u)) {
        XArgs xk = x;
        xk.store_ds = use_ds ? 1 : 0;
        xk.ds = a.ds;
        xk.store_p = p_mode ? 1 : 0;
        xk.p = a.p;
        if ((e = launch_xchg(XOP_DK, xk, st)) != cudaSuccess) return e;
        x.pdl = 1;
    }
    if (!kv_empty && (a.stages & 2u) && p_mode && (e = tile_gemm(true)) != cudaSuccess) return e;
    const bool dq_from_ds = use_ds && ((a.stages & 16u) || ((a.stages & 4u) && (a.stages & 8u)));
    if (!q_empty && dq_from_ds) {
        if ((e = tile_gemm(false)) != cudaSuccess) return e;
    } else if (!q_empty && (a.stages & 4u) && (e = launch_xchg(XOP_DQ, x, st)) != cudaSuccess) {
        return e;
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
