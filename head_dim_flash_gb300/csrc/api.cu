// C ABI entry points (declared in include/ffpa.h): argument validation,
// workspace carving, device status word, and dispatch to the kernels.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/ffpa.h"
#include "kernels.h"
#include "ptx.cuh"

namespace {

thread_local std::string g_err;
std::atomic<uint64_t> g_limit_ns{2000000000ull};

ffpa_status fail(ffpa_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

ffpa_status ok()
{
    g_err.clear();
    return FFPA_OK;
}

}  // namespace

// One status word per device; kernels record the first failing wait here.
__device__ uint32_t g_ffpa_status_word;

namespace {

constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices];
int g_cc_ok[kMaxDevices];  // 0 unknown, 1 yes, -1 no
std::mutex g_dev_mu;

// Device address of the status word on the current device (looked up once).
bool device_state(uint32_t** status, bool* cc_ok)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ffpa_status_word) != cudaSuccess) return false;
        g_status_ptr[dev] = static_cast<uint32_t*>(p);
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    *status = g_status_ptr[dev];
    *cc_ok = g_cc_ok[dev] == 1;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ffpa_status check_common(ffpa_dtype dt, int Hq, int Hkv, int D, float scale)
{
    if (dt != FFPA_BF16 && dt != FFPA_FP16) return fail(FFPA_ERR_NOT_SUPPORTED, "dtype %d: only bf16 (0) and fp16 (1)", (int)dt);
    if (D < 64 || D > 1024 || D % 32 != 0)
        return fail(FFPA_ERR_NOT_SUPPORTED, "head dim D=%d: supported D is a multiple of 32 in [64, 1024]", D);
    if (Hq < 0 || Hkv < 0) return fail(FFPA_ERR_INVALID_VALUE, "negative head count Hq=%d Hkv=%d", Hq, Hkv);
    if (Hq > 0 && (Hkv == 0 || Hq % Hkv != 0))
        return fail(FFPA_ERR_INVALID_VALUE, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
    if (!std::isfinite(scale)) return fail(FFPA_ERR_INVALID_VALUE, "scale must be finite");
    return FFPA_OK;
}

ffpa_status check_ptr(const void* p, bool needed, const char* name)
{
    if (!needed) return FFPA_OK;
    if (!p) return fail(FFPA_ERR_INVALID_VALUE, "%s is NULL", name);
    if (!aligned16(p)) return fail(FFPA_ERR_INVALID_VALUE, "%s is not 16-byte aligned", name);
    return FFPA_OK;
}

ffpa_status device_ctl(ffpa::DeviceCtl* ctl)
{
    bool cc_ok = false;
    uint32_t* st = nullptr;
    if (!device_state(&st, &cc_ok)) return fail(FFPA_ERR_CUDA, "no usable CUDA device");
    if (!cc_ok) return fail(FFPA_ERR_NOT_SUPPORTED, "device is not compute capability 10.3 (sm_103)");
    if (!ffpa::encode_fn()) return fail(FFPA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    ctl->status = st;
    ctl->limit_ns = g_limit_ns.load();
    return FFPA_OK;
}

ffpa_status launch_result(cudaError_t e, const char* what)
{
    if (e != cudaSuccess) return fail(FFPA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Work units one launch can index (unit_grid: 65535 x 65535 clusters).
constexpr long long kMaxUnits = 65535LL * 65535LL;

size_t ws_bytes(long rows) { return rows <= 0 ? 0 : 2 * align256(static_cast<size_t>(rows) * sizeof(float)); }

// Strides of a contiguous [B, H, N, D] tensor, and of a packed [T, H, D] one.
ffpa::View contiguous_view(int H, int N, int D)
{
    return ffpa::View{static_cast<long long>(H) * N * D, static_cast<long long>(N) * D, D};
}

ffpa::View packed_view(int H, int D) { return ffpa::View{0, D, static_cast<long long>(H) * D}; }

// A strided view as the ABI describes it: strides are multiples of 8 elements
// (16 bytes), non-negative, positive along every dimension with more than one
// entry, and below 2^39 elements (the tensor-map limit of 2^40 bytes).
ffpa_status check_view(const ffpa_view& v, bool needed, const char* name, int B, int H, int N)
{
    if (!needed) return FFPA_OK;
    if (!v.data) return fail(FFPA_ERR_INVALID_VALUE, "%s: data is NULL", name);
    if (reinterpret_cast<uintptr_t>(v.data) & 15u) return fail(FFPA_ERR_INVALID_VALUE, "%s: data is not 16-byte aligned", name);
    const int64_t st[3] = {v.stride_b, v.stride_h, v.stride_n};
    const int ext[3] = {B, H, N};
    const char* dim[3] = {"stride_b", "stride_h", "stride_n"};
    for (int i = 0; i < 3; ++i) {
        if (st[i] < 0 || st[i] % 8 != 0 || st[i] >= (int64_t(1) << 39))
            return fail(FFPA_ERR_INVALID_VALUE, "%s: %s=%lld must be a non-negative multiple of 8 below 2^39", name, dim[i],
                        (long long)st[i]);
        if (ext[i] > 1 && st[i] == 0) return fail(FFPA_ERR_INVALID_VALUE, "%s: %s is 0 for an extent of %d", name, dim[i], ext[i]);
    }
    return FFPA_OK;
}

ffpa::View to_view(const ffpa_view& v) { return ffpa::View{v.stride_b, v.stride_h, v.stride_n}; }

ffpa::Problem dense_problem(int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale)
{
    ffpa::Problem pb{};
    pb.varlen = 0;
    pb.B = B;
    pb.Hq = Hq;
    pb.Hkv = Hkv;
    pb.Nq = Nq;
    pb.Nkv = Nkv;
    pb.D = D;
    pb.causal = causal ? 1 : 0;
    pb.scale = scale;
    pb.scale_log2 = scale * 1.4426950408889634f;
    pb.vq = pb.vo = pb.vdo = pb.vdq = contiguous_view(Hq, Nq, D);
    pb.vk = pb.vv = pb.vdk = pb.vdv = contiguous_view(Hkv, Nkv, D);
    return pb;
}

ffpa_status check_dense_sizes(int B, int Hq, int Nq, int Nkv)
{
    if (B < 0 || Nq < 0 || Nkv < 0) return fail(FFPA_ERR_INVALID_VALUE, "negative size B=%d Nq=%d Nkv=%d", B, Nq, Nkv);
    // (batch, head) pairs index the launch grids as int
    if (static_cast<long>(B) * Hq > INT_MAX || static_cast<long>(B) * Hq * ((Nq > Nkv ? Nq : Nkv) / 128 + 1) > kMaxUnits)
        return fail(FFPA_ERR_NOT_SUPPORTED, "B*Hq=%ld with N=%d exceeds the launch grid's %lld work units", (long)B * Hq,
                    Nq > Nkv ? Nq : Nkv, kMaxUnits);
    return FFPA_OK;
}

ffpa_status check_varlen_sizes(int batch, int total_q, int total_k, int max_q, int max_k, int Hq, const int* cu_q,
                               const int* cu_k)
{
    if (batch < 0 || total_q < 0 || total_k < 0 || max_q < 0 || max_k < 0)
        return fail(FFPA_ERR_INVALID_VALUE, "negative varlen size");
    if (static_cast<long>(batch) * Hq > INT_MAX ||
        static_cast<long>(batch) * Hq * ((max_q > max_k ? max_q : max_k) / 128 + 1) > kMaxUnits)
        return fail(FFPA_ERR_NOT_SUPPORTED, "batch*Hq=%ld with max_seqlen %d exceeds the launch grid's %lld work units",
                    (long)batch * Hq, max_q > max_k ? max_q : max_k, kMaxUnits);
    if (batch > 0 && (!cu_q || !cu_k))
        return fail(FFPA_ERR_INVALID_VALUE, "cu_seqlens_q and cu_seqlens_k are both required (varlen-one-sided)");
    if ((reinterpret_cast<uintptr_t>(cu_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_k) & 3u))
        return fail(FFPA_ERR_INVALID_VALUE, "cu_seqlens must be 4-byte aligned");
    return FFPA_OK;
}

#define FFPA_TRY(x)                              \
    do {                                         \
        const ffpa_status s_ = (x);              \
        if (s_ != FFPA_OK) return s_;            \
    } while (0)

ffpa_status run_fwd(ffpa_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                    const ffpa::Problem& pb, long q_rows, long k_rows, ffpa_stream_t stream)
{
    FFPA_TRY(check_ptr(q, q_rows > 0, "q"));
    FFPA_TRY(check_ptr(o, q_rows > 0, "o"));
    FFPA_TRY(check_ptr(lse, q_rows > 0, "lse"));
    FFPA_TRY(check_ptr(k, q_rows > 0 && k_rows > 0, "k"));
    FFPA_TRY(check_ptr(v, q_rows > 0 && k_rows > 0, "v"));
    if (q_rows == 0) return ok();
    // the forward operation of the cluster-exchange kernel: each unit of a
    // cluster scores its own key tiles, the units agree on the running row
    // maximum and exchange P, and every unit accumulates its head-dim slab of O
    ffpa::XArgs a{};
    a.pb = pb;
    FFPA_TRY(device_ctl(&a.ctl));
    a.bf16 = dt == FFPA_BF16;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    return launch_result(ffpa::launch_xchg(ffpa::XOP_FWD, a, reinterpret_cast<cudaStream_t>(stream)),
                         "forward launch");
}

// Layout of the stored-tile part of a backward workspace (byte offsets; 0 =
// absent) for a workspace of `bytes` whose row statistics take `need`.
struct StoredPlan {
    size_t ds_off, p_off;
    int chunk_groups;  // > 0: chunks of this many kv groups
    size_t used;       // bytes the plan uses
};

StoredPlan stored_plan(const ffpa::Problem& pb, size_t need, size_t bytes, bool chunks_allowed)
{
    StoredPlan s{0, 0, 0, need};
    if (!ffpa::dsq_supported(pb)) return s;
    const size_t t_all = ffpa::dsq_ds_bytes(pb), t_g = ffpa::dsq_group_bytes(pb);
    if (bytes >= need + align256(t_all) + t_all) {  // every head at once
        s.ds_off = need;
        s.p_off = need + align256(t_all);
        s.used = s.p_off + t_all;
        return s;
    }
    if (chunks_allowed && t_g > 0 && bytes >= need + align256(t_g) + t_g) {
        // as many kv groups per chunk as fit, then the chunks evened out
        // (ceil(Hkv / chunks) groups each), so that no launch is a small tail
        long ng = static_cast<long>((bytes - need) / (2 * t_g + 256));
        if (ng < 1) ng = 1;
        while (ng > 1 && need + align256(ng * t_g) + ng * t_g > bytes) --ng;
        const long chunks = (pb.Hkv + ng - 1) / ng;
        ng = (pb.Hkv + chunks - 1) / chunks;
        s.chunk_groups = static_cast<int>(ng);
        s.ds_off = need;
        s.p_off = need + align256(ng * t_g);
        s.used = s.p_off + ng * t_g;
        return s;
    }
    if (bytes >= need + t_all) {  // dS^T of every head
        s.ds_off = need;
        s.used = need + t_all;
    }
    return s;
}

// Largest useful backward workspace within `budget` bytes: every head's tiles
// if they fit, else the largest chunk of kv groups that fits (evened out),
// else the row statistics alone.
size_t budget_bytes(const ffpa::Problem& pb, size_t need, size_t budget)
{
    if (budget <= need) return need;
    return stored_plan(pb, need, budget, true).used;
}

ffpa_status run_bwd(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                    const ffpa::Problem& pb, long q_rows, long k_rows, long stat_rows, unsigned stages,
                    ffpa_stream_t stream)
{
    const bool any = q_rows > 0 || k_rows > 0;
    FFPA_TRY(check_ptr(q, q_rows > 0, "q"));
    FFPA_TRY(check_ptr(o, q_rows > 0, "o"));
    FFPA_TRY(check_ptr(lse, q_rows > 0, "lse"));
    FFPA_TRY(check_ptr(dO, q_rows > 0, "dO"));
    FFPA_TRY(check_ptr(dq, q_rows > 0, "dq"));
    FFPA_TRY(check_ptr(k, k_rows > 0, "k"));
    FFPA_TRY(check_ptr(v, k_rows > 0, "v"));
    FFPA_TRY(check_ptr(dk, k_rows > 0, "dk"));
    FFPA_TRY(check_ptr(dv, k_rows > 0, "dv"));
    const size_t need = ws_bytes(stat_rows);
    if (workspace_bytes < need)
        return fail(FFPA_ERR_INVALID_VALUE, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(FFPA_ERR_INVALID_VALUE, "workspace must be non-NULL and 256-byte aligned");
    if (!any) return ok();
    ffpa::BwdArgs a{};
    a.pb = pb;
    a.stages = stages & 63u;
    // The workspace after the row statistics decides the stored-tile path
    // (where it applies): room for dS^T and P^T of every head has the dK
    // launch store both, and dV and dQ are GEMMs over them; room for both
    // tile sets of at least one kv group (and a call that runs dV, dK and dQ)
    // runs that path in chunks of as many groups as fit; room for dS^T of
    // every head alone stores dS only (dV recomputes); less recomputes.
    a.ds = nullptr;
    a.p = nullptr;
    a.chunk_groups = 0;
    const StoredPlan plan = stored_plan(pb, need, workspace_bytes, (stages & 14u) == 14u && !(stages & 48u));
    if (plan.ds_off) a.ds = static_cast<char*>(workspace) + plan.ds_off;
    if (plan.p_off) a.p = static_cast<char*>(workspace) + plan.p_off;
    a.chunk_groups = plan.chunk_groups;
    if ((a.stages & 16u) && a.ds == nullptr)
        return fail(FFPA_ERR_INVALID_VALUE, "stage bit 4 (dQ from stored dS) needs the larger workspace of "
                                            "ffpa_bwd_workspace_bytes_ds on a dense problem with D % 64 == 0, D <= 1024");
    if ((a.stages & 32u) && a.p == nullptr)
        return fail(FFPA_ERR_INVALID_VALUE, "stage bit 5 (stored P) needs the workspace of "
                                            "ffpa_bwd_workspace_bytes_ds on a dense problem with D % 64 == 0, D <= 1024");
    FFPA_TRY(device_ctl(&a.ctl));
    a.bf16 = dt == FFPA_BF16;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.dO = dO;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.delta = static_cast<float*>(workspace);
    a.lse_log2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + need / 2);
    return launch_result(ffpa::launch_bwd(a, reinterpret_cast<cudaStream_t>(stream)), "backward launch");
}

ffpa::Problem varlen_problem(int batch, int total_q, int total_k, int max_q, int max_k, int Hq, int Hkv, int D,
                             int causal, float scale, const int* cu_q, const int* cu_k)
{
    ffpa::Problem pb = dense_problem(batch, Hq, Hkv, max_q, max_k, D, causal, scale);
    pb.varlen = 1;
    pb.total_q = total_q;
    pb.total_k = total_k;
    pb.cu_q = cu_q;
    pb.cu_k = cu_k;
    pb.vq = pb.vo = pb.vdo = pb.vdq = packed_view(Hq, D);
    pb.vk = pb.vv = pb.vdk = pb.vdv = packed_view(Hkv, D);
    return pb;
}

__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ffpa::mbar_init(&bar, 1);
        abort_flag = 0;
        ffpa::fence_barrier_init();
        // nothing ever arrives on `bar`: the wait must give up by itself
        ffpa::mbar_wait(&bar, 0, &abort_flag, status, limit_ns, 255);
    }
}

}  // namespace

int ffpa::set_error(int status, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return status;
}

extern "C" {

ffpa_status ffpa_fwd(ffpa_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                     int Hkv, int Nq, int Nkv, int D, int causal, float scale, ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_dense_sizes(B, Hq, Nq, Nkv));
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    const long k_rows = static_cast<long>(B) * Hkv * Nkv;
    return run_fwd(dt, q, k, v, o, lse, dense_problem(B, Hq, Hkv, Nq, Nkv, D, causal, scale), q_rows, k_rows, stream);
}

ffpa_status ffpa_fwd_strided(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, ffpa_view o, float* lse, int B,
                             int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale, ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_dense_sizes(B, Hq, Nq, Nkv));
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    const long k_rows = static_cast<long>(B) * Hkv * Nkv;
    FFPA_TRY(check_view(q, q_rows > 0, "q", B, Hq, Nq));
    FFPA_TRY(check_view(o, q_rows > 0, "o", B, Hq, Nq));
    FFPA_TRY(check_view(k, q_rows > 0 && k_rows > 0, "k", B, Hkv, Nkv));
    FFPA_TRY(check_view(v, q_rows > 0 && k_rows > 0, "v", B, Hkv, Nkv));
    ffpa::Problem pb = dense_problem(B, Hq, Hkv, Nq, Nkv, D, causal, scale);
    pb.vq = to_view(q);
    pb.vo = to_view(o);
    pb.vk = to_view(k);
    pb.vv = to_view(v);
    return run_fwd(dt, q.data, k.data, v.data, o.data, lse, pb, q_rows, k_rows, stream);
}

size_t ffpa_decode_workspace_bytes(ffpa_dtype, int B, int Hq, int Hkv, int Nq, int Nkv, int D)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nkv < 0 || D <= 0 || Hq % Hkv != 0) return 0;
    return ffpa::decode_plan(dense_problem(B, Hq, Hkv, Nq, Nkv, D, 0, 1.f)).workspace_bytes;
}

ffpa_status ffpa_decode_fwd(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, ffpa_view o, float* lse,
                            void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                            int causal, float scale, ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_dense_sizes(B, Hq, Nq, Nkv));
    if (D % 64 != 0) return fail(FFPA_ERR_NOT_SUPPORTED, "decode path: D=%d must be a multiple of 64", D);
    if (Hq > 0 && static_cast<long long>(B) * Hkv * ((static_cast<long long>(Hq / Hkv) * Nq + ffpa::kDecodeRows - 1) /
                                                     ffpa::kDecodeRows) > kMaxUnits)
        return fail(FFPA_ERR_NOT_SUPPORTED, "decode path: B*Hkv*ceil((Hq/Hkv)*Nq/%d) exceeds the grid's %lld units",
                    ffpa::kDecodeRows, kMaxUnits);
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    const long k_rows = static_cast<long>(B) * Hkv * Nkv;
    FFPA_TRY(check_view(q, q_rows > 0, "q", B, Hq, Nq));
    FFPA_TRY(check_view(o, q_rows > 0, "o", B, Hq, Nq));
    FFPA_TRY(check_view(k, q_rows > 0 && k_rows > 0, "k", B, Hkv, Nkv));
    FFPA_TRY(check_view(v, q_rows > 0 && k_rows > 0, "v", B, Hkv, Nkv));
    FFPA_TRY(check_ptr(lse, q_rows > 0, "lse"));
    if (q_rows == 0) return ok();
    ffpa::Problem pb = dense_problem(B, Hq, Hkv, Nq, Nkv, D, causal, scale);
    pb.vq = to_view(q);
    pb.vo = to_view(o);
    pb.vk = to_view(k);
    pb.vv = to_view(v);
    const size_t need = ffpa::decode_plan(pb).workspace_bytes;
    if (workspace_bytes < need)
        return fail(FFPA_ERR_INVALID_VALUE, "decode workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(FFPA_ERR_INVALID_VALUE, "decode workspace must be non-NULL and 256-byte aligned");
    ffpa::FwdArgs a{};
    a.pb = pb;
    FFPA_TRY(device_ctl(&a.ctl));
    a.bf16 = dt == FFPA_BF16;
    a.q = q.data;
    a.k = k.data;
    a.v = v.data;
    a.o = o.data;
    a.lse = lse;
    return launch_result(ffpa::launch_decode(a, workspace, reinterpret_cast<cudaStream_t>(stream)), "decode launch");
}

size_t ffpa_fp8_workspace_layout(int B, int Hq, int Hkv, int Nq, int Nkv, int D, size_t* offsets)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nkv < 0 || D < 64 || D > 1024 || Hq % Hkv != 0 || D % 32 != 0)
        return 0;
    const ffpa::Fp8Layout L = ffpa::fp8_layout(B, Hq, Hkv, Nq, Nkv, D);
    if (offsets) {
        offsets[0] = L.q8;
        offsets[1] = L.k8;
        offsets[2] = L.v8t;
        offsets[3] = L.sq;
        offsets[4] = L.sk;
        offsets[5] = L.sv;
        offsets[6] = static_cast<size_t>(L.ldv);
        offsets[7] = L.total;
    }
    return L.total;
}

size_t ffpa_fp8_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nkv, int D)
{
    return ffpa_fp8_workspace_layout(B, Hq, Hkv, Nq, Nkv, D, nullptr);
}

}  // extern "C"

namespace {

// Validation shared by the FP8 entry points; fills `pb` on success.
ffpa_status check_fp8(ffpa_dtype dt, const ffpa_view& q, const ffpa_view& k, const ffpa_view& v, const void* ws,
                      size_t ws_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D, float scale, ffpa::Problem* pb)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_dense_sizes(B, Hq, Nq, Nkv));
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    if (q_rows > 0 && Nkv < 1) return fail(FFPA_ERR_NOT_SUPPORTED, "fp8 forward: Nkv must be >= 1");
    FFPA_TRY(check_view(q, q_rows > 0, "q", B, Hq, Nq));
    FFPA_TRY(check_view(k, q_rows > 0, "k", B, Hkv, Nkv));
    FFPA_TRY(check_view(v, q_rows > 0, "v", B, Hkv, Nkv));
    if (q_rows > 0) {
        const size_t need = ffpa::fp8_layout(B, Hq, Hkv, Nq, Nkv, D).total;
        if (ws_bytes < need)
            return fail(FFPA_ERR_INVALID_VALUE, "fp8 workspace too small: %zu < %zu bytes", ws_bytes, need);
        if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u))
            return fail(FFPA_ERR_INVALID_VALUE, "fp8 workspace must be non-NULL and 256-byte aligned");
    }
    *pb = dense_problem(B, Hq, Hkv, Nq, Nkv, D, 0, scale);
    pb->vq = to_view(q);
    pb->vk = to_view(k);
    pb->vv = to_view(v);
    return ok();
}

}  // namespace

extern "C" {

ffpa_status ffpa_fp8_quantize(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, void* workspace,
                              size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                              ffpa_stream_t stream)
{
    ffpa::Problem pb;
    FFPA_TRY(check_fp8(dt, q, k, v, workspace, workspace_bytes, B, Hq, Hkv, Nq, Nkv, D, 1.f, &pb));
    if (static_cast<long>(B) * Hq * Nq == 0) return ok();
    ffpa::FwdArgs a{};
    a.pb = pb;
    FFPA_TRY(device_ctl(&a.ctl));
    a.bf16 = dt == FFPA_BF16;
    a.q = q.data;
    a.k = k.data;
    a.v = v.data;
    return launch_result(ffpa::launch_fp8_quantize(a, workspace, reinterpret_cast<cudaStream_t>(stream)),
                         "fp8 quantize launch");
}

ffpa_status ffpa_fwd_fp8(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, ffpa_view o, float* lse,
                         void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D,
                         int causal, float scale, ffpa_stream_t stream)
{
    ffpa::Problem pb;
    FFPA_TRY(check_fp8(dt, q, k, v, workspace, workspace_bytes, B, Hq, Hkv, Nq, Nkv, D, scale, &pb));
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    FFPA_TRY(check_view(o, q_rows > 0, "o", B, Hq, Nq));
    FFPA_TRY(check_ptr(lse, q_rows > 0, "lse"));
    if (q_rows == 0) return ok();
    pb.causal = causal != 0;
    pb.vo = to_view(o);
    ffpa::FwdArgs a{};
    a.pb = pb;
    FFPA_TRY(device_ctl(&a.ctl));
    a.bf16 = dt == FFPA_BF16;
    a.q = q.data;
    a.k = k.data;
    a.v = v.data;
    a.o = o.data;
    a.lse = lse;
    return launch_result(ffpa::launch_fwd_fp8(a, workspace, reinterpret_cast<cudaStream_t>(stream), true),
                         "fp8 launch");
}

ffpa_status ffpa_fwd_fp8_quantized(ffpa_dtype dt, ffpa_view o, float* lse, const void* workspace,
                                   size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal,
                                   float scale, ffpa_stream_t stream)
{
    // the views of q/k/v are not read: validate with dense views over the workspace
    void* ws = const_cast<void*>(workspace);
    const ffpa_view vq{ws, static_cast<long long>(Hq) * Nq * D, static_cast<long long>(Nq) * D, D};
    const ffpa_view vk{ws, static_cast<long long>(Hkv) * Nkv * D, static_cast<long long>(Nkv) * D, D};
    ffpa::Problem pb;
    FFPA_TRY(check_fp8(dt, vq, vk, vk, workspace, workspace_bytes, B, Hq, Hkv, Nq, Nkv, D, scale, &pb));
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    FFPA_TRY(check_view(o, q_rows > 0, "o", B, Hq, Nq));
    FFPA_TRY(check_ptr(lse, q_rows > 0, "lse"));
    if (q_rows == 0) return ok();
    pb.causal = causal != 0;
    pb.vo = to_view(o);
    ffpa::FwdArgs a{};
    a.pb = pb;
    FFPA_TRY(device_ctl(&a.ctl));
    a.bf16 = dt == FFPA_BF16;
    a.o = o.data;
    a.lse = lse;
    return launch_result(ffpa::launch_fwd_fp8(a, const_cast<void*>(workspace),
                                              reinterpret_cast<cudaStream_t>(stream), false),
                         "fp8 launch");
}

size_t ffpa_varlen_fp8_workspace_bytes(int batch, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int Hq,
                                       int Hkv, int D)
{
    if (batch <= 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || Hq <= 0 || Hkv <= 0 ||
        D < 64 || D > 1024 || Hq % Hkv != 0 || D % 32 != 0)
        return 0;
    return ffpa::fp8_varlen_layout(batch, Hq, Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, D).total;
}

ffpa_status ffpa_varlen_fwd_fp8(ffpa_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                                const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int total_q,
                                int total_k, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D, int causal,
                                float scale, void* workspace, size_t workspace_bytes, ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_varlen_sizes(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, cu_seqlens_q, cu_seqlens_k));
    const long q_rows = batch > 0 ? static_cast<long>(total_q) * Hq : 0;
    if (q_rows > 0 && total_k < 1) return fail(FFPA_ERR_NOT_SUPPORTED, "fp8 forward: total_k must be >= 1");
    FFPA_TRY(check_ptr(q, q_rows > 0, "q"));
    FFPA_TRY(check_ptr(k, q_rows > 0, "k"));
    FFPA_TRY(check_ptr(v, q_rows > 0, "v"));
    FFPA_TRY(check_ptr(o, q_rows > 0, "o"));
    FFPA_TRY(check_ptr(lse, q_rows > 0, "lse"));
    if (q_rows == 0) return ok();
    const size_t need =
        ffpa::fp8_varlen_layout(batch, Hq, Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, D).total;
    if (workspace_bytes < need)
        return fail(FFPA_ERR_INVALID_VALUE, "fp8 workspace too small: %zu < %zu bytes", workspace_bytes, need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(FFPA_ERR_INVALID_VALUE, "fp8 workspace must be non-NULL and 256-byte aligned");
    ffpa::FwdArgs a{};
    a.pb = varlen_problem(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, causal, scale, cu_seqlens_q,
                          cu_seqlens_k);
    FFPA_TRY(device_ctl(&a.ctl));
    a.bf16 = dt == FFPA_BF16;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    return launch_result(ffpa::launch_fwd_fp8(a, workspace, reinterpret_cast<cudaStream_t>(stream), true),
                         "fp8 varlen launch");
}

size_t ffpa_bwd_workspace_bytes_ds(ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal)
{
    const size_t small = ffpa_bwd_workspace_bytes(dt, B, Hq, Hkv, Nq, Nkv, D);
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nkv <= 0 || Hq % Hkv != 0) return small;
    const ffpa::Problem pb = dense_problem(B, Hq, Hkv, Nq, Nkv, D, causal, 1.f);
    // dS^T, then P^T at the next 256-byte boundary
    return ffpa::dsq_supported(pb) ? small + align256(ffpa::dsq_ds_bytes(pb)) + ffpa::dsq_ds_bytes(pb) : small;
}

size_t ffpa_bwd_workspace_bytes_budget(ffpa_dtype dt, int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal,
                                       size_t budget)
{
    const size_t small = ffpa_bwd_workspace_bytes(dt, B, Hq, Hkv, Nq, Nkv, D);
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nkv <= 0 || Hq % Hkv != 0) return small;
    return budget_bytes(dense_problem(B, Hq, Hkv, Nq, Nkv, D, causal, 1.f), small, budget);
}

size_t ffpa_bwd_workspace_bytes(ffpa_dtype, int B, int Hq, int, int Nq, int, int)
{
    if (B < 0 || Hq < 0 || Nq < 0) return 0;
    return ws_bytes(static_cast<long>(B) * Hq * Nq);
}

ffpa_status ffpa_bwd(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B,
                     int Hq, int Hkv, int Nq, int Nkv, int D, int causal, float scale, ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_dense_sizes(B, Hq, Nq, Nkv));
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    const long k_rows = static_cast<long>(B) * Hkv * Nkv;
    return run_bwd(dt, q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes,
                   dense_problem(B, Hq, Hkv, Nq, Nkv, D, causal, scale), q_rows, k_rows, q_rows, 15u, stream);
}

ffpa_status ffpa_bwd_strided(ffpa_dtype dt, ffpa_view q, ffpa_view k, ffpa_view v, ffpa_view o, const float* lse,
                             ffpa_view dO, ffpa_view dq, ffpa_view dk, ffpa_view dv, void* workspace,
                             size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal,
                             float scale, ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_dense_sizes(B, Hq, Nq, Nkv));
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    const long k_rows = static_cast<long>(B) * Hkv * Nkv;
    FFPA_TRY(check_view(q, q_rows > 0, "q", B, Hq, Nq));
    FFPA_TRY(check_view(o, q_rows > 0, "o", B, Hq, Nq));
    FFPA_TRY(check_view(dO, q_rows > 0, "dO", B, Hq, Nq));
    FFPA_TRY(check_view(dq, q_rows > 0, "dq", B, Hq, Nq));
    FFPA_TRY(check_view(k, k_rows > 0, "k", B, Hkv, Nkv));
    FFPA_TRY(check_view(v, k_rows > 0, "v", B, Hkv, Nkv));
    FFPA_TRY(check_view(dk, k_rows > 0, "dk", B, Hkv, Nkv));
    FFPA_TRY(check_view(dv, k_rows > 0, "dv", B, Hkv, Nkv));
    ffpa::Problem pb = dense_problem(B, Hq, Hkv, Nq, Nkv, D, causal, scale);
    pb.vq = to_view(q);
    pb.vo = to_view(o);
    pb.vdo = to_view(dO);
    pb.vdq = to_view(dq);
    pb.vk = to_view(k);
    pb.vv = to_view(v);
    pb.vdk = to_view(dk);
    pb.vdv = to_view(dv);
    return run_bwd(dt, q.data, k.data, v.data, o.data, lse, dO.data, dq.data, dk.data, dv.data, workspace,
                   workspace_bytes, pb, q_rows, k_rows, q_rows, 15u, stream);
}

ffpa_status ffpa_bwd_stages(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, int B, int Hq, int Hkv, int Nq, int Nkv, int D, int causal,
                            float scale, unsigned stages, ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_dense_sizes(B, Hq, Nq, Nkv));
    if (stages > 63u) return fail(FFPA_ERR_INVALID_VALUE, "stages mask %u: only bits 0..5", stages);
    const long q_rows = static_cast<long>(B) * Hq * Nq;
    const long k_rows = static_cast<long>(B) * Hkv * Nkv;
    return run_bwd(dt, q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes,
                   dense_problem(B, Hq, Hkv, Nq, Nkv, D, causal, scale), q_rows, k_rows, q_rows, stages, stream);
}

ffpa_status ffpa_varlen_fwd(ffpa_dtype dt, const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k, int batch, int total_q, int total_k,
                            int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D, int causal, float scale,
                            ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_varlen_sizes(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, cu_seqlens_q, cu_seqlens_k));
    const long q_rows = batch > 0 ? static_cast<long>(total_q) * Hq : 0;
    const long k_rows = batch > 0 ? static_cast<long>(total_k) * Hkv : 0;
    return run_fwd(dt, q, k, v, o, lse,
                   varlen_problem(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, causal, scale,
                                  cu_seqlens_q, cu_seqlens_k),
                   q_rows, k_rows, stream);
}

size_t ffpa_varlen_bwd_workspace_bytes(ffpa_dtype, int batch, int total_q, int, int, int, int Hq, int, int)
{
    if (batch <= 0 || total_q < 0 || Hq < 0) return 0;
    return ws_bytes(static_cast<long>(total_q) * Hq);
}

size_t ffpa_varlen_bwd_workspace_bytes_ds(ffpa_dtype dt, int batch, int total_q, int total_k, int max_seqlen_q,
                                          int max_seqlen_k, int Hq, int Hkv, int D, int causal)
{
    const size_t small =
        ffpa_varlen_bwd_workspace_bytes(dt, batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, Hkv, D);
    if (batch <= 0 || total_q <= 0 || total_k <= 0 || max_seqlen_q <= 0 || max_seqlen_k <= 0 || Hq <= 0 ||
        Hkv <= 0 || Hq % Hkv != 0)
        return small;
    const ffpa::Problem pb = varlen_problem(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, causal,
                                            1.f, nullptr, nullptr);
    // dS^T, then P^T at the next 256-byte boundary
    return ffpa::dsq_supported(pb) ? small + align256(ffpa::dsq_ds_bytes(pb)) + ffpa::dsq_ds_bytes(pb) : small;
}

size_t ffpa_varlen_bwd_workspace_bytes_budget(ffpa_dtype dt, int batch, int total_q, int total_k, int max_seqlen_q,
                                              int max_seqlen_k, int Hq, int Hkv, int D, int causal, size_t budget)
{
    const size_t small =
        ffpa_varlen_bwd_workspace_bytes(dt, batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, Hkv, D);
    if (batch <= 0 || total_q <= 0 || total_k <= 0 || max_seqlen_q <= 0 || max_seqlen_k <= 0 || Hq <= 0 ||
        Hkv <= 0 || Hq % Hkv != 0)
        return small;
    return budget_bytes(varlen_problem(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, causal, 1.f,
                                       nullptr, nullptr),
                        small, budget);
}

ffpa_status ffpa_varlen_bwd(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                            const int* cu_seqlens_k, int batch, int total_q, int total_k, int max_seqlen_q,
                            int max_seqlen_k, int Hq, int Hkv, int D, int causal, float scale, void* workspace,
                            size_t workspace_bytes, ffpa_stream_t stream)
{
    FFPA_TRY(check_common(dt, Hq, Hkv, D, scale));
    FFPA_TRY(check_varlen_sizes(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, cu_seqlens_q, cu_seqlens_k));
    const long q_rows = batch > 0 ? static_cast<long>(total_q) * Hq : 0;
    const long k_rows = batch > 0 ? static_cast<long>(total_k) * Hkv : 0;
    return run_bwd(dt, q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes,
                   varlen_problem(batch, total_q, total_k, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, causal, scale,
                                  cu_seqlens_q, cu_seqlens_k),
                   q_rows, k_rows, q_rows, 15u, stream);
}

ffpa_status ffpa_get_status(ffpa_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(FFPA_ERR_CUDA, "stream error: %s", cudaGetErrorString(e));
    uint32_t word = 0;
    e = cudaMemcpyFromSymbol(&word, g_ffpa_status_word, sizeof(word));
    if (e != cudaSuccess) return fail(FFPA_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
    if (word == 0) return ok();
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_ffpa_status_word, &zero, sizeof(zero));
    if ((word & 0xffu) == ffpa::DEV_TIMEOUT)
        return fail(FFPA_ERR_TIMEOUT, "a device wait timed out (site %u, block %u)", (word >> 8) & 0xffu, word >> 16);
    if ((word & 0xffu) == ffpa::DEV_INVALID)
        return fail(FFPA_ERR_INVALID_VALUE,
                    "packed sequence %u breaks the varlen contract: its cu_seqlens entries are negative, decrease or "
                    "run past total_q / total_k, or its length exceeds max_seqlen_q / max_seqlen_k (which size the "
                    "launch); the outputs of that call are undefined (site 0x%02x)",
                    word >> 16, (word >> 8) & 0xffu);
    return fail(FFPA_ERR_CUDA, "device status word 0x%08x", word);
}

const char* ffpa_last_error(void) { return g_err.c_str(); }

void ffpa_set_wait_limit_ns(uint64_t ns) { g_limit_ns.store(ns ? ns : 2000000000ull); }

ffpa_status ffpa_selftest_wait_timeout(uint64_t limit_ns, ffpa_stream_t stream)
{
    bool cc_ok = false;
    uint32_t* st = nullptr;
    if (!device_state(&st, &cc_ok)) return fail(FFPA_ERR_CUDA, "no usable CUDA device");
    selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(st, limit_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(FFPA_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
    return ffpa_get_status(stream);
}

int ffpa_num_sms(void) { return ffpa::num_sms(); }

}  // extern "C"
