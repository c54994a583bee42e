// ffpa_bwd_noalloc: the dense backward for callers that cannot allocate
// device memory.
//
// ffpa_bwd needs a few bytes of fp32 scratch per query row (the row sums
// delta = dO.O and the scaled LSE) and asks the caller for it. Some callers
// have no way to provide it: code running inside a fixed, pre-planned memory
// pool with no spare buffer (inference servers, plugin hosts of other
// frameworks, embedded runtimes), or code on a latency path where a
// cudaMalloc/cudaFree pair would synchronise the device. For them this entry
// point takes its scratch from one array that lives in this library's device
// image, so the call allocates nothing at all.
//
// The array holds kNoAllocMaxRows query rows; every GPU that loads the
// library keeps those 4 MiB until the process exits. All calls on a device
// share it, so two calls whose kernels overlap on the GPU (different streams
// without ordering between them) race on it; calls on one stream are fine.
// Each call hands ffpa_bwd exactly the workspace size that ffpa_bwd asks for
// (the per-row statistics only), never the whole array: the backward then
// always runs the same kernels (preprocess, dV, dK, dQ, each recomputing its
// scores), whatever the problem size, and never the stored-tile path that a
// larger workspace would select. Nothing in the array has to start at zero:
// the preprocess kernel of each call writes delta and the scaled LSE of every
// row before the gradient kernels of that call read them, and the contents
// left by the previous call are never read.
#include <mutex>

#include "../../include/ffpa.h"
#include "kernels.h"

namespace {

constexpr long kNoAllocMaxRows = 1L << 19;  // B*Hq*Nq limit: 524288 query rows
constexpr size_t kNoAllocBytes = 2 * kNoAllocMaxRows * sizeof(float);
constexpr int kMaxDevices = 64;

// delta[kNoAllocMaxRows] followed by lse2[kNoAllocMaxRows]. In host code this
// name is only a stand-in for the device symbol: its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[2 * kNoAllocMaxRows];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device. Looked up once
// per device, with that device current, on the first call that needs it.
// A cudaDeviceReset unloads the library's device image, after which that
// address is stale: the call is not valid after a reset of its device in the
// same process.
void* scratch_address(const char** why)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *why = "no usable CUDA device";
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            *why = cudaGetErrorString(e);
            return nullptr;
        }
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

ffpa_status ffpa_bwd_noalloc(ffpa_dtype dt, const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                             int Nq, int Nkv, int D, int causal, float scale, ffpa_stream_t stream)
{
    const long rows = static_cast<long>(B) * Hq * Nq;
    if (rows > kNoAllocMaxRows)
        return static_cast<ffpa_status>(ffpa::set_error(
            FFPA_ERR_INVALID_VALUE,
            "ffpa_bwd_noalloc: B*Hq*Nq = %ld query rows exceeds its built-in scratch of %ld rows; "
            "use ffpa_bwd with a caller-provided workspace",
            rows, kNoAllocMaxRows));
    if (rows <= 0)  // no query rows: no scratch is read; ffpa_bwd validates and zero-fills dK/dV
        return ffpa_bwd(dt, q, k, v, o, lse, dO, dq, dk, dv, nullptr, 0, B, Hq, Hkv, Nq, Nkv, D, causal, scale,
                        stream);
    const char* why = "";
    void* scratch = scratch_address(&why);
    if (!scratch)
        return static_cast<ffpa_status>(
            ffpa::set_error(FFPA_ERR_CUDA, "ffpa_bwd_noalloc: scratch address lookup failed: %s", why));
    // the size ffpa_bwd asks for (row statistics only; within kNoAllocBytes by the check above)
    const size_t bytes = ffpa_bwd_workspace_bytes(dt, B, Hq, Hkv, Nq, Nkv, D);
    return ffpa_bwd(dt, q, k, v, o, lse, dO, dq, dk, dv, scratch, bytes, B, Hq, Hkv, Nq, Nkv, D, causal, scale,
                    stream);
}

}  // extern "C"
