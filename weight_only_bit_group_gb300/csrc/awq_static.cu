// awq_static.cu -- awq_search for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they want to run the
// search: code that runs inside a memory-pool or arena owned by someone else,
// plug-ins of a host framework that forbids allocations on its worker threads,
// or code paths that must not synchronise the device (cudaMalloc can).  This
// entry point takes the same inputs and outputs as awq_search but needs no
// caller workspace: its scratch lives in a fixed array compiled into this
// library, which every GPU that loads the library holds until the process exits.
//
// How it works: on the first call in a CUDA context of a device (that device
// must be current), the device address of the array is looked up once with
// cudaGetSymbolAddress and cached together with the context's unique id; in host
// code the array's name is only a host-side stand-in, so the kernels must be
// handed that looked-up address.  Make that first call before any stream capture
// on the device.  A later call in a new context of the same device (after
// cudaDeviceReset, say) sees a different context id and looks the address up
// again.  A stream that belongs to another device than the current one is
// refused.  The call then runs the ordinary awq_search with the array as its
// workspace.  Every call shares the array and leaves the previous call's
// contents in it; no byte of it needs to start at zero, because each call writes
// every scratch byte it later reads (the arrival counter is cleared by a memset
// on the stream).  Calls that overlap on the GPU (other streams, other host
// threads) race on the array and must be serialised by the caller.
#include <mutex>

#include "wq_common.cuh"

namespace {

constexpr int64_t kStaticMaxK = 16384;
constexpr int kStaticMaxAlpha = 16;

// Workspace layout of awq_search for k = 16384, n_alpha = 16 (see
// wq_workspace_bytes): control block, two [16][16384] binary32 tables,
// a_c [16384], ln(an) and an [16384], 4096 x 16 binary64 partials.
constexpr size_t kStaticScratchBytes =
    256 + 2 * (size_t)kStaticMaxAlpha * kStaticMaxK * 4 + (size_t)kStaticMaxK * 4 +
    (size_t)kStaticMaxK * 12 + (size_t)4096 * kStaticMaxAlpha * 8;

static __device__ __align__(256) unsigned char g_awq_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_addr[64] = {nullptr};
unsigned long long g_ctx[64] = {0};

// cuCtxGetId through the runtime's driver entry point (no link-time dependency
// on the driver library): a context id that is unique for the life of the process.
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);
CtxGetIdFn ctx_get_id() {
    static CtxGetIdFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        cudaGetLastError();
        return (CtxGetIdFn)p;
    }();
    return fn;
}

// Device address of g_awq_scratch in the current context (looked up once per
// context), after checking that `stream` belongs to the current device.
wq_status scratch_address(cudaStream_t stream, void** out) {
    int dev = 0, sdev = 0;
    wq_status s = wqh::cuda_status(cudaGetDevice(&dev));
    if (s != WQ_OK) return s;
    if (dev < 0 || dev >= 64) return WQ_ERR_UNSUPPORTED;
    s = wqh::cuda_status(cudaStreamGetDevice(stream, &sdev));
    if (s != WQ_OK) return s;
    if (sdev != dev) return WQ_ERR_UNSUPPORTED;  // the stream of another device
    CtxGetIdFn get_id = ctx_get_id();
    if (!get_id) return WQ_ERR_UNSUPPORTED;
    unsigned long long id = 0;
    if (get_id(nullptr, &id) != 0 || id == 0) {
        // no context current on this thread yet: the symbol lookup makes the
        // runtime create (or bind) the device's primary context
        void* p = nullptr;
        s = wqh::cuda_status(cudaGetSymbolAddress(&p, g_awq_scratch));
        if (s != WQ_OK) return s;
        if (get_id(nullptr, &id) != 0 || id == 0) return WQ_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev] || g_ctx[dev] != id) {
        void* p = nullptr;
        s = wqh::cuda_status(cudaGetSymbolAddress(&p, g_awq_scratch));
        if (s != WQ_OK) return s;
        g_addr[dev] = p;
        g_ctx[dev] = id;
    }
    *out = g_addr[dev];
    return WQ_OK;
}

}  // namespace

extern "C" wq_status awq_search_static_scratch(const uint16_t* w, int64_t n, int64_t k,
                                               const float* a, const float* alphas_host,
                                               int n_alpha, int max_rows, int tie_mode,
                                               float* best_s, int32_t* best_idx,
                                               float* best_alpha, double* errs, void* stream) {
    // the same codes as awq_search for the same conditions; then the array's limit
    if (n <= 0 || k <= 0 || k % 32 != 0) return WQ_ERR_BAD_SHAPE;
    if (n_alpha < 1 || n_alpha > kStaticMaxAlpha || max_rows < 1) return WQ_ERR_UNSUPPORTED;
    if (k > kStaticMaxK) return WQ_ERR_BAD_SHAPE;
    const size_t need = wq_workspace_bytes(WQ_OP_AWQ_SEARCH, n, k, n_alpha);
    if (need > kStaticScratchBytes) return WQ_ERR_BAD_SHAPE;
    if (!w || !a || !alphas_host) return WQ_ERR_NULL_PTR;
    void* scratch = nullptr;
    wq_status s = scratch_address((cudaStream_t)stream, &scratch);
    if (s != WQ_OK) return s;
    return awq_search(w, n, k, a, alphas_host, n_alpha, max_rows, tie_mode, best_s, best_idx,
                      best_alpha, errs, scratch, kStaticScratchBytes, stream);
}
