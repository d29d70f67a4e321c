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
// How it works: on the first call on a device (that device must be current),
// the device address of the array is looked up once with cudaGetSymbolAddress
// and cached; in host code the array's name is only a host-side stand-in, so
// the kernels must be handed that looked-up address.  Make that first call
// before any stream capture on the device.  The call then runs the ordinary
// awq_search with the array as its workspace.  Every call shares the array and
// leaves the previous call's contents in it; no byte of it needs to start at
// zero, because each call writes every scratch byte it later reads.  Calls that
// overlap on the GPU (other streams, other host threads) race on the array and
// must be serialised by the caller.
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

// Device address of g_awq_scratch on the current device (looked up once).
wq_status scratch_address(void** out) {
    int dev = 0;
    wq_status s = wqh::cuda_status(cudaGetDevice(&dev));
    if (s != WQ_OK) return s;
    if (dev < 0 || dev >= 64) return WQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        s = wqh::cuda_status(cudaGetSymbolAddress(&p, g_awq_scratch));
        if (s != WQ_OK) return s;
        g_addr[dev] = p;
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
    if (k > kStaticMaxK || n_alpha > kStaticMaxAlpha) return WQ_ERR_BAD_SHAPE;
    const size_t need = wq_workspace_bytes(WQ_OP_AWQ_SEARCH, n, k, n_alpha);
    if (need > kStaticScratchBytes) return WQ_ERR_BAD_SHAPE;
    if (n <= 0 || k <= 0 || k % 32 != 0) return WQ_ERR_BAD_SHAPE;
    if (!w || !a || !alphas_host) return WQ_ERR_NULL_PTR;
    void* scratch = nullptr;
    wq_status s = scratch_address(&scratch);
    if (s != WQ_OK) return s;
    return awq_search(w, n, k, a, alphas_host, n_alpha, max_rows, tie_mode, best_s, best_idx,
                      best_alpha, errs, scratch, kStaticScratchBytes, stream);
}
