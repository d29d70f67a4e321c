// common.cu -- host-side helpers of the C ABI: status strings, launch sizing,
// CUDA error capture and the pure-arithmetic size queries.
#include <mutex>
#include <string.h>

#include "wq_common.cuh"

namespace {
thread_local char g_last_cuda_error[256] = "";

struct KernelKey {
    const void* fn;
    int device;
    int threads;
    size_t smem;
};
std::mutex g_mu;
constexpr int kMaxCache = 128;
KernelKey g_keys[kMaxCache];
int g_vals[kMaxCache];
int g_ncache = 0;
int g_sms[64] = {0};
}  // namespace

namespace wqh {

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (g_sms[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 1;
        g_sms[dev] = v;
    }
    return g_sms[dev];
}

// Grid for a grid-stride kernel: enough CTAs to fill every SM to its occupancy
// limit, never more than the work needs or than `cap`.
int grid_for(const void* kernel, int threads, size_t smem, int64_t work_items, int cap) {
    int dev = 0;
    cudaGetDevice(&dev);
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        for (int i = 0; i < g_ncache; ++i)
            if (g_keys[i].fn == kernel && g_keys[i].device == dev && g_keys[i].threads == threads &&
                g_keys[i].smem == smem)
                per_sm = g_vals[i];
    }
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
                cudaSuccess ||
            per_sm <= 0) {
            cudaGetLastError();
            per_sm = 1;
        }
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_ncache < kMaxCache) {
            g_keys[g_ncache] = KernelKey{kernel, dev, threads, smem};
            g_vals[g_ncache] = per_sm;
            ++g_ncache;
        }
    }
    int64_t g = (int64_t)sm_count() * per_sm;
    if (g > work_items) g = work_items;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

wq_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return WQ_OK;
    strncpy(g_last_cuda_error, cudaGetErrorString(e), sizeof(g_last_cuda_error) - 1);
    g_last_cuda_error[sizeof(g_last_cuda_error) - 1] = 0;
    return WQ_ERR_CUDA;
}

wq_status check_launch() { return cuda_status(cudaGetLastError()); }

}  // namespace wqh

extern "C" const char* wq_status_string(wq_status s) {
    switch (s) {
        case WQ_OK: return "ok";
        case WQ_ERR_NULL_PTR: return "null pointer argument";
        case WQ_ERR_BAD_SHAPE: return "unsupported or inconsistent shape";
        case WQ_ERR_BAD_DTYPE: return "unsupported dtype";
        case WQ_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case WQ_ERR_UNSUPPORTED: return "unsupported parameter value";
        case WQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case WQ_ERR_CUDA: return "CUDA error";
        case WQ_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

extern "C" const char* wq_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char* wq_version(void) { return "wqgb300 0.1 sm_103a"; }

extern "C" int64_t uintx_packed_bytes(int64_t numel, int nbits) {
    if (numel < 0 || nbits < 1 || nbits > 8) return -1;
    int64_t total = 0;
    for (int kb = 8; kb >= 1; kb /= 2)
        if (nbits & kb) total += (numel + (8 / kb) - 1) / (8 / kb);
    return total;
}

// Workspace layouts (all offsets 256-byte aligned):
//   GPTQ quantize with SNR, quant_snr, mxfp4_quantize_err, uintx_quantize_err:
//               control block (arrival counter) |
//               kMaxPartials x 16-byte per-CTA float-float pairs.
//   awq_search: control block | s table [n_alpha][k] f32 | a_c/s table
//               [n_alpha][k] f32 | a_c [k] f32 | ln(an) [k] f64 + an [k] f32 |
//               per-CTA partials kMaxPartials x n_alpha doubles.
extern "C" size_t wq_workspace_bytes(int op, int64_t n, int64_t k, int arg) {
    (void)n;
    auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
    switch (op) {
        case WQ_OP_GPTQ_QUANTIZE:
        case WQ_OP_QUANT_SNR:
        case WQ_OP_MXFP4_ERR:
        case WQ_OP_UINTX_ERR:
            return wqh::kCtrlBytes + up((size_t)wqh::kMaxPartials * 2 * sizeof(double));
        case WQ_OP_AWQ_SEARCH: {
            if (arg < 1 || k < 0) return 0;
            size_t tab = up((size_t)arg * (size_t)k * sizeof(float));
            return wqh::kCtrlBytes + 2 * tab + up((size_t)k * sizeof(float)) +
                   up((size_t)k * (sizeof(double) + sizeof(float))) +
                   up((size_t)wqh::kMaxPartials * (size_t)arg * sizeof(double));
        }
        default:
            return 0;
    }
}

namespace wqh {
unsigned gptq_stage_polls_exchange(unsigned polls);  // gptq.cu
unsigned gemm_mma_slices_exchange(unsigned slices);  // gemm.cu
}  // namespace wqh

extern "C" unsigned wq_set_wait_budget(int site, unsigned budget) {
    switch (site) {
        case WQ_WAIT_GPTQ_STAGE: return wqh::gptq_stage_polls_exchange(budget);
        case WQ_WAIT_GEMM_MMA: return wqh::gemm_mma_slices_exchange(budget);
        default: return 0xFFFFFFFFu;
    }
}
