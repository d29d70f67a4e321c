// fold.cu -- the AWQ scale fold that follows the alpha search
// (quantize_dflash_mxfp4.py, main(): once search_scale has chosen s, the norm
// weights are divided by s, the conv kernel projections and the q/k/v, gate/up
// and down columns are multiplied by s, and up's rows are divided by down's s).
//
// out[r][c] = bf16(w[r][c] op s), op a binary32 multiply or IEEE division of the
// exact bf16 value, s per column (axis 0) or per row (axis 1): the page's
// (W.float() op s).to(bfloat16), two roundings (binary32, then bf16).
//
// A thread owns 8 consecutive columns (one 16-byte load and store) and walks the
// rows with the grid's row stride, so the column scales are loaded once per
// thread and a row scale is the same for the whole CTA.  HBM bound: 2 B read and
// 2 B written per weight.  out may be w (in-place fold): the weights are read
// through the ordinary data path, each element by the thread that writes it.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;

template <int AXIS, int OP>
__global__ void __launch_bounds__(kThreads) awq_fold_kernel(const uint16_t* w, int64_t n, int64_t k,
                                                            const float* __restrict__ s,
                                                            uint16_t* out) {
    const int64_t kc = k / 8;
    const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x;  // 8-column chunk
    if (c >= kc) return;
    float sv[8];
    if (AXIS == 0) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(s) + 2 * c);
        const float4 b = __ldg(reinterpret_cast<const float4*>(s) + 2 * c + 1);
        sv[0] = a.x; sv[1] = a.y; sv[2] = a.z; sv[3] = a.w;
        sv[4] = b.x; sv[5] = b.y; sv[6] = b.z; sv[7] = b.w;
    }
    for (int64_t r = blockIdx.y; r < n; r += gridDim.y) {
        if (AXIS == 1) {
            const float v = __ldg(s + r);
#pragma unroll
            for (int i = 0; i < 8; ++i) sv[i] = v;
        }
        const uint4 u = *reinterpret_cast<const uint4*>(w + r * k + 8 * c);
        const uint32_t x[4] = {u.x, u.y, u.z, u.w};
        uint32_t y[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = wq::bf_lo(x[j]), hi = wq::bf_hi(x[j]);
            const float a = OP == 0 ? __fmul_rn(lo, sv[2 * j]) : __fdiv_rn(lo, sv[2 * j]);
            const float b = OP == 0 ? __fmul_rn(hi, sv[2 * j + 1]) : __fdiv_rn(hi, sv[2 * j + 1]);
            y[j] = wq::f2_to_bf2(a, b);
        }
        *reinterpret_cast<uint4*>(out + r * k + 8 * c) = make_uint4(y[0], y[1], y[2], y[3]);
    }
}

template <int AXIS, int OP>
wq_status launch_fold(const uint16_t* w, int64_t n, int64_t k, const float* s, uint16_t* out,
                      cudaStream_t st) {
    const void* fn = (const void*)awq_fold_kernel<AXIS, OP>;
    const int64_t gx = (k / 8 + kThreads - 1) / kThreads;
    // enough CTAs to fill every SM, split between column chunks and row slices
    const int64_t full = wqh::grid_for(fn, kThreads, 0, (int64_t)1 << 30, 1 << 30);
    int64_t gy = full / gx;
    if (gy < 1) gy = 1;
    if (gy > n) gy = n;
    if (gy > 65535) gy = 65535;
    awq_fold_kernel<AXIS, OP><<<dim3((unsigned)gx, (unsigned)gy), kThreads, 0, st>>>(w, n, k, s, out);
    return wqh::check_launch();
}

}  // namespace

extern "C" wq_status awq_fold(const uint16_t* w, int64_t n, int64_t k, const float* s, int axis,
                              int op, uint16_t* out, void* stream) {
    if (n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if ((axis != WQ_FOLD_COLUMNS && axis != WQ_FOLD_ROWS) || (op != WQ_FOLD_MUL && op != WQ_FOLD_DIV))
        return WQ_ERR_UNSUPPORTED;
    if (k % 8 != 0 || k / 8 / kThreads >= ((int64_t)1 << 31)) return WQ_ERR_BAD_SHAPE;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !s || !out) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(w) || !wqh::aligned16(out) ||
        (axis == WQ_FOLD_COLUMNS ? !wqh::aligned16(s) : !wqh::aligned_to(s, 4)))
        return WQ_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    if (axis == WQ_FOLD_COLUMNS)
        return op == WQ_FOLD_MUL ? launch_fold<0, 0>(w, n, k, s, out, st) : launch_fold<0, 1>(w, n, k, s, out, st);
    return op == WQ_FOLD_MUL ? launch_fold<1, 0>(w, n, k, s, out, st) : launch_fold<1, 1>(w, n, k, s, out, st);
}
