// awq.cu -- AWQ alpha search for MXFP4 (quantize_dflash_mxfp4.py: search_scale,
// with quantize_mxfp4 / dequantize_mxfp4 as the inner step).
//
//   a_c = max(a, 1e-8); an = a_c / mean(a_c)
//   for each alpha: t = clamp(an^alpha, 1e-2, 1e2); s = t / exp(mean(log t))
//                   err = sum over the row subsample of ((deq(quant(W*s)) / s - W) * a_c)^2
//   best = first alpha with the strictly smallest err
//
// Four kernels on the caller's stream:
//   awq_tables    grid (k/256, n_alpha): t = clamp(an^alpha, 1e-2, 1e2) and log t
//                 per column and alpha (pow/log in binary64 rounded once to
//                 binary32; mean(a_c) as a binary64 sum in a fixed order, the
//                 same in every CTA), a_c [k].
//   awq_norm      one CTA per alpha: exp(mean(log t)) (fixed-order binary64
//                 sum), s = t / gm and RN(1/s).
//   awq_err       every subsampled weight is read once; all alphas are evaluated
//                 in registers (4 rows x 8 columns per lane, s/1-s loaded once per
//                 alpha for those 4 rows).  Per element and alpha: W*s, the
//                 32-block amax by 2 quad shuffles, the exact block exponent,
//                 hardware e2m1 rounding, exact dequant, the quotient by s (exact
//                 reciprocal + one FMA correction), the weighted square.  Per-CTA
//                 binary64 partials go to the workspace.
//   awq_finalize  one CTA: partials added in index order, argmin, best_s copy.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxAlpha = 16;
constexpr int kRowsPerLane = 4;

struct AlphaList {
    float v[kMaxAlpha];
};

// Fixed-order sum over a 256-thread CTA (every thread gets the result).
__device__ double block_sum_256(double v, double* red) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int i = 0; i < kThreads / 32; ++i) t += red[i];
        red[kThreads / 32] = t;
    }
    __syncthreads();
    return red[kThreads / 32];
}

// Grid (ceil(k/256), n_alpha).  Every CTA forms mean(a_c) in the same fixed
// order (so all agree bit for bit), then for its 256 columns and its alpha:
// t = clamp(an^alpha, 1e-2, 1e2) -> t_tab, log(t) rounded to binary32 -> l_tab.
__global__ void __launch_bounds__(kThreads) awq_tables(const float* __restrict__ a, int64_t k,
                                                       AlphaList al, float* __restrict__ t_tab,
                                                       float* __restrict__ l_tab,
                                                       float* __restrict__ a_c) {
    __shared__ double red[kThreads / 32 + 1];
    double part = 0.0;
    for (int64_t c = threadIdx.x; c < k; c += kThreads) part += (double)fmaxf(__ldg(a + c), 1e-8f);
    const float mean = (float)(block_sum_256(part, red) / (double)k);
    const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int i = blockIdx.y;
    if (c < k) {
        const float ac = fmaxf(__ldg(a + c), 1e-8f);
        if (i == 0) a_c[c] = ac;
        const float an = __fdiv_rn(ac, mean);
        float t = (float)pow((double)an, (double)al.v[i]);
        t = fminf(fmaxf(t, 1e-2f), 1e2f);
        t_tab[(int64_t)i * k + c] = t;
        l_tab[(int64_t)i * k + c] = (float)log((double)t);
    }
}

// One CTA per alpha: gm = exp(mean(log t)) from the binary32 logs (binary64 sum
// in a fixed order), then s = t / gm and r = RN(1/s).  r_tab holds the logs on
// entry (all read before any is overwritten).
__global__ void __launch_bounds__(kThreads) awq_norm(int64_t k, float* __restrict__ s_tab,
                                                     float* __restrict__ r_tab) {
    __shared__ double red[kThreads / 32 + 1];
    const int i = blockIdx.x;
    float* s = s_tab + (int64_t)i * k;
    float* r = r_tab + (int64_t)i * k;
    double part = 0.0;
    for (int64_t c = threadIdx.x; c < k; c += kThreads) part += (double)r[c];
    const float lmean = (float)(block_sum_256(part, red) / (double)k);
    const float gm = (float)exp((double)lmean);
    for (int64_t c = threadIdx.x; c < k; c += kThreads) {
        const float sv = __fdiv_rn(s[c], gm);
        s[c] = sv;
        r[c] = __frcp_rn(sv);
    }
}

// exp = clamp(floor(log2(amax)) - 2, -127, 127) for a binary32 amax >= 0 (0 -> 0).
__device__ __forceinline__ int exp_from_f32(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const uint32_t ef = b >> 23;
    if (ef == 0) return b == 0 ? 0 : -127;  // subnormal: floor(log2) <= -127
    const int e = (int)ef - 129;
    return e < -127 ? -127 : e;
}

__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void e2m1x2_to_f(uint32_t byte, float& lo, float& hi) {
    uint32_t h2;
    uint16_t in = (uint16_t)byte;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "h"(in));
    lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
    hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

__device__ __forceinline__ uint32_t page_tie(uint32_t nib, float v) {
    const float m = fabsf(v);
    return (m == 0.75f || m == 1.75f || m == 3.5f) ? nib - 2u : nib;
}

template <int TIE>
__global__ void __launch_bounds__(kThreads) awq_err(const uint16_t* __restrict__ w, int64_t k,
                                                    int64_t rows, int64_t row_stride, int n_alpha,
                                                    const float* __restrict__ s_tab,
                                                    const float* __restrict__ r_tab,
                                                    const float* __restrict__ a_c,
                                                    double* __restrict__ slots) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gwarp = (int64_t)blockIdx.x * (kThreads / 32) + warp;
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    const int64_t col_chunks = (k + 255) / 256;
    const int64_t row_batches = (rows + kRowsPerLane - 1) / kRowsPerLane;

    double acc[kMaxAlpha];
#pragma unroll
    for (int i = 0; i < kMaxAlpha; ++i) acc[i] = 0.0;

    for (int64_t it = gwarp; it < col_chunks * row_batches; it += nwarps) {
        const int64_t col = (it % col_chunks) * 256 + 8 * lane;
        const int64_t r0 = (it / col_chunks) * kRowsPerLane;
        const bool cval = col < k;  // k % 32 == 0: a lane quad is valid or not as a whole
        uint4 wv[kRowsPerLane];
#pragma unroll
        for (int q = 0; q < kRowsPerLane; ++q) {
            const int64_t r = r0 + q;
            wv[q] = (cval && r < rows) ? wq::ld_stream(w + (r * row_stride) * k + col)
                                       : make_uint4(0, 0, 0, 0);
        }
        float ac[8];
        {
            const float4 a0 = cval ? __ldg(reinterpret_cast<const float4*>(a_c + col)) : make_float4(0, 0, 0, 0);
            const float4 a1 = cval ? __ldg(reinterpret_cast<const float4*>(a_c + col) + 1) : make_float4(0, 0, 0, 0);
            ac[0] = a0.x; ac[1] = a0.y; ac[2] = a0.z; ac[3] = a0.w;
            ac[4] = a1.x; ac[5] = a1.y; ac[6] = a1.z; ac[7] = a1.w;
        }
#pragma unroll
        for (int i = 0; i < kMaxAlpha; ++i) {
            if (i >= n_alpha) break;
            float s[8], rr[8];
            {
                const float4* sp = reinterpret_cast<const float4*>(s_tab + (int64_t)i * k + (cval ? col : 0));
                const float4* rp = reinterpret_cast<const float4*>(r_tab + (int64_t)i * k + (cval ? col : 0));
                const float4 s0 = __ldg(sp), s1 = __ldg(sp + 1), q0 = __ldg(rp), q1 = __ldg(rp + 1);
                s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
                s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
                rr[0] = q0.x; rr[1] = q0.y; rr[2] = q0.z; rr[3] = q0.w;
                rr[4] = q1.x; rr[5] = q1.y; rr[6] = q1.z; rr[7] = q1.w;
            }
            float part = 0.0f;
#pragma unroll
            for (int q = 0; q < kRowsPerLane; ++q) {
                const uint32_t u[4] = {wv[q].x, wv[q].y, wv[q].z, wv[q].w};
                float x[8], ws[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    x[2 * j] = wq::bf_lo(u[j]);
                    x[2 * j + 1] = wq::bf_hi(u[j]);
                }
                float amax = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    ws[j] = __fmul_rn(x[j], s[j]);
                    amax = fmaxf(amax, fabsf(ws[j]));
                }
                amax = fmaxf(amax, wq::shfl_xor(amax, 1));
                amax = fmaxf(amax, wq::shfl_xor(amax, 2));
                const int ex = exp_from_f32(amax);
                const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-exp, normal
                const float sc = __uint_as_float(ex == -127 ? 0x00400000u : (uint32_t)(ex + 127) << 23);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float v0 = __fmul_rn(ws[2 * j], inv), v1 = __fmul_rn(ws[2 * j + 1], inv);
                    uint32_t b = e2m1x2(v0, v1);
                    if (TIE == WQ_TIE_PAGE_LITERAL) b = page_tie(b & 15u, v0) | (page_tie(b >> 4, v1) << 4);
                    float m0, m1;
                    e2m1x2_to_f(b, m0, m1);
                    const float d0 = __fmul_rn(m0, sc), d1 = __fmul_rn(m1, sc);
                    const float q0 = wq::div_by_recip(d0, s[2 * j], rr[2 * j]);
                    const float q1 = wq::div_by_recip(d1, s[2 * j + 1], rr[2 * j + 1]);
                    const float e0 = __fmul_rn(__fsub_rn(q0, x[2 * j]), ac[2 * j]);
                    const float e1 = __fmul_rn(__fsub_rn(q1, x[2 * j + 1]), ac[2 * j + 1]);
                    part = __fadd_rn(part, __fmul_rn(e0, e0));
                    part = __fadd_rn(part, __fmul_rn(e1, e1));
                }
            }
            acc[i] += (double)part;
        }
    }

    // CTA partial per alpha, fixed order
    __shared__ double red[kThreads / 32][kMaxAlpha];
#pragma unroll
    for (int i = 0; i < kMaxAlpha; ++i) {
        double v = acc[i];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
        if (lane == 0) red[warp][i] = v;
    }
    __syncthreads();
    if (threadIdx.x < n_alpha) {
        double t = 0.0;
        for (int wgi = 0; wgi < kThreads / 32; ++wgi) t += red[wgi][threadIdx.x];
        slots[(int64_t)blockIdx.x * n_alpha + threadIdx.x] = t;
    }
}

__global__ void __launch_bounds__(kThreads) awq_finalize(const double* __restrict__ slots, int nslots,
                                                         int n_alpha, AlphaList al, int64_t k,
                                                         const float* __restrict__ s_tab,
                                                         float* __restrict__ best_s,
                                                         int32_t* __restrict__ best_idx,
                                                         float* __restrict__ best_alpha,
                                                         double* __restrict__ errs) {
    __shared__ double e[kMaxAlpha];
    __shared__ int best;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // warp w sums alphas w, w + 8: lane-strided slots, then a fixed shuffle tree
    for (int i = warp; i < n_alpha; i += kThreads / 32) {
        double t = 0.0;
        for (int b = lane; b < nslots; b += 32) t += slots[(int64_t)b * n_alpha + i];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) t += __shfl_xor_sync(0xffffffffu, t, m);
        if (lane == 0) e[i] = t;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int bi = 0;
        for (int i = 1; i < n_alpha; ++i)
            if (e[i] < e[bi]) bi = i;  // strict: the first of equal errors wins
        best = bi;
        if (best_idx) *best_idx = bi;
        if (best_alpha) *best_alpha = al.v[bi];
    }
    __syncthreads();
    if (errs && threadIdx.x < n_alpha) errs[threadIdx.x] = e[threadIdx.x];
    if (best_s)
        for (int64_t c = threadIdx.x; c < k; c += kThreads) best_s[c] = s_tab[(int64_t)best * k + c];
}

}  // namespace

extern "C" wq_status awq_search(const uint16_t* w, int64_t n, int64_t k, const float* a,
                                const float* alphas_host, int n_alpha, int max_rows, int tie_mode,
                                float* best_s, int32_t* best_idx, float* best_alpha, double* errs,
                                void* workspace, size_t workspace_bytes, void* stream) {
    if (n <= 0 || k <= 0 || k % 32 != 0) return WQ_ERR_BAD_SHAPE;
    if (n_alpha < 1 || n_alpha > kMaxAlpha || max_rows < 1) return WQ_ERR_UNSUPPORTED;
    if (tie_mode != WQ_TIE_HALF_EVEN && tie_mode != WQ_TIE_PAGE_LITERAL) return WQ_ERR_UNSUPPORTED;
    if (!w || !a || !alphas_host || !workspace) return WQ_ERR_NULL_PTR;
    if (workspace_bytes < wq_workspace_bytes(WQ_OP_AWQ_SEARCH, n, k, n_alpha))
        return WQ_ERR_WORKSPACE_TOO_SMALL;
    if (!wqh::aligned16(w) || !wqh::aligned_to(a, 4) || !wqh::aligned_to(workspace, 256) ||
        (best_s && !wqh::aligned_to(best_s, 4)) || (errs && !wqh::aligned_to(errs, 8)))
        return WQ_ERR_MISALIGNED;

    int64_t stride = 1, rows = n;
    if (n > max_rows) {
        stride = n / max_rows;
        if (stride < 1) stride = 1;
        rows = (n + stride - 1) / stride;
        if (rows > max_rows) rows = max_rows;
    }
    AlphaList al;
    for (int i = 0; i < kMaxAlpha; ++i) al.v[i] = i < n_alpha ? alphas_host[i] : 0.0f;

    auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
    char* ws = (char*)workspace + wqh::kCtrlBytes;
    float* s_tab = (float*)ws;
    float* r_tab = (float*)(ws + up((size_t)n_alpha * k * sizeof(float)));
    float* a_c = (float*)(ws + 2 * up((size_t)n_alpha * k * sizeof(float)));
    double* slots = (double*)(ws + 2 * up((size_t)n_alpha * k * sizeof(float)) + up((size_t)k * sizeof(float)));

    cudaStream_t st = (cudaStream_t)stream;
    awq_tables<<<dim3((unsigned)((k + kThreads - 1) / kThreads), (unsigned)n_alpha), kThreads, 0, st>>>(
        a, k, al, s_tab, r_tab, a_c);
    wq_status s = wqh::check_launch();
    if (s != WQ_OK) return s;
    awq_norm<<<n_alpha, kThreads, 0, st>>>(k, s_tab, r_tab);
    s = wqh::check_launch();
    if (s != WQ_OK) return s;

    const int64_t items = ((k + 255) / 256) * ((rows + kRowsPerLane - 1) / kRowsPerLane);
    const int64_t ctas = (items + (kThreads / 32) - 1) / (kThreads / 32);
    int grid;
    if (tie_mode == WQ_TIE_HALF_EVEN) {
        grid = wqh::grid_for((const void*)awq_err<WQ_TIE_HALF_EVEN>, kThreads, 0, ctas, wqh::kMaxPartials);
        awq_err<WQ_TIE_HALF_EVEN><<<grid, kThreads, 0, st>>>(w, k, rows, stride, n_alpha, s_tab, r_tab, a_c, slots);
    } else {
        grid = wqh::grid_for((const void*)awq_err<WQ_TIE_PAGE_LITERAL>, kThreads, 0, ctas, wqh::kMaxPartials);
        awq_err<WQ_TIE_PAGE_LITERAL><<<grid, kThreads, 0, st>>>(w, k, rows, stride, n_alpha, s_tab, r_tab, a_c, slots);
    }
    s = wqh::check_launch();
    if (s != WQ_OK) return s;
    awq_finalize<<<1, kThreads, 0, st>>>(slots, grid, n_alpha, al, k, s_tab, best_s, best_idx, best_alpha, errs);
    return wqh::check_launch();
}
