// awq.cu -- AWQ alpha search for MXFP4 (quantize_dflash_mxfp4.py: search_scale,
// with quantize_mxfp4 / dequantize_mxfp4 as the inner step).
//
//   a_c = max(a, 1e-8); an = a_c / mean(a_c)
//   for each alpha: t = clamp(an^alpha, 1e-2, 1e2); s = t / exp(mean(log t))
//                   err = sum over the row subsample of ((deq(quant(W*s)) / s - W) * a_c)^2
//   best = first alpha with the strictly smallest err
//
// Four kernels on the caller's stream (plus one memset of the arrival counter):
//   awq_logs      a_c [k] and ln(an) per column (binary64; mean(a_c) as a
//                 binary64 sum in a fixed order, the same in every CTA).
//   awq_tables    grid (k/256, n_alpha): t = clamp(an^alpha, 1e-2, 1e2) per
//                 column and alpha (binary64, rounded once to binary32) and
//                 gm = exp(mean ln t) per alpha from the last CTA.
//   awq_scale     s = t / gm and a_c / s for every column and alpha.
//   awq_err       every subsampled weight is read once; all alphas are evaluated
//                 in registers (4 rows x 8 columns per lane, s and a_c/s loaded
//                 once per alpha for those 4 rows).  Per element and alpha: W*s,
//                 the 32-block amax by 2 quad shuffles, the exact block exponent,
//                 hardware e2m1 rounding, the exact quantization error, the
//                 weighted square.  Per-CTA binary64 partials go to the
//                 workspace; the last CTA adds them in index order, takes the
//                 argmin and copies best_s.
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

// Grid ceil(k/256).  Every CTA forms mean(a_c) in the same fixed order (so all
// agree bit for bit), then for its columns a_c and L = ln(an) in binary64.
__global__ void __launch_bounds__(kThreads) awq_logs(const float* __restrict__ a, int64_t k,
                                                     float* __restrict__ a_c,
                                                     double* __restrict__ lan) {
    __shared__ double red[kThreads / 32 + 1];
    double ps = 0.0;
    for (int64_t c = threadIdx.x; c < k; c += kThreads) ps += (double)fmaxf(__ldg(a + c), 1e-8f);
    const float mean = (float)(block_sum_256(ps, red) / (double)k);
    const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (c < k) {
        const float ac = fmaxf(__ldg(a + c), 1e-8f);
        a_c[c] = ac;
        const float an = __fdiv_rn(ac, mean);
        lan[c] = log((double)an);
        reinterpret_cast<float*>(lan + k)[c] = an;  // an itself, for alpha = 1
    }
}

// Grid (ceil(k/256), n_alpha): t = an^alpha = exp(alpha * L) in binary64 (alpha
// = 0 and 1 give exactly 1 and an), rounded once to binary32 and clamped to
// [1e-2, 1e2]; then ln t of the binary32 t, rounded to binary32.  ln t comes from
// the binary64 exp already at hand: ln(t32) = alpha*L + ln(t32/t64) and
// t32/t64 - 1 is below 2^-24, so the first-order term carries it to far below
// binary32 resolution.  Each CTA adds its columns' logs (fixed order) into its
// own slot; the last CTA to finish adds, per alpha, the slots in index order and
// stores gm[alpha] = exp(mean ln t) rounded to binary32.
__global__ void __launch_bounds__(kThreads) awq_tables(int64_t k, AlphaList al, int n_alpha,
                                                       const double* __restrict__ lan,
                                                       float* __restrict__ t_tab,
                                                       double* __restrict__ part,
                                                       float* __restrict__ gm,
                                                       unsigned* __restrict__ counter) {
    __shared__ double red[kThreads / 32 + 1];
    __shared__ bool last;
    const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int i = blockIdx.y;
    const bool valid = c < k;
    const float alpha = al.v[i];
    double td = 1.0, lt = 0.0;
    if (valid) {
        const double L = lan[c];
        if (alpha == 1.0f) {
            td = (double)reinterpret_cast<const float*>(lan + k)[c];
            lt = L;
        } else if (alpha != 0.0f) {
            lt = (double)alpha * L;
            td = exp(lt);
        }
    }
    float t = (float)td;
    if (t < 1e-2f) {
        t = 1e-2f;
        lt = log((double)1e-2f);
    } else if (t > 1e2f) {
        t = 1e2f;
        lt = log((double)1e2f);
    } else {
        lt += ((double)t - td) / td;
    }
    if (valid) t_tab[(int64_t)i * k + c] = t;
    const double cta = block_sum_256(valid ? (double)(float)lt : 0.0, red);
    if (threadIdx.x == 0) {
        part[(int64_t)i * gridDim.x + blockIdx.x] = cta;
        __threadfence();
        last = atomicAdd(counter, 1u) == gridDim.x * gridDim.y - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (threadIdx.x < n_alpha) {
        double v = 0.0;
        for (unsigned b = 0; b < gridDim.x; ++b) v += __ldcg(part + (int64_t)threadIdx.x * gridDim.x + b);
        const float lmean = (float)(v / (double)k);
        gm[threadIdx.x] = (float)exp((double)lmean);
    }
    if (threadIdx.x == 0) *counter = 0u;  // every other CTA has counted itself in: ready for awq_err
}

// Grid (ceil(k/256), n_alpha): s = t / gm (IEEE) and q = (a_c / s)^2, the
// column weight of the squared error term.
__global__ void __launch_bounds__(kThreads) awq_scale(int64_t k, const float* __restrict__ gm,
                                                      const float* __restrict__ a_c,
                                                      float* __restrict__ s_tab,
                                                      float* __restrict__ q_tab) {
    const int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int i = blockIdx.y;
    if (c >= k) return;
    const float sv = __fdiv_rn(s_tab[(int64_t)i * k + c], __ldcg(gm + i));
    s_tab[(int64_t)i * k + c] = sv;
    const float q = __fdiv_rn(a_c[c], sv);
    q_tab[(int64_t)i * k + c] = __fmul_rn(q, q);
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

// Two e2m1 nibbles of one byte -> their values as f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte) {
    uint32_t h2;
    uint16_t in = (uint16_t)byte;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "h"(in));
    return h2;
}

// (m - v) for the f16x2 grid values m and the binary32 pair v, by mixed-precision
// subtractions that read the f16 halves in place (exact: see awq_err).
__device__ __forceinline__ wq::f2_t grid_minus(uint32_t h2, wq::f2_t v) {
    float d0, d1;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "sub.rn.f32.f16 %0, lo, %3;\n\tsub.rn.f32.f16 %1, hi, %4;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(h2), "f"(v.x), "f"(v.y));
    return wq::f2(d0, d1);
}

// e2m1 rounding of (lo, hi) straight back to f16x2 values (round half even,
// saturating at 6): the nearest grid values, sign included.
__device__ __forceinline__ uint32_t e2m1_round2(float lo, float hi) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2)
        : "f"(hi), "f"(lo));
    return h2;
}

__device__ __forceinline__ uint32_t page_tie(uint32_t nib, float v) {
    const float m = fabsf(v);
    return (m == 0.75f || m == 1.75f || m == 3.5f) ? nib - 2u : nib;
}

// Per element and alpha the page's error term is e = (deq/s - w) * a_c.  Here it
// is evaluated as (deq - ws) * (a_c/s) with ws = w*s the value that was
// quantized: algebraically the same product, without a division per element;
// its square is formed as (e2m1(v) - v)^2 * (a_c/s)^2 per element (v = ws *
// 2^-exp), summed over the lane's 8 columns of one block row and scaled by
// 2^exp twice (two steps, so that an exact zero stays zero under a huge scale).
// deq - ws is exact: with v = ws * 2^-exp (exact), deq - ws = (e2m1(v) - v) *
// 2^exp and e2m1(v) - v is an exact difference (the two lie within a factor two
// of each other, or e2m1(v) = 0).  The terms therefore differ from the page's
// only by the rounding of ws and of the final products (relative 1e-7), far
// inside the 1e-4 agreement required of the errors.
template <int TIE>
__global__ void __launch_bounds__(kThreads, 2) awq_err(const uint16_t* __restrict__ w, int64_t k,
                                                    int64_t rows, int64_t row_stride, int n_alpha,
                                                    AlphaList al, const float* __restrict__ s_tab,
                                                    const float* __restrict__ q_tab,
                                                    float2* __restrict__ slots,
                                                    unsigned* __restrict__ counter,
                                                    float* __restrict__ best_s,
                                                    int32_t* __restrict__ best_idx,
                                                    float* __restrict__ best_alpha,
                                                    double* __restrict__ errs) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gwarp = (int64_t)blockIdx.x * (kThreads / 32) + warp;
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    const int64_t col_chunks = (k + 255) / 256;
    const int64_t row_batches = (rows + kRowsPerLane - 1) / kRowsPerLane;

    wq::KSum acc[kMaxAlpha];  // compensated binary32 sums (the binary64 pipe is narrow)

    for (int64_t it = gwarp; it < col_chunks * row_batches; it += nwarps) {
        const int64_t rb = it / col_chunks;  // once per 32 x 4 values, all alphas
        const int64_t col = (it - rb * col_chunks) * 256 + 8 * lane;
        const int64_t r0 = rb * kRowsPerLane;
        const bool cval = col < k;  // k % 32 == 0: a lane quad is valid or not as a whole
        // the lane's 4 x 8 weights as binary32 pairs, shared by every alpha
        wq::f2_t wf[kRowsPerLane][4];
#pragma unroll
        for (int q = 0; q < kRowsPerLane; ++q) {
            const int64_t r = r0 + q;
            const uint4 u = (cval && r < rows) ? wq::ld_stream(w + (r * row_stride) * k + col)
                                               : make_uint4(0, 0, 0, 0);
            wf[q][0] = wq::bf2_to_f2(u.x);
            wf[q][1] = wq::bf2_to_f2(u.y);
            wf[q][2] = wq::bf2_to_f2(u.z);
            wf[q][3] = wq::bf2_to_f2(u.w);
        }
        // the column tables of alpha i + 1 are read while alpha i is evaluated (their
        // L2 latency was the kernel's main stall)
        auto tables = [&](int i, float4 (&t)[4]) {
            const int64_t off = (int64_t)i * k + (cval ? col : 0);
            t[0] = __ldg(reinterpret_cast<const float4*>(s_tab + off));
            t[1] = __ldg(reinterpret_cast<const float4*>(s_tab + off) + 1);
            t[2] = cval ? __ldg(reinterpret_cast<const float4*>(q_tab + off)) : make_float4(0, 0, 0, 0);
            t[3] = cval ? __ldg(reinterpret_cast<const float4*>(q_tab + off) + 1) : make_float4(0, 0, 0, 0);
        };
        float4 tn[4];
        tables(0, tn);
#pragma unroll
        for (int i = 0; i < kMaxAlpha; ++i) {
            if (i >= n_alpha) break;
            wq::f2_t S[4], Q[4];
            {
                const float4 s0 = tn[0], s1 = tn[1], q0 = tn[2], q1 = tn[3];
                if (i + 1 < n_alpha) tables(i + 1, tn);
                S[0] = wq::f2(s0.x, s0.y); S[1] = wq::f2(s0.z, s0.w);
                S[2] = wq::f2(s1.x, s1.y); S[3] = wq::f2(s1.z, s1.w);
                Q[0] = wq::f2(q0.x, q0.y); Q[1] = wq::f2(q0.z, q0.w);
                Q[2] = wq::f2(q1.x, q1.y); Q[3] = wq::f2(q1.z, q1.w);
            }
            float part = 0.0f;
#pragma unroll
            for (int q = 0; q < kRowsPerLane; ++q) {
                wq::f2_t ws[4];
                float am[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ws[j] = wq::mul2(wf[q][j], S[j]);
                    am[j] = fmaxf(fabsf(ws[j].x), fabsf(ws[j].y));
                }
                float amax = fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3]));  // a tree: short chain
                amax = fmaxf(amax, wq::shfl_xor(amax, 1));
                amax = fmaxf(amax, wq::shfl_xor(amax, 2));
                // 2^-exp and 2^exp.  With amax >= 2^-124 (every lane of the warp)
                // exp = floor(log2 amax) - 2 >= -126 and both are bit arithmetic on
                // the exponent field of amax; otherwise the clamped general form
                float inv, sc;
                const uint32_t ab = __float_as_uint(amax);
                if (__all_sync(0xffffffffu, ab >= 0x01800000u)) {
                    const uint32_t pe = ab & 0x7F800000u;         // 2^floor(log2 amax)
                    inv = __uint_as_float(0x80000000u - pe);      // 2^(2 - floor(log2 amax))
                    sc = __uint_as_float(pe - 0x01000000u);       // 2^(floor(log2 amax) - 2)
                } else {
                    const int ex = exp_from_f32(amax);
                    inv = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-exp, normal
                    sc = __uint_as_float(ex == -127 ? 0x00400000u : (uint32_t)(ex + 127) << 23);
                }
                const wq::f2_t INV = wq::f2(inv, inv);
                wq::f2_t loc = wq::f2(0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const wq::f2_t v = wq::mul2(ws[j], INV);
                    uint32_t h2;  // the e2m1 grid values of v as f16x2
                    if (TIE == WQ_TIE_PAGE_LITERAL) {
                        uint32_t b = e2m1x2(v.x, v.y);
                        b = page_tie(b & 15u, v.x) | (page_tie(b >> 4, v.y) << 4);
                        h2 = e2m1x2_to_h2(b);
                    } else {
                        h2 = e2m1_round2(v.x, v.y);
                    }
                    const wq::f2_t d = grid_minus(h2, v);  // m - v, exact
                    loc = wq::fma2(wq::mul2(d, d), Q[j], loc);
                }
                part = __fadd_rn(part, __fmul_rn(__fmul_rn(__fadd_rn(loc.x, loc.y), sc), sc));
            }
            acc[i].add(part);
        }
    }

    // CTA partial per alpha, fixed order, in float-float (binary32 hi + lo pairs on
    // the FP32 pipes); the last CTA to finish reduces them all.  Within a warp a
    // transposed butterfly halves the number of values per lane at each step, so
    // that lane l ends with the warp's sum for alpha l / 2.
    __shared__ float2 red[kThreads / 32][kMaxAlpha];
    __shared__ double e[kMaxAlpha];
    __shared__ bool last;
    __shared__ int best;
    wq::FF v[kMaxAlpha];
#pragma unroll
    for (int i = 0; i < kMaxAlpha; ++i) v[i] = wq::ff_of(acc[i]);
#pragma unroll
    for (int h = kMaxAlpha / 2, m = 16; h >= 1; h >>= 1, m >>= 1) {
        const bool upper = (lane & m) != 0;  // keeps the upper half of its values
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const wq::FF keep = upper ? v[i + h] : v[i];
            const wq::FF send = upper ? v[i] : v[i + h];
            v[i] = wq::ff_add(keep, wq::ff_shfl_xor(send, m));
        }
    }
    v[0] = wq::ff_add(v[0], wq::ff_shfl_xor(v[0], 1));
    if ((lane & 1) == 0) red[warp][lane >> 1] = make_float2(v[0].hi, v[0].lo);
    __syncthreads();
    if (threadIdx.x < n_alpha) {
        wq::FF t{0.f, 0.f};
        for (int wgi = 0; wgi < kThreads / 32; ++wgi) {
            const float2 r = red[wgi][threadIdx.x];
            t = wq::ff_add(t, wq::FF{r.x, r.y});
        }
        slots[(int64_t)blockIdx.x * n_alpha + threadIdx.x] = make_float2(t.hi, t.lo);
        __threadfence();
    }
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(counter, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    // warp w sums alphas w, w + 8: lane-strided slots, then a fixed shuffle tree
    for (int i = warp; i < n_alpha; i += kThreads / 32) {
        wq::FF t{0.f, 0.f};
        for (unsigned b = lane; b < gridDim.x; b += 32) {
            const float2 r = __ldcg(slots + (int64_t)b * n_alpha + i);
            t = wq::ff_add(t, wq::FF{r.x, r.y});
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) t = wq::ff_add(t, wq::ff_shfl_xor(t, m));
        if (lane == 0) e[i] = wq::ff_value(t);
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
        for (int64_t c = threadIdx.x; c < k; c += kThreads) best_s[c] = __ldcg(s_tab + (int64_t)best * k + c);
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
    float* r_tab = (float*)(ws + up((size_t)n_alpha * k * sizeof(float)));  // a_c / s
    float* a_c = (float*)(ws + 2 * up((size_t)n_alpha * k * sizeof(float)));
    double* lan = (double*)(ws + 2 * up((size_t)n_alpha * k * sizeof(float)) + up((size_t)k * sizeof(float)));
    float2* slots = (float2*)((char*)lan + up((size_t)k * (sizeof(double) + sizeof(float))));

    cudaStream_t st = (cudaStream_t)stream;
    unsigned* counter = (unsigned*)workspace;
    float* gm = (float*)((char*)workspace + 64);  // n_alpha <= 16 floats in the control block
    wq_status s = wqh::cuda_status(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
    if (s != WQ_OK) return s;
    const unsigned col_ctas = (unsigned)((k + kThreads - 1) / kThreads);
    awq_logs<<<col_ctas, kThreads, 0, st>>>(a, k, a_c, lan);
    s = wqh::check_launch();
    if (s != WQ_OK) return s;
    awq_tables<<<dim3(col_ctas, (unsigned)n_alpha), kThreads, 0, st>>>(k, al, n_alpha, lan, s_tab,
                                                                        reinterpret_cast<double*>(slots), gm,
                                                                        counter);
    s = wqh::check_launch();
    if (s != WQ_OK) return s;
    awq_scale<<<dim3(col_ctas, (unsigned)n_alpha), kThreads, 0, st>>>(k, gm, a_c, s_tab, r_tab);
    s = wqh::check_launch();
    if (s != WQ_OK) return s;
    const int64_t items = ((k + 255) / 256) * ((rows + kRowsPerLane - 1) / kRowsPerLane);
    // at least two items per warp: the per-CTA reduction is then a small part of the work
    const int64_t ctas = (items + 2 * (kThreads / 32) - 1) / (2 * (kThreads / 32));
    if (tie_mode == WQ_TIE_HALF_EVEN) {
        const int grid = wqh::grid_for((const void*)awq_err<WQ_TIE_HALF_EVEN>, kThreads, 0, ctas, wqh::kMaxPartials);
        awq_err<WQ_TIE_HALF_EVEN><<<grid, kThreads, 0, st>>>(w, k, rows, stride, n_alpha, al, s_tab, r_tab,
                                                             slots, counter, best_s, best_idx, best_alpha, errs);
    } else {
        const int grid = wqh::grid_for((const void*)awq_err<WQ_TIE_PAGE_LITERAL>, kThreads, 0, ctas, wqh::kMaxPartials);
        awq_err<WQ_TIE_PAGE_LITERAL><<<grid, kThreads, 0, st>>>(w, k, rows, stride, n_alpha, al, s_tab, r_tab,
                                                                slots, counter, best_s, best_idx, best_alpha, errs);
    }
    return wqh::check_launch();
}
