// mxfp4.cu -- OCP MXFP4 quantize / dequantize (quantize_dflash_mxfp4.py:
// E2M1 table, GROUP = 32, quantize_mxfp4, dequantize_mxfp4).
//
// Layout: k % 32 == 0, so the 32-value blocks of a row-major [n, k] matrix are
// consecutive in memory and the whole matrix is a flat stream of blocks.  One
// thread takes one 16-byte chunk (8 bf16 values), four lanes make one block:
//   load   uint4 (8 bf16) by cp.async into a two-stage per-thread shared-memory
//          pipeline (the next chunks stream in while these are coded)
//   amax   16-bit SIMD max of |bf16| bit patterns, 2 shuffles over 4 lanes
//   code   v = w * 2^-exp (exact), hardware cvt to e2m1x2 (round half even,
//          saturate at 6) -- the e2m1 encoding IS the page's magnitude index
//   store  one uint32 of 8 nibbles per lane (128 B per warp), one e8m0 byte per
//          block.
// HBM bound: 2 B read + 0.53 B written per weight.
//
// mxfp4_quantize_err runs the same kernel with ERR = 1: each lane also decodes
// its codes back (hardware e2m1 -> f16x2, times 2^exp: the values
// dequantize_mxfp4 returns), forms the binary32 terms w^2 and (w - deq)^2 that
// quantize_dflash_mxfp4.py main() reduces into its relative error, and the grid
// finishes both sums with the last-CTA float-float reduction: no second read of
// w and no dequantized tensor in memory.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // independent 16-byte chunks in flight per thread

// exp = clamp(floor(log2(amax)) - 2, -127, 127), 0 for amax == 0, from the
// 15-bit magnitude pattern of a bf16 amax.  A bf16 subnormal has
// floor(log2) <= -127 so it always clamps.
__device__ __forceinline__ int exp_from_bf16_mag(uint32_t a) {
    uint32_t ef = a >> 7;
    if (ef == 0) return a == 0 ? 0 : -127;
    int e = (int)ef - 129;
    return e < -127 ? -127 : e;
}

// Two binary32 -> two e2m1 nibbles, round to nearest even, saturating at +-6.
// `lo` lands in bits 0..3, `hi` in bits 4..7 (the first source operand of the
// cvt goes to the upper nibble).
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Two e2m1 nibbles of one byte -> two binary32 magnitudes with sign (exact).
__device__ __forceinline__ void e2m1x2_to_f(uint32_t byte, float& lo, float& hi) {
    uint32_t h2;
    uint16_t in = (uint16_t)byte;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "h"(in));
    lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
    hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
}

// 2^(e - 127) in binary32: e = 0 is the subnormal 2^-127, e = 255 is inf
// (as exp2(128.0) is in binary32).
__device__ __forceinline__ float e8m0_scale(uint32_t e) {
    return __uint_as_float(e == 0 ? 0x00400000u : (e << 23));
}

// Page-literal tie rewrite: exact midpoints 0.75, 1.75 and 3.5 go two grid steps
// down from the half-even choice ((argmin // 2) * 2 with argmin the lower
// neighbour); the other midpoints already agree with half-even.
__device__ __forceinline__ uint32_t page_tie(uint32_t nib, float v) {
    float m = fabsf(v);
    return (m == 0.75f || m == 1.75f || m == 3.5f) ? nib - 2u : nib;
}

template <int TIE>
__device__ __forceinline__ uint32_t code_pair(float x0, float x1, float inv) {
    float a0 = __fmul_rn(x0, inv), a1 = __fmul_rn(x1, inv);
    uint32_t b = e2m1x2(a0, a1);
    if (TIE == WQ_TIE_PAGE_LITERAL) b = page_tie(b & 15u, a0) | (page_tie(b >> 4, a1) << 4);
    return b;
}

// Error terms of one packed pair: sw += x*x, se += (x - deq)^2 with deq = e2m1
// value * 2^exp.  x - deq is formed by one FMA of the exact product q * 2^exp
// (a power-of-two scaling, never rounded for these magnitudes), so it is the
// binary32 difference the page's (deq - w) computes.
__device__ __forceinline__ void err_pair(uint32_t xbits, uint32_t byte, wq::f2_t ns2, wq::f2_t& sw,
                                         wq::f2_t& se) {
    float q0, q1;
    e2m1x2_to_f(byte, q0, q1);
    const wq::f2_t x = wq::bf2_to_f2(xbits);
    const wq::f2_t d = wq::fma2(wq::f2(q0, q1), ns2, x);
    se = wq::fma2(d, d, se);
    sw = wq::fma2(x, x, sw);
}

template <int TIE, int ERR>
__global__ void __launch_bounds__(kThreads) mxfp4_quant_kernel(const uint4* __restrict__ w,
                                                               int64_t nchunks,
                                                               uint32_t* __restrict__ packed,
                                                               uint8_t* __restrict__ e8m0,
                                                               float4* __restrict__ slots,
                                                               unsigned* __restrict__ counter,
                                                               double* __restrict__ snr_db,
                                                               double* __restrict__ rel_err) {
    // two pipeline stages of kUnroll 16-byte chunks, private to each thread
    __shared__ __align__(16) uint4 stage_buf[2][kUnroll][kThreads];
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int64_t step = nwarps * 32 * kUnroll;
    wq::KSum dw, de;

    auto issue = [&](int64_t wb, int st) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t c = wb + (int64_t)u * nwarps * 32 + lane;
            if (c < nchunks) wq::cp_async16(&stage_buf[st][u][threadIdx.x], w + c);
        }
        wq::cp_async_commit();
    };

    // Every lane of a warp runs the same trip count (shuffles below); lanes past
    // the end compute on zeros and store nothing.  nchunks % 4 == 0 and chunk
    // indices are 4-aligned per lane quad, so a quad is all-valid or all-invalid.
    issue(warp * 32, 0);
    int j = 0;
    for (int64_t wb = warp * 32; wb < nchunks; wb += step, ++j) {
        issue(wb + step, (j + 1) & 1);
        wq::cp_async_wait<1>();
        uint4 v[kUnroll];
        int64_t ch[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            ch[u] = wb + (int64_t)u * nwarps * 32 + lane;
            v[u] = ch[u] < nchunks ? stage_buf[j & 1][u][threadIdx.x] : make_uint4(0, 0, 0, 0);
        }
        wq::f2_t sw = wq::f2(0.f, 0.f), se = wq::f2(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t M = 0x7fff7fffu;
            uint32_t m2 = __vmaxu2(__vmaxu2(v[u].x & M, v[u].y & M), __vmaxu2(v[u].z & M, v[u].w & M));
            uint32_t a = max(m2 & 0xffffu, m2 >> 16);
            a = max(a, wq::shfl_xor(a, 1));
            a = max(a, wq::shfl_xor(a, 2));
            const int ex = exp_from_bf16_mag(a);
            const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-exp, normal
            uint32_t word = code_pair<TIE>(wq::bf_lo(v[u].x), wq::bf_hi(v[u].x), inv);
            word |= code_pair<TIE>(wq::bf_lo(v[u].y), wq::bf_hi(v[u].y), inv) << 8;
            word |= code_pair<TIE>(wq::bf_lo(v[u].z), wq::bf_hi(v[u].z), inv) << 16;
            word |= code_pair<TIE>(wq::bf_lo(v[u].w), wq::bf_hi(v[u].w), inv) << 24;
            if (ERR) {
                // lanes past the end hold zeros: zero codes, zero terms
                const float ns = -e8m0_scale((uint32_t)(ex + 127));
                const wq::f2_t ns2 = wq::f2(ns, ns);
                err_pair(v[u].x, word & 0xffu, ns2, sw, se);
                err_pair(v[u].y, (word >> 8) & 0xffu, ns2, sw, se);
                err_pair(v[u].z, (word >> 16) & 0xffu, ns2, sw, se);
                err_pair(v[u].w, word >> 24, ns2, sw, se);
            }
            if (ch[u] < nchunks) {
                packed[ch[u]] = word;
                if ((lane & 3) == 0) e8m0[ch[u] >> 2] = (uint8_t)(ex + 127);
            }
        }
        if (ERR) {
            dw.add(__fadd_rn(sw.x, sw.y));
            de.add(__fadd_rn(se.x, se.y));
        }
    }
    wq::cp_async_wait<0>();
    if (ERR) wq::finish_snr(wq::ff_of(dw), wq::ff_of(de), slots, counter, snr_db, rel_err);
}

template <int OUT_BF16>
__global__ void __launch_bounds__(kThreads) mxfp4_dequant_kernel(const uint32_t* __restrict__ packed,
                                                                 const uint8_t* __restrict__ e8m0,
                                                                 int64_t nchunks, void* __restrict__ out) {
    // kUnroll independent 8-value chunks per thread: their loads are all in
    // flight before the first is decoded
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < nchunks;
         base += stride * kUnroll) {
        uint32_t word[kUnroll], ex[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t c = base + u * stride;
            word[u] = c < nchunks ? wq::ld_stream1(packed + c) : 0u;
            ex[u] = c < nchunks ? (uint32_t)__ldg(e8m0 + (c >> 2)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t c = base + u * stride;
            if (c >= nchunks) break;
            const float s = e8m0_scale(ex[u]);
            float f[8];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                float lo, hi;
                e2m1x2_to_f((word[u] >> (8 * p)) & 0xffu, lo, hi);
                f[2 * p] = __fmul_rn(lo, s);
                f[2 * p + 1] = __fmul_rn(hi, s);
            }
            if (OUT_BF16) {
                uint4 o;
                o.x = wq::f2_to_bf2(f[0], f[1]);
                o.y = wq::f2_to_bf2(f[2], f[3]);
                o.z = wq::f2_to_bf2(f[4], f[5]);
                o.w = wq::f2_to_bf2(f[6], f[7]);
                reinterpret_cast<uint4*>(out)[c] = o;
            } else {
                float4* o = reinterpret_cast<float4*>(out) + 2 * c;
                o[0] = make_float4(f[0], f[1], f[2], f[3]);
                o[1] = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    }
}

template <int TIE, int ERR>
wq_status launch_quant(const uint16_t* w, int64_t nchunks, uint8_t* packed, uint8_t* e8m0,
                       void* workspace, double* snr_db, double* rel_err, cudaStream_t st) {
    const void* fn = (const void*)mxfp4_quant_kernel<TIE, ERR>;
    // with the error sums every CTA owns one partial-sum slot
    const int grid = wqh::grid_for(fn, kThreads, 0, (nchunks + kThreads - 1) / kThreads,
                                   ERR ? wqh::kMaxPartials : 1 << 30);
    unsigned* counter = nullptr;
    float4* slots = nullptr;
    if (ERR) {
        counter = (unsigned*)workspace;
        slots = (float4*)((char*)workspace + wqh::kCtrlBytes);
        wq_status s = wqh::cuda_status(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
        if (s != WQ_OK) return s;
    }
    mxfp4_quant_kernel<TIE, ERR><<<grid, kThreads, 0, st>>>((const uint4*)w, nchunks, (uint32_t*)packed,
                                                            e8m0, slots, counter, snr_db, rel_err);
    return wqh::check_launch();
}

}  // namespace

extern "C" wq_status mxfp4_quantize(const uint16_t* w, int64_t n, int64_t k, int tie_mode,
                                    uint8_t* packed, uint8_t* e8m0, void* stream) {
    if (n < 0 || k < 0 || k % 32 != 0) return WQ_ERR_BAD_SHAPE;
    if (tie_mode != WQ_TIE_HALF_EVEN && tie_mode != WQ_TIE_PAGE_LITERAL) return WQ_ERR_UNSUPPORTED;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !packed || !e8m0) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(w) || !wqh::aligned16(packed)) return WQ_ERR_MISALIGNED;
    const int64_t nchunks = n * k / 8;
    cudaStream_t st = (cudaStream_t)stream;
    if (tie_mode == WQ_TIE_HALF_EVEN)
        return launch_quant<WQ_TIE_HALF_EVEN, 0>(w, nchunks, packed, e8m0, nullptr, nullptr, nullptr, st);
    return launch_quant<WQ_TIE_PAGE_LITERAL, 0>(w, nchunks, packed, e8m0, nullptr, nullptr, nullptr, st);
}

extern "C" wq_status mxfp4_quantize_err(const uint16_t* w, int64_t n, int64_t k, int tie_mode,
                                        uint8_t* packed, uint8_t* e8m0, double* snr_db,
                                        double* rel_err, void* workspace, size_t workspace_bytes,
                                        void* stream) {
    if (!snr_db && !rel_err) return mxfp4_quantize(w, n, k, tie_mode, packed, e8m0, stream);
    if (n < 0 || k < 0 || k % 32 != 0) return WQ_ERR_BAD_SHAPE;
    if (tie_mode != WQ_TIE_HALF_EVEN && tie_mode != WQ_TIE_PAGE_LITERAL) return WQ_ERR_UNSUPPORTED;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !packed || !e8m0 || !workspace) return WQ_ERR_NULL_PTR;
    if (workspace_bytes < wq_workspace_bytes(WQ_OP_MXFP4_ERR, n, k, 0)) return WQ_ERR_WORKSPACE_TOO_SMALL;
    if (!wqh::aligned16(w) || !wqh::aligned16(packed) || !wqh::aligned_to(workspace, 16) ||
        (snr_db && !wqh::aligned_to(snr_db, 8)) || (rel_err && !wqh::aligned_to(rel_err, 8)))
        return WQ_ERR_MISALIGNED;
    const int64_t nchunks = n * k / 8;
    cudaStream_t st = (cudaStream_t)stream;
    if (tie_mode == WQ_TIE_HALF_EVEN)
        return launch_quant<WQ_TIE_HALF_EVEN, 1>(w, nchunks, packed, e8m0, workspace, snr_db, rel_err, st);
    return launch_quant<WQ_TIE_PAGE_LITERAL, 1>(w, nchunks, packed, e8m0, workspace, snr_db, rel_err, st);
}

extern "C" wq_status mxfp4_dequantize(const uint8_t* packed, const uint8_t* e8m0, int64_t n,
                                      int64_t k, int out_dtype, void* out, void* stream) {
    if (n < 0 || k < 0 || k % 32 != 0) return WQ_ERR_BAD_SHAPE;
    if (out_dtype != WQ_DTYPE_F32 && out_dtype != WQ_DTYPE_BF16) return WQ_ERR_BAD_DTYPE;
    if (n == 0 || k == 0) return WQ_OK;
    if (!packed || !e8m0 || !out) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(packed) || !wqh::aligned16(out)) return WQ_ERR_MISALIGNED;
    const int64_t nchunks = n * k / 8;
    cudaStream_t st = (cudaStream_t)stream;
    if (out_dtype == WQ_DTYPE_BF16) {
        int grid = wqh::grid_for((const void*)mxfp4_dequant_kernel<1>, kThreads, 0,
                                 (nchunks + kThreads * kUnroll - 1) / (kThreads * kUnroll), 1 << 30);
        mxfp4_dequant_kernel<1><<<grid, kThreads, 0, st>>>((const uint32_t*)packed, e8m0, nchunks, out);
    } else {
        int grid = wqh::grid_for((const void*)mxfp4_dequant_kernel<0>, kThreads, 0,
                                 (nchunks + kThreads * kUnroll - 1) / (kThreads * kUnroll), 1 << 30);
        mxfp4_dequant_kernel<0><<<grid, kThreads, 0, st>>>((const uint32_t*)packed, e8m0, nchunks, out);
    }
    return wqh::check_launch();
}
