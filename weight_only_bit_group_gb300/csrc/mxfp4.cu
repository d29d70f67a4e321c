// mxfp4.cu -- OCP MXFP4 quantize / dequantize (quantize_dflash_mxfp4.py:
// E2M1 table, GROUP = 32, quantize_mxfp4, dequantize_mxfp4).
//
// Layout: k % 32 == 0, so the 32-value blocks of a row-major [n, k] matrix are
// consecutive in memory and the whole matrix is a flat stream of blocks.  One
// lane codes one block (64 bytes of bf16) per step:
//   load   four 16-byte loads, the next block's issued before this one is coded
//   amax   bf16x2 max tree of |w| inside the lane
//   code   v = w * 2^-exp (exact: one mixed bf16 x bf16 -> binary32 FMA per value,
//          read straight from the packed bf16 pair), hardware cvt to e2m1x2
//          (round half even, saturate at 6) -- the e2m1 encoding IS the page's
//          magnitude index
//   store  one 16-byte word of 32 codes and one E8M0 byte per lane.
// HBM bound: 2 B read + 0.53 B written per weight.
//
// mxfp4_quantize_err runs the same kernel with ERR = 1: each lane also decodes
// its codes back (hardware e2m1 -> f16x2: the values dequantize_mxfp4 returns,
// before the block scale), forms the terms w^2 and (w - deq)^2 that
// quantize_dflash_mxfp4.py main() reduces into its relative error (see
// code_pair_err), and the grid finishes both sums with the last-CTA float-float
// reduction: no second read of w and no dequantized tensor in memory.
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

// Codes of one packed pair of weights (the two bf16 values of `u`; inv_h =
// 2^-exp as bf16 bits) and, with ERR, the pair's error terms in the block's
// scaled domain.  Both halves go straight into mixed-precision FMAs (bf16 x bf16
// + binary32): a = w * 2^-exp is exact (a product of two bf16 values), so no
// bf16 -> binary32 unpacking runs on the integer pipe.  With ERR: sa += a^2 and
// se += (q - a)^2, q the e2m1 value of the chosen code (back from the code byte
// through the hardware e2m1 -> f16x2 conversion; q - a is one mixed f16 /
// binary32 subtraction, exact).  a * 2^exp = w and (q - a) * 2^exp = deq - w
// exactly, so a block's two sums, scaled by 2^exp twice, are the sums of the
// page's binary32 terms w^2 and (deq - w)^2 up to the rounding of each square
// (relative 2^-24).
template <int TIE, int ERR>
__device__ __forceinline__ uint32_t code_pair_err(uint32_t u, uint16_t inv_h, wq::f2_t& sa, wq::f2_t& se) {
    float a0, a1;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "fma.rn.f32.bf16 %0, lo, %3, %4;\n\tfma.rn.f32.bf16 %1, hi, %3, %4;\n\t}"
        : "=f"(a0), "=f"(a1)
        : "r"(u), "h"(inv_h), "f"(-0.0f));
    uint32_t b = e2m1x2(a0, a1);
    if (TIE == WQ_TIE_PAGE_LITERAL) b = page_tie(b & 15u, a0) | (page_tie(b >> 4, a1) << 4);
    if (ERR) {
        uint32_t h2;
        const uint16_t in = (uint16_t)b;
        asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "h"(in));
        float r0, r1;
        asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "sub.rn.f32.f16 %0, lo, %3;\n\tsub.rn.f32.f16 %1, hi, %4;\n\t}"
            : "=f"(r0), "=f"(r1)
            : "r"(h2), "f"(a0), "f"(a1));
        const wq::f2_t a = wq::f2(a0, a1), r = wq::f2(r0, r1);  // r = q - a, exact
        se = wq::fma2(r, r, se);
        sa = wq::fma2(a, a, sa);
    }
    return b;
}

// One lane codes one whole 32-value block per step: four 16-byte loads (the
// next block's are issued before this one is coded), the block |amax| by a
// bf16x2 max tree inside the lane (no shuffles), 16 code pairs, one 16-byte
// store of the 32 codes and one E8M0 byte.  Consecutive lanes take consecutive
// blocks, so a warp reads 2 KB and writes 512 + 32 bytes contiguously per
// step; the four loads of a lane hit the same L1 lines.
template <int TIE, int ERR>
__global__ void __launch_bounds__(kThreads) mxfp4_quant_kernel(const uint4* __restrict__ w,
                                                               int64_t nblocks,
                                                               uint4* __restrict__ packed,
                                                               uint8_t* __restrict__ e8m0,
                                                               float4* __restrict__ slots,
                                                               unsigned* __restrict__ counter,
                                                               double* __restrict__ snr_db,
                                                               double* __restrict__ rel_err) {
    const int64_t nth = (int64_t)gridDim.x * kThreads;
    int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    wq::KSum dw, de;
    uint4 nx[4];
    if (b < nblocks) {
#pragma unroll
        for (int q = 0; q < 4; ++q) nx[q] = __ldg(w + 4 * b + q);
    }
    for (; b < nblocks; b += nth) {
        uint4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = nx[q];
        if (b + nth < nblocks) {
#pragma unroll
            for (int q = 0; q < 4; ++q) nx[q] = __ldg(w + 4 * (b + nth) + q);
        }
        // block |amax| as bf16 magnitudes (max.xorsign.abs leaves garbage sign bits)
        uint32_t m2[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            m2[q] = wq::babsmax2(wq::babsmax2(v[q].x, v[q].y), wq::babsmax2(v[q].z, v[q].w));
        uint32_t m = wq::babsmax2(wq::babsmax2(m2[0], m2[1]), wq::babsmax2(m2[2], m2[3])) & 0x7fff7fffu;
        const int ex = exp_from_bf16_mag(max(m & 0xffffu, m >> 16));
        const uint16_t inv_h = (uint16_t)((127 - ex) << 7);  // 2^-exp as bf16 (normal)
        wq::f2_t sa = wq::f2(0.f, 0.f), se = wq::f2(0.f, 0.f);
        uint32_t word[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            word[q] = code_pair_err<TIE, ERR>(v[q].x, inv_h, sa, se);
            word[q] |= code_pair_err<TIE, ERR>(v[q].y, inv_h, sa, se) << 8;
            word[q] |= code_pair_err<TIE, ERR>(v[q].z, inv_h, sa, se) << 16;
            word[q] |= code_pair_err<TIE, ERR>(v[q].w, inv_h, sa, se) << 24;
        }
        packed[b] = make_uint4(word[0], word[1], word[2], word[3]);
        e8m0[b] = (uint8_t)(ex + 127);
        if (ERR) {
            // back to the weights' scale: times 2^exp twice (2^(2 exp) itself may
            // leave the binary32 range)
            const float sc = e8m0_scale((uint32_t)(ex + 127));
            dw.add(__fmul_rn(__fmul_rn(__fadd_rn(sa.x, sa.y), sc), sc));
            de.add(__fmul_rn(__fmul_rn(__fadd_rn(se.x, se.y), sc), sc));
        }
    }
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
    const int64_t nblocks = nchunks / 4;
    // with the error sums every CTA owns one partial-sum slot
    const int grid = wqh::grid_for(fn, kThreads, 0, (nblocks + kThreads - 1) / kThreads,
                                   ERR ? wqh::kMaxPartials : 1 << 30);
    unsigned* counter = nullptr;
    float4* slots = nullptr;
    if (ERR) {
        counter = (unsigned*)workspace;
        slots = (float4*)((char*)workspace + wqh::kCtrlBytes);
        wq_status s = wqh::cuda_status(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
        if (s != WQ_OK) return s;
    }
    mxfp4_quant_kernel<TIE, ERR><<<grid, kThreads, 0, st>>>((const uint4*)w, nblocks, (uint4*)packed, e8m0,
                                                            slots, counter, snr_db, rel_err);
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
