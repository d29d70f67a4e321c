// quant_wide.cu -- GPTQ and MXFP4 quantization of fp16 and fp32 weights.
//
// export_gptq_cpu.py (quantize_sym, quantize_asym) and quantize_dflash_mxfp4.py
// (quantize_mxfp4) both start from w.float(): an fp16 or fp32 weight reaches
// the same binary32 arithmetic as a bf16 one, only with more significant bits.
// GPTQ: argument checks here, the warp-tiled TMA kernel in gptq.cu
// (gptq_quant_wide_kernel).  MXFP4: one thread per 32-value block, below.
// bf16 weights go to the bf16 kernels.
#include <cuda_fp16.h>

#include "wq_common.cuh"

namespace {

constexpr int kWideThreads = 128;

// Eight consecutive values from element idx (a multiple of 8) as binary32; the
// widening of fp16 is exact.
template <int DT>
__device__ __forceinline__ void load8(const void* base, int64_t idx, float (&v)[8]) {
    if (DT == WQ_DTYPE_F32) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
        const float4 a = __ldg(p), b = __ldg(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx));
        const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
}

// Two binary32 values -> two e2m1 nibbles (round half to even, saturating at
// 6); `lo` in bits 0..3.  Same rule as the bf16 kernel's.
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi) {
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r;
}
// The page's literal tie rule differs from half-even at the midpoints 0.75,
// 1.75 and 3.5 only: there it takes the grid point two steps down.
__device__ __forceinline__ uint32_t literal_tie(uint32_t nib, float v) {
    const float m = fabsf(v);
    return (m == 0.75f || m == 1.75f || m == 3.5f) ? nib - 2u : nib;
}

// One thread per 32-value block: amax, the block exponent from the binary32 bits
// of amax (floor(log2 amax) - 2, clamped to [-127, 127], 0 for amax == 0), the
// values scaled by the exact power of two and converted in pairs.
template <int TIE, int DT>
__global__ void __launch_bounds__(kWideThreads)
mxfp4_quant_wide_kernel(const void* __restrict__ w, int64_t nblocks, uint4* __restrict__ packed,
                        uint8_t* __restrict__ e8m0) {
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float t[8];
            load8<DT>(w, b * 32 + 8 * q, t);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[8 * q + i] = t[i];
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        int ex = 0;
        if (amax > 0.f) {
            const int eb = (int)((__float_as_uint(amax) >> 23) & 0xffu);
            ex = eb == 0 ? -127 : max(eb - 127 - 2, -127);  // subnormal amax: floor(log2) <= -127
            ex = min(ex, 127);
        }
        const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-ex, a normal number
        uint32_t word[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float a0 = __fmul_rn(v[2 * i], inv), a1 = __fmul_rn(v[2 * i + 1], inv);
            uint32_t byte = e2m1_pair(a0, a1);
            if (TIE == WQ_TIE_PAGE_LITERAL) byte = literal_tie(byte & 15u, a0) | (literal_tie(byte >> 4, a1) << 4);
            word[i >> 2] |= byte << (8 * (i & 3));
        }
        packed[b] = make_uint4(word[0], word[1], word[2], word[3]);
        e8m0[b] = (uint8_t)(ex + 127);
    }
}

}  // namespace

extern "C" {

wq_status gptq_quantize_ex(const void* w, int w_dtype, int64_t n, int64_t k, int group, int sym,
                           int32_t* qweight, int32_t* qzeros, uint16_t* scales, int32_t* g_idx,
                           double* snr_db, void* workspace, size_t workspace_bytes, void* stream) {
    if (w_dtype == WQ_DTYPE_BF16)
        return sym ? gptq_quantize_sym((const uint16_t*)w, n, k, group, qweight, qzeros, scales, g_idx, snr_db,
                                       workspace, workspace_bytes, stream)
                   : gptq_quantize_asym((const uint16_t*)w, n, k, group, qweight, qzeros, scales, g_idx, snr_db,
                                        workspace, workspace_bytes, stream);
    if (w_dtype != WQ_DTYPE_F32 && w_dtype != WQ_DTYPE_F16) return WQ_ERR_BAD_DTYPE;
    if (n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (group != 32 && group != 64 && group != 128 && group != 256) return WQ_ERR_UNSUPPORTED;
    if (k % group != 0 || n % 8 != 0) return WQ_ERR_BAD_SHAPE;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !qweight || !scales) return WQ_ERR_NULL_PTR;
    if (snr_db && !workspace) return WQ_ERR_NULL_PTR;
    if (snr_db && workspace_bytes < wq_workspace_bytes(WQ_OP_GPTQ_QUANTIZE, n, k, group))
        return WQ_ERR_WORKSPACE_TOO_SMALL;
    if (!wqh::aligned16(w) || !wqh::aligned_to(qweight, 4) || !wqh::aligned_to(scales, 2) ||
        (qzeros && !wqh::aligned_to(qzeros, 4)) || (g_idx && !wqh::aligned_to(g_idx, 4)) ||
        (snr_db && !wqh::aligned_to(workspace, 256)))
        return WQ_ERR_MISALIGNED;
    return wqh::gptq_quantize_wide(w, w_dtype, n, k, group, sym != 0, qweight, qzeros, scales, g_idx, snr_db,
                                   workspace, (cudaStream_t)stream);
}

wq_status mxfp4_quantize_ex(const void* w, int w_dtype, int64_t n, int64_t k, int tie_mode, uint8_t* packed,
                            uint8_t* e8m0, void* stream) {
    if (w_dtype == WQ_DTYPE_BF16) return mxfp4_quantize((const uint16_t*)w, n, k, tie_mode, packed, e8m0, stream);
    if (w_dtype != WQ_DTYPE_F32 && w_dtype != WQ_DTYPE_F16) return WQ_ERR_BAD_DTYPE;
    if (n < 0 || k < 0 || k % 32 != 0) return WQ_ERR_BAD_SHAPE;
    if (tie_mode != WQ_TIE_HALF_EVEN && tie_mode != WQ_TIE_PAGE_LITERAL) return WQ_ERR_UNSUPPORTED;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !packed || !e8m0) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(w) || !wqh::aligned16(packed)) return WQ_ERR_MISALIGNED;
    const int64_t nblocks = n * k / 32;
    const int64_t want = (nblocks + kWideThreads - 1) / kWideThreads;
    const int grid = (int)(want < (1 << 20) ? want : (1 << 20));
    cudaStream_t st = (cudaStream_t)stream;
    const bool f32 = w_dtype == WQ_DTYPE_F32;
    if (tie_mode == WQ_TIE_HALF_EVEN) {
        if (f32) mxfp4_quant_wide_kernel<WQ_TIE_HALF_EVEN, WQ_DTYPE_F32><<<grid, kWideThreads, 0, st>>>(w, nblocks, (uint4*)packed, e8m0);
        else mxfp4_quant_wide_kernel<WQ_TIE_HALF_EVEN, WQ_DTYPE_F16><<<grid, kWideThreads, 0, st>>>(w, nblocks, (uint4*)packed, e8m0);
    } else {
        if (f32) mxfp4_quant_wide_kernel<WQ_TIE_PAGE_LITERAL, WQ_DTYPE_F32><<<grid, kWideThreads, 0, st>>>(w, nblocks, (uint4*)packed, e8m0);
        else mxfp4_quant_wide_kernel<WQ_TIE_PAGE_LITERAL, WQ_DTYPE_F16><<<grid, kWideThreads, 0, st>>>(w, nblocks, (uint4*)packed, e8m0);
    }
    return wqh::check_launch();
}

}  // extern "C"
