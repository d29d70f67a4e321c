// uintx_wide.cu -- uintx quantization and dequantization of fp16 and fp32
// weights in the weight's own dtype (uintx_quant.py: UIntXQuantizer works in the
// weight dtype; _quantize_impl, pack_uintx, _dequantize_native).
//
// Every op is the binary32 op on the operands rounded once to the weight dtype
// (for fp32 the op's own rounding), as the bf16 kernels do for bf16.  Three
// plain kernels, correctness first (bf16 weights go to the fused bf16 kernels):
//   stats  thread = one (row, group): min/max, scale and zero point
//   pack   thread = one byte of one power-of-two bit shard: the byte's 8/k_s
//          elements are e = i + j * L_s; each element's code is recomputed from
//          its group's stored scale and zero point (no workspace)
//   deq    thread = one element: its bits gathered from every shard, then
//          (q - zp) and times the scale in the weight dtype
#include <cuda_fp16.h>

#include "wq_common.cuh"

namespace {

constexpr int kUxThreads = 256;

template <int DT>
__device__ __forceinline__ float rd(float x) {  // one rounding to the weight dtype
    return DT == WQ_DTYPE_F16 ? __half2float(__float2half_rn(x)) : x;
}
template <int DT>
__device__ __forceinline__ float load_w(const void* w, int64_t i) {
    if (DT == WQ_DTYPE_F16) return __half2float(__ushort_as_half(__ldg(static_cast<const unsigned short*>(w) + i)));
    return __ldg(static_cast<const float*>(w) + i);
}
template <int DT>
__device__ __forceinline__ void store_w(void* out, int64_t i, float v) {
    if (DT == WQ_DTYPE_F16) static_cast<unsigned short*>(out)[i] = __half_as_ushort(__float2half_rn(v));
    else static_cast<float*>(out)[i] = v;
}

template <int DT>
__global__ void __launch_bounds__(kUxThreads)
uintx_stats_wide(const void* __restrict__ w, int64_t n, int64_t k, int group, int qmax, void* __restrict__ scale,
                 uint8_t* __restrict__ zp) {
    const int64_t ngr = k / group, items = n * ngr;
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = it / ngr, gi = it - r * ngr, base = r * k + gi * group;
        float mn = INFINITY, mx = -INFINITY;
        for (int j = 0; j < group; ++j) {
            const float x = load_w<DT>(w, base + j);
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
        const float mn_neg = fminf(mn, 0.f), mx_pos = fmaxf(mx, 0.f);
        float sc = rd<DT>(__fsub_rn(mx_pos, mn_neg));
        sc = rd<DT>(__fdiv_rn(sc, (float)qmax));
        sc = fmaxf(sc, 0x1p-23f);  // float32 eps, exact in fp16 and fp32
        const float ratio = rd<DT>(__fdiv_rn(mn_neg, sc));
        float z = rd<DT>(__fsub_rn(0.f, rintf(ratio)));
        z = fminf(fmaxf(z, 0.f), (float)qmax);
        store_w<DT>(scale, it, sc);
        zp[it] = (uint8_t)z;
    }
}

template <int DT>
__device__ __forceinline__ uint32_t code_of(const void* w, const void* scale, const uint8_t* zp, int64_t e,
                                            int64_t k, int group, int qmax) {
    const int64_t r = e / k, c = e - r * k, gi = r * (k / group) + c / group;
    const float sc = load_w<DT>(scale, gi), z = (float)zp[gi];
    const float inv = rd<DT>(__fdiv_rn(1.0f, sc));
    const float p = rd<DT>(__fmul_rn(load_w<DT>(w, e), inv));
    const float q = rd<DT>(__fadd_rn(rintf(p), z));
    return (uint32_t)fminf(fmaxf(q, 0.f), (float)qmax);
}

// One shard of kb bits per element: L bytes from out, element e = i + j L in
// bits j*kb .. j*kb+kb-1 of byte i; the shard holds code bits off .. off+kb-1.
template <int DT>
__global__ void __launch_bounds__(kUxThreads)
uintx_pack_wide(const void* __restrict__ w, const void* __restrict__ scale, const uint8_t* __restrict__ zp,
                int64_t numel, int64_t k, int group, int qmax, int kb, int off, int64_t L, uint8_t* __restrict__ out) {
    const int vpb = 8 / kb;
    const uint32_t mask = (1u << kb) - 1u;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < L; i += (int64_t)gridDim.x * blockDim.x) {
        uint32_t byte = 0;
        for (int j = 0; j < vpb; ++j) {
            const int64_t e = i + (int64_t)j * L;
            if (e < numel) byte |= ((code_of<DT>(w, scale, zp, e, k, group, qmax) >> off) & mask) << (j * kb);
        }
        out[i] = (uint8_t)byte;
    }
}

template <int DT>
__global__ void __launch_bounds__(kUxThreads)
uintx_deq_wide(const uint8_t* __restrict__ packed, const void* __restrict__ scale, const uint8_t* __restrict__ zp,
               int64_t numel, int64_t k, int group, int nbits, void* __restrict__ out) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < numel; e += (int64_t)gridDim.x * blockDim.x) {
        uint32_t q = 0;
        int off = 0;
        int64_t base = 0;
        for (int kb = 4; kb >= 1; kb >>= 1) {
            if (!(nbits & kb)) continue;
            const int64_t L = (numel + 8 / kb - 1) / (8 / kb);
            const int64_t j = e / L, i = e - j * L;
            q |= (((uint32_t)packed[base + i] >> (j * kb)) & ((1u << kb) - 1u)) << off;
            off += kb;
            base += L;
        }
        const int64_t r = e / k, c = e - r * k, gi = r * (k / group) + c / group;
        const float d = rd<DT>(__fsub_rn((float)q, (float)zp[gi]));
        store_w<DT>(out, e, rd<DT>(__fmul_rn(d, load_w<DT>(scale, gi))));
    }
}

int grid_of(int64_t items) {
    const int64_t g = (items + kUxThreads - 1) / kUxThreads;
    return (int)(g < (1 << 20) ? (g > 0 ? g : 1) : (1 << 20));
}

}  // namespace

extern "C" {

wq_status uintx_quantize_ex(const void* w, int w_dtype, int64_t n, int64_t k, int nbits, int group,
                            uint8_t* packed, void* scale, uint8_t* zp, void* stream) {
    if (w_dtype == WQ_DTYPE_BF16)
        return uintx_quantize((const uint16_t*)w, n, k, nbits, group, packed, (uint16_t*)scale, zp, stream);
    if (w_dtype != WQ_DTYPE_F32 && w_dtype != WQ_DTYPE_F16) return WQ_ERR_BAD_DTYPE;
    if (nbits < 2 || nbits > 7) return WQ_ERR_UNSUPPORTED;
    if (n < 0 || k < 0 || group <= 0 || group % 8 != 0 || k % group != 0) return WQ_ERR_BAD_SHAPE;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !packed || !scale || !zp) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned_to(w, w_dtype == WQ_DTYPE_F32 ? 4 : 2) || !wqh::aligned_to(scale, w_dtype == WQ_DTYPE_F32 ? 4 : 2))
        return WQ_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    const int qmax = (1 << nbits) - 1;
    const int64_t numel = n * k;
    const bool f32 = w_dtype == WQ_DTYPE_F32;
    if (f32) uintx_stats_wide<WQ_DTYPE_F32><<<grid_of(n * (k / group)), kUxThreads, 0, st>>>(w, n, k, group, qmax, scale, zp);
    else uintx_stats_wide<WQ_DTYPE_F16><<<grid_of(n * (k / group)), kUxThreads, 0, st>>>(w, n, k, group, qmax, scale, zp);
    int off = 0;
    int64_t base = 0;
    for (int kb = 4; kb >= 1; kb >>= 1) {
        if (!(nbits & kb)) continue;
        const int64_t L = (numel + 8 / kb - 1) / (8 / kb);
        if (f32)
            uintx_pack_wide<WQ_DTYPE_F32><<<grid_of(L), kUxThreads, 0, st>>>(w, scale, zp, numel, k, group, qmax, kb, off, L, packed + base);
        else
            uintx_pack_wide<WQ_DTYPE_F16><<<grid_of(L), kUxThreads, 0, st>>>(w, scale, zp, numel, k, group, qmax, kb, off, L, packed + base);
        off += kb;
        base += L;
    }
    return wqh::check_launch();
}

wq_status uintx_dequantize_ex(const uint8_t* packed, const void* scale, int w_dtype, const uint8_t* zp, int64_t n,
                              int64_t k, int nbits, int group, void* out, void* stream) {
    if (w_dtype == WQ_DTYPE_BF16)
        return uintx_dequantize(packed, (const uint16_t*)scale, zp, n, k, nbits, group, WQ_DTYPE_BF16, out, stream);
    if (w_dtype != WQ_DTYPE_F32 && w_dtype != WQ_DTYPE_F16) return WQ_ERR_BAD_DTYPE;
    if (nbits < 2 || nbits > 7) return WQ_ERR_UNSUPPORTED;
    if (n < 0 || k < 0 || group <= 0 || group % 8 != 0 || k % group != 0) return WQ_ERR_BAD_SHAPE;
    if (n == 0 || k == 0) return WQ_OK;
    if (!packed || !scale || !zp || !out) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned_to(out, w_dtype == WQ_DTYPE_F32 ? 4 : 2) || !wqh::aligned_to(scale, w_dtype == WQ_DTYPE_F32 ? 4 : 2))
        return WQ_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t numel = n * k;
    if (w_dtype == WQ_DTYPE_F32)
        uintx_deq_wide<WQ_DTYPE_F32><<<grid_of(numel), kUxThreads, 0, st>>>(packed, scale, zp, numel, k, group, nbits, out);
    else
        uintx_deq_wide<WQ_DTYPE_F16><<<grid_of(numel), kUxThreads, 0, st>>>(packed, scale, zp, numel, k, group, nbits, out);
    return wqh::check_launch();
}

}  // extern "C"
