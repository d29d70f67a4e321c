// snr.cu -- reconstruction SNR and relative error (export_gptq_cpu.py,
// quantize_sym / quantize_asym: snr = 20*log10(||w|| / max(||w - deq||, 1e-12));
// quantize_dflash_mxfp4.py main(): rel = ||deq - w|| / ||w||).
//
// One pass, deterministic for a given grid: every CTA writes its (sum w^2,
// sum e^2) to its own workspace slot; the last CTA to finish adds the slots in
// index order and evaluates the formulas in binary64 (nothing waits).  Terms are
// binary32 (as the page computes them); each thread sums at most 32 terms in
// binary32 and adds those partials into a compensated binary32 running sum; the
// CTA and final sums are float-float (hi + lo binary32 pairs, about 44 bits) on
// the FP32 pipes, since the binary64 pipe of this GPU is too narrow for a whole
// wave of CTAs to reduce in binary64.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <int DEQ_BF16>
__device__ __forceinline__ void load_deq8(const void* deq, int64_t c, float d[8]) {
    if (DEQ_BF16) {
        uint4 u = wq::ld_stream(reinterpret_cast<const uint4*>(deq) + c);
        d[0] = wq::bf_lo(u.x); d[1] = wq::bf_hi(u.x); d[2] = wq::bf_lo(u.y); d[3] = wq::bf_hi(u.y);
        d[4] = wq::bf_lo(u.z); d[5] = wq::bf_hi(u.z); d[6] = wq::bf_lo(u.w); d[7] = wq::bf_hi(u.w);
    } else {
        const uint4* p = reinterpret_cast<const uint4*>(deq) + 2 * c;
        uint4 u0 = wq::ld_stream(p), u1 = wq::ld_stream(p + 1);
        d[0] = __uint_as_float(u0.x); d[1] = __uint_as_float(u0.y);
        d[2] = __uint_as_float(u0.z); d[3] = __uint_as_float(u0.w);
        d[4] = __uint_as_float(u1.x); d[5] = __uint_as_float(u1.y);
        d[6] = __uint_as_float(u1.z); d[7] = __uint_as_float(u1.w);
    }
}

// deq laid out like w ([n, k]): a flat stream of 8-value chunks.
template <int DEQ_BF16>
__global__ void __launch_bounds__(kThreads) snr_partial_nk(const uint4* __restrict__ w,
                                                           const void* __restrict__ deq,
                                                           int64_t nchunks, float4* __restrict__ slots,
                                                           unsigned* __restrict__ counter,
                                                           double* __restrict__ snr_db,
                                                           double* __restrict__ rel_err) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    wq::KSum dw, de;
    for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < nchunks;
         base += stride * kUnroll) {
        float sw = 0.0f, se = 0.0f;
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) {
            const int64_t c = base + (int64_t)j * stride;
            if (c < nchunks) {
                uint4 u = wq::ld_stream(w + c);
                float d[8];
                load_deq8<DEQ_BF16>(deq, c, d);
                float x[8] = {wq::bf_lo(u.x), wq::bf_hi(u.x), wq::bf_lo(u.y), wq::bf_hi(u.y),
                              wq::bf_lo(u.z), wq::bf_hi(u.z), wq::bf_lo(u.w), wq::bf_hi(u.w)};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float e = __fsub_rn(x[i], d[i]);
                    sw = __fmaf_rn(x[i], x[i], sw);
                    se = __fmaf_rn(e, e, se);
                }
            }
        }
        dw.add(sw);
        de.add(se);
    }
    wq::finish_snr(wq::ff_of(dw), wq::ff_of(de), slots, counter, snr_db, rel_err);
}

// deq laid out [k, n] (the GPTQ page's layout): 64 x 64 tiles, the deq tile is
// staged in shared memory so that both reads stay coalesced.
constexpr int kT = 64;

template <int DEQ_BF16>
__global__ void __launch_bounds__(kThreads) snr_partial_kn(const uint16_t* __restrict__ w,
                                                           const void* __restrict__ deq, int64_t n,
                                                           int64_t k, float4* __restrict__ slots,
                                                           unsigned* __restrict__ counter,
                                                           double* __restrict__ snr_db,
                                                           double* __restrict__ rel_err) {
    __shared__ float sd[kT][kT + 1];  // [k][n]
    const int64_t tiles_n = (n + kT - 1) / kT, tiles_k = (k + kT - 1) / kT;
    wq::KSum dw, de;
    for (int64_t t = blockIdx.x; t < tiles_n * tiles_k; t += gridDim.x) {
        const int64_t n0 = (t % tiles_n) * kT, k0 = (t / tiles_n) * kT;
        __syncthreads();
        // deq rows k0..k0+63, columns n0..n0+63: 4 consecutive columns per thread
        for (int i = threadIdx.x; i < kT * (kT / 4); i += kThreads) {
            const int kr = i / (kT / 4), nc = (i % (kT / 4)) * 4;
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            const int64_t kk = k0 + kr;
            if (kk < k) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t nn = n0 + nc + q;
                    if (nn < n) {
                        v[q] = DEQ_BF16 ? wq::bf_to_f(reinterpret_cast<const uint16_t*>(deq)[kk * n + nn])
                                        : reinterpret_cast<const float*>(deq)[kk * n + nn];
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) sd[kr][nc + q] = v[q];
        }
        __syncthreads();
        // w rows n0..n0+63, columns k0..k0+63: 8 consecutive k per thread
        float sw = 0.0f, se = 0.0f;
        for (int i = threadIdx.x; i < kT * (kT / 8); i += kThreads) {
            const int nr = i / (kT / 8), kc = (i % (kT / 8)) * 8;
            const int64_t nn = n0 + nr;
            if (nn < n) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int64_t kk = k0 + kc + q;
                    if (kk < k) {
                        float x = wq::bf_to_f(w[nn * k + kk]);
                        float e = __fsub_rn(x, sd[kc + q][nr]);
                        sw = __fmaf_rn(x, x, sw);
                        se = __fmaf_rn(e, e, se);
                    }
                }
            }
        }
        dw.add(sw);
        de.add(se);
    }
    wq::finish_snr(wq::ff_of(dw), wq::ff_of(de), slots, counter, snr_db, rel_err);
}

}  // namespace

extern "C" wq_status quant_snr(const uint16_t* w, const void* deq, int deq_dtype, int deq_layout,
                               int64_t n, int64_t k, double* snr_db, double* rel_err,
                               void* workspace, size_t workspace_bytes, void* stream) {
    if (n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (deq_dtype != WQ_DTYPE_F32 && deq_dtype != WQ_DTYPE_BF16) return WQ_ERR_BAD_DTYPE;
    if (deq_layout != WQ_LAYOUT_NK && deq_layout != WQ_LAYOUT_KN) return WQ_ERR_UNSUPPORTED;
    if (!snr_db && !rel_err) return WQ_OK;
    if (!w || !deq || !workspace) return WQ_ERR_NULL_PTR;
    if (workspace_bytes < wq_workspace_bytes(WQ_OP_QUANT_SNR, n, k, 0)) return WQ_ERR_WORKSPACE_TOO_SMALL;
    if (!wqh::aligned16(w) || !wqh::aligned16(deq) || !wqh::aligned_to(workspace, 8))
        return WQ_ERR_MISALIGNED;
    if (deq_layout == WQ_LAYOUT_NK && (n * k) % 8 != 0) return WQ_ERR_BAD_SHAPE;
    if (n == 0 || k == 0) {
        // empty tensor: 20*log10(0 / 1e-12) = -inf, 0/0 = NaN, as torch gives
        const double v[2] = {-INFINITY, NAN};
        if (snr_db) {
            wq_status s0 = wqh::cuda_status(cudaMemcpyAsync(snr_db, &v[0], sizeof(double),
                                                            cudaMemcpyHostToDevice, (cudaStream_t)stream));
            if (s0 != WQ_OK) return s0;
        }
        if (rel_err)
            return wqh::cuda_status(cudaMemcpyAsync(rel_err, &v[1], sizeof(double),
                                                    cudaMemcpyHostToDevice, (cudaStream_t)stream));
        return WQ_OK;
    }
    cudaStream_t st = (cudaStream_t)stream;
    unsigned* counter = (unsigned*)workspace;
    float4* slots = (float4*)((char*)workspace + wqh::kCtrlBytes);
    wq_status s = wqh::cuda_status(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
    if (s != WQ_OK) return s;
    if (deq_layout == WQ_LAYOUT_NK) {
        const int64_t nchunks = n * k / 8;
        const void* fn = deq_dtype == WQ_DTYPE_BF16 ? (const void*)snr_partial_nk<1>
                                                    : (const void*)snr_partial_nk<0>;
        const int grid = wqh::grid_for(fn, kThreads, 0, (nchunks + kThreads - 1) / kThreads,
                                       wqh::kMaxPartials);
        if (deq_dtype == WQ_DTYPE_BF16)
            snr_partial_nk<1><<<grid, kThreads, 0, st>>>((const uint4*)w, deq, nchunks, slots, counter,
                                                          snr_db, rel_err);
        else
            snr_partial_nk<0><<<grid, kThreads, 0, st>>>((const uint4*)w, deq, nchunks, slots, counter,
                                                          snr_db, rel_err);
    } else {
        const int64_t tiles = ((n + kT - 1) / kT) * ((k + kT - 1) / kT);
        const void* fn = deq_dtype == WQ_DTYPE_BF16 ? (const void*)snr_partial_kn<1>
                                                    : (const void*)snr_partial_kn<0>;
        const int grid = wqh::grid_for(fn, kThreads, 0, tiles, wqh::kMaxPartials);
        if (deq_dtype == WQ_DTYPE_BF16)
            snr_partial_kn<1><<<grid, kThreads, 0, st>>>(w, deq, n, k, slots, counter, snr_db, rel_err);
        else
            snr_partial_kn<0><<<grid, kThreads, 0, st>>>(w, deq, n, k, slots, counter, snr_db, rel_err);
    }
    return wqh::check_launch();
}
