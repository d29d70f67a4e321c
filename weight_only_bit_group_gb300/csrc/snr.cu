// snr.cu -- reconstruction SNR and relative error (export_gptq_cpu.py,
// quantize_sym / quantize_asym: snr = 20*log10(||w|| / max(||w - deq||, 1e-12));
// quantize_dflash_mxfp4.py main(): rel = ||deq - w|| / ||w||).
//
// Two passes, no atomics, deterministic for a given grid: every CTA writes its
// (sum w^2, sum e^2) to its own workspace slot; one CTA adds the slots in index
// order and evaluates the formulas.  Terms are binary32 (as the page computes
// them); sums are binary32 over at most 32 terms per thread and binary64 above.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// Sum two doubles over the CTA in a fixed order; thread 0 writes the slot.
__device__ __forceinline__ void cta_store_pair(double a, double b, double* slot) {
    __shared__ double sa[kThreads / 32], sb[kThreads / 32];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, m);
        b += __shfl_xor_sync(0xffffffffu, b, m);
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) { sa[warp] = a; sb[warp] = b; }
    __syncthreads();
    if (threadIdx.x == 0) {
        double ta = 0.0, tb = 0.0;
        for (int i = 0; i < kThreads / 32; ++i) { ta += sa[i]; tb += sb[i]; }
        slot[0] = ta;
        slot[1] = tb;
    }
}

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
                                                           int64_t nchunks, double* __restrict__ slots) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    double dw = 0.0, de = 0.0;
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
                    sw = __fadd_rn(sw, __fmul_rn(x[i], x[i]));
                    se = __fadd_rn(se, __fmul_rn(e, e));
                }
            }
        }
        dw += (double)sw;
        de += (double)se;
    }
    cta_store_pair(dw, de, slots + 2 * blockIdx.x);
}

// deq laid out [k, n] (the GPTQ page's layout): 64 x 64 tiles, the deq tile is
// staged in shared memory so that both reads stay coalesced.
constexpr int kT = 64;

template <int DEQ_BF16>
__global__ void __launch_bounds__(kThreads) snr_partial_kn(const uint16_t* __restrict__ w,
                                                           const void* __restrict__ deq, int64_t n,
                                                           int64_t k, double* __restrict__ slots) {
    __shared__ float sd[kT][kT + 1];  // [k][n]
    const int64_t tiles_n = (n + kT - 1) / kT, tiles_k = (k + kT - 1) / kT;
    double dw = 0.0, de = 0.0;
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
                        sw = __fadd_rn(sw, __fmul_rn(x, x));
                        se = __fadd_rn(se, __fmul_rn(e, e));
                    }
                }
            }
        }
        dw += (double)sw;
        de += (double)se;
    }
    cta_store_pair(dw, de, slots + 2 * blockIdx.x);
}

__global__ void __launch_bounds__(kThreads) snr_finalize(const double* __restrict__ slots, int nslots,
                                                         double* __restrict__ snr_db,
                                                         double* __restrict__ rel_err) {
    __shared__ double sa[kThreads], sb[kThreads];
    double a = 0.0, b = 0.0;
    for (int i = threadIdx.x; i < nslots; i += kThreads) {
        a += slots[2 * i];
        b += slots[2 * i + 1];
    }
    sa[threadIdx.x] = a;
    sb[threadIdx.x] = b;
    __syncthreads();
    for (int s = kThreads / 2; s >= 1; s >>= 1) {
        if (threadIdx.x < s) {
            sa[threadIdx.x] += sa[threadIdx.x + s];
            sb[threadIdx.x] += sb[threadIdx.x + s];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double nw = sqrt(sa[0]), ne = sqrt(sb[0]);
        if (snr_db) *snr_db = 20.0 * log10(nw / fmax(ne, 1e-12));
        if (rel_err) *rel_err = ne / nw;
    }
}

}  // namespace

namespace wqh {
wq_status launch_snr_finalize(const double* slots, int nslots, double* snr_db, double* rel_err,
                              cudaStream_t st) {
    snr_finalize<<<1, kThreads, 0, st>>>(slots, nslots, snr_db, rel_err);
    return check_launch();
}
}  // namespace wqh

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
    cudaStream_t st = (cudaStream_t)stream;
    double* slots = (double*)workspace;
    int grid = 1;
    if (n * k > 0) {
        if (deq_layout == WQ_LAYOUT_NK) {
            const int64_t nchunks = n * k / 8;
            const void* fn = deq_dtype == WQ_DTYPE_BF16 ? (const void*)snr_partial_nk<1>
                                                        : (const void*)snr_partial_nk<0>;
            grid = wqh::grid_for(fn, kThreads, 0, (nchunks + kThreads - 1) / kThreads, wqh::kMaxPartials);
            if (deq_dtype == WQ_DTYPE_BF16)
                snr_partial_nk<1><<<grid, kThreads, 0, st>>>((const uint4*)w, deq, nchunks, slots);
            else
                snr_partial_nk<0><<<grid, kThreads, 0, st>>>((const uint4*)w, deq, nchunks, slots);
        } else {
            const int64_t tiles = ((n + kT - 1) / kT) * ((k + kT - 1) / kT);
            const void* fn = deq_dtype == WQ_DTYPE_BF16 ? (const void*)snr_partial_kn<1>
                                                        : (const void*)snr_partial_kn<0>;
            grid = wqh::grid_for(fn, kThreads, 0, tiles, wqh::kMaxPartials);
            if (deq_dtype == WQ_DTYPE_BF16)
                snr_partial_kn<1><<<grid, kThreads, 0, st>>>(w, deq, n, k, slots);
            else
                snr_partial_kn<0><<<grid, kThreads, 0, st>>>(w, deq, n, k, slots);
        }
        wq_status s = wqh::check_launch();
        if (s != WQ_OK) return s;
    } else {
        // empty tensor: one zero slot, so the finalize gives 20*log10(0/1e-12) = -inf
        wq_status s = wqh::cuda_status(cudaMemsetAsync(slots, 0, 2 * sizeof(double), st));
        if (s != WQ_OK) return s;
    }
    return wqh::launch_snr_finalize(slots, grid, snr_db, rel_err, st);
}
