// linear.cu -- the consumer of an exported GPTQ checkpoint, for decode batches:
// y = x deq(W)^T straight from the packed int4 weights (export_gptq_cpu.py,
// module docstring: the checkpoint is served by vLLM's W4A16 uint4b8 layer,
// which reads qweight [K/8, N], scales [K/G, N] and qzeros [K/G, N/8]).
//
// Only the codes (0.5 B per weight) and the group scale / zero point are read,
// a quarter of the bytes of a bf16 weight, so for m = 1 the kernel is HBM bound.
//
// Grid: ceil(N/256) column blocks x S slices of whole groups along K.  Thread =
// one output column.  The CTA stages its slice of x (all m rows) in shared
// memory as binary32, read by broadcast.  Per qweight word the 8 codes become
// binary32 1.5*2^23 + c by byte permutes; subtracting 1.5*2^23 + zp gives the
// exact c - zp, and f32x2 FMAs accumulate x (c - zp) over the group; the group
// sum times the fp16 scale is added to the column's sum.  Partials go to a
// workspace slot per (slice, row, column); the last CTA of a column block to
// finish adds the S slices in order (deterministic, no waiting), writes y and
// sets the block's arrival counter back to zero, so that a call needs no
// separate reset of the workspace.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr int kMaxSlices = 64;
constexpr int kMaxM = 8;
constexpr int kXSmemBytes = 40 * 1024;  // staged x: under the default 48 KB dynamic limit

__device__ __forceinline__ float code_f(uint32_t bytes, int j) {
    return __uint_as_float(__byte_perm(bytes, 0x4B400000u, 0x7640u + (unsigned)j));
}

template <bool SYM, int M, int G>
__global__ void __launch_bounds__(kThreads) gptq_linear_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ qweight,
    const int32_t* __restrict__ qzeros, const uint16_t* __restrict__ scales, int64_t n, int64_t k,
    int gps, float* __restrict__ part, unsigned* __restrict__ counters, int out_bf16,
    void* __restrict__ out) {
    extern __shared__ __align__(16) float xs[];  // [M][gps * G]
    const int64_t groups = k / G;
    const int64_t g0 = (int64_t)blockIdx.y * gps;
    const int64_t g1 = min(g0 + gps, groups);
    const int len = (int)((g1 - g0) * G);  // this slice's input channels
    const int S = gridDim.y;

    const int64_t col = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const bool colv = col < n;
    constexpr int WPG = G / 8;  // qweight words per group
    // the first group's words are requested before x is staged (independent
    // loads in flight together); each later group's while the previous is summed
    uint32_t nx[WPG];
    if (colv) {
#pragma unroll
        for (int r = 0; r < WPG; ++r) nx[r] = (uint32_t)__ldg(qweight + (g0 * WPG + r) * n + col);
    }

    // x[m][g0*G .. g1*G) -> binary32 in shared memory (8 values per thread step)
    for (int i = threadIdx.x; i < M * len / 8; i += kThreads) {
        const int m = i / (len / 8), c = i % (len / 8);
        const uint4 u = *reinterpret_cast<const uint4*>(x + m * k + g0 * G + 8 * c);
        float4* d = reinterpret_cast<float4*>(xs + m * (gps * G) + 8 * c);
        d[0] = make_float4(wq::bf_lo(u.x), wq::bf_hi(u.x), wq::bf_lo(u.y), wq::bf_hi(u.y));
        d[1] = make_float4(wq::bf_lo(u.z), wq::bf_hi(u.z), wq::bf_lo(u.w), wq::bf_hi(u.w));
    }
    __syncthreads();

    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.0f;
    if (colv) {
        for (int64_t g = g0; g < g1; ++g) {
            uint32_t wd[WPG];
#pragma unroll
            for (int r = 0; r < WPG; ++r) wd[r] = nx[r];
            if (g + 1 < g1) {
#pragma unroll
                for (int r = 0; r < WPG; ++r) nx[r] = (uint32_t)__ldg(qweight + ((g + 1) * WPG + r) * n + col);
            }
            const float s = __half2float(__ushort_as_half(__ldg(scales + g * n + col)));
            float zp = 8.0f;
            if (!SYM) zp = (float)((__ldg(qzeros + g * (n / 8) + col / 8) >> (4 * (col & 7))) & 15);
            const wq::f2_t Z2 = wq::f2(-(kMagic + zp), -(kMagic + zp));
            wq::f2_t ag[M];
#pragma unroll
            for (int m = 0; m < M; ++m) ag[m] = wq::f2(0.0f, 0.0f);
            const float* xg = xs + (g - g0) * G;
#pragma unroll
            for (int r = 0; r < WPG; ++r) {
                const uint32_t lo = wd[r] & 0x0F0F0F0Fu, hi = (wd[r] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // c - zp of input channels 8r + 4h .. 8r + 4h + 3 (exact)
                    const wq::f2_t d0 = wq::add2(wq::f2(code_f(lo, 2 * h), code_f(hi, 2 * h)), Z2);
                    const wq::f2_t d1 = wq::add2(wq::f2(code_f(lo, 2 * h + 1), code_f(hi, 2 * h + 1)), Z2);
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const float4 xv = *reinterpret_cast<const float4*>(xg + m * (gps * G) + 8 * r + 4 * h);
                        ag[m] = wq::fma2(d0, wq::f2(xv.x, xv.y), ag[m]);
                        ag[m] = wq::fma2(d1, wq::f2(xv.z, xv.w), ag[m]);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < M; ++m) acc[m] = __fmaf_rn(__fadd_rn(ag[m].x, ag[m].y), s, acc[m]);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) part[((int64_t)blockIdx.y * M + m) * n + col] = acc[m];
    }
    // the last CTA of this column block adds the slices in order
    // (the barrier orders every thread's partial before thread 0's fence, which
    // makes them visible device-wide before the arrival is counted)
    __shared__ bool last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(counters + blockIdx.x, 1u) == (unsigned)S - 1;
    }
    __syncthreads();
    if (!last) return;
    if (threadIdx.x == 0) counters[blockIdx.x] = 0u;  // ready for the next call
    if (!colv) return;
    __threadfence();
#pragma unroll
    for (int m = 0; m < M; ++m) {
        // slices in order; loads issued 16 at a time, not one per dependent add
        float y = 0.0f;
        for (int s0 = 0; s0 < S; s0 += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                v[i] = s0 + i < S ? __ldcg(part + ((int64_t)(s0 + i) * M + m) * n + col) : 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (s0 + i < S) y = __fadd_rn(y, v[i]);
        }
        if (out_bf16)
            reinterpret_cast<uint16_t*>(out)[m * n + col] = (uint16_t)wq::f_to_bf(y);
        else
            reinterpret_cast<float*>(out)[m * n + col] = y;
    }
}

template <bool SYM, int M, int G>
wq_status launch_linear(const uint16_t* x, const int32_t* qweight, const int32_t* qzeros,
                        const uint16_t* scales, int64_t n, int64_t k, int out_bf16, void* out,
                        char* ws, cudaStream_t st) {
    const void* fn = (const void*)gptq_linear_kernel<SYM, M, G>;
    const int64_t col_blocks = (n + kThreads - 1) / kThreads;
    const int64_t groups = k / G;
    const int64_t target = wqh::grid_for(fn, kThreads, 0, (int64_t)1 << 30, 1 << 30);
    int64_t S = target / col_blocks;
    if (S < 1) S = 1;
    if (S > kMaxSlices) S = kMaxSlices;
    if (S > groups) S = groups;
    int64_t gps = (groups + S - 1) / S;
    const int64_t max_gps = kXSmemBytes / (M * G * 4);
    if (gps > max_gps) return WQ_ERR_BAD_SHAPE;  // k beyond kMaxSlices * max_gps groups
    S = (groups + gps - 1) / gps;
    // arrival counters: zero before the first call (the caller zeroes the
    // workspace once), reset to zero by the last CTA of every column block
    unsigned* counters = reinterpret_cast<unsigned*>(ws);
    float* part = reinterpret_cast<float*>(ws + ((col_blocks * 4 + 255) & ~(int64_t)255));
    const size_t smem = (size_t)M * gps * G * sizeof(float);
    gptq_linear_kernel<SYM, M, G><<<dim3((unsigned)col_blocks, (unsigned)S), kThreads, smem, st>>>(
        x, qweight, qzeros, scales, n, k, (int)gps, part, counters, out_bf16, out);
    return wqh::check_launch();
}

template <bool SYM, int G>
wq_status dispatch_m(int64_t m, const uint16_t* x, const int32_t* qw, const int32_t* qz,
                     const uint16_t* sc, int64_t n, int64_t k, int ob, void* out, char* ws,
                     cudaStream_t st) {
    switch (m) {
        case 1: return launch_linear<SYM, 1, G>(x, qw, qz, sc, n, k, ob, out, ws, st);
        case 2: return launch_linear<SYM, 2, G>(x, qw, qz, sc, n, k, ob, out, ws, st);
        case 3: return launch_linear<SYM, 3, G>(x, qw, qz, sc, n, k, ob, out, ws, st);
        case 4: return launch_linear<SYM, 4, G>(x, qw, qz, sc, n, k, ob, out, ws, st);
        case 5: return launch_linear<SYM, 5, G>(x, qw, qz, sc, n, k, ob, out, ws, st);
        case 6: return launch_linear<SYM, 6, G>(x, qw, qz, sc, n, k, ob, out, ws, st);
        case 7: return launch_linear<SYM, 7, G>(x, qw, qz, sc, n, k, ob, out, ws, st);
        default: return launch_linear<SYM, 8, G>(x, qw, qz, sc, n, k, ob, out, ws, st);
    }
}

template <bool SYM>
wq_status dispatch_g(int group, int64_t m, const uint16_t* x, const int32_t* qw, const int32_t* qz,
                     const uint16_t* sc, int64_t n, int64_t k, int ob, void* out, char* ws,
                     cudaStream_t st) {
    switch (group) {
        case 32: return dispatch_m<SYM, 32>(m, x, qw, qz, sc, n, k, ob, out, ws, st);
        case 64: return dispatch_m<SYM, 64>(m, x, qw, qz, sc, n, k, ob, out, ws, st);
        case 128: return dispatch_m<SYM, 128>(m, x, qw, qz, sc, n, k, ob, out, ws, st);
        default: return dispatch_m<SYM, 256>(m, x, qw, qz, sc, n, k, ob, out, ws, st);
    }
}

// ------------------------------------------------------------------ MXFP4
// y = x deq(W)^T from the packed e2m1 codes [n, k/2] and the E8M0 bytes
// [n, k/32] (quantize_dflash_mxfp4.py: the drafter's linears are served in this
// format; deq as dequantize_mxfp4).  A CTA of 4 warps owns kRowsMx output rows
// and all of k; the warps take interleaved K steps; lane = WPL consecutive
// weights of one 32-weight block (one 16-, 8- or 4-byte code load and one E8M0
// byte per row), with all rows' loads issued together and the lane's x values
// converted once and reused for every row.  WPL is 32 for m <= 2, 16 for m <= 4
// and 8 above (the x values of a lane stay in registers).  Codes -> f16x2 by
// the hardware e2m1 conversion (exact); products with x are exact in binary32
// and summed per lane and block, times 2^(e - 127), added per row; then
// fixed-order warp shuffles and a shared-memory sum over the 4 warps
// (deterministic, no workspace).

constexpr int kRowsMx = 8;
constexpr int kThreadsMx = 128;

__device__ __forceinline__ wq::f2_t e2m1_pair(uint32_t byte) {
    uint32_t h2;
    const uint16_t in = (uint16_t)byte;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "h"(in));
    return __half22float2(*reinterpret_cast<const __half2*>(&h2));  // (low nibble, high nibble)
}

template <int NW>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[NW]) {
    if (NW == 4) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        w[0] = v.x; w[NW > 1 ? 1 : 0] = v.y; w[NW > 2 ? 2 : 0] = v.z; w[NW > 3 ? 3 : 0] = v.w;
    } else if (NW == 2) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
        w[0] = v.x; w[NW > 1 ? 1 : 0] = v.y;
    } else {
        w[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
    }
}

template <int M, int WPL>
__global__ void __launch_bounds__(kThreadsMx) mxfp4_linear_kernel(const uint16_t* __restrict__ x,
                                                                  const uint8_t* __restrict__ packed,
                                                                  const uint8_t* __restrict__ e8m0,
                                                                  int64_t n, int64_t k, int out_bf16,
                                                                  void* __restrict__ out) {
    constexpr int WARPS = kThreadsMx / 32;
    constexpr int NW = WPL / 8;  // 32-bit code words (8 codes) per lane and row
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t r0 = (int64_t)blockIdx.x * kRowsMx;
    float acc[kRowsMx][M];
#pragma unroll
    for (int r = 0; r < kRowsMx; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;
    for (int64_t kk = ((int64_t)warp * 32 + lane) * WPL; kk < k; kk += (int64_t)WARPS * 32 * WPL) {
        // every row's codes and scale byte requested before any is decoded (rows
        // past n read row n - 1 and are never written)
        uint32_t w[kRowsMx][NW], eb[kRowsMx];
#pragma unroll
        for (int r = 0; r < kRowsMx; ++r) {
            const int64_t row = min(r0 + r, n - 1);
            load_words<NW>(packed + row * (k / 2) + kk / 2, w[r]);
            eb[r] = __ldg(e8m0 + row * (k / 32) + kk / 32);
        }
        wq::f2_t xv[M][WPL / 2];
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int q = 0; q < WPL / 8; ++q) {
                const uint4 u = *reinterpret_cast<const uint4*>(x + m * k + kk + 8 * q);
                xv[m][4 * q + 0] = wq::bf2_to_f2(u.x);
                xv[m][4 * q + 1] = wq::bf2_to_f2(u.y);
                xv[m][4 * q + 2] = wq::bf2_to_f2(u.z);
                xv[m][4 * q + 3] = wq::bf2_to_f2(u.w);
            }
#pragma unroll
        for (int r = 0; r < kRowsMx; ++r) {
            const uint32_t e = eb[r];
            const float sc = __uint_as_float(e == 0 ? 0x00400000u : (e << 23));  // 2^(e-127); 255 -> inf
            wq::f2_t pm[M];
#pragma unroll
            for (int m = 0; m < M; ++m) pm[m] = wq::f2(0.0f, 0.0f);
#pragma unroll
            for (int q = 0; q < NW; ++q)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const wq::f2_t c = e2m1_pair((w[r][q] >> (8 * j)) & 0xffu);
#pragma unroll
                    for (int m = 0; m < M; ++m) pm[m] = wq::fma2(c, xv[m][4 * q + j], pm[m]);
                }
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = __fmaf_rn(__fadd_rn(pm[m].x, pm[m].y), sc, acc[r][m]);
        }
    }
    __shared__ float red[WARPS][kRowsMx][kMaxM];
#pragma unroll
    for (int r = 0; r < kRowsMx; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) red[warp][r][m] = v;
        }
    __syncthreads();
    if (threadIdx.x < kRowsMx * M) {
        const int r = threadIdx.x / M, m = threadIdx.x % M;
        const int64_t row = r0 + r;
        if (row < n) {
            float y = 0.0f;
#pragma unroll
            for (int w2 = 0; w2 < WARPS; ++w2) y = __fadd_rn(y, red[w2][r][m]);
            if (out_bf16)
                reinterpret_cast<uint16_t*>(out)[m * n + row] = (uint16_t)wq::f_to_bf(y);
            else
                reinterpret_cast<float*>(out)[m * n + row] = y;
        }
    }
}

template <int M>
wq_status launch_mx_linear(const uint16_t* x, const uint8_t* packed, const uint8_t* e8m0, int64_t n,
                           int64_t k, int out_bf16, void* out, cudaStream_t st) {
    constexpr int WPL = M <= 2 ? 32 : (M <= 4 ? 16 : 8);
    const int64_t grid = (n + kRowsMx - 1) / kRowsMx;
    mxfp4_linear_kernel<M, WPL><<<(unsigned)grid, kThreadsMx, 0, st>>>(x, packed, e8m0, n, k, out_bf16, out);
    return wqh::check_launch();
}

}  // namespace

extern "C" wq_status mxfp4_linear(const uint16_t* x, int64_t m, const uint8_t* packed,
                                  const uint8_t* e8m0, int64_t n, int64_t k, int out_dtype,
                                  void* out, void* stream) {
    if (m < 0 || n < 0 || k < 0 || k % 32 != 0) return WQ_ERR_BAD_SHAPE;
    if (m > kMaxM) return WQ_ERR_UNSUPPORTED;
    if (out_dtype != WQ_DTYPE_F32 && out_dtype != WQ_DTYPE_BF16) return WQ_ERR_BAD_DTYPE;
    if ((n + kRowsMx - 1) / kRowsMx >= ((int64_t)1 << 31)) return WQ_ERR_BAD_SHAPE;
    if (m == 0 || n == 0) return WQ_OK;
    if (!out) return WQ_ERR_NULL_PTR;
    cudaStream_t st = (cudaStream_t)stream;
    if (k == 0)  // an empty sum: y = 0
        return wqh::cuda_status(cudaMemsetAsync(out, 0, (size_t)(m * n) * (out_dtype == WQ_DTYPE_BF16 ? 2 : 4), st));
    if (!x || !packed || !e8m0) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(x) || !wqh::aligned16(packed) || !wqh::aligned_to(out, 4)) return WQ_ERR_MISALIGNED;
    const int ob = out_dtype == WQ_DTYPE_BF16;
    switch (m) {
        case 1: return launch_mx_linear<1>(x, packed, e8m0, n, k, ob, out, st);
        case 2: return launch_mx_linear<2>(x, packed, e8m0, n, k, ob, out, st);
        case 3: return launch_mx_linear<3>(x, packed, e8m0, n, k, ob, out, st);
        case 4: return launch_mx_linear<4>(x, packed, e8m0, n, k, ob, out, st);
        case 5: return launch_mx_linear<5>(x, packed, e8m0, n, k, ob, out, st);
        case 6: return launch_mx_linear<6>(x, packed, e8m0, n, k, ob, out, st);
        case 7: return launch_mx_linear<7>(x, packed, e8m0, n, k, ob, out, st);
        default: return launch_mx_linear<8>(x, packed, e8m0, n, k, ob, out, st);
    }
}

extern "C" size_t gptq_linear_workspace_bytes(int64_t m, int64_t n) {
    if (m < 1 || m > kMaxM || n < 0) return 0;
    const size_t col_blocks = (size_t)((n + kThreads - 1) / kThreads);
    return ((col_blocks * 4 + 255) & ~(size_t)255) + (size_t)kMaxSlices * m * n * sizeof(float);
}

extern "C" wq_status gptq_linear(const uint16_t* x, int64_t m, const int32_t* qweight,
                                 const int32_t* qzeros, const uint16_t* scales, int64_t n,
                                 int64_t k, int group, int sym, int out_dtype, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    if (m < 0 || n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (m > kMaxM) return WQ_ERR_UNSUPPORTED;
    if (group != 32 && group != 64 && group != 128 && group != 256) return WQ_ERR_UNSUPPORTED;
    if (k % group != 0 || n % 8 != 0) return WQ_ERR_BAD_SHAPE;
    if (out_dtype != WQ_DTYPE_F32 && out_dtype != WQ_DTYPE_BF16) return WQ_ERR_BAD_DTYPE;
    if (m == 0 || n == 0) return WQ_OK;
    if (!out) return WQ_ERR_NULL_PTR;
    if (k == 0)  // an empty sum: y = 0
        return wqh::cuda_status(cudaMemsetAsync(out, 0, (size_t)(m * n) * (out_dtype == WQ_DTYPE_BF16 ? 2 : 4),
                                                (cudaStream_t)stream));
    if (!x || !qweight || !scales || !workspace || (!sym && !qzeros)) return WQ_ERR_NULL_PTR;
    if (workspace_bytes < gptq_linear_workspace_bytes(m, n)) return WQ_ERR_WORKSPACE_TOO_SMALL;
    if (!wqh::aligned16(x) || !wqh::aligned_to(qweight, 4) || !wqh::aligned_to(scales, 2) ||
        (!sym && !wqh::aligned_to(qzeros, 4)) || !wqh::aligned_to(out, 4) ||
        !wqh::aligned_to(workspace, 256))
        return WQ_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    char* ws = (char*)workspace;
    const int ob = out_dtype == WQ_DTYPE_BF16;
    return sym ? dispatch_g<true>(group, m, x, qweight, qzeros, scales, n, k, ob, out, ws, st)
               : dispatch_g<false>(group, m, x, qweight, qzeros, scales, n, k, ob, out, ws, st);
}
