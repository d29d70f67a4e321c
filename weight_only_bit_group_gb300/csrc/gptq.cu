// gptq.cu -- GPTQ int4 quantize (sym / asym) and dequantize
// (export_gptq_cpu.py: pack_int32, quantize_sym, quantize_asym; module docstring
// for the uint4b8 dequant rule).
//
// Quantize tile: 64 output channels (rows of w) x 256 input channels.  Lane l of
// a warp reads w[row][k0 + 8l .. 8l+7] (one 16-byte load); warp j owns rows
// j, j+8, ..., j+56, so a CTA keeps 32 KB of loads in flight.  The eight codes of
// a lane are one qweight word (row r = (k0 + 8l)/8, column = row of w); words go
// through shared memory so that each qweight row segment [r][n0 .. n0+63] leaves
// as 256 contiguous bytes.  Per (group, column) parameters: the max/min is a
// shuffle reduction over the group's G/8 lanes; the divisions are then done once
// per group (not once per lane) and broadcast back by shuffle.  Per element the
// quotient x / scale uses a correctly rounded reciprocal and one FMA correction
// (bit-identical to IEEE division), round-half-even comes from the binary32
// adder, and the clamp to [0, 15] is applied before rounding (exact because the
// bounds are integers).
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kNT = 64;   // rows of w (columns of qweight) per tile
constexpr int kKT = 256;  // input channels per tile
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

struct GroupParams {
    float s;   // binary32 scale
    float r;   // RN(1 / s)
    float zp;  // zero point as a float (8 for sym)
};

template <bool SYM>
__device__ __forceinline__ GroupParams make_params(float a, float b) {
    // SYM: a = amax.  ASYM: a = wmax, b = wmin.
    GroupParams p;
    if (SYM) {
        p.s = fmaxf(__fdiv_rn(a, 8.0f), 1e-9f);
        p.zp = 8.0f;
    } else {
        p.s = __fdiv_rn(fmaxf(__fsub_rn(a, b), 1e-9f), 15.0f);
        p.zp = fminf(fmaxf(rintf(__fdiv_rn(-b, p.s)), 0.0f), 15.0f);
    }
    p.r = __frcp_rn(p.s);
    return p;
}

template <bool SYM, int G, bool SNR>
__global__ void __launch_bounds__(kThreads) gptq_quant_kernel(
    const uint16_t* __restrict__ w, int64_t n, int64_t k, int32_t* __restrict__ qweight,
    int32_t* __restrict__ qzeros, uint16_t* __restrict__ scales, int32_t* __restrict__ g_idx,
    double* __restrict__ slots) {
    constexpr int LPG = G / 8;                    // lanes per group
    constexpr int RPL = LPG >= 8 ? 1 : 8 / LPG;   // rows whose parameters each lane computes
    constexpr int GPT = kKT / G;                  // groups per tile along k
    __shared__ uint32_t s_qw[kKT / 8][kNT + 1];
    __shared__ uint16_t s_sc[GPT][kNT];
    __shared__ uint8_t s_zp[GPT][kNT];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t tiles_n = (n + kNT - 1) / kNT, tiles_k = (k + kKT - 1) / kKT;
    double dw = 0.0, de = 0.0;

    for (int64_t t = blockIdx.x; t < tiles_n * tiles_k; t += gridDim.x) {
        const int64_t n0 = (t % tiles_n) * kNT, k0 = (t / tiles_n) * kKT;
        const int64_t kk = k0 + 8 * lane;
        const bool kval = kk < k;  // k % G == 0: a group is all-valid or all-invalid

        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = n0 + warp + 8 * i;
            v[i] = (kval && row < n) ? wq::ld_stream(w + row * k + kk) : make_uint4(0, 0, 0, 0);
        }

        // per-row group statistics, reduced over the LPG lanes of the group
        float ra[8], rb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float x[8] = {wq::bf_lo(v[i].x), wq::bf_hi(v[i].x), wq::bf_lo(v[i].y), wq::bf_hi(v[i].y),
                          wq::bf_lo(v[i].z), wq::bf_hi(v[i].z), wq::bf_lo(v[i].w), wq::bf_hi(v[i].w)};
            float a, b = 0.0f;
            if (SYM) {
                a = fabsf(x[0]);
#pragma unroll
                for (int j = 1; j < 8; ++j) a = fmaxf(a, fabsf(x[j]));
#pragma unroll
                for (int m = 1; m < LPG; m <<= 1) a = fmaxf(a, wq::shfl_xor(a, m));
            } else {
                a = x[0];
                b = x[0];
#pragma unroll
                for (int j = 1; j < 8; ++j) { a = fmaxf(a, x[j]); b = fminf(b, x[j]); }
#pragma unroll
                for (int m = 1; m < LPG; m <<= 1) {
                    a = fmaxf(a, wq::shfl_xor(a, m));
                    b = fminf(b, wq::shfl_xor(b, m));
                }
            }
            ra[i] = a;
            rb[i] = b;
        }

        // each lane derives the parameters of the rows i with i % LPG == lane % LPG
        // (once per group instead of once per lane), then they are broadcast
        GroupParams own[RPL];
#pragma unroll
        for (int p = 0; p < RPL; ++p) {
            const int sel = LPG >= 8 ? ((lane % LPG) & 7) : (lane % LPG) + p * LPG;
            float a = ra[0], b = rb[0];
#pragma unroll
            for (int i = 1; i < 8; ++i)
                if (sel == i) { a = ra[i]; b = rb[i]; }
            own[p] = make_params<SYM>(a, b);
        }

        float sw = 0.0f, se = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int src = (lane & ~(LPG - 1)) | (i % LPG);
            const GroupParams& o = own[LPG >= 8 ? 0 : i / LPG];
            GroupParams P;
            P.s = __shfl_sync(0xffffffffu, o.s, src);
            P.r = __shfl_sync(0xffffffffu, o.r, src);
            P.zp = __shfl_sync(0xffffffffu, o.zp, src);
            const float lo = -P.zp, hi = 15.0f - P.zp;
            const uint32_t zpi = (uint32_t)P.zp;
            float x[8] = {wq::bf_lo(v[i].x), wq::bf_hi(v[i].x), wq::bf_lo(v[i].y), wq::bf_hi(v[i].y),
                          wq::bf_lo(v[i].z), wq::bf_hi(v[i].z), wq::bf_lo(v[i].w), wq::bf_hi(v[i].w)};
            const bool exact_path = P.s <= 0x1p100f;  // r stays normal
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float q = exact_path ? wq::div_by_recip(x[j], P.s, P.r) : __fdiv_rn(x[j], P.s);
                q = fminf(fmaxf(q, lo), hi);
                const float tq = __fadd_rn(q, kMagic);  // rint(q) + 1.5*2^23, exact
                const uint32_t code = (uint32_t)(__float_as_int(tq) - 0x4B400000) + zpi;
                word |= code << (4 * j);
                if (SNR) {
                    const float deq = __fmul_rn(__fsub_rn(tq, kMagic), P.s);  // (code - zp) * s
                    const float e = __fsub_rn(x[j], deq);
                    sw = __fadd_rn(sw, __fmul_rn(x[j], x[j]));
                    se = __fadd_rn(se, __fmul_rn(e, e));
                }
            }
            const int col = warp + 8 * i;
            s_qw[lane][col] = word;
            if ((lane % LPG) == 0) {
                s_sc[lane / LPG][col] = __half_as_ushort(__float2half_rn(P.s));
                s_zp[lane / LPG][col] = (uint8_t)zpi;
            }
        }
        if (SNR) {
            dw += (double)sw;
            de += (double)se;
        }
        __syncthreads();

        // qweight rows r = k0/8 + rl, columns n0 .. n0+63, 16 bytes per thread
        const int64_t rows_q = k / 8;
        for (int idx = threadIdx.x; idx < (kKT / 8) * (kNT / 4); idx += kThreads) {
            const int rl = idx / (kNT / 4), c4 = (idx % (kNT / 4)) * 4;
            const int64_t r = k0 / 8 + rl, c = n0 + c4;
            if (r < rows_q && c < n) {
                uint4 o = make_uint4(s_qw[rl][c4], s_qw[rl][c4 + 1], s_qw[rl][c4 + 2], s_qw[rl][c4 + 3]);
                *reinterpret_cast<uint4*>(qweight + r * n + c) = o;
            }
        }
        const int64_t gk = k / G;
        for (int idx = threadIdx.x; idx < GPT * kNT; idx += kThreads) {
            const int gl = idx / kNT, c = idx % kNT;
            const int64_t g = k0 / G + gl;
            if (g < gk && n0 + c < n) scales[g * n + n0 + c] = s_sc[gl][c];
        }
        if (qzeros) {
            for (int idx = threadIdx.x; idx < GPT * (kNT / 8); idx += kThreads) {
                const int gl = idx / (kNT / 8), c8 = idx % (kNT / 8);
                const int64_t g = k0 / G + gl;
                if (g < gk && n0 + 8 * c8 < n) {
                    uint32_t word = 0x77777777u;
                    if (!SYM) {
                        word = 0;
#pragma unroll
                        for (int j = 0; j < 8; ++j) word |= (uint32_t)s_zp[gl][8 * c8 + j] << (4 * j);
                    }
                    qzeros[g * (n / 8) + n0 / 8 + c8] = (int32_t)word;
                }
            }
        }
        if (g_idx && n0 == 0) {
            for (int idx = threadIdx.x; idx < kKT; idx += kThreads)
                if (k0 + idx < k) g_idx[k0 + idx] = (int32_t)((k0 + idx) / G);
        }
        __syncthreads();
    }

    if (SNR) {
        __shared__ double sa[kThreads / 32], sb[kThreads / 32];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            dw += __shfl_xor_sync(0xffffffffu, dw, m);
            de += __shfl_xor_sync(0xffffffffu, de, m);
        }
        if (lane == 0) { sa[warp] = dw; sb[warp] = de; }
        __syncthreads();
        if (threadIdx.x == 0) {
            double ta = 0.0, tb = 0.0;
            for (int i = 0; i < kThreads / 32; ++i) { ta += sa[i]; tb += sb[i]; }
            slots[2 * blockIdx.x] = ta;
            slots[2 * blockIdx.x + 1] = tb;
        }
    }
}

template <bool SYM, int G, bool SNR>
wq_status launch_quant(const uint16_t* w, int64_t n, int64_t k, int32_t* qweight, int32_t* qzeros,
                       uint16_t* scales, int32_t* g_idx, double* slots, int* grid_out,
                       cudaStream_t st) {
    const int64_t tiles = ((n + kNT - 1) / kNT) * ((k + kKT - 1) / kKT);
    const void* fn = (const void*)gptq_quant_kernel<SYM, G, SNR>;
    const int grid = wqh::grid_for(fn, kThreads, 0, tiles, wqh::kMaxPartials);
    gptq_quant_kernel<SYM, G, SNR><<<grid, kThreads, 0, st>>>(w, n, k, qweight, qzeros, scales, g_idx, slots);
    *grid_out = grid;
    return wqh::check_launch();
}

template <bool SYM>
wq_status quantize(const uint16_t* w, int64_t n, int64_t k, int group, int32_t* qweight,
                   int32_t* qzeros, uint16_t* scales, int32_t* g_idx, double* snr_db, void* ws,
                   size_t ws_bytes, void* stream) {
    if (n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (group != 32 && group != 64 && group != 128 && group != 256) return WQ_ERR_UNSUPPORTED;
    if (k % group != 0 || n % 8 != 0) return WQ_ERR_BAD_SHAPE;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !qweight || !scales) return WQ_ERR_NULL_PTR;
    if (snr_db && !ws) return WQ_ERR_NULL_PTR;
    if (snr_db && ws_bytes < wq_workspace_bytes(WQ_OP_GPTQ_QUANTIZE, n, k, group))
        return WQ_ERR_WORKSPACE_TOO_SMALL;
    if (!wqh::aligned16(w) || !wqh::aligned16(qweight) || !wqh::aligned_to(scales, 2) ||
        (qzeros && !wqh::aligned_to(qzeros, 4)) || (g_idx && !wqh::aligned_to(g_idx, 4)) ||
        (snr_db && !wqh::aligned_to(ws, 8)))
        return WQ_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    double* slots = (double*)ws;
    int grid = 0;
    wq_status s;
#define WQ_GPTQ_CASE(GG)                                                                          \
    case GG:                                                                                      \
        s = snr_db ? launch_quant<SYM, GG, true>(w, n, k, qweight, qzeros, scales, g_idx, slots,  \
                                                 &grid, st)                                       \
                   : launch_quant<SYM, GG, false>(w, n, k, qweight, qzeros, scales, g_idx, slots, \
                                                  &grid, st);                                     \
        break;
    switch (group) {
        WQ_GPTQ_CASE(32)
        WQ_GPTQ_CASE(64)
        WQ_GPTQ_CASE(128)
        WQ_GPTQ_CASE(256)
        default: return WQ_ERR_UNSUPPORTED;
    }
#undef WQ_GPTQ_CASE
    if (s != WQ_OK || !snr_db) return s;
    return wqh::launch_snr_finalize(slots, grid, snr_db, nullptr, st);
}

// ------------------------------------------------------------------ dequant
// (code - zp) * scale16, exact in binary32 (a 5-bit integer times an 11-bit
// significand).

__device__ __forceinline__ int zp_of(const int32_t* __restrict__ qzeros, int64_t g, int64_t n,
                                     int64_t col, bool sym) {
    if (sym) return 8;
    const uint32_t zw = (uint32_t)__ldg(qzeros + g * (n / 8) + col / 8);
    return (int)((zw >> (4 * (col % 8))) & 15u);
}

// [k, n] output: thread = (qweight row r, two adjacent columns); the 8 output
// rows 8r..8r+7 are written at those two columns (coalesced along n).
template <bool SYM, bool BF16>
__global__ void __launch_bounds__(kThreads) gptq_dequant_kn(const int32_t* __restrict__ qweight,
                                                            const int32_t* __restrict__ qzeros,
                                                            const uint16_t* __restrict__ scales,
                                                            int64_t n, int64_t k, int group,
                                                            void* __restrict__ out) {
    const int64_t pairs = n / 2, items = (k / 8) * pairs;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t it = (int64_t)blockIdx.x * kThreads + threadIdx.x; it < items; it += stride) {
        const int64_t r = it / pairs, c = (it % pairs) * 2;
        const uint2 wd = wq::ld_stream2(qweight + r * n + c);
        const int64_t g = (8 * r) / group;
        const uint32_t sc2 = __ldg(reinterpret_cast<const uint32_t*>(scales + g * n + c));
        const float s0 = __half2float(__ushort_as_half((unsigned short)(sc2 & 0xffffu)));
        const float s1 = __half2float(__ushort_as_half((unsigned short)(sc2 >> 16)));
        const int z0 = zp_of(qzeros, g, n, c, SYM), z1 = zp_of(qzeros, g, n, c + 1, SYM);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float v0 = __fmul_rn((float)((int)((wd.x >> (4 * i)) & 15u) - z0), s0);
            const float v1 = __fmul_rn((float)((int)((wd.y >> (4 * i)) & 15u) - z1), s1);
            const int64_t o = (8 * r + i) * n + c;
            if (BF16)
                *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(out) + o) = wq::f2_to_bf2(v0, v1);
            else
                *reinterpret_cast<float2*>(reinterpret_cast<float*>(out) + o) = make_float2(v0, v1);
        }
    }
}

// [n, k] output: 32 qweight rows x 64 columns per tile, transposed through
// shared memory; thread = (column, qweight row) writes 8 consecutive k values.
template <bool SYM, bool BF16>
__global__ void __launch_bounds__(kThreads) gptq_dequant_nk(const int32_t* __restrict__ qweight,
                                                            const int32_t* __restrict__ qzeros,
                                                            const uint16_t* __restrict__ scales,
                                                            int64_t n, int64_t k, int group,
                                                            void* __restrict__ out) {
    constexpr int RT = 32, CT = 64;
    __shared__ uint32_t s_w[RT][CT + 1];
    const int64_t rows_q = k / 8;
    const int64_t tiles_c = (n + CT - 1) / CT, tiles_r = (rows_q + RT - 1) / RT;
    for (int64_t t = blockIdx.x; t < tiles_c * tiles_r; t += gridDim.x) {
        const int64_t c0 = (t % tiles_c) * CT, r0 = (t / tiles_c) * RT;
        __syncthreads();
        for (int idx = threadIdx.x; idx < RT * CT; idx += kThreads) {
            const int rl = idx / CT, cl = idx % CT;
            const int64_t r = r0 + rl, c = c0 + cl;
            s_w[rl][cl] = (r < rows_q && c < n) ? (uint32_t)__ldg(qweight + r * n + c) : 0u;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < RT * CT; idx += kThreads) {
            const int cl = idx / RT, rl = idx % RT;
            const int64_t r = r0 + rl, c = c0 + cl;
            if (r >= rows_q || c >= n) continue;
            const int64_t g = (8 * r) / group;
            const float s = __half2float(__ushort_as_half(__ldg(scales + g * n + c)));
            const int z = zp_of(qzeros, g, n, c, SYM);
            const uint32_t wd = s_w[rl][cl];
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fmul_rn((float)((int)((wd >> (4 * i)) & 15u) - z), s);
            const int64_t o = c * k + 8 * r;
            if (BF16) {
                uint4 q = make_uint4(wq::f2_to_bf2(v[0], v[1]), wq::f2_to_bf2(v[2], v[3]),
                                     wq::f2_to_bf2(v[4], v[5]), wq::f2_to_bf2(v[6], v[7]));
                *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(out) + o) = q;
            } else {
                float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o);
                p[0] = make_float4(v[0], v[1], v[2], v[3]);
                p[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
    }
}

template <bool SYM, bool BF16>
wq_status launch_dequant(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                         int64_t n, int64_t k, int group, int layout, void* out, cudaStream_t st) {
    if (layout == WQ_LAYOUT_KN) {
        const void* fn = (const void*)gptq_dequant_kn<SYM, BF16>;
        const int64_t items = (k / 8) * (n / 2);
        const int grid = wqh::grid_for(fn, kThreads, 0, (items + kThreads - 1) / kThreads, 1 << 30);
        gptq_dequant_kn<SYM, BF16><<<grid, kThreads, 0, st>>>(qweight, qzeros, scales, n, k, group, out);
    } else {
        const void* fn = (const void*)gptq_dequant_nk<SYM, BF16>;
        const int64_t tiles = ((n + 63) / 64) * ((k / 8 + 31) / 32);
        const int grid = wqh::grid_for(fn, kThreads, 0, tiles, 1 << 30);
        gptq_dequant_nk<SYM, BF16><<<grid, kThreads, 0, st>>>(qweight, qzeros, scales, n, k, group, out);
    }
    return wqh::check_launch();
}

}  // namespace

extern "C" wq_status gptq_quantize_sym(const uint16_t* w, int64_t n, int64_t k, int group,
                                       int32_t* qweight, int32_t* qzeros, uint16_t* scales,
                                       int32_t* g_idx, double* snr_db, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    return quantize<true>(w, n, k, group, qweight, qzeros, scales, g_idx, snr_db, workspace,
                          workspace_bytes, stream);
}

extern "C" wq_status gptq_quantize_asym(const uint16_t* w, int64_t n, int64_t k, int group,
                                        int32_t* qweight, int32_t* qzeros, uint16_t* scales,
                                        int32_t* g_idx, double* snr_db, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    return quantize<false>(w, n, k, group, qweight, qzeros, scales, g_idx, snr_db, workspace,
                           workspace_bytes, stream);
}

extern "C" wq_status gptq_dequantize(const int32_t* qweight, const int32_t* qzeros,
                                     const uint16_t* scales, int64_t n, int64_t k, int group,
                                     int sym, int out_dtype, int out_layout, void* out,
                                     void* stream) {
    if (n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (group <= 0 || group % 8 != 0) return WQ_ERR_UNSUPPORTED;
    if (k % group != 0 || n % 8 != 0) return WQ_ERR_BAD_SHAPE;
    if (out_dtype != WQ_DTYPE_F32 && out_dtype != WQ_DTYPE_BF16) return WQ_ERR_BAD_DTYPE;
    if (out_layout != WQ_LAYOUT_NK && out_layout != WQ_LAYOUT_KN) return WQ_ERR_UNSUPPORTED;
    if (n == 0 || k == 0) return WQ_OK;
    if (!qweight || !scales || !out || (!sym && !qzeros)) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(qweight) || !wqh::aligned16(out) || !wqh::aligned_to(scales, 4) ||
        (!sym && !wqh::aligned_to(qzeros, 4)))
        return WQ_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    const bool bf = out_dtype == WQ_DTYPE_BF16;
    if (sym)
        return bf ? launch_dequant<true, true>(qweight, qzeros, scales, n, k, group, out_layout, out, st)
                  : launch_dequant<true, false>(qweight, qzeros, scales, n, k, group, out_layout, out, st);
    return bf ? launch_dequant<false, true>(qweight, qzeros, scales, n, k, group, out_layout, out, st)
              : launch_dequant<false, false>(qweight, qzeros, scales, n, k, group, out_layout, out, st);
}
