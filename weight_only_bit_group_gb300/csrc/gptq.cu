// gptq.cu -- GPTQ int4 quantize (sym / asym) and dequantize
// (export_gptq_cpu.py: pack_int32, quantize_sym, quantize_asym; module docstring
// for the uint4b8 dequant rule).
//
// Quantize: a warp owns a tile of 32 output channels (rows of w) x KT input
// channels (KT = 128, or the group when it is larger) and lane l owns row
// n0 + l.  The tile arrives in shared memory through a two-stage per-warp
// cp.async pipeline (each copy instruction moves two whole 256-byte row
// segments, fully coalesced; rows are padded to 272 bytes so the per-lane
// reads are bank-conflict free) while the previous tile is computed.  A lane
// holds whole groups of its row, so the group max/min is an in-thread bf16x2
// reduction and the scale / zero point are computed once per group with true
// IEEE divisions.  Per element: the quotient by the scale from a correctly
// rounded reciprocal plus one FMA correction (bit-identical to IEEE division),
// the clamp to [-zp, 15-zp] (exact before rounding, the bounds are integers),
// round-half-even by the binary32 adder (x + 1.5*2^23), and the nibble pack as
// one IMAD per element.  The eight codes along k of one row are one qweight
// word, so the 32 lanes store 32 consecutive qweight columns (128 bytes) per
// word row -- the [K/8, N] transpose costs nothing.  Packed-pair (f32x2) math
// halves the issue slots of the arithmetic.  The optional reconstruction SNR
// is accumulated from the same registers and reduced by the last CTA.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;  // dequant kernels
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

template <int G>
struct QTile {
    static constexpr int KT = G < 128 ? 128 : G;     // input channels per warp tile
    static constexpr int CH = KT / 8;                 // 16-byte chunks per row
    static constexpr int ROWB = KT * 2 + 16;          // padded shared-memory row
    static constexpr int STAGE = 32 * ROWB;           // one stage of one warp
    static constexpr int NS = 2;                      // pipeline stages
    static constexpr int WARPS = KT > 128 ? 2 : 4;    // warps per CTA
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int SMEM = NS * WARPS * STAGE;
};

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

template <bool SYM, int G, bool SNR>
__global__ void __launch_bounds__(QTile<G>::THREADS, 3) gptq_quant_kernel(
    const uint16_t* __restrict__ w, int64_t n, int64_t k, int32_t* __restrict__ qweight,
    int32_t* __restrict__ qzeros, uint16_t* __restrict__ scales, int32_t* __restrict__ g_idx,
    double* __restrict__ slots, unsigned* __restrict__ counter, double* __restrict__ snr_db) {
    using T = QTile<G>;
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned char* wsm = smem + warp * (T::NS * T::STAGE);
    const int64_t tn = (n + 31) / 32, tk = (k + T::KT - 1) / T::KT, ntiles = tn * tk;
    const int64_t gwarp = (int64_t)blockIdx.x * T::WARPS + warp;
    const int64_t nwarps = (int64_t)gridDim.x * T::WARPS;

    auto issue = [&](int64_t t, int stage) {
        if (t < ntiles) {
            const int64_t n0 = (t % tn) * 32, k0 = (t / tn) * T::KT;
            unsigned char* dst = wsm + stage * T::STAGE;
#pragma unroll
            for (int i = 0; i < T::CH; ++i) {
                const int idx = i * 32 + lane, row = idx / T::CH, ch = idx % T::CH;
                const int64_t gr = n0 + row, gk = k0 + 8 * ch;
                if (gr < n && gk < k) wq::cp_async16(dst + row * T::ROWB + 16 * ch, w + gr * k + gk);
            }
        }
        wq::cp_async_commit();
    };

    double dw = 0.0, de = 0.0;
    int64_t t = gwarp;
    issue(t, 0);
    for (int j = 0; t < ntiles; ++j, t += nwarps) {
        issue(t + nwarps, (j + 1) & 1);
        wq::cp_async_wait<1>();
        __syncwarp();
        const int64_t n0 = (t % tn) * 32, k0 = (t / tn) * T::KT;
        const int64_t col = n0 + lane;
        const bool rowv = col < n;
        const unsigned char* rsm = wsm + (j & 1) * T::STAGE + lane * T::ROWB;
#pragma unroll
        for (int g = 0; g < T::KT / G; ++g) {
            if (k0 + g * G >= k) break;  // k % G == 0: warp-uniform
            uint4 v[G / 8];
#pragma unroll
            for (int c = 0; c < G / 8; ++c) v[c] = *reinterpret_cast<const uint4*>(rsm + 16 * (g * (G / 8) + c));
            float s, zp;
            if (SYM) {
                const uint32_t M = 0x7fff7fffu;
                uint32_t m = __vmaxu2(v[0].x & M, v[0].y & M);
#pragma unroll
                for (int c = 0; c < G / 8; ++c)
                    m = __vmaxu2(m, __vmaxu2(__vmaxu2(v[c].x & M, v[c].y & M), __vmaxu2(v[c].z & M, v[c].w & M)));
                const float amax = wq::bf_to_f(max(m & 0xffffu, m >> 16));
                s = fmaxf(__fdiv_rn(amax, 8.0f), 1e-9f);
                zp = 8.0f;
            } else {
                uint32_t mx = v[0].x, mn = v[0].x;
#pragma unroll
                for (int c = 0; c < G / 8; ++c) {
                    mx = bmax2(mx, bmax2(bmax2(v[c].x, v[c].y), bmax2(v[c].z, v[c].w)));
                    mn = bmin2(mn, bmin2(bmin2(v[c].x, v[c].y), bmin2(v[c].z, v[c].w)));
                }
                const float wmax = fmaxf(wq::bf_lo(mx), wq::bf_hi(mx));
                const float wmin = fminf(wq::bf_lo(mn), wq::bf_hi(mn));
                s = __fdiv_rn(fmaxf(__fsub_rn(wmax, wmin), 1e-9f), 15.0f);
                zp = fminf(fmaxf(rintf(__fdiv_rn(-wmin, s)), 0.0f), 15.0f);
            }
            const float r = __frcp_rn(s);
            const float lo = -zp, hi = 15.0f - zp;
            const uint32_t cg = (uint32_t)((int)zp - 0x4B400000) * 0x11111111u;
            const wq::f2_t R2 = wq::f2(r, r), NS2 = wq::f2(-s, -s), M2 = wq::f2(kMagic, kMagic);
            const wq::f2_t NM2 = wq::f2(-kMagic, -kMagic);
            const bool exact = s <= 0x1p100f;  // r stays normal: the correction step is exact
            wq::f2_t sw2 = wq::f2(0.0f, 0.0f), se2 = sw2;
            const int64_t r0 = (k0 + g * G) / 8;
#pragma unroll
            for (int c = 0; c < G / 8; ++c) {
                const uint32_t u[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
                uint32_t word = cg;
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const wq::f2_t x = wq::bf2_to_f2(u[p]);
                    float q0, q1;
                    if (exact) {
                        const wq::f2_t qa = wq::mul2(x, R2);
                        const wq::f2_t rem = wq::fma2(qa, NS2, x);
                        wq::f2u(wq::fma2(rem, R2, qa), q0, q1);
                    } else {
                        float x0, x1;
                        wq::f2u(x, x0, x1);
                        q0 = __fdiv_rn(x0, s);
                        q1 = __fdiv_rn(x1, s);
                    }
                    q0 = fminf(fmaxf(q0, lo), hi);
                    q1 = fminf(fmaxf(q1, lo), hi);
                    const wq::f2_t tq = wq::add2(wq::f2(q0, q1), M2);  // rint(q) + 1.5*2^23
                    float t0, t1;
                    wq::f2u(tq, t0, t1);
                    word += (uint32_t)__float_as_int(t0) << (8 * p);
                    word += (uint32_t)__float_as_int(t1) << (8 * p + 4);
                    if (SNR) {
                        const wq::f2_t e = wq::fma2(wq::add2(tq, NM2), NS2, x);  // x - (code-zp)*s
                        se2 = wq::fma2(e, e, se2);
                        sw2 = wq::fma2(x, x, sw2);
                    }
                }
                if (rowv) qweight[(r0 + c) * n + col] = (int32_t)word;
            }
            if (SNR) {
                float a0, a1, b0, b1;
                wq::f2u(sw2, a0, a1);
                wq::f2u(se2, b0, b1);
                if (rowv) {
                    dw += (double)a0 + (double)a1;
                    de += (double)b0 + (double)b1;
                }
            }
            const int64_t gi = (k0 + g * G) / G;
            if (rowv) scales[gi * n + col] = __half_as_ushort(__float2half_rn(s));
            if (qzeros) {
                uint32_t zw = SYM ? 0x77777777u : ((uint32_t)zp << (4 * (lane & 7)));
                if (!SYM) {
                    zw |= __shfl_xor_sync(0xffffffffu, zw, 1);
                    zw |= __shfl_xor_sync(0xffffffffu, zw, 2);
                    zw |= __shfl_xor_sync(0xffffffffu, zw, 4);
                }
                if (rowv && (lane & 7) == 0) qzeros[gi * (n / 8) + col / 8] = (int32_t)zw;
            }
        }
        if (g_idx && n0 == 0) {
#pragma unroll
            for (int i = lane; i < T::KT; i += 32)
                if (k0 + i < k) g_idx[k0 + i] = (int32_t)((k0 + i) / G);
        }
        __syncwarp();
    }
    wq::cp_async_wait<0>();
    if (SNR) wq::finish_snr(dw, de, slots, counter, snr_db, nullptr);
}

template <bool SYM, int G, bool SNR>
wq_status launch_quant(const uint16_t* w, int64_t n, int64_t k, int32_t* qweight, int32_t* qzeros,
                       uint16_t* scales, int32_t* g_idx, double* slots, unsigned* counter,
                       double* snr_db, cudaStream_t st) {
    using T = QTile<G>;
    const void* fn = (const void*)gptq_quant_kernel<SYM, G, SNR>;
    static bool attr_set = false;  // per-process; the attribute is per function
    if (!attr_set) {
        wq_status s = wqh::cuda_status(
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM));
        if (s != WQ_OK) return s;
        attr_set = true;
    }
    const int64_t warp_tiles = ((n + 31) / 32) * ((k + T::KT - 1) / T::KT);
    const int grid = wqh::grid_for(fn, T::THREADS, T::SMEM, (warp_tiles + T::WARPS - 1) / T::WARPS,
                                   wqh::kMaxPartials);
    gptq_quant_kernel<SYM, G, SNR><<<grid, T::THREADS, T::SMEM, st>>>(
        w, n, k, qweight, qzeros, scales, g_idx, slots, counter, snr_db);
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
        (snr_db && !wqh::aligned_to(ws, 256)))
        return WQ_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    unsigned* counter = snr_db ? (unsigned*)ws : nullptr;
    double* slots = snr_db ? (double*)((char*)ws + wqh::kCtrlBytes) : nullptr;
    if (snr_db) {
        wq_status s0 = wqh::cuda_status(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
        if (s0 != WQ_OK) return s0;
    }
#define WQ_GPTQ_CASE(GG)                                                                          \
    case GG:                                                                                      \
        return snr_db ? launch_quant<SYM, GG, true>(w, n, k, qweight, qzeros, scales, g_idx,      \
                                                    slots, counter, snr_db, st)                   \
                      : launch_quant<SYM, GG, false>(w, n, k, qweight, qzeros, scales, g_idx,     \
                                                     slots, counter, snr_db, st);
    switch (group) {
        WQ_GPTQ_CASE(32)
        WQ_GPTQ_CASE(64)
        WQ_GPTQ_CASE(128)
        WQ_GPTQ_CASE(256)
        default: return WQ_ERR_UNSUPPORTED;
    }
#undef WQ_GPTQ_CASE
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
