// uintx.cu -- affine uintx quantization with power-of-two bit-shard packing and
// its inverse (uintx_quant.py: module docstring, _pack_shard, pack_uintx,
// unpack_uintx, UIntXQuantizer._quantize_impl, _dequantize_native).
//
// Shard geometry.  numel = n*k is a multiple of 8 (group % 8 == 0 divides k), so
// with L1 = numel/8 the 1-bit shard has L1 bytes, the 2-bit shard 2*L1 and the
// 4-bit shard 4*L1.  Byte i of the 1-bit shard takes element i + j*L1 (j < 8) as
// bit j; byte h*L1 + d of the 2-bit shard takes elements (2jj + h)*L1 + d (jj < 4)
// at bits 2jj; byte m*L1 + d of the 4-bit shard takes elements m*L1 + d and
// (m+4)*L1 + d.  Hence one thread that holds, for 8 consecutive positions d, the
// codes of all 8 "segments" m*L1 + d (m < 8) completes every shard byte of those
// positions in registers: one read of w, no atomics, 8-byte coalesced stores.
//
// Fused path (group 64, numel % 512 == 0, so segment starts are group-aligned):
// a warp takes 256 consecutive positions d; lane l holds d = d0 + 8l .. 8l+7 of
// all 8 segments (8 coalesced 16-byte loads).  The 8 lanes of an octet together
// hold 8 whole groups (one per segment): a 3-round reduce-scatter leaves lane c
// with the min/max of segment c's group, lane c derives that group's bf16
// qparams (once per group) and an 8-shuffle all-gather hands every lane the
// (1/scale, zp) of all 8 groups.
//
// bf16 arithmetic: every page step is the binary32 operation on bf16 operands
// rounded once to bf16 (cvt.rn).  w * (1/scale) is an exact binary32 product of
// two bf16 values, so rounding it with cvt.rn.bf16 reproduces the bf16 multiply.
//
// uintx_quantize_err runs the same kernels with ERR = 1: from the code bytes in
// registers each lane rebuilds the page's bf16 dequantized value
// (_dequantize_native: bf16(bf16(q - zp) * scale)) and accumulates the binary32
// terms w^2 and (w - deq)^2; the grid finishes both sums with the last-CTA
// float-float reduction, so the reconstruction error costs no second pass.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t kB192x2 = 0x43404340u;  // bf16 192 = 1.5 * 2^7, both halves

struct QParams {
    uint32_t scale_bits;  // bf16 bits of the scale
    uint32_t inv_bits;    // bf16 bits of 1/scale
    uint32_t zp;
};

// choose_qparams_affine as the page states it, in bf16 (preserve_zero, eps =
// binary32 eps, integer zero point).
template <int QMAX>
__device__ __forceinline__ QParams qparams(float mn, float mx) {
    const float mnn = fminf(mn, 0.0f), mxp = fmaxf(mx, 0.0f);
    float sc = wq::bfr(__fsub_rn(mxp, mnn));
    sc = wq::bfr(__fdiv_rn(sc, (float)QMAX));
    sc = fmaxf(sc, 0x1p-23f);
    const float ratio = wq::bfr(__fdiv_rn(mnn, sc));
    float zpf = wq::bfr(__fsub_rn(0.0f, rintf(ratio)));
    zpf = fminf(fmaxf(zpf, 0.0f), (float)QMAX);
    QParams p;
    p.scale_bits = wq::f_to_bf(sc);
    p.inv_bits = wq::f_to_bf(__fdiv_rn(1.0f, sc));
    p.zp = (uint32_t)zpf;
    return p;
}

template <int NBITS>
struct Shards {
    static constexpr bool has4 = (NBITS & 4) != 0;
    static constexpr bool has2 = (NBITS & 2) != 0;
    static constexpr bool has1 = (NBITS & 1) != 0;
    static constexpr int off2 = has4 ? 4 : 0;
    static constexpr int off1 = (has4 ? 4 : 0) + (has2 ? 2 : 0);
};

// Build and store every shard byte of 8 positions d .. d+7 from the code bytes
// B[m] (8 bytes: codes of elements m*L1 + d .. d+7).
template <int NBITS>
__device__ __forceinline__ void store_shards(const uint32_t (&blo)[8], const uint32_t (&bhi)[8],
                                             uint8_t* __restrict__ packed, int64_t numel,
                                             int64_t L1, int64_t d) {
    using S = Shards<NBITS>;
    const int64_t base2 = S::has4 ? numel / 2 : 0;
    const int64_t base1 = base2 + (S::has2 ? numel / 4 : 0);
    if (S::has4) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint2 o;
            o.x = (blo[m] & 0x0F0F0F0Fu) | ((blo[m + 4] & 0x0F0F0F0Fu) << 4);
            o.y = (bhi[m] & 0x0F0F0F0Fu) | ((bhi[m + 4] & 0x0F0F0F0Fu) << 4);
            *reinterpret_cast<uint2*>(packed + m * L1 + d) = o;
        }
    }
    if (S::has2) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint2 o = make_uint2(0, 0);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                o.x |= ((blo[2 * jj + h] >> S::off2) & 0x03030303u) << (2 * jj);
                o.y |= ((bhi[2 * jj + h] >> S::off2) & 0x03030303u) << (2 * jj);
            }
            *reinterpret_cast<uint2*>(packed + base2 + h * L1 + d) = o;
        }
    }
    if (S::has1) {
        uint2 o = make_uint2(0, 0);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            o.x |= ((blo[m] >> S::off1) & 0x01010101u) << m;
            o.y |= ((bhi[m] >> S::off1) & 0x01010101u) << m;
        }
        *reinterpret_cast<uint2*>(packed + base1 + d) = o;
    }
}

// Error terms of one packed pair: x the two bf16 weights, r the two bf16 values
// q - zp (exact integers), s2 the group's bf16 scale in both halves.  deq =
// bf16(r * s) is the page's bf16 multiply (mul.rn.bf16x2); the binary32 values
// of w and the difference w - deq come from mixed-precision FMAs that read the
// bf16 halves in place (w * 1 and deq * -1 + w, each exact or rounded once as
// the binary32 subtraction is), so the integer pipe, which the code
// computation keeps busy, does no unpacking.
__device__ __forceinline__ void err_pair(uint32_t x, uint32_t r, uint32_t s2, wq::f2_t& sw,
                                         wq::f2_t& se) {
    const uint32_t dq = wq::bmul2(r, s2);  // the page's bf16 deq
    float x0, x1, d0, d1;
    asm("{\n\t.reg .b16 xl, xh, ql, qh, one, m1;\n\t"
        "mov.b32 {xl, xh}, %4;\n\tmov.b32 {ql, qh}, %5;\n\t"
        "mov.b16 one, 0x3F80;\n\tmov.b16 m1, 0xBF80;\n\t"
        "fma.rn.f32.bf16 %0, xl, one, %6;\n\tfma.rn.f32.bf16 %1, xh, one, %6;\n\t"
        "fma.rn.f32.bf16 %2, ql, m1, %0;\n\tfma.rn.f32.bf16 %3, qh, m1, %1;\n\t}"
        : "=f"(x0), "=f"(x1), "=f"(d0), "=f"(d1)
        : "r"(x), "r"(dq), "f"(-0.0f));
    const wq::f2_t xf = wq::f2(x0, x1), d = wq::f2(d0, d1);  // w and RN(w - deq)
    se = wq::fma2(d, d, se);
    sw = wq::fma2(xf, xf, sw);
}

template <int NBITS, int ERR>
__global__ void __launch_bounds__(kThreads, 2) uintx_quant_fused(const uint16_t* __restrict__ w,
                                                                 int64_t numel, uint8_t* __restrict__ packed,
                                                                 uint16_t* __restrict__ scale,
                                                                 uint8_t* __restrict__ zp,
                                                                 float4* __restrict__ slots,
                                                                 unsigned* __restrict__ counter,
                                                                 double* __restrict__ snr_db,
                                                                 double* __restrict__ rel_err) {
    constexpr int QMAX = (1 << NBITS) - 1;
    // two pipeline stages x 8 segments x 16 bytes, private to each thread
    extern __shared__ __align__(16) uint4 dyn_smem[];
    uint4 (*stage_buf)[8][kThreads] = reinterpret_cast<uint4 (*)[8][kThreads]>(dyn_smem);
    const int64_t L1 = numel / 8;  // multiple of 64
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    const int64_t items = (L1 + 255) / 256;
    wq::KSum dw, de;

    auto issue = [&](int64_t it, int st) {
        const int64_t d = it * 256 + 8 * lane;
        if (it < items && d < L1) {
#pragma unroll
            for (int m = 0; m < 8; ++m) wq::cp_async16(&stage_buf[st][m][threadIdx.x], w + m * L1 + d);
        }
        wq::cp_async_commit();
    };

    issue(warp, 0);
    int j = 0;
    for (int64_t it = warp; it < items; it += nwarps, ++j) {
        issue(it + nwarps, (j + 1) & 1);
        wq::cp_async_wait<1>();
        const int64_t d0 = it * 256, d = d0 + 8 * lane;
        const bool valid = d < L1;  // uniform over an octet (64 positions)
        uint4 v[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) v[m] = valid ? stage_buf[j & 1][m][threadIdx.x] : make_uint4(0, 0, 0, 0);

        // group min and max as one bf16x2 word (min, -max): every combining step
        // is a single min.bf16x2
        uint32_t st[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            uint32_t lo = wq::bmin2(wq::bmin2(v[m].x, v[m].y), wq::bmin2(v[m].z, v[m].w));
            uint32_t hi = wq::bmax2(wq::bmax2(v[m].x, v[m].y), wq::bmax2(v[m].z, v[m].w));
            lo = wq::bmin2(lo, wq::bswap2(lo));
            hi = wq::bmax2(hi, wq::bswap2(hi));
            st[m] = __byte_perm(lo, hi ^ 0x80008000u, 0x7610);  // (min, -max)
        }
        // reduce-scatter over the octet: lane c ends with segment c's group
#pragma unroll
        for (int h = 4, msk = 4; h >= 1; h >>= 1, msk >>= 1) {
            const bool hb = (lane & msk) != 0;  // keeps the upper half of its values
#pragma unroll
            for (int j = 0; j < h; ++j) {
                const uint32_t keep = hb ? st[j + h] : st[j];
                const uint32_t send = hb ? st[j] : st[j + h];
                st[j] = wq::bmin2(keep, wq::shfl_xor(send, msk));
            }
        }
        const float gmn = wq::bf_lo(st[0]), gmx = -wq::bf_hi(st[0]);
        const int c = lane & 7;
        const QParams qp = qparams<QMAX>(gmn, gmx);
        if (valid) {
            const int64_t g = (c * L1 + d0) / 64 + (lane >> 3);
            scale[g] = (uint16_t)qp.scale_bits;
            zp[g] = (uint8_t)qp.zp;
        }
        const uint32_t mine = qp.inv_bits | (qp.zp << 16);

        uint32_t blo[8], bhi[8];
        wq::f2_t sw = wq::f2(0.f, 0.f), se = wq::f2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const uint32_t P = __shfl_sync(0xffffffffu, mine, (lane & ~7) | m);
            // the group's scale (bf16) in both halves, for the error terms only
            const uint32_t s2 = ERR ? __shfl_sync(0xffffffffu, qp.scale_bits, (lane & ~7) | m) * 0x10001u : 0u;
            const uint32_t z = P >> 16;
            // bf16(w * inv) clamped to [-zp, qmax - zp] (bf16x2, exact bounds)
            const uint32_t inv2 = (P & 0xffffu) * 0x10001u;
            const uint32_t lo2 = wq::f2_to_bf2(-(float)z, -(float)z);
            const uint32_t hi2 = wq::f2_to_bf2((float)(QMAX - (int)z), (float)(QMAX - (int)z));
            const uint32_t u[4] = {v[m].x, v[m].y, v[m].z, v[m].w};
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = wq::bmin2(wq::bmax2(wq::bmul2(u[i], inv2), lo2), hi2);
            if (QMAX <= 63) {
                // + 192 in bf16: the sum lies in [129, 255], where bf16 has unit
                // spacing, so the addition rounds half to even and the low byte of
                // each half is 64 + round(.)
                const uint32_t zadd = (uint32_t)((int)z - 64) * 0x01010101u;
#pragma unroll
                for (int i = 0; i < 4; ++i) q[i] = wq::badd2(q[i], kB192x2);
                blo[m] = __byte_perm(q[0], q[1], 0x6420) + zadd;
                bhi[m] = __byte_perm(q[2], q[3], 0x6420) + zadd;
                if (ERR) {
                    // (192 + round(.)) - 192 = the exact integer q - zp, in bf16
#pragma unroll
                    for (int i = 0; i < 4; ++i) err_pair(u[i], wq::bsub2(q[i], kB192x2), s2, sw, se);
                }
            } else {
                // + (1.5 * 2^23 + 128) in binary32: the adder rounds half to even (the
                // offset is even) and the low byte of the sum is 128 + round(.)
                const uint32_t zadd = (uint32_t)((int)z - 128) * 0x01010101u;
                const wq::f2_t M2 = wq::f2(kMagic + 128.0f, kMagic + 128.0f);
                uint32_t b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const wq::f2_t t = wq::add2(wq::bf2_to_f2(q[i]), M2);
                    b[i] = __byte_perm(__float_as_uint(t.x), __float_as_uint(t.y), 0x0040);
                    if (ERR) {
                        // t - (1.5 * 2^23 + 128) = the exact integer q - zp
                        const wq::f2_t r = wq::add2(t, wq::f2(-(kMagic + 128.0f), -(kMagic + 128.0f)));
                        err_pair(u[i], wq::f2_to_bf2(r.x, r.y), s2, sw, se);
                    }
                }
                blo[m] = __byte_perm(b[0], b[1], 0x5410) + zadd;
                bhi[m] = __byte_perm(b[2], b[3], 0x5410) + zadd;
            }
        }
        if (valid) store_shards<NBITS>(blo, bhi, packed, numel, L1, d);
        if (ERR) {  // lanes past the end hold zeros: zero terms
            dw.add(__fadd_rn(sw.x, sw.y));
            de.add(__fadd_rn(se.x, se.y));
        }
    }
    wq::cp_async_wait<0>();
    if (ERR) wq::finish_snr(wq::ff_of(dw), wq::ff_of(de), slots, counter, snr_db, rel_err);
}

// ----------------------------------------------------------- general path
// (any group % 8 == 0 dividing k; numel % 8 == 0)

template <int QMAX>
__global__ void __launch_bounds__(kThreads) uintx_qparams_kernel(const uint16_t* __restrict__ w,
                                                                 int64_t ngroups, int group,
                                                                 uint16_t* __restrict__ scale,
                                                                 uint8_t* __restrict__ zp) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < ngroups; g += stride) {
        const uint4* p = reinterpret_cast<const uint4*>(w + g * group);
        float a = INFINITY, b = -INFINITY;
        for (int i = 0; i < group / 8; ++i) {
            const uint4 u = __ldg(p + i);
            const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                a = fminf(a, fminf(wq::bf_lo(q[j]), wq::bf_hi(q[j])));
                b = fmaxf(b, fmaxf(wq::bf_lo(q[j]), wq::bf_hi(q[j])));
            }
        }
        const QParams qp = qparams<QMAX>(a, b);
        scale[g] = (uint16_t)qp.scale_bits;
        zp[g] = (uint8_t)qp.zp;
    }
}

template <int NBITS, int ERR>
__global__ void __launch_bounds__(kThreads) uintx_pack_general(const uint16_t* __restrict__ w,
                                                               int64_t numel, int group,
                                                               const uint16_t* __restrict__ scale,
                                                               const uint8_t* __restrict__ zp,
                                                               uint8_t* __restrict__ packed,
                                                               float4* __restrict__ slots,
                                                               unsigned* __restrict__ counter,
                                                               double* __restrict__ snr_db,
                                                               double* __restrict__ rel_err) {
    using S = Shards<NBITS>;
    constexpr int QMAX = (1 << NBITS) - 1;
    const int64_t L1 = numel / 8;
    const int64_t base2 = S::has4 ? numel / 2 : 0;
    const int64_t base1 = base2 + (S::has2 ? numel / 4 : 0);
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    wq::KSum dw, de;
    for (int64_t d = (int64_t)blockIdx.x * kThreads + threadIdx.x; d < L1; d += stride) {
        uint32_t c[8];
        float sw = 0.f, se = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int64_t e = m * L1 + d, g = e / group;
            const float sc = wq::bf_to_f(__ldg(scale + g));
            const uint32_t z = __ldg(zp + g);
            const float inv = wq::bfr(__fdiv_rn(1.0f, sc));
            const float x = wq::bf_to_f(__ldg(w + e));
            const float p = wq::bfr(__fmul_rn(x, inv));
            const float pc = fminf(fmaxf(p, -(float)z), (float)(QMAX - (int)z));
            const int r = __float_as_int(__fadd_rn(pc, kMagic)) - 0x4B400000;  // q - zp
            c[m] = (uint32_t)r + z;
            if (ERR) {
                // _dequantize_native: bf16(q - zp) is exact, times the bf16 scale, one rounding
                const float dq = wq::bfr(__fmul_rn((float)r, sc));
                const float df = __fsub_rn(x, dq);
                se = __fmaf_rn(df, df, se);
                sw = __fmaf_rn(x, x, sw);
            }
        }
        if (ERR) {
            dw.add(sw);
            de.add(se);
        }
        if (S::has4) {
#pragma unroll
            for (int m = 0; m < 4; ++m) packed[m * L1 + d] = (uint8_t)((c[m] & 15u) | ((c[m + 4] & 15u) << 4));
        }
        if (S::has2) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t b = 0;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) b |= ((c[2 * jj + h] >> S::off2) & 3u) << (2 * jj);
                packed[base2 + h * L1 + d] = (uint8_t)b;
            }
        }
        if (S::has1) {
            uint32_t b = 0;
#pragma unroll
            for (int m = 0; m < 8; ++m) b |= ((c[m] >> S::off1) & 1u) << m;
            packed[base1 + d] = (uint8_t)b;
        }
    }
    if (ERR) wq::finish_snr(wq::ff_of(dw), wq::ff_of(de), slots, counter, snr_db, rel_err);
}

// ----------------------------------------------------------- dequant
// Codes of positions d .. d+7 of all 8 segments from the shard bytes, then
// out = bf16(bf16(q - zp) * scale): q - zp is an exact small integer and the
// product of two bf16 values is exact in binary32, so one rounding to bf16 (of
// the binary32 product, or of mul.rn.bf16x2) gives the page's bf16 result.
template <int NBITS>
__device__ __forceinline__ void load_codes(const uint8_t* __restrict__ packed, int64_t numel,
                                           int64_t L1, int64_t d, uint32_t (&blo)[8],
                                           uint32_t (&bhi)[8]) {
    using S = Shards<NBITS>;
    const int64_t base2 = S::has4 ? numel / 2 : 0;
    const int64_t base1 = base2 + (S::has2 ? numel / 4 : 0);
#pragma unroll
    for (int m = 0; m < 8; ++m) { blo[m] = 0; bhi[m] = 0; }
    if (S::has4) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const uint2 s = wq::ld_stream2(packed + m * L1 + d);
            blo[m] |= s.x & 0x0F0F0F0Fu;
            bhi[m] |= s.y & 0x0F0F0F0Fu;
            blo[m + 4] |= (s.x >> 4) & 0x0F0F0F0Fu;
            bhi[m + 4] |= (s.y >> 4) & 0x0F0F0F0Fu;
        }
    }
    if (S::has2) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint2 s = wq::ld_stream2(packed + base2 + h * L1 + d);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                blo[2 * jj + h] |= ((s.x >> (2 * jj)) & 0x03030303u) << S::off2;
                bhi[2 * jj + h] |= ((s.y >> (2 * jj)) & 0x03030303u) << S::off2;
            }
        }
    }
    if (S::has1) {
        const uint2 s = wq::ld_stream2(packed + base1 + d);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            blo[m] |= ((s.x >> m) & 0x01010101u) << S::off1;
            bhi[m] |= ((s.y >> m) & 0x01010101u) << S::off1;
        }
    }
}

__device__ __forceinline__ float deq1(uint32_t q, float zf, float sc) {
    return __fmul_rn(__fsub_rn((float)q, zf), sc);
}

// numel % 64 == 0 and a power-of-two group: 8 positions per thread, 16-byte
// output stores.
template <int NBITS, bool BF16>
__global__ void __launch_bounds__(kThreads) uintx_dequant_vec(const uint8_t* __restrict__ packed,
                                                              const uint16_t* __restrict__ scale,
                                                              const uint8_t* __restrict__ zp,
                                                              int64_t numel, int lg_group,
                                                              void* __restrict__ out) {
    const int64_t L1 = numel / 8, items = L1 / 8;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < items; t += stride) {
        const int64_t d = 8 * t;
        uint32_t blo[8], bhi[8];
        load_codes<NBITS>(packed, numel, L1, d, blo, bhi);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int64_t e = m * L1 + d, g = e >> lg_group;  // 8 | group: one group
            // bf16x2 arithmetic: the code byte under 0x43 is the bf16 128 + q, so
            // (128 + q) - (128 + zp) is the exact bf16 q - zp and mul.rn rounds the
            // exact product with the scale once, as the page's bf16 multiply does
            const uint32_t s2 = (uint32_t)__ldg(scale + g) * 0x10001u;
            const float zb = 128.0f + (float)__ldg(zp + g);
            const uint32_t z2 = wq::f2_to_bf2(zb, zb);
            const uint4 o = make_uint4(
                wq::bmul2(wq::bsub2(__byte_perm(blo[m], 0x43434343u, 0x4140), z2), s2),
                wq::bmul2(wq::bsub2(__byte_perm(blo[m], 0x43434343u, 0x4342), z2), s2),
                wq::bmul2(wq::bsub2(__byte_perm(bhi[m], 0x43434343u, 0x4140), z2), s2),
                wq::bmul2(wq::bsub2(__byte_perm(bhi[m], 0x43434343u, 0x4342), z2), s2));
            if (BF16) {
                reinterpret_cast<uint4*>(out)[e / 8] = o;
            } else {
                float4* p = reinterpret_cast<float4*>(out) + e / 4;
                p[0] = make_float4(wq::bf_lo(o.x), wq::bf_hi(o.x), wq::bf_lo(o.y), wq::bf_hi(o.y));
                p[1] = make_float4(wq::bf_lo(o.z), wq::bf_hi(o.z), wq::bf_lo(o.w), wq::bf_hi(o.w));
            }
        }
    }
}

// any numel % 8 == 0: one position per thread, byte loads.
template <int NBITS, bool BF16>
__global__ void __launch_bounds__(kThreads) uintx_dequant_general(const uint8_t* __restrict__ packed,
                                                                  const uint16_t* __restrict__ scale,
                                                                  const uint8_t* __restrict__ zp,
                                                                  int64_t numel, int group,
                                                                  void* __restrict__ out) {
    using S = Shards<NBITS>;
    const int64_t L1 = numel / 8;
    const int64_t base2 = S::has4 ? numel / 2 : 0;
    const int64_t base1 = base2 + (S::has2 ? numel / 4 : 0);
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t d = (int64_t)blockIdx.x * kThreads + threadIdx.x; d < L1; d += stride) {
        uint32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (S::has4) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t b = __ldg(packed + m * L1 + d);
                c[m] |= b & 15u;
                c[m + 4] |= b >> 4;
            }
        }
        if (S::has2) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t b = __ldg(packed + base2 + h * L1 + d);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) c[2 * jj + h] |= ((b >> (2 * jj)) & 3u) << S::off2;
            }
        }
        if (S::has1) {
            const uint32_t b = __ldg(packed + base1 + d);
#pragma unroll
            for (int m = 0; m < 8; ++m) c[m] |= ((b >> m) & 1u) << S::off1;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int64_t e = m * L1 + d, g = e / group;
            const float v = deq1(c[m], (float)__ldg(zp + g), wq::bf_to_f(__ldg(scale + g)));
            const uint32_t h = wq::f_to_bf(v);
            if (BF16) reinterpret_cast<uint16_t*>(out)[e] = (uint16_t)h;
            else reinterpret_cast<float*>(out)[e] = wq::bf_to_f(h);
        }
    }
}

// Error outputs of uintx_quantize_err (all null for uintx_quantize).
struct ErrOut {
    void* workspace = nullptr;
    double* snr_db = nullptr;
    double* rel_err = nullptr;
};

template <int NBITS, int ERR>
wq_status quant_nbits(const uint16_t* w, int64_t numel, int group, uint8_t* packed, uint16_t* scale,
                      uint8_t* zp, const ErrOut& eo, cudaStream_t st) {
    constexpr int QMAX = (1 << NBITS) - 1;
    unsigned* counter = nullptr;
    float4* slots = nullptr;
    if (ERR) {
        counter = (unsigned*)eo.workspace;
        slots = (float4*)((char*)eo.workspace + wqh::kCtrlBytes);
        wq_status s = wqh::cuda_status(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
        if (s != WQ_OK) return s;
    }
    // with the error sums every CTA owns one partial-sum slot
    const int cap = ERR ? wqh::kMaxPartials : 1 << 30;
    if (group == 64 && numel % 512 == 0) {
        const int64_t items = (numel / 8 + 255) / 256;  // one per warp
        const void* fn = (const void*)uintx_quant_fused<NBITS, ERR>;
        constexpr int smem = 2 * 8 * kThreads * 16;
        static bool attr_set = false;
        if (!attr_set) {
            wq_status s = wqh::cuda_status(
                cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
            if (s != WQ_OK) return s;
            attr_set = true;
        }
        const int grid = wqh::grid_for(fn, kThreads, smem, (items + 7) / 8, cap);
        uintx_quant_fused<NBITS, ERR><<<grid, kThreads, smem, st>>>(w, numel, packed, scale, zp, slots,
                                                                    counter, eo.snr_db, eo.rel_err);
        return wqh::check_launch();
    }
    const int64_t ngroups = numel / group;
    int grid = wqh::grid_for((const void*)uintx_qparams_kernel<QMAX>, kThreads, 0,
                             (ngroups + kThreads - 1) / kThreads, 1 << 30);
    uintx_qparams_kernel<QMAX><<<grid, kThreads, 0, st>>>(w, ngroups, group, scale, zp);
    wq_status s = wqh::check_launch();
    if (s != WQ_OK) return s;
    const int64_t L1 = numel / 8;
    grid = wqh::grid_for((const void*)uintx_pack_general<NBITS, ERR>, kThreads, 0,
                         (L1 + kThreads - 1) / kThreads, cap);
    uintx_pack_general<NBITS, ERR><<<grid, kThreads, 0, st>>>(w, numel, group, scale, zp, packed, slots,
                                                              counter, eo.snr_db, eo.rel_err);
    return wqh::check_launch();
}

template <int ERR>
wq_status quant_dispatch(const uint16_t* w, int64_t numel, int nbits, int group, uint8_t* packed,
                         uint16_t* scale, uint8_t* zp, const ErrOut& eo, cudaStream_t st) {
    switch (nbits) {
        case 2: return quant_nbits<2, ERR>(w, numel, group, packed, scale, zp, eo, st);
        case 3: return quant_nbits<3, ERR>(w, numel, group, packed, scale, zp, eo, st);
        case 4: return quant_nbits<4, ERR>(w, numel, group, packed, scale, zp, eo, st);
        case 5: return quant_nbits<5, ERR>(w, numel, group, packed, scale, zp, eo, st);
        case 6: return quant_nbits<6, ERR>(w, numel, group, packed, scale, zp, eo, st);
        case 7: return quant_nbits<7, ERR>(w, numel, group, packed, scale, zp, eo, st);
        default: return WQ_ERR_UNSUPPORTED;
    }
}

template <int NBITS, bool BF16>
wq_status dequant_nbits(const uint8_t* packed, const uint16_t* scale, const uint8_t* zp,
                        int64_t numel, int group, void* out, cudaStream_t st) {
    if (numel % 64 == 0 && (group & (group - 1)) == 0) {
        const int64_t items = numel / 64;
        const int grid = wqh::grid_for((const void*)uintx_dequant_vec<NBITS, BF16>, kThreads, 0,
                                       (items + kThreads - 1) / kThreads, 1 << 30);
        uintx_dequant_vec<NBITS, BF16><<<grid, kThreads, 0, st>>>(packed, scale, zp, numel,
                                                                  __builtin_ctz(group), out);
    } else {
        const int64_t L1 = numel / 8;
        const int grid = wqh::grid_for((const void*)uintx_dequant_general<NBITS, BF16>, kThreads, 0,
                                       (L1 + kThreads - 1) / kThreads, 1 << 30);
        uintx_dequant_general<NBITS, BF16><<<grid, kThreads, 0, st>>>(packed, scale, zp, numel, group, out);
    }
    return wqh::check_launch();
}

wq_status check_common(int64_t n, int64_t k, int nbits, int group) {
    if (n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (nbits < 2 || nbits > 7) return WQ_ERR_UNSUPPORTED;  // uint8 is refused, as the page does
    if (group <= 0 || group % 8 != 0) return WQ_ERR_UNSUPPORTED;
    if (k % group != 0) return WQ_ERR_BAD_SHAPE;
    return WQ_OK;
}

}  // namespace

extern "C" wq_status uintx_quantize(const uint16_t* w, int64_t n, int64_t k, int nbits, int group,
                                    uint8_t* packed, uint16_t* scale, uint8_t* zp, void* stream) {
    wq_status s = check_common(n, k, nbits, group);
    if (s != WQ_OK) return s;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !packed || !scale || !zp) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(w) || !wqh::aligned16(packed) || !wqh::aligned_to(scale, 2))
        return WQ_ERR_MISALIGNED;
    return quant_dispatch<0>(w, n * k, nbits, group, packed, scale, zp, ErrOut{}, (cudaStream_t)stream);
}

extern "C" wq_status uintx_quantize_err(const uint16_t* w, int64_t n, int64_t k, int nbits, int group,
                                        uint8_t* packed, uint16_t* scale, uint8_t* zp, double* snr_db,
                                        double* rel_err, void* workspace, size_t workspace_bytes,
                                        void* stream) {
    if (!snr_db && !rel_err) return uintx_quantize(w, n, k, nbits, group, packed, scale, zp, stream);
    wq_status s = check_common(n, k, nbits, group);
    if (s != WQ_OK) return s;
    if (n == 0 || k == 0) return WQ_OK;
    if (!w || !packed || !scale || !zp || !workspace) return WQ_ERR_NULL_PTR;
    if (workspace_bytes < wq_workspace_bytes(WQ_OP_UINTX_ERR, n, k, nbits)) return WQ_ERR_WORKSPACE_TOO_SMALL;
    if (!wqh::aligned16(w) || !wqh::aligned16(packed) || !wqh::aligned_to(scale, 2) ||
        !wqh::aligned_to(workspace, 16) || (snr_db && !wqh::aligned_to(snr_db, 8)) ||
        (rel_err && !wqh::aligned_to(rel_err, 8)))
        return WQ_ERR_MISALIGNED;
    ErrOut eo;
    eo.workspace = workspace;
    eo.snr_db = snr_db;
    eo.rel_err = rel_err;
    return quant_dispatch<1>(w, n * k, nbits, group, packed, scale, zp, eo, (cudaStream_t)stream);
}

extern "C" wq_status uintx_dequantize(const uint8_t* packed, const uint16_t* scale, const uint8_t* zp,
                                      int64_t n, int64_t k, int nbits, int group, int out_dtype,
                                      void* out, void* stream) {
    wq_status s = check_common(n, k, nbits, group);
    if (s != WQ_OK) return s;
    if (out_dtype != WQ_DTYPE_F32 && out_dtype != WQ_DTYPE_BF16) return WQ_ERR_BAD_DTYPE;
    if (n == 0 || k == 0) return WQ_OK;
    if (!packed || !scale || !zp || !out) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(packed) || !wqh::aligned16(out) || !wqh::aligned_to(scale, 2))
        return WQ_ERR_MISALIGNED;
    const int64_t numel = n * k;
    cudaStream_t st = (cudaStream_t)stream;
    const bool bf = out_dtype == WQ_DTYPE_BF16;
#define WQ_UX_DQ(NB) \
    case NB: return bf ? dequant_nbits<NB, true>(packed, scale, zp, numel, group, out, st) \
                       : dequant_nbits<NB, false>(packed, scale, zp, numel, group, out, st);
    switch (nbits) {
        WQ_UX_DQ(2)
        WQ_UX_DQ(3)
        WQ_UX_DQ(4)
        WQ_UX_DQ(5)
        WQ_UX_DQ(6)
        WQ_UX_DQ(7)
        default: return WQ_ERR_UNSUPPORTED;
    }
#undef WQ_UX_DQ
}
