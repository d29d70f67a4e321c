// gptq.cu -- GPTQ int4 quantize (sym / asym) and dequantize
// (export_gptq_cpu.py: pack_int32, quantize_sym, quantize_asym; module docstring
// for the uint4b8 dequant rule).
//
// Quantize.  For groups up to 128 a warp owns a tile of 32 output channels (rows
// of w) x 128 input channels and lane r owns row n0 + r, so each group lies in
// one lane; for group 256 the tile is 16 rows x 256 channels and lane h*16 + r
// owns half h of row n0 + r.  Tiles are numbered K-fastest, so the warps that
// run at the same time sweep long contiguous stretches of the same rows.  A
// tile arrives in shared memory through a two-stage per-warp TMA pipeline: one
// lane arms the stage's mbarrier and issues 2D tensor-map loads of (32 or 16) x
// 64 bf16 boxes with the 128-byte swizzle, which makes the per-lane 16-byte
// reads bank conflict free; the next tile streams in while the current one is
// coded.  The group max/min is a bf16x2 reduction inside the lane (plus one
// shuffle when a group spans both halves); scale and zero point use true IEEE
// divisions once per group (warp-uniformly through the rare large-scale path).
// Per element pair, with packed binary32 pairs (f32x2): where a clamp to the
// code range can act (always for sym; for asym only in warps where some group's
// extreme code leaves [0, 15], tested exactly per group) it is applied to w
// itself, in bf16x2, with bounds bf16(lo*s) and bf16(hi*s) (exact, see bound2);
// the quotient by the scale is a correctly rounded reciprocal plus one FMA
// correction step (bit-identical to IEEE division); round-half-even comes from
// the binary32 adder (q + 1.5*2^23); the nibble pack is one shift-add per code.
// The eight codes along k of one row are one qweight word, so the [K/8, N]
// transpose costs nothing.  The optional reconstruction SNR is accumulated from
// the same registers and reduced by the last CTA to finish.  fp16 and fp32
// weights take the same pipeline with their own kernel (gptq_quant_wide_kernel,
// below).  Every wait on an mbarrier is bounded: a wait that runs out records
// WQ_ERR_DEVICE_TIMEOUT in a device status word (read by wq_device_status) and
// the kernel finishes without touching the stage again.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <atomic>
#include <type_traits>
#include <mutex>

#include "wq_common.cuh"

namespace wqh {
unsigned gemm_status_take();  // gemm.cu
}

namespace {

constexpr int kThreads = 256;  // dequant kernels
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kRcp15 = 1.0f / 15.0f;  // RN(1/15), correctly rounded by the compiler

template <int G>
struct QTile {
    static constexpr int KT = G > 128 ? G : 128;      // input channels per warp tile
    static constexpr int P = G > 128 ? 2 : 1;          // lanes per row
    static constexpr int R = 32 / P;                   // output channels per warp tile
    static constexpr int HALF = KT / P;                // input channels per lane
    static constexpr int GL = G < HALF ? G : HALF;     // group elements one lane holds
    static constexpr int LPG = G / GL;                 // lanes per group (1 or 2)
    static constexpr int NB = KT / 64;                 // TMA boxes (R rows x 64 bf16) per tile
    static constexpr int BOXB = R * 128;               // bytes per box
    static constexpr int STAGE = NB * BOXB;            // one stage of one warp (8 KB)
    static constexpr int NS = 2;                       // pipeline stages
    static constexpr int WARPS = 4;                    // warps per CTA
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int BARS = WARPS * NS * 8;        // mbarriers after the stages
    static constexpr int SMEM = NS * WARPS * STAGE + BARS + 1024;  // + room to align to 1 KB
    // CTAs per SM: shared memory allows 3
    static constexpr int minb(bool) { return 3; }
};

// Per-group constants of the code computation.
struct GroupConst {
    float s;        // binary32 scale
    float zp;       // zero point (8 for sym)
    uint32_t lo2;   // bf16x2 lower clamp bound on w: bf16(-zp * s), both halves
    uint32_t hi2;   // bf16x2 upper clamp bound on w: bf16((15 - zp) * s)
};

// Clamping w to [bf16(lo*s), bf16(hi*s)] before dividing gives exactly the
// page's clamp(round(w/s), lo, hi): a bf16 bound is off lo*s (hi*s) by at most
// 2^-8 relative, i.e. by less than 15 * 2^-8 < 0.5 code steps, so every w that
// moves rounds to the same end code either way.
__device__ __forceinline__ uint32_t bound2(float v) {
    const uint32_t b = wq::f_to_bf(v);
    return b | (b << 16);
}

// Codes of one 8-value chunk (one qweight word) and the SNR terms, on packed
// binary32 pairs.  Per value: clamp (bf16x2, on w), q = RN(w/s) by reciprocal +
// correction, t = rint(q) + 1.5*2^23 from the binary32 adder; the low bits of
// t hold rint(q), and the word is sum over i of bits(t_i) << 4i plus the
// per-group constant cg = (zp - bits(1.5*2^23)) * 0x11111111 (mod 2^32).
// SNR terms as the page forms them: deq = RN((code - zp) * s), e = RN(w - deq),
// e^2 and w^2 summed (each a single-rounding FMA).
// CLAMP selects the clamps applied to w before the division:
//   0  none: every code of the warp's groups is already in [0, 15], so the
//      unpacked x is w itself and the SNR terms come from it in f32x2
//   1  the upper one (sym: the positive extreme amax / s = 8 rounds to code 16)
//   2  both (asym groups whose extreme codes leave [0, 15]).  rint(w/s) + zp < 0
//      needs w/s below -zp - 1/2; as the quotients round monotonically and
//      rint(RN(wmin/s)) = -rint(RN(-wmin/s)), that happens only when the zero
//      point was clamped down from above 15 (an all-negative group); the upper
//      end, rint(RN(wmax/s)) + zp > 15, is tested exactly per group
// With a clamp, x may differ from w, so e and w^2 read w's bf16 halves by
// mixed-precision FMAs instead.
template <int CLAMP, bool SNR>
__device__ __forceinline__ uint32_t quant_chunk(const uint4 v, const GroupConst& gc, const wq::f2_t R2,
                                                const wq::f2_t NS2, uint32_t cg, wq::f2_t& sw2,
                                                wq::f2_t& se2) {
    const wq::f2_t M2 = wq::f2(kMagic, kMagic), NM2 = wq::f2(-kMagic, -kMagic);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
    uint32_t word = cg;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t uc = u[p];
        if (CLAMP >= 1) uc = wq::bmin2(uc, gc.hi2);
        if (CLAMP == 2) uc = wq::bmax2(uc, gc.lo2);
        // bf16 pair -> binary32 pair on the integer pipe (byte permute, mask): the
        // FMA pipe already carries the packed quotient and SNR arithmetic
        const wq::f2_t x = wq::f2(__uint_as_float(__byte_perm(uc, 0u, 0x1044)), __uint_as_float(uc & 0xffff0000u));
        const wq::f2_t qa = wq::mul2(x, R2);
        const wq::f2_t rem = wq::fma2(qa, NS2, x);                          // x - qa*s, exact
        const wq::f2_t tq = wq::add2(wq::fma2(rem, R2, qa), M2);            // rint(RN(x/s)) + 1.5*2^23
        float t0, t1;
        wq::f2u(tq, t0, t1);
        word += (uint32_t)__float_as_int(t0) << (8 * p);
        word += (uint32_t)__float_as_int(t1) << (8 * p + 4);
        if (SNR && CLAMP == 0) {
            const wq::f2_t nd = wq::mul2_kept(wq::add2(tq, NM2), NS2);  // -deq = -RN((code - zp) * s)
            const wq::f2_t e = wq::add2(x, nd);                    // RN(w - deq)
            se2 = wq::fma2(e, e, se2);
            sw2 = wq::fma2(x, x, sw2);
        } else if (SNR) {
            const wq::f2_t nd = wq::mul2(wq::add2(tq, NM2), NS2);  // -deq = -RN((code - zp) * s)
            float e0, e1, w0, w1;
            asm("{\n\t.reg .b16 l, h, one;\n\tmov.b32 {l, h}, %4;\n\tmov.b16 one, 0x3F80;\n\t"
                "fma.rn.f32.bf16 %0, l, one, %5;\n\tfma.rn.f32.bf16 %1, h, one, %6;\n\t"
                "fma.rn.f32.bf16 %2, l, l, %7;\n\tfma.rn.f32.bf16 %3, h, h, %8;\n\t}"
                : "=f"(e0), "=f"(e1), "=f"(w0), "=f"(w1)
                : "r"(u[p]), "f"(nd.x), "f"(nd.y), "f"(sw2.x), "f"(sw2.y));
            const wq::f2_t e = wq::f2(e0, e1);  // RN(w - deq)
            se2 = wq::fma2(e, e, se2);
            sw2 = wq::f2(w0, w1);
        }
    }
    return word;
}

__device__ unsigned g_device_status;  // WQ_ERR_DEVICE_TIMEOUT once a bounded wait ran out

// Wait for phase `parity` of the mbarrier at shared address `bar`, giving up
// after `polls` polls (each poll may itself suspend for a while).
constexpr unsigned kMaxPolls = 1u << 22;
__device__ __forceinline__ bool wait_stage(uint32_t bar, uint32_t parity, unsigned polls) {
    for (unsigned i = 0; i < polls; ++i)
        if (wq::mbar_try_wait(bar, parity)) return true;
    return false;
}

// Poll budget of the stage waits for the next launches (kernel argument; a
// diagnostic lowers it to make the timeout path run, see wq_set_wait_budget).
// The drain of loads still in flight after a timeout always uses kMaxPolls.
std::atomic<unsigned> g_stage_polls{kMaxPolls};

template <bool SYM, int G, bool SNR>
__global__ void __launch_bounds__(QTile<G>::THREADS, QTile<G>::minb(SNR)) gptq_quant_kernel(
    const __grid_constant__ CUtensorMap wmap, int64_t n, int64_t k, int32_t* __restrict__ qweight,
    int32_t* __restrict__ qzeros, uint16_t* __restrict__ scales, int32_t* __restrict__ g_idx,
    float4* __restrict__ slots, unsigned* __restrict__ counter, double* __restrict__ snr_db,
    unsigned max_polls) {
    using T = QTile<G>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // the 128-byte swizzle needs 1 KB aligned boxes
    // pointer arithmetic on the shared array (no integer round trip) keeps the
    // shared address space visible, so the chunk reads below compile to 32-bit
    // shared loads
    unsigned char* smem =
        smem_raw + ((1024u - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 1023u)) & 1023u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = lane % T::R, half = lane / T::R;  // half: which part of the row (P = 2 only)
    unsigned char* wsm = smem + warp * (T::NS * T::STAGE);
    const uint32_t wsm_s = (uint32_t)__cvta_generic_to_shared(wsm);
    const uint32_t bar_s = (uint32_t)__cvta_generic_to_shared(smem + T::WARPS * T::NS * T::STAGE) + warp * T::NS * 8;
    // tile coordinates fit in 32 bits (n, k < 2^31)
    const int tn = (int)((n + T::R - 1) / T::R), tk = (int)((k + T::KT - 1) / T::KT);
    const int gwarp = blockIdx.x * T::WARPS + warp;
    const int nwarps = gridDim.x * T::WARPS;
    const int dn = nwarps / tk, dk = nwarps % tk;  // tile step, once
    if (lane == 0) {
        for (int i = 0; i < T::NS; ++i) wq::mbar_init(bar_s + 8 * i, 1);
        wq::mbar_fence_init();
    }
    __syncwarp();

    // this lane's reads: chunk c of its half-row sits at roff8[c % 8] + (c / 8) boxes
    // (the swizzle permutes the 16-byte chunks of each 128-byte box row by row % 8)
    uint32_t roff8[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        roff8[c] = (uint32_t)(half * (T::NB / T::P) * T::BOXB + row * 128 + 16 * (c ^ (row & 7)));
#define WQ_CHUNK(c) (*reinterpret_cast<const uint4*>(stage + roff8[(c) & 7] + ((c) >> 3) * T::BOXB))

    unsigned inflight = 0;  // bit i: a load into stage i has been issued and not yet waited for
    auto issue = [&](int nb, int kb, int st) {
        if (nb < tn) {  // warp-uniform
            if (lane == 0) {
                const uint32_t bar = bar_s + 8 * st, dst = wsm_s + st * T::STAGE;
                wq::mbar_expect_tx(bar, T::STAGE);
#pragma unroll
                for (int b = 0; b < T::NB; ++b)
                    wq::tma_load_2d(dst + b * T::BOXB, &wmap, kb * T::KT + 64 * b, nb * T::R, bar);
            }
            inflight |= 1u << st;
        }
    };

    wq::KSum ksw, kse;
    bool ok = true;
    // (nb, kb): tile being coded; (na, ka): tile NS - 1 steps ahead, being loaded
    int nb = gwarp / tk, kb = gwarp % tk;
    int na = nb, ka = kb;
    auto step = [&](int& x, int& y) {
        x += dn;
        y += dk;
        if (y >= tk) { y -= tk; ++x; }
    };
#pragma unroll
    for (int i = 0; i < T::NS - 1; ++i) {
        issue(na, ka, i);
        step(na, ka);
    }
    int st = 0, ahead = T::NS - 1;  // stage of the current tile / of the tile ahead
    uint32_t parity = 0;            // phase parity of the current stage's barrier
    for (; nb < tn;) {
        issue(na, ka, ahead);
        step(na, ka);
        ahead = ahead + 1 == T::NS ? 0 : ahead + 1;
        if (!wait_stage(bar_s + 8 * st, parity, max_polls)) {
            atomicExch(&g_device_status, (unsigned)WQ_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
        }
        inflight &= ~(1u << st);
        const int64_t n0 = (int64_t)nb * T::R, k0 = (int64_t)kb * T::KT;
        const int64_t col = n0 + row;
        const bool rowv = col < n;
        const int64_t kl = k0 + half * T::HALF;  // first input channel of this lane
        const unsigned char* stage = wsm + st * T::STAGE;
        int32_t* qp = qweight + (kl / 8) * n + col;  // qweight word of the lane's first chunk
#pragma unroll
        for (int g = 0; g < T::HALF / T::GL; ++g) {
            const int64_t kg = kl + g * T::GL;
            // group validity is uniform over the lanes sharing a group (k % G == 0) but
            // may differ between the two halves: shuffles below run on every lane
            const bool gval = kg < k;
            constexpr int GC = T::GL / 8;  // chunks per group part
            const int c0 = g * GC;
            float s, zp, rcp;
            bool big;  // warp-uniform: some lane's scale is beyond 2^100 (IEEE divisions then)
            bool need_clamp = false;  // asym: some code of this lane's group leaves [0, 15]
            if (SYM) {
                uint32_t m = 0;
#pragma unroll
                for (int c = 0; c < GC; ++c) {
                    const uint4 v = WQ_CHUNK(c0 + c);
                    m = wq::babsmax2(m, wq::babsmax2(wq::babsmax2(v.x, v.y), wq::babsmax2(v.z, v.w)));
                }
                if (T::LPG == 2) m = wq::babsmax2(m, __shfl_xor_sync(0xffffffffu, m, 16));
                m &= 0x7fff7fffu;
                const float amax = wq::bf_to_f(max(m & 0xffffu, m >> 16));
                s = fmaxf(__fmul_rn(amax, 0.125f), 1e-9f);  // amax / 8: exact for any bf16 amax
                zp = 8.0f;
                big = __any_sync(0xffffffffu, s > 0x1p100f);
                rcp = big ? 0.0f : __frcp_rn(s);
            } else {
                const uint4 v0 = WQ_CHUNK(c0);
                uint32_t mx = v0.x, mn = v0.x;
#pragma unroll
                for (int c = 0; c < GC; ++c) {
                    const uint4 v = WQ_CHUNK(c0 + c);
                    mx = wq::bmax2(mx, wq::bmax2(wq::bmax2(v.x, v.y), wq::bmax2(v.z, v.w)));
                    mn = wq::bmin2(mn, wq::bmin2(wq::bmin2(v.x, v.y), wq::bmin2(v.z, v.w)));
                }
                if (T::LPG == 2) {
                    mx = wq::bmax2(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    mn = wq::bmin2(mn, __shfl_xor_sync(0xffffffffu, mn, 16));
                }
                const float wmax = fmaxf(wq::bf_lo(mx), wq::bf_hi(mx));
                const float wmin = fminf(wq::bf_lo(mn), wq::bf_hi(mn));
                const float range = fmaxf(__fsub_rn(wmax, wmin), 1e-9f);
                // range / 15 and -wmin / s as IEEE quotients: reciprocal + one FMA
                // correction (exact while the operands stay in the normal range:
                // range <= 2^100 keeps s, 1/s and the quotients there); a warp with
                // a larger range anywhere takes true divisions on every lane, so
                // that no lane branches around them alone
                big = __any_sync(0xffffffffu, range > 0x1p100f);
                float q;
                if (!big) {
                    s = wq::div_by_recip(range, 15.0f, kRcp15);
                    rcp = __frcp_rn(s);
                    q = wq::div_by_recip(-wmin, s, rcp);
                } else {
                    s = __fdiv_rn(range, 15.0f);
                    rcp = 0.0f;
                    q = __fdiv_rn(-wmin, s);
                }
                const float zr = rintf(q);
                zp = fminf(fmaxf(zr, 0.0f), 15.0f);
                // the largest code is the one of wmax (the same correctly rounded
                // quotient as the coding pass; ignored on the IEEE-division path)
                const float cmax = big ? 0.0f : __fadd_rn(rintf(wq::div_by_recip(wmax, s, rcp)), zp);
                need_clamp = zr > 15.0f || cmax > 15.0f;
            }
            // the coding pass reads the chunks from shared memory again: holding all
            // of the group's chunks in registers between the two passes left too few
            // registers to interleave the per-pair chains (measured: sym 74.2 -> 68.2 us
            // on a 16384 x 8192 weight together with the integer-pipe unpacking)
            asm volatile("" ::: "memory");
            // warp-uniform: asym clamps only in warps where some group needs it
            const bool clamp_any = !SYM && __any_sync(0xffffffffu, need_clamp);
            if (gval) {
                GroupConst gc;
                gc.s = s;
                gc.zp = zp;
                gc.lo2 = bound2(__fmul_rn(-zp, s));
                gc.hi2 = bound2(__fmul_rn(15.0f - zp, s));
                wq::f2_t sw2 = wq::f2(0.0f, 0.0f), se2 = sw2;
                if (!big) {  // 1/s normal: the reciprocal + correction step is exact
                    const wq::f2_t R2 = wq::f2(rcp, rcp), NS2 = wq::f2(-s, -s);
                    const uint32_t cg = (uint32_t)((int)zp - 0x4B400000) * 0x11111111u;
                    int32_t* qc = qp + (int64_t)c0 * n;
                    if (SYM || clamp_any) {
#pragma unroll(SYM ? GC : 8)
                        for (int c = 0; c < GC; ++c) {
                            const uint4 v = WQ_CHUNK(c0 + c);
                            const uint32_t word =
                                quant_chunk<SYM ? 1 : 2, SNR>(v, gc, R2, NS2, cg, sw2, se2);
                            if (rowv) *qc = (int32_t)word;
                            qc += n;
                        }
                    } else {
#pragma unroll 8
                        for (int c = 0; c < GC; ++c) {
                            const uint4 v = WQ_CHUNK(c0 + c);
                            const uint32_t word = quant_chunk<0, SNR>(v, gc, R2, NS2, cg, sw2, se2);
                            if (rowv) *qc = (int32_t)word;
                            qc += n;
                        }
                    }
                } else {  // astronomically large scales somewhere in the warp: IEEE division
                    const float lo = -zp, hi = 15.0f - zp;
                    float sw = 0.f, se = 0.f;
#pragma unroll 1
                    for (int c = 0; c < GC; ++c) {
                        const int cc = c0 + c;
                        const uint4 v = *reinterpret_cast<const uint4*>(
                            stage + half * (T::NB / T::P) * T::BOXB + (cc >> 3) * T::BOXB + row * 128 +
                            16 * ((cc & 7) ^ (row & 7)));
                        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
                        uint32_t word = 0;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float x = (e & 1) ? wq::bf_hi(u[e >> 1]) : wq::bf_lo(u[e >> 1]);
                            const float rq = rintf(fminf(fmaxf(__fdiv_rn(x, s), lo), hi));
                            word |= (uint32_t)((int)rq + (int)zp) << (4 * e);
                            const float dd = __fsub_rn(x, __fmul_rn(rq, s));
                            sw = __fmaf_rn(x, x, sw);
                            se = __fmaf_rn(dd, dd, se);
                        }
                        if (rowv) qp[(int64_t)(c0 + c) * n] = (int32_t)word;
                    }
                    sw2 = wq::f2(sw, 0.f);
                    se2 = wq::f2(se, 0.f);
                }
                if (SNR) {  // rows past n hold zeros (the tensor map fills them): zero terms
                    float a0, a1, b0, b1;
                    wq::f2u(sw2, a0, a1);
                    wq::f2u(se2, b0, b1);
                    ksw.add(__fadd_rn(a0, a1));
                    kse.add(__fadd_rn(b0, b1));
                }
            }
            const int64_t gi = kg / G;
            const bool owner = T::LPG == 1 || half == 0;  // one lane writes per group
            if (gval && rowv && owner) scales[gi * n + col] = __half_as_ushort(__float2half_rn(s));
            if (qzeros) {
                // zero points of 8 consecutive rows (8 consecutive lanes of one part)
                uint32_t zw = SYM ? 0x77777777u : ((uint32_t)zp << (4 * (row & 7)));
                if (!SYM) {
                    zw |= __shfl_xor_sync(0xffffffffu, zw, 1);
                    zw |= __shfl_xor_sync(0xffffffffu, zw, 2);
                    zw |= __shfl_xor_sync(0xffffffffu, zw, 4);
                }
                if (gval && rowv && owner && (row & 7) == 0) qzeros[gi * (n / 8) + col / 8] = (int32_t)zw;
            }
        }
        if (g_idx && n0 == 0) {
            for (int i = lane; i < T::KT; i += 32)
                if (k0 + i < k) g_idx[k0 + i] = (int32_t)((k0 + i) / G);
        }
        __syncwarp();
        step(nb, kb);
        if (++st == T::NS) { st = 0; parity ^= 1u; }
    }
    if (!ok && lane == 0) {
        // loads still in flight (the stage that timed out, the one ahead of it):
        // wait for them with the full budget before the CTA's shared memory can be
        // handed to another CTA.  Stages are used round-robin, so a stage at or
        // after the current one completes with the current parity, one before it
        // (already refilled for the next round) with the other.
        for (int i = 0; i < T::NS; ++i)
            if ((inflight >> i) & 1u) wait_stage(bar_s + 8 * i, i >= st ? parity : parity ^ 1u, kMaxPolls);
    }
    __syncwarp();
    if (SNR) wq::finish_snr(wq::ff_of(ksw), wq::ff_of(kse), slots, counter, snr_db, nullptr);
}
#undef WQ_CHUNK

// ------------------------------------------------------------------ fp16 / fp32 weights
// export_gptq_cpu.py quantizes w.float(): an fp16 or fp32 weight takes the same
// binary32 steps with more significant bits, so the bf16 kernel's shortcuts
// (bf16x2 clamps on w, exact squares) do not carry over.  Same warp-tile
// pipeline: a warp stage is 8 KB, i.e. R rows x KT channels with R = 32 (fp16)
// or 16 (fp32) for KT = 128; a row spans P = 32 / R lanes.  The clamp acts on
// the rounded quotient t = rint(RN(w/s)) + 1.5*2^23 (exact for |w/s| < 2^22,
// which the per-group test below guarantees), and only in warps where some
// group's extreme code leaves [0, 15].
template <int DT, int G>
struct WTile {
    static constexpr int ES = DT == WQ_DTYPE_F32 ? 4 : 2;  // element bytes
    static constexpr int BI = 128 / ES;                     // elements per 128-byte box row
    static constexpr int KT = G > 128 ? G : 128;            // input channels per warp tile
    static constexpr int R = 8192 / (KT * ES);              // output channels per warp tile
    static constexpr int P = 32 / R;                        // lanes per row
    static constexpr int HALF = KT / P;                     // input channels per lane
    static constexpr int GL = G < HALF ? G : HALF;          // group elements one lane holds
    static constexpr int LPG = G / GL;                      // lanes per group
    static constexpr int NB = KT / BI;                      // TMA boxes (R rows x 128 B) per tile
    static constexpr int BOXB = R * 128;
    static constexpr int STAGE = NB * BOXB;
    static constexpr int CPW = ES / 2;                      // 16-byte chunks per qweight word
    static constexpr int PPC = 4 / CPW;                     // binary32 pairs per chunk
    static constexpr int NS = 2, WARPS = 4, THREADS = 32 * WARPS;
    static constexpr int SMEM = NS * WARPS * STAGE + WARPS * NS * 8 + 1024;
    static_assert(STAGE == 8192 && R >= 8 && R <= 32 && HALF % BI == 0, "warp tile");
};

// The 16-byte chunk `c` of w values held by this lane, as binary32 pairs
// (fp16 widens exactly): two pairs per chunk for fp32, four for fp16.
template <int DT>
__device__ __forceinline__ void chunk_pairs(const uint4 v, wq::f2_t (&x)[4]) {
    if (DT == WQ_DTYPE_F32) {
        x[0] = wq::f2(__uint_as_float(v.x), __uint_as_float(v.y));
        x[1] = wq::f2(__uint_as_float(v.z), __uint_as_float(v.w));
    } else {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
            x[i] = wq::f2(f.x, f.y);
        }
    }
}

// Codes (4 bits each, added into `word` from nibble `nib`) and SNR terms of one
// binary32 pair.  CLAMP: 0 none, 1 the upper end, 2 both.
template <int CLAMP, bool SNR>
__device__ __forceinline__ void wide_pair(const wq::f2_t x, const wq::f2_t R2, const wq::f2_t NS2, float tlo,
                                          float thi, uint32_t& word, int nib, wq::f2_t& sw2, wq::f2_t& se2) {
    const wq::f2_t qa = wq::mul2(x, R2);
    const wq::f2_t rem = wq::fma2(qa, NS2, x);                                 // x - qa*s, exact
    const wq::f2_t tq = wq::add2(wq::fma2(rem, R2, qa), wq::f2(kMagic, kMagic));  // rint(RN(x/s)) + 1.5*2^23
    float t0, t1;
    wq::f2u(tq, t0, t1);
    if (CLAMP >= 1) { t0 = fminf(t0, thi); t1 = fminf(t1, thi); }
    if (CLAMP == 2) { t0 = fmaxf(t0, tlo); t1 = fmaxf(t1, tlo); }
    word += (uint32_t)__float_as_int(t0) << (4 * nib);
    word += (uint32_t)__float_as_int(t1) << (4 * nib + 4);
    if (SNR) {
        // deq = RN((code - zp) * s), e = RN(w - deq); squares summed by FMAs
        const wq::f2_t nd = wq::mul2_kept(wq::add2(wq::f2(t0, t1), wq::f2(-kMagic, -kMagic)), NS2);
        const wq::f2_t e = wq::add2(x, nd);
        se2 = wq::fma2(e, e, se2);
        sw2 = wq::fma2(x, x, sw2);
    }
}

template <bool SYM, int DT, int G, bool SNR>
__global__ void __launch_bounds__(WTile<DT, G>::THREADS, 3) gptq_quant_wide_kernel(
    const __grid_constant__ CUtensorMap wmap, int64_t n, int64_t k, int32_t* __restrict__ qweight,
    int32_t* __restrict__ qzeros, uint16_t* __restrict__ scales, int32_t* __restrict__ g_idx,
    float4* __restrict__ slots, unsigned* __restrict__ counter, double* __restrict__ snr_db,
    unsigned max_polls) {
    using T = WTile<DT, G>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char* smem =
        smem_raw + ((1024u - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 1023u)) & 1023u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = lane % T::R, part = lane / T::R;
    unsigned char* wsm = smem + warp * (T::NS * T::STAGE);
    const uint32_t wsm_s = (uint32_t)__cvta_generic_to_shared(wsm);
    const uint32_t bar_s =
        (uint32_t)__cvta_generic_to_shared(smem + T::WARPS * T::NS * T::STAGE) + warp * T::NS * 8;
    const int tn = (int)((n + T::R - 1) / T::R), tk = (int)((k + T::KT - 1) / T::KT);
    const int gwarp = blockIdx.x * T::WARPS + warp;
    const int nwarps = gridDim.x * T::WARPS;
    const int dn = nwarps / tk, dk = nwarps % tk;
    if (lane == 0) {
        for (int i = 0; i < T::NS; ++i) wq::mbar_init(bar_s + 8 * i, 1);
        wq::mbar_fence_init();
    }
    __syncwarp();
    // chunk c of this lane's part of its row: box part * (HALF / BI) + c / 8, with
    // the 128-byte swizzle permuting the 16-byte chunks of each box row by row % 8
    uint32_t roff8[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        roff8[c] = (uint32_t)(part * (T::HALF / T::BI) * T::BOXB + row * 128 + 16 * (c ^ (row & 7)));
#define WQ_WCHUNK(c) (*reinterpret_cast<const uint4*>(stage + roff8[(c) & 7] + ((c) >> 3) * T::BOXB))

    unsigned inflight = 0;
    auto issue = [&](int nb, int kb, int st) {
        if (nb < tn) {
            if (lane == 0) {
                const uint32_t bar = bar_s + 8 * st, dst = wsm_s + st * T::STAGE;
                wq::mbar_expect_tx(bar, T::STAGE);
#pragma unroll
                for (int b = 0; b < T::NB; ++b)
                    wq::tma_load_2d(dst + b * T::BOXB, &wmap, kb * T::KT + T::BI * b, nb * T::R, bar);
            }
            inflight |= 1u << st;
        }
    };
    wq::KSum ksw, kse;
    bool ok = true;
    int nb = gwarp / tk, kb = gwarp % tk;
    int na = nb, ka = kb;
    auto step = [&](int& x, int& y) {
        x += dn;
        y += dk;
        if (y >= tk) { y -= tk; ++x; }
    };
    issue(na, ka, 0);
    step(na, ka);
    int st = 0, ahead = 1;
    uint32_t parity = 0;
    constexpr int GC = T::GL * T::ES / 16;  // chunks per group part
    constexpr unsigned FULL = 0xffffffffu;
    for (; nb < tn;) {
        issue(na, ka, ahead);
        step(na, ka);
        ahead ^= 1;
        if (!wait_stage(bar_s + 8 * st, parity, max_polls)) {
            atomicExch(&g_device_status, (unsigned)WQ_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
        }
        inflight &= ~(1u << st);
        const int64_t n0 = (int64_t)nb * T::R, k0 = (int64_t)kb * T::KT;
        const int64_t col = n0 + row;
        const bool rowv = col < n;
        const int64_t kl = k0 + part * T::HALF;
        const unsigned char* stage = wsm + st * T::STAGE;
        int32_t* qp = qweight + (kl / 8) * n + col;
#pragma unroll
        for (int g = 0; g < T::HALF / T::GL; ++g) {
            const int64_t kg = kl + g * T::GL;
            const bool gval = kg < k;
            const int c0 = g * GC;
            // group statistics (exact: fp16 pairs by half2 max / min, fp32 values
            // one by one)
            float wmax = -INFINITY, wmin = INFINITY;
            if (DT == WQ_DTYPE_F16) {
                const uint4 v0 = WQ_WCHUNK(c0);
                __half2 mx = *reinterpret_cast<const __half2*>(&v0.x), mn = mx;
#pragma unroll
                for (int c = 0; c < GC; ++c) {
                    const uint4 v = WQ_WCHUNK(c0 + c);
                    const __half2* h = reinterpret_cast<const __half2*>(&v);
                    mx = __hmax2(mx, __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3])));
                    mn = __hmin2(mn, __hmin2(__hmin2(h[0], h[1]), __hmin2(h[2], h[3])));
                }
                const float2 fx = __half22float2(mx), fn = __half22float2(mn);
                wmax = fmaxf(fx.x, fx.y);
                wmin = fminf(fn.x, fn.y);
            } else {
#pragma unroll
                for (int c = 0; c < GC; ++c) {
                    wq::f2_t x[4];
                    chunk_pairs<DT>(WQ_WCHUNK(c0 + c), x);
#pragma unroll
                    for (int i = 0; i < T::PPC; ++i) {
                        wmax = fmaxf(wmax, fmaxf(x[i].x, x[i].y));
                        wmin = fminf(wmin, fminf(x[i].x, x[i].y));
                    }
                }
            }
#pragma unroll
            for (int o = T::R; o < T::R * T::LPG; o <<= 1) {
                wmax = fmaxf(wmax, __shfl_xor_sync(FULL, wmax, o));
                wmin = fminf(wmin, __shfl_xor_sync(FULL, wmin, o));
            }
            float s, zp, rcp = 0.0f, q0 = 0.0f;
            bool big, need = false;
            if (SYM) {
                const float amax = fmaxf(wmax, -wmin);
                s = fmaxf(__fmul_rn(amax, 0.125f), 1e-9f);  // amax / 8: exact
                zp = 8.0f;
                big = __any_sync(FULL, s > 0x1p100f);
                if (!big) rcp = __frcp_rn(s);
            } else {
                const float range = fmaxf(__fsub_rn(wmax, wmin), 1e-9f);
                // the fast path needs normal quotients and |w / s| < 2^22 (the
                // adder rounding): range <= 2^100 and |w| <= 2^16 range
                big = __any_sync(FULL, range > 0x1p100f || fmaxf(wmax, -wmin) > __fmul_rn(range, 0x1p16f));
                if (!big) {
                    s = wq::div_by_recip(range, 15.0f, kRcp15);
                    rcp = __frcp_rn(s);
                    q0 = wq::div_by_recip(-wmin, s, rcp);
                } else {
                    s = __fdiv_rn(range, 15.0f);
                    q0 = __fdiv_rn(-wmin, s);
                }
                const float zr = rintf(q0);
                zp = fminf(fmaxf(zr, 0.0f), 15.0f);
                // the extreme codes: wmin's is -rint(q0) + zp (< 0 only when zp was
                // clamped down), wmax's from the same quotient as the coding pass
                const float cmax = big ? 0.0f : __fadd_rn(rintf(wq::div_by_recip(wmax, s, rcp)), zp);
                need = zr > 15.0f || cmax > 15.0f;
            }
            asm volatile("" ::: "memory");  // the coding pass reads the chunks again
            const bool clamp_any = !SYM && __any_sync(FULL, need);
            if (gval) {
                wq::f2_t sw2 = wq::f2(0.0f, 0.0f), se2 = sw2;
                if (!big) {
                    const wq::f2_t R2 = wq::f2(rcp, rcp), NS2 = wq::f2(-s, -s);
                    const float tlo = __fsub_rn(kMagic, zp), thi = __fadd_rn(kMagic, __fsub_rn(15.0f, zp));
                    const uint32_t cg = (uint32_t)((int)zp - 0x4B400000) * 0x11111111u;
                    int32_t* qc = qp + (int64_t)(c0 / T::CPW) * n;
                    auto code = [&](auto clamp_tag) {
                        constexpr int CL = decltype(clamp_tag)::value;
#pragma unroll(SYM ? GC / T::CPW : 8)
                        for (int wd = 0; wd < GC / T::CPW; ++wd) {
                            uint32_t word = cg;
#pragma unroll
                            for (int h = 0; h < T::CPW; ++h) {
                                wq::f2_t x[4];
                                chunk_pairs<DT>(WQ_WCHUNK(c0 + wd * T::CPW + h), x);
#pragma unroll
                                for (int i = 0; i < T::PPC; ++i)
                                    wide_pair<CL, SNR>(x[i], R2, NS2, tlo, thi, word, 2 * (h * T::PPC + i),
                                                       sw2, se2);
                            }
                            if (rowv) *qc = (int32_t)word;
                            qc += n;
                        }
                    };
                    if (SYM) code(std::integral_constant<int, 1>());
                    else if (clamp_any) code(std::integral_constant<int, 2>());
                    else code(std::integral_constant<int, 0>());
                } else {  // astronomical ratios somewhere in the warp: IEEE division
                    const float lo = -zp, hi = 15.0f - zp;
                    float sw = 0.f, se = 0.f;
#pragma unroll 1
                    for (int wd = 0; wd < GC / T::CPW; ++wd) {
                        uint32_t word = 0;
                        for (int h = 0; h < T::CPW; ++h) {
                            const int cc = c0 + wd * T::CPW + h;
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                stage + part * (T::HALF / T::BI) * T::BOXB + (cc >> 3) * T::BOXB + row * 128 +
                                16 * ((cc & 7) ^ (row & 7)));
                            wq::f2_t x[4];
                            chunk_pairs<DT>(v, x);
                            for (int i = 0; i < T::PPC; ++i) {
                                const float xv[2] = {x[i].x, x[i].y};
                                for (int e = 0; e < 2; ++e) {
                                    const float rq = rintf(fminf(fmaxf(__fdiv_rn(xv[e], s), lo), hi));
                                    const int nibble = 2 * (h * T::PPC + i) + e;
                                    word |= (uint32_t)((int)rq + (int)zp) << (4 * nibble);
                                    const float dd = __fsub_rn(xv[e], __fmul_rn(rq, s));
                                    sw = __fmaf_rn(xv[e], xv[e], sw);
                                    se = __fmaf_rn(dd, dd, se);
                                }
                            }
                        }
                        if (rowv) qp[(int64_t)(c0 / T::CPW + wd) * n] = (int32_t)word;
                    }
                    sw2 = wq::f2(sw, 0.f);
                    se2 = wq::f2(se, 0.f);
                }
                if (SNR) {  // rows past n hold zeros (the tensor map fills them): zero terms
                    float a0, a1, b0, b1;
                    wq::f2u(sw2, a0, a1);
                    wq::f2u(se2, b0, b1);
                    ksw.add(__fadd_rn(a0, a1));
                    kse.add(__fadd_rn(b0, b1));
                }
            }
            const int64_t gi = kg / G;
            const bool owner = part % T::LPG == 0;  // one lane writes per group
            if (gval && rowv && owner) scales[gi * n + col] = __half_as_ushort(__float2half_rn(s));
            if (qzeros) {
                uint32_t zw = SYM ? 0x77777777u : ((uint32_t)zp << (4 * (row & 7)));
                if (!SYM) {
                    zw |= __shfl_xor_sync(FULL, zw, 1);
                    zw |= __shfl_xor_sync(FULL, zw, 2);
                    zw |= __shfl_xor_sync(FULL, zw, 4);
                }
                if (gval && rowv && owner && (row & 7) == 0) qzeros[gi * (n / 8) + col / 8] = (int32_t)zw;
            }
        }
        if (g_idx && n0 == 0) {
            for (int i = lane; i < T::KT; i += 32)
                if (k0 + i < k) g_idx[k0 + i] = (int32_t)((k0 + i) / G);
        }
        __syncwarp();
        step(nb, kb);
        if (++st == T::NS) { st = 0; parity ^= 1u; }
    }
    if (!ok && lane == 0) {
        for (int i = 0; i < T::NS; ++i)
            if ((inflight >> i) & 1u) wait_stage(bar_s + 8 * i, i >= st ? parity : parity ^ 1u, kMaxPolls);
    }
    __syncwarp();
    if (SNR) wq::finish_snr(wq::ff_of(ksw), wq::ff_of(kse), slots, counter, snr_db, nullptr);
}
#undef WQ_WCHUNK

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on the driver library).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

// Tensor map of w [n, k] bf16 (row-major): boxes of box_rows rows x 64 values with the
// 128-byte swizzle; reads outside the tensor return zeros.
wq_status weight_map(const uint16_t* w, int64_t n, int64_t k, int box_rows, CUtensorMap* map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return wqh::cuda_status(cudaErrorNotSupported);
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(w), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? WQ_OK : wqh::cuda_status(cudaErrorInvalidValue);
}

template <bool SYM, int G, bool SNR>
wq_status launch_quant(const uint16_t* w, int64_t n, int64_t k, int32_t* qweight, int32_t* qzeros,
                       uint16_t* scales, int32_t* g_idx, float4* slots, unsigned* counter,
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
    CUtensorMap map;
    wq_status s = weight_map(w, n, k, T::R, &map);
    if (s != WQ_OK) return s;
    const int64_t warp_tiles = ((n + T::R - 1) / T::R) * ((k + T::KT - 1) / T::KT);
    const int grid = wqh::grid_for(fn, T::THREADS, T::SMEM, (warp_tiles + T::WARPS - 1) / T::WARPS,
                                   wqh::kMaxPartials);
    gptq_quant_kernel<SYM, G, SNR><<<grid, T::THREADS, T::SMEM, st>>>(
        map, n, k, qweight, qzeros, scales, g_idx, slots, counter, snr_db, g_stage_polls.load());
    return wqh::check_launch();
}

// Tensor map of an fp16 / fp32 weight [n, k]: boxes of box_rows rows x 128 bytes
// with the 128-byte swizzle; reads outside the tensor return zeros.
wq_status wide_map(const void* w, int dt, int64_t n, int64_t k, int box_rows, CUtensorMap* map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return wqh::cuda_status(cudaErrorNotSupported);
    const int es = dt == WQ_DTYPE_F32 ? 4 : 2;
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)k * es};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, dt == WQ_DTYPE_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           2, const_cast<void*>(w), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? WQ_OK : wqh::cuda_status(cudaErrorInvalidValue);
}

template <bool SYM, int DT, int G, bool SNR>
wq_status launch_wide(const void* w, int64_t n, int64_t k, int32_t* qweight, int32_t* qzeros,
                      uint16_t* scales, int32_t* g_idx, float4* slots, unsigned* counter, double* snr_db,
                      cudaStream_t st) {
    using T = WTile<DT, G>;
    const void* fn = (const void*)gptq_quant_wide_kernel<SYM, DT, G, SNR>;
    static bool attr_set = false;
    if (!attr_set) {
        wq_status s = wqh::cuda_status(
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM));
        if (s != WQ_OK) return s;
        attr_set = true;
    }
    CUtensorMap map;
    wq_status s = wide_map(w, DT, n, k, T::R, &map);
    if (s != WQ_OK) return s;
    const int64_t warp_tiles = ((n + T::R - 1) / T::R) * ((k + T::KT - 1) / T::KT);
    const int grid = wqh::grid_for(fn, T::THREADS, T::SMEM, (warp_tiles + T::WARPS - 1) / T::WARPS,
                                   wqh::kMaxPartials);
    gptq_quant_wide_kernel<SYM, DT, G, SNR><<<grid, T::THREADS, T::SMEM, st>>>(
        map, n, k, qweight, qzeros, scales, g_idx, slots, counter, snr_db, g_stage_polls.load());
    return wqh::check_launch();
}

template <bool SYM, int DT>
wq_status wide_group(int group, bool snr, const void* w, int64_t n, int64_t k, int32_t* qweight,
                     int32_t* qzeros, uint16_t* scales, int32_t* g_idx, float4* slots, unsigned* counter,
                     double* snr_db, cudaStream_t st) {
#define WQ_WIDE_CASE(GG)                                                                                   \
    case GG:                                                                                               \
        return snr ? launch_wide<SYM, DT, GG, true>(w, n, k, qweight, qzeros, scales, g_idx, slots, counter, \
                                                    snr_db, st)                                            \
                   : launch_wide<SYM, DT, GG, false>(w, n, k, qweight, qzeros, scales, g_idx, slots,       \
                                                     counter, snr_db, st);
    switch (group) {
        WQ_WIDE_CASE(32)
        WQ_WIDE_CASE(64)
        WQ_WIDE_CASE(128)
        WQ_WIDE_CASE(256)
        default: return WQ_ERR_UNSUPPORTED;
    }
#undef WQ_WIDE_CASE
}

template <bool SYM>
wq_status quantize(const uint16_t* w, int64_t n, int64_t k, int group, int32_t* qweight,
                   int32_t* qzeros, uint16_t* scales, int32_t* g_idx, double* snr_db, void* ws,
                   size_t ws_bytes, void* stream) {
    if (n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (group != 32 && group != 64 && group != 128 && group != 256) return WQ_ERR_UNSUPPORTED;
    if (k % group != 0 || n % 8 != 0) return WQ_ERR_BAD_SHAPE;
    if (n > INT32_MAX || k > INT32_MAX) return WQ_ERR_BAD_SHAPE;  // TMA coordinates are 32-bit
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
    float4* slots = snr_db ? (float4*)((char*)ws + wqh::kCtrlBytes) : nullptr;
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

// Codes of one qweight word as binary32 values 1.5*2^23 + code, two at a time:
// byte j of lo = nibble 2j, byte j of hi = nibble 2j + 1, and one byte permute
// places a byte under the exponent bits 0x4B40.
__device__ __forceinline__ uint32_t code_f(uint32_t bytes, int j) {
    return __byte_perm(bytes, 0x4B400000u, 0x7640u + (unsigned)j);
}

// [k, n] output.  A CTA tile is one qweight row r (output rows 8r .. 8r+7) x
// 1024 columns, 4 per thread (one 16-byte load; per output row one 8-byte bf16
// or 16-byte fp32 store, coalesced along n).  CTA tiles are walked with
// incremental, block-uniform coordinates.  Value = (code - zp) * fp16 scale,
// exact in binary32, computed on column pairs with f32x2 arithmetic.
template <bool SYM, bool BF16>
__global__ void __launch_bounds__(kThreads) gptq_dequant_kn(const int32_t* __restrict__ qweight,
                                                            const int32_t* __restrict__ qzeros,
                                                            const uint16_t* __restrict__ scales,
                                                            int64_t n, int64_t k, int lg_group,
                                                            void* __restrict__ out) {
    constexpr int CB = kThreads * 4;  // columns per CTA tile
    const int64_t rows = k / 8, ncb = (n + CB - 1) / CB;
    const int64_t dr = gridDim.x / ncb, dcb = gridDim.x % ncb;
    int64_t r = blockIdx.x / ncb, cb = blockIdx.x % ncb;
    for (; r < rows;) {
        const int64_t c = cb * CB + 4 * threadIdx.x;
        if (c < n) {  // n % 8 == 0: four columns are all valid or all not
            const uint4 wd = wq::ld_stream(qweight + r * n + c);
            const int64_t g = (8 * r) >> lg_group;
            const uint32_t s01 = __ldg(reinterpret_cast<const uint32_t*>(scales + g * n + c));
            const uint32_t s23 = __ldg(reinterpret_cast<const uint32_t*>(scales + g * n + c + 2));
            float z[4] = {8.f, 8.f, 8.f, 8.f};
            if (!SYM) {
                const uint32_t zw = (uint32_t)__ldg(qzeros + g * (n / 8) + c / 8) >> (4 * (c & 4));
#pragma unroll
                for (int j = 0; j < 4; ++j) z[j] = (float)((zw >> (4 * j)) & 15u);
            }
            const wq::f2_t S01 = wq::f2(__half2float(__ushort_as_half((unsigned short)(s01 & 0xffffu))),
                                        __half2float(__ushort_as_half((unsigned short)(s01 >> 16))));
            const wq::f2_t S23 = wq::f2(__half2float(__ushort_as_half((unsigned short)(s23 & 0xffffu))),
                                        __half2float(__ushort_as_half((unsigned short)(s23 >> 16))));
            const wq::f2_t Z01 = wq::f2(-(kMagic + z[0]), -(kMagic + z[1]));
            const wq::f2_t Z23 = wq::f2(-(kMagic + z[2]), -(kMagic + z[3]));
            const uint32_t lo[4] = {wd.x & 0x0F0F0F0Fu, wd.y & 0x0F0F0F0Fu, wd.z & 0x0F0F0F0Fu, wd.w & 0x0F0F0F0Fu};
            const uint32_t hi[4] = {(wd.x >> 4) & 0x0F0F0F0Fu, (wd.y >> 4) & 0x0F0F0F0Fu,
                                    (wd.z >> 4) & 0x0F0F0F0Fu, (wd.w >> 4) & 0x0F0F0F0Fu};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t* src = (i & 1) ? hi : lo;
                const int j = i >> 1;
                const wq::f2_t q01 = wq::f2(__uint_as_float(code_f(src[0], j)), __uint_as_float(code_f(src[1], j)));
                const wq::f2_t q23 = wq::f2(__uint_as_float(code_f(src[2], j)), __uint_as_float(code_f(src[3], j)));
                const wq::f2_t v01 = wq::mul2(wq::add2(q01, Z01), S01);
                const wq::f2_t v23 = wq::mul2(wq::add2(q23, Z23), S23);
                float a0, a1, a2, a3;
                wq::f2u(v01, a0, a1);
                wq::f2u(v23, a2, a3);
                const int64_t o = (8 * r + i) * n + c;
                if (BF16)
                    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(out) + o) =
                        make_uint2(wq::f2_to_bf2(a0, a1), wq::f2_to_bf2(a2, a3));
                else
                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o) = make_float4(a0, a1, a2, a3);
            }
        }
        r += dr;
        cb += dcb;
        if (cb >= ncb) { cb -= ncb; ++r; }
    }
}

// [n, k] output: a warp owns 32 output rows (qweight columns n0 .. n0+31) x 128
// input channels (16 qweight rows); lane l owns output row n0 + l.  Its 16
// qweight words are 16 coalesced 128-byte warp loads; the 128 outputs go through
// a padded per-warp shared tile so that the warp writes whole 256-byte (bf16) or
// 512-byte (fp32) row segments.  Tiles are walked with incremental coordinates.
// A group spans 2^lg_group / 8 words: with groups of 128 or more every tile is
// inside one group and needs one scale (and zero point) per lane.
template <bool SYM, bool BF16>
__global__ void __launch_bounds__(128) gptq_dequant_nk(const int32_t* __restrict__ qweight,
                                                       const int32_t* __restrict__ qzeros,
                                                       const uint16_t* __restrict__ scales,
                                                       int64_t n, int64_t k, int lg_group,
                                                       void* __restrict__ out) {
    constexpr int KT = 128, OB = BF16 ? 2 : 4;
    constexpr int ROWB = KT * OB + 16;   // padded row of the output tile
    constexpr int CPR = KT * OB / 16;    // 16-byte chunks per output row (16 or 32)
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned char* tile = smem + warp * 32 * ROWB;
    unsigned char* mine = tile + lane * ROWB;
    const int64_t tn = (n + 31) / 32, tk = (k + KT - 1) / KT;
    const int64_t gwarp = (int64_t)blockIdx.x * 4 + warp, nwarps = (int64_t)gridDim.x * 4;
    const int64_t dn = nwarps / tk, dk = nwarps % tk;
    const int cpg_mask = lg_group >= 7 ? 15 : (1 << (lg_group - 3)) - 1;  // words per group - 1, capped
    int64_t nb = gwarp / tk, kb = gwarp % tk;
    for (; nb < tn;) {
        const int64_t n0 = nb * 32, k0 = kb * KT;
        const int64_t col = n0 + lane;
        const bool rowv = col < n;
        const int nw = (int)min((int64_t)KT, k - k0) / 8;  // qweight rows in this tile
        const int32_t* qp = qweight + (k0 / 8) * n + col;
        // every load of the tile is issued before the first use: the 16 qweight
        // words and, per group, the fp16 scale and the qzeros word
        uint32_t wd[16], sh[16], zw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const bool cv = rowv && c < nw;
            wd[c] = cv ? wq::ld_stream1(qp + (int64_t)c * n) : 0u;
            sh[c] = 0u;
            zw[c] = 0u;
            if ((c & cpg_mask) == 0 && cv) {  // first word of a group (uniform over the warp)
                const int64_t g = (k0 + 8 * c) >> lg_group;
                sh[c] = __ldg(scales + g * n + col);
                if (!SYM) zw[c] = (uint32_t)__ldg(qzeros + g * (n / 8) + col / 8);
            }
        }
        wq::f2_t S2 = wq::f2(0.f, 0.f), Z2 = wq::f2(-kMagic - 8.f, -kMagic - 8.f);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            if ((c & cpg_mask) == 0) {  // first word of a group (uniform)
                const float sv = __half2float(__ushort_as_half((unsigned short)sh[c]));
                const float z = SYM ? 8.f : (float)((zw[c] >> (4 * (col & 7))) & 15u);
                S2 = wq::f2(sv, sv);
                Z2 = wq::f2(-(kMagic + z), -(kMagic + z));
            }
            const uint32_t lo = wd[c] & 0x0F0F0F0Fu, hi = (wd[c] >> 4) & 0x0F0F0F0Fu;
            float v[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const wq::f2_t q = wq::f2(__uint_as_float(code_f(lo, j)), __uint_as_float(code_f(hi, j)));
                wq::f2u(wq::mul2(wq::add2(q, Z2), S2), v[2 * j], v[2 * j + 1]);  // (code - zp) * s
            }
            if (BF16) {
                *reinterpret_cast<uint4*>(mine + 16 * c) =
                    make_uint4(wq::f2_to_bf2(v[0], v[1]), wq::f2_to_bf2(v[2], v[3]),
                               wq::f2_to_bf2(v[4], v[5]), wq::f2_to_bf2(v[6], v[7]));
            } else {
                *reinterpret_cast<float4*>(mine + 32 * c) = make_float4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<float4*>(mine + 32 * c + 16) = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
        __syncwarp();
        // copy out: row segments of KT*OB bytes, 16 bytes per lane per instruction
        const int valid_chunks = nw * 8 * OB / 16;
        unsigned char* obase = reinterpret_cast<unsigned char*>(out) + (n0 * k + k0) * OB;
#pragma unroll 4
        for (int i = 0; i < CPR; ++i) {
            const int idx = i * 32 + lane, orow = idx / CPR, ch = idx % CPR;
            if (n0 + orow < n && ch < valid_chunks)
                *reinterpret_cast<uint4*>(obase + (int64_t)orow * k * OB + 16 * ch) =
                    *reinterpret_cast<const uint4*>(tile + orow * ROWB + 16 * ch);
        }
        __syncwarp();
        nb += dn;
        kb += dk;
        if (kb >= tk) { kb -= tk; ++nb; }
    }
}

template <bool SYM, bool BF16>
wq_status launch_dequant(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                         int64_t n, int64_t k, int group, int layout, void* out, cudaStream_t st) {
    if (layout == WQ_LAYOUT_KN) {
        const void* fn = (const void*)gptq_dequant_kn<SYM, BF16>;
        const int64_t tiles = (k / 8) * ((n + 4 * kThreads - 1) / (4 * kThreads));
        const int grid = wqh::grid_for(fn, kThreads, 0, tiles, 1 << 30);
        gptq_dequant_kn<SYM, BF16><<<grid, kThreads, 0, st>>>(qweight, qzeros, scales, n, k, __builtin_ctz(group), out);
    } else {
        const void* fn = (const void*)gptq_dequant_nk<SYM, BF16>;
        constexpr int smem = 4 * 32 * (128 * (BF16 ? 2 : 4) + 16);
        static bool attr_set = false;
        if (!attr_set) {
            wq_status s = wqh::cuda_status(
                cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
            if (s != WQ_OK) return s;
            attr_set = true;
        }
        const int64_t warp_tiles = ((n + 31) / 32) * ((k + 127) / 128);
        const int grid = wqh::grid_for(fn, 128, smem, (warp_tiles + 3) / 4, 1 << 30);
        gptq_dequant_nk<SYM, BF16><<<grid, 128, smem, st>>>(qweight, qzeros, scales, n, k, __builtin_ctz(group), out);
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
    if (group < 8 || (group & (group - 1)) != 0) return WQ_ERR_UNSUPPORTED;  // power of two
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

extern "C" wq_status wq_device_status(void) {
    unsigned v = 0;
    wq_status s = wqh::cuda_status(cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v)));
    if (s != WQ_OK) return s;
    const unsigned vg = wqh::gemm_status_take();  // the tensor-core GEMM's own word
    if (v == 0) return vg ? (wq_status)vg : WQ_OK;
    const unsigned zero = 0;
    s = wqh::cuda_status(cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)));
    return s != WQ_OK ? s : (wq_status)v;
}

namespace wqh {
unsigned gptq_stage_polls_exchange(unsigned polls) { return g_stage_polls.exchange(polls); }
}  // namespace wqh

namespace wqh {
// GPTQ quantization of an fp16 / fp32 weight (arguments checked by the caller;
// the workspace, when snr_db is given, holds the SNR's counter and partials).
wq_status gptq_quantize_wide(const void* w, int dt, int64_t n, int64_t k, int group, bool sym,
                             int32_t* qweight, int32_t* qzeros, uint16_t* scales, int32_t* g_idx,
                             double* snr_db, void* ws, cudaStream_t st) {
    if (n > INT32_MAX || k > INT32_MAX) return WQ_ERR_BAD_SHAPE;  // TMA coordinates are 32-bit
    unsigned* counter = snr_db ? (unsigned*)ws : nullptr;
    float4* slots = snr_db ? (float4*)((char*)ws + wqh::kCtrlBytes) : nullptr;
    if (snr_db) {
        const wq_status s0 = wqh::cuda_status(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
        if (s0 != WQ_OK) return s0;
    }
    const bool snr = snr_db != nullptr;
    if (dt == WQ_DTYPE_F32)
        return sym ? wide_group<true, WQ_DTYPE_F32>(group, snr, w, n, k, qweight, qzeros, scales, g_idx, slots,
                                                    counter, snr_db, st)
                   : wide_group<false, WQ_DTYPE_F32>(group, snr, w, n, k, qweight, qzeros, scales, g_idx, slots,
                                                     counter, snr_db, st);
    return sym ? wide_group<true, WQ_DTYPE_F16>(group, snr, w, n, k, qweight, qzeros, scales, g_idx, slots,
                                                counter, snr_db, st)
               : wide_group<false, WQ_DTYPE_F16>(group, snr, w, n, k, qweight, qzeros, scales, g_idx, slots,
                                                 counter, snr_db, st);
}
}  // namespace wqh
