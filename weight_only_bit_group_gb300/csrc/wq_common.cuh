// wq_common.cuh -- device and host helpers shared by the sm_103a kernels of
// libwqgb300.so.  Everything here is exact: no fast-math, the library is built
// with -fmad=false so that only the FMAs written explicitly below are fused.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/wqgb300.h"

namespace wq {

// ------------------------------------------------------------------ memory
// Streaming 128-bit load of data read exactly once (weights): read-only path,
// no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ld_stream2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ld_stream1(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// ------------------------------------------------------------------ bf16 bits
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf_to_f(uint32_t h16) { return __uint_as_float(h16 << 16); }

// binary32 -> bf16 bits, round to nearest even (hardware cvt.rn).
__device__ __forceinline__ uint32_t f_to_bf(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}
// Two binary32 -> packed bf16x2 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// One bf16 operation: the binary32 op result rounded to bf16, back as binary32.
__device__ __forceinline__ float bfr(float x) { return bf_to_f(f_to_bf(x)); }

// ------------------------------------------------------------------ bf16x2
// Packed bf16 pairs.  min/max are exact; mul/add/sub round the exact result once
// to bf16 (nearest even), i.e. they equal the binary32 operation on the bf16
// operands followed by one bf16 rounding whenever that binary32 result is exact
// (always for mul; for add/sub of the small integers used here).
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
// |a| max |b| per bf16 half (sign bits are garbage: callers mask them).
__device__ __forceinline__ uint32_t babsmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t badd2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// The two halves of a bf16x2 word swapped.
__device__ __forceinline__ uint32_t bswap2(uint32_t a) { return __byte_perm(a, 0, 0x1032); }

// ------------------------------------------------------------------ rounding
// Round half to even of |x| < 2^22 via the binary32 adder: (x + 1.5*2^23) has
// unit spacing, so the sum is x rounded to an integer with ties to even (the
// constant is even).  The integer is returned in two's complement.
__device__ __forceinline__ int rint_small(float x) {
    const float magic = 12582912.0f;  // 1.5 * 2^23
    return __float_as_int(__fadd_rn(x, magic)) - 0x4B400000;
}

// Quotient x / s rounded to nearest even, given r = RN(1/s): one Markstein
// correction step (P. Markstein, "IA-64 and Elementary Functions", 2000;
// Muller et al., Handbook of Floating-Point Arithmetic, division by FMA): with r
// correctly rounded and q0 = RN(x*r) within one ulp, the residual x - q0*s is
// exact in one FMA and q0 + residual*r rounds to RN(x/s).  Valid while neither
// s nor 1/s nor the quotient leaves the normal range; callers fall back to
// __fdiv_rn outside it.
__device__ __forceinline__ float div_by_recip(float x, float s, float r) {
    float q0 = __fmul_rn(x, r);
    float rem = __fmaf_rn(-q0, s, x);
    return __fmaf_rn(rem, r, q0);
}

// ------------------------------------------------------------------ cp.async
// 16-byte global -> shared copy that bypasses L1 (LDGSTS); completion is tracked
// per thread by commit groups and awaited in hardware (no spin loop).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ mbarrier + TMA
// Shared-memory operands are 32-bit shared-window addresses.
__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Make initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival that also announces `bytes` of transactions still to land.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// True once the phase with parity `parity` has completed (one poll).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// 2D tiled TMA load of one box at element coordinates (x inner, y outer) into
// shared memory, completing `bytes` on the mbarrier.  x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// ------------------------------------------------------------------ f32x2
// Packed binary32 pairs (Blackwell FFMA2/FMUL2/FADD2 through the float2
// builtins): each half is one IEEE binary32 operation, round to nearest even,
// subnormals kept.
typedef float2 f2_t;
__device__ __forceinline__ f2_t f2(float lo, float hi) { return make_float2(lo, hi); }
__device__ __forceinline__ void f2u(f2_t v, float& lo, float& hi) {
    lo = v.x;
    hi = v.y;
}
__device__ __forceinline__ f2_t mul2(f2_t a, f2_t b) { return __fmul2_rn(a, b); }
// RN(a * b) for a product that is then added to something: a packed multiply
// followed by a packed add was fused into one FMA by the code generator (one
// rounding instead of two, measured in the instruction mix), so the product is
// formed as fma(a, b, +0), which equals RN(a * b) whenever the product is not
// -0 (then +0: the sign of a zero term is irrelevant to the sums it enters) and
// which no rewrite may merge with the following add.
__device__ __forceinline__ f2_t mul2_kept(f2_t a, f2_t b) { return __ffma2_rn(a, b, make_float2(0.0f, 0.0f)); }
__device__ __forceinline__ f2_t add2(f2_t a, f2_t b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ f2_t fma2(f2_t a, f2_t b, f2_t c) { return __ffma2_rn(a, b, c); }
// The two bf16 of a packed word as a binary32 pair (exact).
__device__ __forceinline__ f2_t bf2_to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// ------------------------------------------------------------------ sums
// Compensated (Neumaier) binary32 running sum.  Partial sums of binary32 terms
// are added here instead of in binary64, whose pipe is narrow on this GPU; the
// compensation keeps the running sum accurate to a few binary32 ulps however
// many partials it absorbs.  value() folds the compensation in binary64.
struct KSum {
    float s = 0.0f, c = 0.0f;
    __device__ __forceinline__ void add(float x) {
        const float t = __fadd_rn(s, x);
        c = __fadd_rn(c, fabsf(s) >= fabsf(x) ? __fadd_rn(__fsub_rn(s, t), x) : __fadd_rn(__fsub_rn(x, t), s));
        s = t;
    }
    __device__ __forceinline__ double value() const { return (double)s + (double)c; }
};

// ------------------------------------------------------------------ warp
__device__ __forceinline__ float shfl_xor(float v, int m) {
    return __shfl_xor_sync(0xffffffffu, v, m);
}
__device__ __forceinline__ uint32_t shfl_xor(uint32_t v, int m) {
    return __shfl_xor_sync(0xffffffffu, v, m);
}

// ------------------------------------------------------------------ reductions
// Float-float numbers hi + lo (|lo| <= ulp(hi)/2): sums carried in two binary32
// values with about 44 significant bits, on the FP32 pipes (the binary64 pipe of
// this GPU is far too narrow for a whole wave of CTAs to reduce in binary64).
struct FF {
    float hi, lo;
};
// Knuth's TwoSum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    FF r;
    r.hi = __fadd_rn(s, e);                   // fast renormalisation (|s| >= |e|)
    r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
    return r;
}
__device__ __forceinline__ FF ff_of(const KSum& k) {
    FF r;
    two_sum(k.s, k.c, r.hi, r.lo);
    return r;
}
__device__ __forceinline__ FF ff_shfl_xor(FF v, int m) {
    FF r;
    r.hi = __shfl_xor_sync(0xffffffffu, v.hi, m);
    r.lo = __shfl_xor_sync(0xffffffffu, v.lo, m);
    return r;
}
__device__ __forceinline__ double ff_value(FF v) { return (double)v.hi + (double)v.lo; }

// CTA-wide fixed-order sum of two float-float values (blockDim.x a multiple of
// 32, at most 1024).  `scratch` holds 32 float4; the result is valid in thread 0.
__device__ __forceinline__ void cta_sum_ff2(FF& a, FF& b, float4* scratch) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        a = ff_add(a, ff_shfl_xor(a, m));
        b = ff_add(b, ff_shfl_xor(b, m));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) scratch[warp] = make_float4(a.hi, a.lo, b.hi, b.lo);
    __syncthreads();
    if (warp == 0) {
        const int nw = (int)(blockDim.x >> 5);
        const float4 v = lane < nw ? scratch[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        a = FF{v.x, v.y};
        b = FF{v.z, v.w};
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            a = ff_add(a, ff_shfl_xor(a, m));
            b = ff_add(b, ff_shfl_xor(b, m));
        }
    }
    __syncthreads();
}

// End of a two-level (sum w^2, sum e^2) reduction, with no waiting: each CTA
// stores its float-float pair in its own 16-byte slot, publishes it (fence) and
// counts itself in; the CTA that arrives last adds all slots in index order
// (deterministic for a given grid) and writes, in binary64,
// snr_db = 20*log10(sqrt(Sw)/max(sqrt(Se),1e-12)) and rel_err = sqrt(Se)/sqrt(Sw).
// *counter must be 0 when the kernel starts.
__device__ __forceinline__ void finish_snr(FF a, FF b, float4* slots, unsigned* counter,
                                           double* snr_db, double* rel_err) {
    __shared__ float4 scratch[32];
    __shared__ bool last;
    cta_sum_ff2(a, b, scratch);
    if (threadIdx.x == 0) {
        slots[blockIdx.x] = make_float4(a.hi, a.lo, b.hi, b.lo);
        __threadfence();
        last = atomicAdd(counter, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    FF ta{0.f, 0.f}, tb{0.f, 0.f};
    for (unsigned i = threadIdx.x; i < gridDim.x; i += blockDim.x) {
        const float4 v = __ldcg(slots + i);
        ta = ff_add(ta, FF{v.x, v.y});
        tb = ff_add(tb, FF{v.z, v.w});
    }
    cta_sum_ff2(ta, tb, scratch);
    if (threadIdx.x == 0) {
        const double nw = sqrt(ff_value(ta)), ne = sqrt(ff_value(tb));
        if (snr_db) *snr_db = 20.0 * log10(nw / fmax(ne, 1e-12));
        if (rel_err) *rel_err = ne / nw;
    }
}

}  // namespace wq

// ------------------------------------------------------------------ host side
namespace wqh {

// Number of SMs and resident CTAs of `kernel` at `threads` per CTA on the
// current device (queried once per kernel and device; cached).
int sm_count();
int grid_for(const void* kernel, int threads, size_t smem, int64_t work_items, int cap);

// Record a CUDA error for wq_last_cuda_error and map it to a status.
wq_status cuda_status(cudaError_t e);
wq_status check_launch();

// GPTQ quantization of an fp16 / fp32 weight (gptq.cu; arguments already checked).
wq_status gptq_quantize_wide(const void* w, int dt, int64_t n, int64_t k, int group, bool sym,
                             int32_t* qweight, int32_t* qzeros, uint16_t* scales, int32_t* g_idx,
                             double* snr_db, void* ws, cudaStream_t st);

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline bool aligned_to(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Partial-sum slots: a CTA writes its partial sums to its own 16-byte slot and the
// last CTA to finish adds the slots in index order (deterministic for a given
// grid).  Grids of reduction kernels never exceed this many CTAs.
constexpr int kMaxPartials = 4096;
// Workspace control block (arrival counter) ahead of the slots.
constexpr size_t kCtrlBytes = 256;

}  // namespace wqh
