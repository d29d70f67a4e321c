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

// ------------------------------------------------------------------ warp
__device__ __forceinline__ float shfl_xor(float v, int m) {
    return __shfl_xor_sync(0xffffffffu, v, m);
}
__device__ __forceinline__ uint32_t shfl_xor(uint32_t v, int m) {
    return __shfl_xor_sync(0xffffffffu, v, m);
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

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline bool aligned_to(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// Partial-sum slots: a CTA writes its binary64 partials to its own slot, a
// one-CTA finalize kernel adds the slots in index order (deterministic for a
// given grid).  Grids of reduction kernels never exceed this many CTAs.
constexpr int kMaxPartials = 4096;

// One-CTA reduction of `nslots` (sum w^2, sum e^2) slots into snr_db / rel_err
// (either may be NULL).  Defined in snr.cu.
wq_status launch_snr_finalize(const double* slots, int nslots, double* snr_db, double* rel_err,
                              cudaStream_t st);

}  // namespace wqh
