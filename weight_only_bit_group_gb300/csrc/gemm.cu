// GPTQ W4A16 GEMM for prefill batches on the fifth-generation tensor cores:
// y[t, n] = sum_k x[t, k] * deq(W)[n, k], with deq the export_gptq_cpu.py rule
// (module docstring: w = (code - zp) * scale, zp = 8 for the symmetric uint4b8
// checkpoints, the stored zero point for asym; scale the fp16 group scale).
//
// The product is split at the group boundary so that the tensor cores only ever
// see exact operands: (code - zp) is an integer in [-15, 15], exact in bf16, and
// x is bf16, so every product x * (code - zp) is exact and the MMA accumulates
// them in binary32.  Each group's partial sum P_g lands in its own TMEM
// accumulator; the epilogue folds y += P_g * scale_g with one binary32 FMA per
// group, in group order.  No bf16-rounded weight is ever formed.
//
// One CTA computes 128 output features x 128 tokens over all of K:
//   warps 0-7   dequant: raw qweight rows (TMA) -> (code - zp) bf16, stored by
//               tcgen05.st straight into TMEM as the MMA's A operand (lane =
//               feature row, two K values per column; two threads per row)
//   warps 8-15  epilogue: two warpgroups (token columns 0-63 / 64-127), one
//               feature row per thread, tcgen05.ld of each group's partial
//   warp 16     TMA: x tile [128 tokens x 64] (128-byte swizzle) and qweight
//               rows [8 x 128 features]; owns the TMEM allocation
//   warp 17     MMA: one thread issues tcgen05.mma (A from TMEM, x from shared
//               memory; M 128, N 128, K 16) per 16 values of K, taking K blocks
//               in pairs (one wait, one fence and one stage release per pair),
//               and commits to the stage-pair and group barriers
// Keeping A out of shared memory matters: an N = 128 MMA reading both operands
// from shared memory uses all of its bandwidth by itself.
// Every wait is bounded; on a timeout the CTA records WQ_ERR_DEVICE_TIMEOUT in
// the device status word, lets its copies and MMAs land, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "wq_common.cuh"

namespace {

constexpr int BM = 128;                    // output features per CTA (MMA M)
constexpr int BT = 128;                    // tokens per CTA (MMA N)
constexpr int BK = 64;                     // K per pipeline stage
constexpr int NS = 8;                      // pipeline stages
constexpr int X_BYTES = BT * BK * 2;       // x tile, bf16, 128-byte swizzle
constexpr int Q_BYTES = (BK / 8) * BM * 4; // raw qweight rows
constexpr int STAGE = X_BYTES + Q_BYTES;    // the A operand lives in TMEM
constexpr int BAR_OFF = NS * STAGE;
// barriers: full[NS] (one per K block stage), aready[NS / 2] and empty[NS / 2]
// (one per pair of stages: the MMA thread consumes K blocks two at a time),
// tfull[2] tempty[2] done; then the TMEM address slot and the abort flag
constexpr int NP = NS / 2;                 // stage pairs
constexpr int N_BARS = NS + 2 * NP + 5;
static_assert(NS % 2 == 0, "stages are consumed in pairs");
constexpr int SLOT_OFF = BAR_OFF + 8 * N_BARS;
constexpr int SMEM = SLOT_OFF + 16 + 1024;  // + slack to align the tiles to 1024 bytes
constexpr int DQ_WARPS = 8;                // dequant warps: two per feature row
constexpr int EPI_WARP0 = DQ_WARPS;        // first of the 8 epilogue warps
constexpr int TMA_WARP = EPI_WARP0 + 8;
constexpr int MMA_WARP = TMA_WARP + 1;
constexpr int THREADS = (MMA_WARP + 1) * 32;
constexpr int kBand = 8;                   // token tiles per rasterisation band
// TMEM: two group accumulators (columns 0 .. 2 BT - 1), then the dequantized
// A operand of each stage (BK / 2 columns: two bf16 per 32-bit column, lane =
// feature row)
constexpr int A_COL0 = 2 * BT;
constexpr int TMEM_COLS = 512;
static_assert(STAGE % 1024 == 0 && X_BYTES % 1024 == 0, "swizzle atoms");
static_assert(A_COL0 + NS * (BK / 2) <= TMEM_COLS, "TMEM columns");

__device__ unsigned g_gemm_status;

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tc_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A's rows in TMEM lanes, two bf16 of K per
// 32-bit column.
__device__ __forceinline__ void tc_mma_ta(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes from registers.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Arrive once on the mbarrier when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 16 consecutive binary32 columns of this warp's 32 TMEM lanes, waited for.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Shared-memory matrix descriptor of a K-major tile stored as 8-row x 128-byte
// swizzle atoms (the TMA 128-byte swizzle): start address, stride 1024 bytes
// between 8-row groups, descriptor version 1, swizzle mode 128B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor: binary32 D, bf16 A and B, both K-major, N = BT, M = BM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BT >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for the phase with parity `parity`: the whole poll loop is one
// block of PTX (scoped labels), so every lane that executes it polls on its own
// and no compiler-made convergence barrier surrounds a divergent C++ loop --
// such barriers cost hundreds of cycles per wait.  mbarrier.try_wait suspends the
// thread in the barrier unit until the phase completes or a short time limit
// passes, so a waiting warp takes almost no issue slots.  Returns false after
// `limit` polls without completion (the caller then aborts).
constexpr uint32_t kSuspendNs = 100000;  // per poll; the thread wakes when the phase completes
__device__ __forceinline__ bool poll_bar(uint32_t bar, uint32_t parity, uint32_t limit) {
    uint32_t ok;
    asm volatile(
        "{\n\t"
        ".reg .pred p;\n\t"
        ".reg .u32 c;\n\t"
        "mov.u32 c, 0;\n"
        "WQ_POLL:\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %4;\n\t"
        "@p bra WQ_DONE;\n\t"
        "add.u32 c, c, 1;\n\t"
        "setp.lt.u32 p, c, %3;\n\t"
        "@p bra WQ_POLL;\n"
        "WQ_DONE:\n\t"
        "setp.lt.u32 p, c, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(limit), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}
// One non-blocking test of the phase with parity `parity`.  A completed phase is
// the common case in the pipeline's steady state, and mbarrier.try_wait with a
// suspend hint costs a few hundred cycles even then (measured with clock64
// stamps in the MMA-issuing thread: ~300 cycles per wait on a completed phase,
// against ~250 cycles to issue a K block's four MMAs), so every wait tries this
// first.
__device__ __forceinline__ bool test_bar(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait with the abort protocol: polls in slices, gives up early once another
// role aborted, and records a timeout.  Same outcome on every lane that calls it
// (callers that need a warp-wide decision combine it with __all_sync).
constexpr uint32_t kWaitSlices = 512;  // default budget of a wait: 512 slices of 64 polls
// Budget (slices) of the MMA-issuing thread's waits for the next launches (kernel
// argument; a diagnostic lowers it to make the abort path run, see
// wq_set_wait_budget).  The other roles and every drain keep their own budgets.
std::atomic<unsigned> g_mma_slices{kWaitSlices};
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t slices = kWaitSlices) {
    if (slices != 0 && test_bar(bar, parity)) return true;
    for (uint32_t i = 0; i < slices; ++i) {
        if (poll_bar(bar, parity, 64)) return true;
        if (*abort_flag) return false;
    }
    *abort_flag = 1;
    atomicCAS(&g_gemm_status, 0u, (unsigned)WQ_ERR_DEVICE_TIMEOUT);
    return false;
}
// A warp's wait: every lane polls (uniform control flow), one warp-wide outcome
// so that the warp-collective instructions after it run on all lanes or none.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag));
}
// Drain wait for work already issued (copies, MMAs): bounded, but it does not
// give up when another role aborted, because the hardware is still writing.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    if (test_bar(bar, parity)) return;
    if (!poll_bar(bar, parity, 16384)) atomicCAS(&g_gemm_status, 0u, (unsigned)WQ_ERR_DEVICE_TIMEOUT);
}

// UX == 0: GPTQ (qweight rows by TMA, SYM selects the rule, G the group; one
// accumulator per group, scaled in the epilogue).
// UX in 2..7: uintx of UX bits (uintx_quant.py): the dequant warps read the bit
// shards, scale and zero point themselves and write the page's bf16 deq values;
// one accumulator over all of K (the deq values are the weight, no scaling
// left); ux_group is the uintx group.
template <bool SYM, bool BF16OUT, int G, int UX>
__global__ void __launch_bounds__(THREADS, 1)
gptq_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap qmap,
                 const int32_t* __restrict__ qzeros, const uint16_t* __restrict__ scales, int m, int n,
                 int k, void* __restrict__ out, const uint8_t* __restrict__ ux_packed,
                 const uint8_t* __restrict__ ux_zp, int ux_group, uint32_t mma_slices) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    auto x_at = [&](int s) { return sbase + s * STAGE; };
    auto q_at = [&](int s) { return smem + s * STAGE + X_BYTES; };
    const uint32_t bar0 = sbase + BAR_OFF;
    auto full = [&](int s) { return bar0 + 8 * s; };
    // pair barriers of K blocks kb, kb + 1 (kb even): slot (kb / 2) % NP, used once
    // per NS K blocks, so a wait's parity is (kb / NS) & 1 as for the stages
    auto aready = [&](int kb) { return bar0 + 8 * (NS + (kb >> 1) % NP); };
    auto empty = [&](int kb) { return bar0 + 8 * (NS + NP + (kb >> 1) % NP); };
    auto tfull = [&](int b) { return bar0 + 8 * (NS + 2 * NP + b); };
    auto tempty = [&](int b) { return bar0 + 8 * (NS + 2 * NP + 2 + b); };
    const uint32_t done = bar0 + 8 * (NS + 2 * NP + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SLOT_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SLOT_OFF + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Grouped rasterisation of the 1-D grid: consecutive CTAs sweep the feature
    // tiles of a band of kBand token tiles, so the CTAs resident at one time
    // spread over several x tiles and several weight tiles instead of all
    // reading the same x tile (an L2 hot spot).
    int n0, t0;
    {
        const int ntn = (n + BM - 1) / BM, ntt = (m + BT - 1) / BT;
        const int pid = blockIdx.x, per_band = kBand * ntn;
        const int band = pid / per_band, first = band * kBand;
        const int bsz = min(ntt - first, kBand), in = pid - band * per_band;
        t0 = (first + in % bsz) * BT;
        n0 = (in / bsz) * BM;
    }
    const int nkb = (k + BK - 1) / BK;
    const int ngroups = UX ? 1 : k / G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) wq::mbar_init(full(s), 1);
        for (int q = 0; q < NP; ++q) {
            wq::mbar_init(aready(2 * q), DQ_WARPS);
            wq::mbar_init(empty(2 * q), 1);
        }
        for (int b = 0; b < 2; ++b) {
            wq::mbar_init(tfull(b), 1);
            wq::mbar_init(tempty(b), 8);
        }
        wq::mbar_init(done, 1);
        *abort_flag = 0;
        wq::mbar_fence_init();
    }
    if (warp == TMA_WARP) tc_alloc(sbase + SLOT_OFF, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == TMA_WARP) {
        // ---------------------------------------------------------- TMA
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % NS;
                const uint32_t u = (uint32_t)(kb / NS);
                // both stages of a pair are released together
                if ((kb & 1) == 0 && !wait_bar(empty(kb), (u & 1u) ^ 1u, abort_flag)) break;
                wq::mbar_expect_tx(full(s), UX ? X_BYTES : X_BYTES + Q_BYTES);
                wq::tma_load_2d(x_at(s), &xmap, kb * BK, t0, full(s));
                if (UX == 0)
                    wq::tma_load_2d((uint32_t)__cvta_generic_to_shared(q_at(s)), &qmap, n0, kb * (BK / 8),
                                    full(s));
                ++issued;
            }
            // copies still in flight must land before the shared memory is released
            for (int kb = issued - NS < 0 ? 0 : issued - NS; kb < issued; ++kb)
                drain_wait(full(kb % NS), (uint32_t)(kb / NS) & 1u);
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ---------------------------------------------------------- MMA
        // One thread issues every MMA, so its instruction stream between two
        // issues is on the tensor cores' critical path: group boundaries are
        // compile-time masks of the K-step index and the descriptors advance by
        // constant offsets (no division, no recomputation).
        if (lane == 0) {
            const uint64_t db0 = sw128_desc(x_at(0));
            // issue MMAs for K steps [ks0, ks1) of a stage (A columns da in TMEM, x
            // descriptor db) into accumulator b; the first one starts the
            // accumulator when `fresh`
            auto mmas = [&](uint32_t da, uint64_t db, uint32_t b, int ks0, int ks1, bool fresh) {
#pragma unroll
                for (int ks = ks0; ks < ks1; ++ks)
                    tc_mma_ta(tmem + b * BT, da + (uint32_t)(ks * 8), db + (uint64_t)(ks * 2), kIdesc,
                              (fresh && ks == ks0) ? 0u : 1u);
            };
            // MMAs of one K block; false when a wait for a free accumulator gave up
            auto block = [&](int kb) -> bool {
                const int s = kb % NS;
                const uint32_t da = tmem + (uint32_t)(A_COL0 + s * (BK / 2));
                const uint64_t db = db0 + (uint64_t)((s * STAGE) >> 4);
                if constexpr (UX != 0) {
                    // one accumulator over all of K
                    mmas(da, db, 0u, 0, BK / 16, kb == 0);
                    if (kb == nkb - 1) tc_commit(tfull(0));
                } else if constexpr (G >= BK) {
                    // a group spans G / 64 whole K blocks
                    constexpr int BPG = G / BK;
                    const int g = kb / BPG;
                    const uint32_t b = (uint32_t)g & 1u;
                    const bool gstart = (kb & (BPG - 1)) == 0;
                    if (gstart) {
                        if (!wait_bar(tempty(b), ((uint32_t)(g >> 1) & 1u) ^ 1u, abort_flag, mma_slices))
                            return false;
                        tc_fence_after();
                    }
                    mmas(da, db, b, 0, BK / 16, gstart);
                    if ((kb & (BPG - 1)) == BPG - 1) tc_commit(tfull(b));
                } else {
                    // G == 32: groups 2kb (accumulator 0, K steps 0-1) and 2kb+1
                    // (accumulator 1, K steps 2-3; absent in a half-full last block)
                    const int halves = (k - kb * BK) >= BK ? 2 : 1;
                    for (int hh = 0; hh < halves; ++hh) {
                        const int g = 2 * kb + hh;
                        if (!wait_bar(tempty((uint32_t)hh), ((uint32_t)(g >> 1) & 1u) ^ 1u, abort_flag,
                                      mma_slices))
                            return false;
                        tc_fence_after();
                        mmas(da, db, (uint32_t)hh, 2 * hh, 2 * hh + 2, true);
                        tc_commit(tfull((uint32_t)hh));
                    }
                }
                return true;
            };
            // K blocks two at a time: one wait, one fence and one stage release per
            // pair.  aready completes only after every dequant warp saw both stages'
            // copies land (it waits on full first), so it orders the x tiles too.
            for (int kb = 0; kb < nkb; kb += 2) {
                if (!wait_bar(aready(kb), (uint32_t)(kb / NS) & 1u, abort_flag, mma_slices)) break;
                tc_fence_after();
                if (!block(kb)) break;
                if (kb + 1 < nkb && !block(kb + 1)) break;
                tc_commit(empty(kb));
            }
            // every MMA issued has completed before TMEM can be freed
            tc_commit(done);
            drain_wait(done, 0);
        }
        __syncwarp();
    } else if (warp < DQ_WARPS) {
      if constexpr (UX != 0) {
        // ---------------------------------------------------------- uintx dequant
        // Thread (r, h) writes K values 32h .. 32h+31 of each K block of feature
        // row r.  The codes live in power-of-two bit shards (4, 2, 1 bits, in
        // that order, the first holding the low bits); shard s of L_s bytes puts
        // element e in byte e mod L_s at bit (e div L_s) * k_s.  With k % 64 == 0
        // every L_s and every 8-element run start is a multiple of 8, so a run is
        // one aligned 8-byte load per shard from one chunk.
        const int r = threadIdx.x & (BM - 1), h = threadIdx.x >> 7;
        const int nrow = n0 + r;
        const bool rv = nrow < n;
        constexpr int NSH = ((UX >> 2) & 1) + ((UX >> 1) & 1) + (UX & 1);
        const int64_t numel = (int64_t)n * k;
        int kbits[NSH], boff[NSH];
        int64_t L[NSH], base[NSH], pos[NSH];
        int chunk[NSH];
        {
            int si = 0, off = 0;
            int64_t b = 0;
#pragma unroll
            for (int kb2 = 4; kb2 >= 1; kb2 >>= 1) {
                if (UX & kb2) {
                    kbits[si] = kb2;
                    boff[si] = off;
                    L[si] = numel / (8 / kb2);
                    base[si] = b;
                    b += L[si];
                    off += kb2;
                    ++si;
                }
            }
            const int64_t e0 = (int64_t)nrow * k + 32 * h;  // element of this thread's first run
#pragma unroll
            for (int i = 0; i < NSH; ++i) {
                chunk[i] = rv ? (int)(e0 / L[i]) : 0;
                pos[i] = rv ? e0 - (int64_t)chunk[i] * L[i] : 0;
            }
        }
        const int ngr = k / ux_group;
        // raw words of one K block: [run][shard] plus the group's scale and zero point
        struct Raw {
            uint64_t w[4][NSH];
            uint32_t sh[4][NSH];
            uint32_t sc, zp;
        };
        // With n k % 256 == 0 every shard length and base is a multiple of 32 bytes,
        // so a thread's 32 codes of a K block (32 aligned bytes per shard) never
        // straddle a chunk boundary: two 16-byte loads per shard and one bit offset
        const bool whole = numel % 256 == 0;
        auto fetch = [&](int kb, Raw& o) {
            // positions advance by 64 elements per K block (wrapping into the next chunk)
            if (whole) {
#pragma unroll
                for (int i = 0; i < NSH; ++i) {
                    const uint4* src = reinterpret_cast<const uint4*>(ux_packed + base[i] + pos[i]);
                    const uint4 a = rv ? __ldg(src) : make_uint4(0, 0, 0, 0);
                    const uint4 b = rv ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
                    o.w[0][i] = (uint64_t)a.x | ((uint64_t)a.y << 32);
                    o.w[1][i] = (uint64_t)a.z | ((uint64_t)a.w << 32);
                    o.w[2][i] = (uint64_t)b.x | ((uint64_t)b.y << 32);
                    o.w[3][i] = (uint64_t)b.z | ((uint64_t)b.w << 32);
                    const uint32_t sh = (uint32_t)(chunk[i] * kbits[i]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) o.sh[j][i] = sh;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int i = 0; i < NSH; ++i) {
                        int64_t p = pos[i] + 8 * j;
                        int c = chunk[i];
                        while (p >= L[i]) { p -= L[i]; ++c; }
                        o.sh[j][i] = (uint32_t)(c * kbits[i]);
                        o.w[j][i] = rv ? __ldg(reinterpret_cast<const unsigned long long*>(ux_packed + base[i] + p)) : 0ull;
                    }
                }
            }
            const int gi = (kb * BK + 32 * h) / ux_group;
            o.sc = rv ? (uint32_t)__ldg(scales + (size_t)nrow * ngr + gi) : 0u;
            o.zp = rv ? (uint32_t)__ldg(ux_zp + (size_t)nrow * ngr + gi) : 0u;
#pragma unroll
            for (int i = 0; i < NSH; ++i) {
                pos[i] += BK;
                while (pos[i] >= L[i]) { pos[i] -= L[i]; ++chunk[i]; }
            }
        };
        Raw nxt;
        fetch(0, nxt);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % NS;
            const Raw cur = nxt;  // loaded one K block ago
            if (kb + 1 < nkb) fetch(kb + 1, nxt);
            if (!warp_wait(full(s), (uint32_t)(kb / NS) & 1u, abort_flag)) break;
            const uint32_t zb2 = (0x4300u + cur.zp) * 0x10001u;  // bf16x2 of 128 + zp
            const uint32_t sc2 = cur.sc * 0x10001u;              // bf16x2 of the scale
            uint32_t dv[16];  // this thread's 16 TMEM columns of the stage's A
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint64_t q = 0;  // eight code bytes
#pragma unroll
                for (int i = 0; i < NSH; ++i) {
                    const uint64_t mask = (uint64_t)((1u << kbits[i]) - 1u) * 0x0101010101010101ull;
                    q |= ((cur.w[j][i] >> cur.sh[j][i]) & mask) << boff[i];
                }
                const uint32_t lo = (uint32_t)q, hi = (uint32_t)(q >> 32);
                // bf16 of 128 + q, minus 128 + zp (exact), times the scale: the
                // page's bf16 sub and bf16 multiply, each rounded once
                dv[4 * j + 0] = wq::bmul2(wq::bsub2(__byte_perm(lo, 0x43434343u, 0x4140), zb2), sc2);
                dv[4 * j + 1] = wq::bmul2(wq::bsub2(__byte_perm(lo, 0x43434343u, 0x4342), zb2), sc2);
                dv[4 * j + 2] = wq::bmul2(wq::bsub2(__byte_perm(hi, 0x43434343u, 0x4140), zb2), sc2);
                dv[4 * j + 3] = wq::bmul2(wq::bsub2(__byte_perm(hi, 0x43434343u, 0x4342), zb2), sc2);
            }
            tc_st16(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(A_COL0 + s * (BK / 2) + 16 * h), dv);
            // the stores land before the MMA thread is told the stage is ready
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            // one arrival per pair of K blocks (or for a last, unpaired block)
            if (lane == 0 && ((kb & 1) || kb + 1 == nkb)) mbar_arrive(aready(kb & ~1));
        }
      } else {
        // ---------------------------------------------------------- dequant
        // Two threads per feature row: thread (r, h) converts qweight rows 4h..4h+3
        // of a stage (32 K values, inside one group for every supported group).
        // Two K blocks per round: one proxy fence and one warp barrier serve both.
        const int r = threadIdx.x & (BM - 1), h = threadIdx.x >> 7;
        const int nrow = n0 + r;
        const bool rv = nrow < n;
        // raw qzeros word of this thread's rows of K block kb (asym); issued one
        // round before its use and not touched in between, so the load's latency
        // overlaps a round of work
        auto zword = [&](int kb) -> uint32_t {
            const int kk = kb * (BK / 8) + 4 * h;
            if (SYM || !rv || kb >= nkb || kk * 8 >= k) return 0x88888888u;
            return (uint32_t)__ldg(qzeros + (size_t)(kk * 8 / G) * (n / 8) + nrow / 8);
        };
        auto convert = [&](int kb, uint32_t zw) {
            const int s = kb % NS;
            const uint32_t zp = (zw >> (4 * (nrow & 7))) & 15u;
            const uint32_t zb2 = (0x4300u + zp) * 0x10001u;  // bf16x2 of 128 + zp
            const uint32_t* qsrc = reinterpret_cast<const uint32_t*>(q_at(s)) + 4 * h * BM + r;
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = qsrc[j * BM];
            // column 16h + 4j + i of the stage's A holds K values 2i, 2i+1 of word j
            uint32_t dv[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t t0n = w[j] & 0x0F0F0F0Fu, t1n = (w[j] >> 4) & 0x0F0F0F0Fu;
                const uint32_t lo = __byte_perm(t0n, t1n, 0x5140);  // codes 0..3 as bytes
                const uint32_t hi = __byte_perm(t0n, t1n, 0x7362);  // codes 4..7
                // bytes c | 0x43 << 8 = bf16 of 128 + c; minus 128 + zp is exact
                dv[4 * j + 0] = wq::bsub2(__byte_perm(lo, 0x43434343u, 0x4140), zb2);
                dv[4 * j + 1] = wq::bsub2(__byte_perm(lo, 0x43434343u, 0x4342), zb2);
                dv[4 * j + 2] = wq::bsub2(__byte_perm(hi, 0x43434343u, 0x4140), zb2);
                dv[4 * j + 3] = wq::bsub2(__byte_perm(hi, 0x43434343u, 0x4342), zb2);
            }
            tc_st16(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(A_COL0 + s * (BK / 2) + 16 * h), dv);
        };
        uint32_t za = zword(0), zb = zword(1);
        for (int kb = 0; kb < nkb; kb += 2) {
            const bool two = kb + 1 < nkb;
            if (!warp_wait(full(kb % NS), (uint32_t)(kb / NS) & 1u, abort_flag)) break;
            if (two && !warp_wait(full((kb + 1) % NS), (uint32_t)((kb + 1) / NS) & 1u, abort_flag)) break;
            const uint32_t zcur_a = za, zcur_b = zb;
            za = zword(kb + 2);
            zb = zword(kb + 3);
            convert(kb, zcur_a);
            if (two) convert(kb + 1, zcur_b);
            // the TMEM stores land before the MMA thread is told the stages are ready
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(aready(kb));
        }
      }
    } else {
        // ---------------------------------------------------------- epilogue
        const int quarter = warp & 3, half = (warp - EPI_WARP0) >> 2;
        const int r = quarter * 32 + lane;
        const int nrow = n0 + r;
        const bool rv = nrow < n;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.f;
        bool ok = true;
        float sc_next = UX ? 1.f : ((rv && ngroups > 0) ? __half2float(__ushort_as_half(scales[nrow])) : 0.f);
        for (int g = 0; g < ngroups; ++g) {
            const int b = g & 1;
            const float sc = sc_next;  // uintx: 1 (y = P exactly)
            if (UX == 0 && g + 1 < ngroups && rv)
                sc_next = __half2float(__ushort_as_half(scales[(size_t)(g + 1) * n + nrow]));
            if (!warp_wait(tfull(b), (uint32_t)(g >> 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t col = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * BT + half * 64);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[16];
                tc_ld16(col + c * 16, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[c * 16 + i] = __fmaf_rn(v[i], sc, acc[c * 16 + i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(b));
        }
        if (ok && rv) {
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int t = t0 + half * 64 + i;
                if (t < m) {
                    if (BF16OUT)
                        reinterpret_cast<uint16_t*>(out)[(size_t)t * n + nrow] = (uint16_t)wq::f_to_bf(acc[i]);
                    else
                        reinterpret_cast<float*>(out)[(size_t)t * n + nrow] = acc[i];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == TMA_WARP) {
        tc_fence_after();
        tc_dealloc(tmem, TMEM_COLS);
    }
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
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

template <bool SYM, bool BF16OUT, int G, int UX>
wq_status launch(const uint16_t* x, int64_t m, const int32_t* qweight, const int32_t* qzeros,
                 const uint16_t* scales, int64_t n, int64_t k, void* out, cudaStream_t st,
                 const uint8_t* ux_packed = nullptr, const uint8_t* ux_zp = nullptr, int ux_group = 0) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
    if (!enc) return wqh::cuda_status(cudaErrorNotSupported);
    CUtensorMap xmap, qmap;
    {
        // x [m, k] bf16: boxes of 128 tokens x 64 values, 128-byte swizzle, zeros outside
        const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)m};
        const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
        const cuuint32_t box[2] = {BK, BT};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return WQ_ERR_BAD_SHAPE;
    }
    if (UX == 0) {
        // qweight [k/8, n] int32: boxes of 8 rows x 128 features, unswizzled, zeros outside
        const cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)(k / 8)};
        const cuuint64_t strides[1] = {(cuuint64_t)n * 4};
        const cuuint32_t box[2] = {BM, BK / 8};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(qweight), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return WQ_ERR_BAD_SHAPE;
    } else {
        qmap = xmap;  // not read by the uintx kernels
    }
    const void* fn = (const void*)gptq_gemm_kernel<SYM, BF16OUT, G, UX>;
    static bool attr_set = false;
    if (!attr_set) {
        const wq_status s =
            wqh::cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
        if (s != WQ_OK) return s;
        attr_set = true;
    }
    const dim3 grid((unsigned)(((n + BM - 1) / BM) * ((m + BT - 1) / BT)));
    gptq_gemm_kernel<SYM, BF16OUT, G, UX><<<grid, THREADS, SMEM, st>>>(
        xmap, qmap, qzeros, scales, (int)m, (int)n, (int)k, out, ux_packed, ux_zp, ux_group,
        g_mma_slices.load());
    return wqh::check_launch();
}

template <int G>
wq_status dispatch_rule(bool sym, bool bf, const uint16_t* x, int64_t m, const int32_t* qweight,
                        const int32_t* qzeros, const uint16_t* scales, int64_t n, int64_t k, void* out,
                        cudaStream_t st) {
    if (sym)
        return bf ? launch<true, true, G, 0>(x, m, qweight, qzeros, scales, n, k, out, st)
                  : launch<true, false, G, 0>(x, m, qweight, qzeros, scales, n, k, out, st);
    return bf ? launch<false, true, G, 0>(x, m, qweight, qzeros, scales, n, k, out, st)
              : launch<false, false, G, 0>(x, m, qweight, qzeros, scales, n, k, out, st);
}

template <int UX>
wq_status launch_ux(bool bf, const uint16_t* x, int64_t m, const uint8_t* packed, const uint16_t* scale,
                    const uint8_t* zp, int64_t n, int64_t k, int group, void* out, cudaStream_t st) {
    return bf ? launch<false, true, 64, UX>(x, m, nullptr, nullptr, scale, n, k, out, st, packed, zp, group)
              : launch<false, false, 64, UX>(x, m, nullptr, nullptr, scale, n, k, out, st, packed, zp, group);
}

wq_status dispatch_g(int group, bool sym, bool bf, const uint16_t* x, int64_t m, const int32_t* qweight,
                     const int32_t* qzeros, const uint16_t* scales, int64_t n, int64_t k, void* out,
                     cudaStream_t st) {
    switch (group) {
        case 32: return dispatch_rule<32>(sym, bf, x, m, qweight, qzeros, scales, n, k, out, st);
        case 64: return dispatch_rule<64>(sym, bf, x, m, qweight, qzeros, scales, n, k, out, st);
        case 128: return dispatch_rule<128>(sym, bf, x, m, qweight, qzeros, scales, n, k, out, st);
        default: return dispatch_rule<256>(sym, bf, x, m, qweight, qzeros, scales, n, k, out, st);
    }
}

}  // namespace

namespace wqh {
unsigned gemm_mma_slices_exchange(unsigned slices) { return g_mma_slices.exchange(slices); }

// Read and clear this file's device status word (0 when no wait ran out).
unsigned gemm_status_take() {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (v != 0) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(zero)) != cudaSuccess) cudaGetLastError();
    }
    return v;
}
}  // namespace wqh

extern "C" {

wq_status gptq_gemm(const uint16_t* x, int64_t m, const int32_t* qweight, const int32_t* qzeros,
                    const uint16_t* scales, int64_t n, int64_t k, int group, int sym, int out_dtype,
                    void* out, void* stream) {
    if (m < 0 || n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (group != 32 && group != 64 && group != 128 && group != 256) return WQ_ERR_UNSUPPORTED;
    if (k % group != 0 || n % 8 != 0) return WQ_ERR_BAD_SHAPE;
    if (m >= (1ll << 31) || n >= (1ll << 31) || k >= (1ll << 31) ||
        ((n + BM - 1) / BM) * ((m + BT - 1) / BT) >= (1ll << 31))
        return WQ_ERR_BAD_SHAPE;
    if (out_dtype != WQ_DTYPE_F32 && out_dtype != WQ_DTYPE_BF16) return WQ_ERR_BAD_DTYPE;
    if (m == 0 || n == 0) return WQ_OK;
    if (!out) return WQ_ERR_NULL_PTR;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (k == 0)  // an empty sum: y = 0
        return wqh::cuda_status(
            cudaMemsetAsync(out, 0, (size_t)(m * n) * (out_dtype == WQ_DTYPE_BF16 ? 2 : 4), st));
    if (!x || !qweight || !scales || (!sym && !qzeros)) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(x) || !wqh::aligned16(qweight) || !wqh::aligned_to(scales, 2) ||
        (!sym && !wqh::aligned_to(qzeros, 4)) || !wqh::aligned_to(out, 4))
        return WQ_ERR_MISALIGNED;
    const bool bf = out_dtype == WQ_DTYPE_BF16;
    return dispatch_g(group, sym != 0, bf, x, m, qweight, qzeros, scales, n, k, out, st);
}

wq_status uintx_gemm(const uint16_t* x, int64_t m, const uint8_t* packed, const uint16_t* scale,
                     const uint8_t* zp, int64_t n, int64_t k, int nbits, int group, int out_dtype, void* out,
                     void* stream) {
    if (m < 0 || n < 0 || k < 0) return WQ_ERR_BAD_SHAPE;
    if (nbits < 2 || nbits > 7) return WQ_ERR_UNSUPPORTED;
    if (group != 32 && group != 64 && group != 128 && group != 256) return WQ_ERR_UNSUPPORTED;
    if (k % group != 0) return WQ_ERR_BAD_SHAPE;
    if (k % 64 != 0) return WQ_ERR_UNSUPPORTED;
    if (m >= (1ll << 31) || n >= (1ll << 31) || k >= (1ll << 31) ||
        ((n + BM - 1) / BM) * ((m + BT - 1) / BT) >= (1ll << 31))
        return WQ_ERR_BAD_SHAPE;
    if (out_dtype != WQ_DTYPE_F32 && out_dtype != WQ_DTYPE_BF16) return WQ_ERR_BAD_DTYPE;
    if (m == 0 || n == 0) return WQ_OK;
    if (!out) return WQ_ERR_NULL_PTR;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (k == 0)  // an empty sum: y = 0
        return wqh::cuda_status(
            cudaMemsetAsync(out, 0, (size_t)(m * n) * (out_dtype == WQ_DTYPE_BF16 ? 2 : 4), st));
    if (!x || !packed || !scale || !zp) return WQ_ERR_NULL_PTR;
    if (!wqh::aligned16(x) || !wqh::aligned16(packed) || !wqh::aligned_to(scale, 2) ||
        !wqh::aligned_to(out, 4))
        return WQ_ERR_MISALIGNED;
    const bool bf = out_dtype == WQ_DTYPE_BF16;
    switch (nbits) {
        case 2: return launch_ux<2>(bf, x, m, packed, scale, zp, n, k, group, out, st);
        case 3: return launch_ux<3>(bf, x, m, packed, scale, zp, n, k, group, out, st);
        case 4: return launch_ux<4>(bf, x, m, packed, scale, zp, n, k, group, out, st);
        case 5: return launch_ux<5>(bf, x, m, packed, scale, zp, n, k, group, out, st);
        case 6: return launch_ux<6>(bf, x, m, packed, scale, zp, n, k, group, out, st);
        default: return launch_ux<7>(bf, x, m, packed, scale, zp, n, k, group, out, st);
    }
}

}  // extern "C"
