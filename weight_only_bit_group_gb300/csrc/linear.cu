// linear.cu -- the consumer of an exported GPTQ checkpoint, for decode batches:
// y = x deq(W)^T straight from the packed int4 weights (export_gptq_cpu.py,
// module docstring: the checkpoint is served by vLLM's W4A16 uint4b8 layer,
// which reads qweight [K/8, N], scales [K/G, N] and qzeros [K/G, N/8]).
//
// Only the codes (0.5 B per weight) and the group scale / zero point are read,
// a quarter of the bytes of a bf16 weight, so for m = 1 the kernel is HBM bound.
//
// Grid: ceil(N/128) column blocks x S slices along K.  A CTA is 4 warps over the
// same 128 output columns; lane = 4 adjacent columns, so one 16-byte piece of a
// qweight row holds the 8 codes of each of its 4 columns.  Each warp walks
// `batches` batches of 8 qweight rows (64 input channels) through a 3-stage
// cp.async pipeline of its own: the codes (16 bytes per lane and row) and the
// batch's x rows land in shared memory two batches ahead of their use, so
// the loads stream while earlier batches are computed.  The group scales and
// zero points of the next batch are read into registers one batch ahead.
// Per qweight word the 8 codes become bf16 128 + c by byte permutes (two codes
// per permute); subtracting 128 + zp in bf16x2 gives the exact c - zp; mixed
// bf16 x bf16 -> binary32 FMAs multiply by x (read in place from its bf16
// pairs) and add into two binary32 sums per column and token (even and odd
// input channels): every product is exact and every addition rounds once.  The
// group sum times the fp16 scale is added to the column's sum.  The 4 warps'
// sums meet in shared memory and are added in warp order; each CTA writes its
// slice's partial to a workspace slot per (slice, row, column); the last CTA of
// a column block to finish adds the S slices in order (deterministic, no
// waiting), writes y and sets the block's arrival counter back to zero, so that
// a call needs no separate reset of the workspace.
#include "wq_common.cuh"

namespace {

constexpr int kThreads = 128;   // 4 warps
constexpr int kCols = 128;      // output columns per CTA (4 per lane)
constexpr int kRPW = 8;         // qweight rows per warp batch
constexpr int kNST = 3;         // pipeline stages per warp
constexpr int kMaxSlices = 64;
constexpr int kMaxM = 8;

template <int M>
struct LinSmem {
    static constexpr int W = kRPW * 32 * 16;  // codes of one stage: [row][lane] 16 bytes
    static constexpr int X = kRPW * M * 16;   // x of one stage: [token][row] 8 bf16
    static constexpr int STAGE = W + X;
    static constexpr int WARP = kNST * STAGE;
    static constexpr int CTA = 4 * WARP;
};

// acc_e += sum of c_{2i} x_{2i}, acc_o += sum of c_{2i+1} x_{2i+1} over the 8
// input channels of one word: d0 = (c0, c2), d1 = (c4, c6), d2 = (c1, c3),
// d3 = (c5, c7) as bf16x2 (c - zp, exact), xv the 8 bf16 x values in order.
__device__ __forceinline__ void dot8(uint32_t d0, uint32_t d1, uint32_t d2, uint32_t d3, uint4 xv,
                                     float& e, float& o) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1, c0, c1, f0, f1, x0, x1, x2, x3, x4, x5, x6, x7;\n\t"
        "mov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\tmov.b32 {c0, c1}, %4;\n\tmov.b32 {f0, f1}, %5;\n\t"
        "mov.b32 {x0, x1}, %6;\n\tmov.b32 {x2, x3}, %7;\n\tmov.b32 {x4, x5}, %8;\n\tmov.b32 {x6, x7}, %9;\n\t"
        "fma.rn.f32.bf16 %0, a0, x0, %0;\n\tfma.rn.f32.bf16 %0, a1, x2, %0;\n\t"
        "fma.rn.f32.bf16 %0, b0, x4, %0;\n\tfma.rn.f32.bf16 %0, b1, x6, %0;\n\t"
        "fma.rn.f32.bf16 %1, c0, x1, %1;\n\tfma.rn.f32.bf16 %1, c1, x3, %1;\n\t"
        "fma.rn.f32.bf16 %1, f0, x5, %1;\n\tfma.rn.f32.bf16 %1, f1, x7, %1;\n\t}"
        : "+f"(e), "+f"(o)
        : "r"(d0), "r"(d1), "r"(d2), "r"(d3), "r"(xv.x), "r"(xv.y), "r"(xv.z), "r"(xv.w));
}

template <bool SYM, int M, int G>
__global__ void __launch_bounds__(kThreads) gptq_linear_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ qweight,
    const int32_t* __restrict__ qzeros, const uint16_t* __restrict__ scales, int64_t n, int64_t k,
    int batches, float* __restrict__ part, unsigned* __restrict__ counters, int out_bf16,
    void* __restrict__ out) {
    using L = LinSmem<M>;
    constexpr int RPG = (G / 8) < kRPW ? (G / 8) : kRPW;  // rows of one group inside a batch
    constexpr int GPB = kRPW / RPG;                       // groups (or one group's part) per batch
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned char* wsm = smem + warp * L::WARP;
    const int64_t c0 = (int64_t)blockIdx.x * kCols + 4 * lane;
    const bool cv = c0 < n;  // n % 8 == 0: a lane's 4 columns are all valid or all not
    const int64_t rows = k / 8;
    const int S = gridDim.y;
    // first qweight row of batch bt of this warp (the CTA's 4 warps take
    // consecutive 8-row pieces of each 32-row step of the slice)
    auto rowof = [&](int bt) -> int64_t { return (((int64_t)blockIdx.y * batches + bt) * 4 + warp) * kRPW; };

    auto issue = [&](int bt) {
        if (bt < batches) {
            const int64_t r0 = rowof(bt);
            unsigned char* sw = wsm + (bt % kNST) * L::STAGE;
#pragma unroll
            for (int r = 0; r < kRPW; ++r)
                if (cv && r0 + r < rows) wq::cp_async16(sw + (r * 32 + lane) * 16, qweight + (r0 + r) * n + c0);
            for (int p = lane; p < kRPW * M; p += 32) {  // piece p: token p / 8, row p % 8
                const int m = p / kRPW, r = p % kRPW;
                if (r0 + r < rows) wq::cp_async16(sw + L::W + p * 16, x + m * k + (r0 + r) * 8);
            }
        }
        wq::cp_async_commit();  // every lane commits a group per batch, empty or not
    };
    // the group constants of a batch: 4 scales and the qzeros word of each group
    auto consts = [&](int bt, uint32_t (&sh)[GPB][4], uint32_t (&zw)[GPB]) {
        const int64_t r0 = rowof(bt);
#pragma unroll
        for (int gi = 0; gi < GPB; ++gi) {
            const bool gv = bt < batches && cv && r0 + gi * RPG < rows;
            const int64_t g = ((r0 + gi * RPG) * 8) / G;
#pragma unroll
            for (int j = 0; j < 4; ++j) sh[gi][j] = gv ? (uint32_t)__ldg(scales + g * n + c0 + j) : 0u;
            zw[gi] = (!SYM && gv) ? (uint32_t)__ldg(qzeros + g * (n / 8) + c0 / 8) : 0u;
        }
    };

    float acc[M][4];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[m][j] = 0.0f;

#pragma unroll
    for (int i = 0; i < kNST - 1; ++i) issue(i);
    uint32_t shn[GPB][4], zwn[GPB];
    consts(0, shn, zwn);
    for (int bt = 0; bt < batches; ++bt) {
        issue(bt + kNST - 1);
        uint32_t sh[GPB][4], zw[GPB];
#pragma unroll
        for (int gi = 0; gi < GPB; ++gi) {
            zw[gi] = zwn[gi];
#pragma unroll
            for (int j = 0; j < 4; ++j) sh[gi][j] = shn[gi][j];
        }
        consts(bt + 1, shn, zwn);
        wq::cp_async_wait<kNST - 1>();  // this lane's copies of batch bt have landed
        __syncwarp();                    // ... and every other lane's (the x pieces)
        const int64_t r0 = rowof(bt);
        const unsigned char* sw = wsm + (bt % kNST) * L::STAGE;
#pragma unroll
        for (int gi = 0; gi < GPB; ++gi) {
            uint32_t zb2[4];  // bf16x2 of 128 + zp, per column
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t zp = SYM ? 8u : (zw[gi] >> (4 * ((c0 + j) & 7))) & 15u;
                zb2[j] = (0x4300u + zp) * 0x10001u;
            }
            float ge[M][4], go[M][4];
#pragma unroll
            for (int m = 0; m < M; ++m)
#pragma unroll
                for (int j = 0; j < 4; ++j) ge[m][j] = go[m][j] = 0.0f;
#pragma unroll
            for (int rr = 0; rr < RPG; ++rr) {
                const int r = gi * RPG + rr;
                if (r0 + r >= rows) break;  // uniform over the warp
                const uint4 wv = *reinterpret_cast<const uint4*>(sw + (r * 32 + lane) * 16);
                uint4 xv[M];
#pragma unroll
                for (int m = 0; m < M; ++m) xv[m] = *reinterpret_cast<const uint4*>(sw + L::W + (m * kRPW + r) * 16);
                const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // byte q of lo / hi: the codes of input channels 2q / 2q + 1
                    const uint32_t lo = wd[j] & 0x0F0F0F0Fu, hi = (wd[j] >> 4) & 0x0F0F0F0Fu;
                    // bytes c | 0x43 << 8 = bf16 of 128 + c; minus 128 + zp is exact
                    const uint32_t d0 = wq::bsub2(__byte_perm(lo, 0x43434343u, 0x4140), zb2[j]);
                    const uint32_t d1 = wq::bsub2(__byte_perm(lo, 0x43434343u, 0x4342), zb2[j]);
                    const uint32_t d2 = wq::bsub2(__byte_perm(hi, 0x43434343u, 0x4140), zb2[j]);
                    const uint32_t d3 = wq::bsub2(__byte_perm(hi, 0x43434343u, 0x4342), zb2[j]);
#pragma unroll
                    for (int m = 0; m < M; ++m) dot8(d0, d1, d2, d3, xv[m], ge[m][j], go[m][j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float sc = __half2float(__ushort_as_half((unsigned short)sh[gi][j]));
#pragma unroll
                for (int m = 0; m < M; ++m) acc[m][j] = __fmaf_rn(__fadd_rn(ge[m][j], go[m][j]), sc, acc[m][j]);
            }
        }
        __syncwarp();  // every lane is done with this stage before it is refilled
    }
    wq::cp_async_wait<0>();

    // the 4 warps' sums of each column, added in warp order
    __shared__ float red[4][M][kCols];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j) red[warp][m][4 * lane + j] = acc[m][j];
    __syncthreads();
    const int64_t col = (int64_t)blockIdx.x * kCols + threadIdx.x;
    const bool colv = col < n;
    if (colv) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float v = red[0][m][threadIdx.x];
#pragma unroll
            for (int w2 = 1; w2 < 4; ++w2) v = __fadd_rn(v, red[w2][m][threadIdx.x]);
            part[((int64_t)blockIdx.y * M + m) * n + col] = v;
        }
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
    using L = LinSmem<M>;
    const void* fn = (const void*)gptq_linear_kernel<SYM, M, G>;
    static bool attr_set = false;  // per process; the attribute is per function
    if (!attr_set) {
        const wq_status s =
            wqh::cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::CTA));
        if (s != WQ_OK) return s;
        attr_set = true;
    }
    const int64_t col_blocks = (n + kCols - 1) / kCols;
    const int64_t rows = k / 8;
    const int64_t nbw = (rows + kRPW - 1) / kRPW;  // 8-row warp batches per column block
    // one wave: about as many CTAs as fit on the GPU at once, each warp walking
    // several batches through its pipeline (and never more slices than the
    // kMaxSlices the workspace holds)
    const int64_t resident = wqh::grid_for(fn, kThreads, L::CTA, (int64_t)1 << 30, 1 << 30);
    int64_t want = resident / col_blocks;
    if (want < 1) want = 1;
    if (want > kMaxSlices) want = kMaxSlices;
    const int64_t batches = (nbw + 4 * want - 1) / (4 * want);
    const int64_t S = (nbw + 4 * batches - 1) / (4 * batches);
    if (S < 1 || batches >= (1ll << 31) || col_blocks >= (1ll << 31)) return WQ_ERR_BAD_SHAPE;
    // arrival counters: zero before the first call (the caller zeroes the
    // workspace once), reset to zero by the last CTA of every column block
    unsigned* counters = reinterpret_cast<unsigned*>(ws);
    float* part = reinterpret_cast<float*>(ws + ((col_blocks * 4 + 255) & ~(int64_t)255));
    gptq_linear_kernel<SYM, M, G><<<dim3((unsigned)col_blocks, (unsigned)S), kThreads, L::CTA, st>>>(
        x, qweight, qzeros, scales, n, k, (int)batches, part, counters, out_bf16, out);
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
    if (!wqh::aligned16(x) || !wqh::aligned16(qweight) || !wqh::aligned_to(scales, 2) ||
        (!sym && !wqh::aligned_to(qzeros, 4)) || !wqh::aligned_to(out, 4) ||
        !wqh::aligned_to(workspace, 256))
        return WQ_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    char* ws = (char*)workspace;
    const int ob = out_dtype == WQ_DTYPE_BF16;
    return sym ? dispatch_g<true>(group, m, x, qweight, qzeros, scales, n, k, ob, out, ws, st)
               : dispatch_g<false>(group, m, x, qweight, qzeros, scales, n, k, ob, out, ws, st);
}
