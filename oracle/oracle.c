/*
 * oracle.c -- plain, slow CPU oracle for group-wise low-bit weight quantization.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check in
 * __graft_entry__ and the CPU-baseline leg of bench.py may load this library.  It
 * shares no source, header, table or helper with the CUDA library; the two meet
 * only through byte buffers produced by the seeded input generators.
 *
 * Every floating-point operation below is ONE IEEE-754 operation (binary32 unless
 * stated), rounded to nearest-even and never fused: the file is built with
 * -ffp-contract=off -fno-fast-math.  bf16 and fp16 roundings are written out by
 * hand (orc_f32_to_bf16, orc_f32_to_f16) and pinned against independent library
 * conversions in the tests.
 *
 * Sources, cited by page title and the function / docstring on that page:
 *   [GPTQ] export_gptq_cpu.py         -- pack_int32, quantize_sym, quantize_asym,
 *                                        the module docstring (uint4b8 dequant rule)
 *   [MX]   quantize_dflash_mxfp4.py   -- E2M1 table, quantize_mxfp4,
 *                                        dequantize_mxfp4, search_scale, the
 *                                        relative-error report in main()
 *   [UX]   uintx_quant.py             -- module docstring, _pack_shard,
 *                                        _unpack_shard, pack_uintx, unpack_uintx,
 *                                        UIntXQuantizer._quantize_impl and
 *                                        UIntXQuantizer._dequantize_native
 *
 * Readings taken where a page is silent or ambiguous (each one is listed in the
 * design notes and pinned by a test):
 *   - MXFP4 block exponent: floor(log2(amax)) is taken as the exact binary
 *     exponent of amax (frexp).  For every bf16 amax this equals what a log2
 *     evaluation gives; for fp32 amax just below a power of two a rounded log2
 *     would overshoot by one.
 *   - MXFP4 ties: mode 0 (round-half-even) sends an exact midpoint to the even
 *     e2m1 index of its two neighbours; mode 1 reproduces the page's literal
 *     "(argmin // 2) * 2" tie rewrite byte for byte.
 *   - AWQ scale preparation: sums run in binary64 in index order and are rounded
 *     once to binary32; pow/log/exp are evaluated in binary64 and rounded once to
 *     binary32 (see orc_awq_prepare_scales).
 *   - Reductions (SNR, AWQ error): binary32 terms, binary64 accumulation.
 *   - uintx: every bf16 operation is the binary32 operation on the bf16 operands
 *     followed by one round-to-nearest-even to bf16; divisions are true IEEE
 *     divisions; "1.0 / scale" is a bf16 reciprocal.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

/* ------------------------------------------------------------------------- */
/* scalar formats                                                             */
/* ------------------------------------------------------------------------- */

static float f_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the top half of a binary32. */
float orc_bf16_to_f32(uint16_t h) { return f_from_bits((uint32_t)h << 16); }

/* binary32 -> bf16, round to nearest, ties to even.  The 16 discarded bits decide:
 * above half -> up, below half -> down, exactly half -> up only if the kept
 * half is odd.  Rounding the magnitude up may carry into the exponent, which is
 * the correct result (including the carry from the largest finite value to inf). */
uint16_t orc_f32_to_bf16(float x) {
    uint32_t u = bits_of(x);
    if (isnan(x)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16, dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
    return (uint16_t)kept;
}

/* binary16 -> binary32 (exact). */
float orc_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return (float)(sign ? -v : v);
}

/* binary32 -> binary16, round to nearest, ties to even, with subnormals and
 * overflow to infinity.  Works on the magnitude in binary64, where every step
 * below is exact except the explicit nearbyint() (default mode: ties-to-even). */
uint16_t orc_f32_to_f16(float x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    if (isinf(x)) return (uint16_t)(sign | 0x7c00u);
    double a = fabs((double)x);
    if (a < 0x1p-14) {
        /* subnormal range: an integer multiple of 2^-24; 1024 * 2^-24 is the
         * smallest normal and encodes correctly as 0x0400. */
        double q = nearbyint(a * 0x1p24);
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    m *= 2.0;
    e -= 1; /* a = m * 2^e, m in [1, 2) */
    double frac = nearbyint((m - 1.0) * 1024.0);
    if (frac == 1024.0) { frac = 0.0; e += 1; }
    if (e > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)frac);
}

/* Round a binary32 value to bf16 and return it as binary32: one "bf16 op". */
static float bf(float x) { return orc_bf16_to_f32(orc_f32_to_bf16(x)); }

/* torch.round / rint: round half to even (default rounding mode). */
static float rne(float x) { return nearbyintf(x); }

static float clampf(float x, float lo, float hi) { return fminf(fmaxf(x, lo), hi); }

/* ------------------------------------------------------------------------- */
/* [GPTQ] export_gptq_cpu.py                                                  */
/* ------------------------------------------------------------------------- */

/* pack_int32: 8 nibbles per int32, low-order nibble first.  codes is [k, n]
 * row-major.  dim 0 packs along k giving [k/8, n]; dim 1 packs along n giving
 * [k, n/8]. */
void orc_pack_int32(const int32_t* codes, int64_t k, int64_t n, int dim, int32_t* out) {
    if (dim == 0) {
        for (int64_t r = 0; r < k / 8; ++r)
            for (int64_t c = 0; c < n; ++c) {
                uint32_t word = 0;
                for (int i = 0; i < 8; ++i)
                    word |= ((uint32_t)codes[(8 * r + i) * n + c] & 0xfu) << (4 * i);
                out[r * n + c] = (int32_t)word;
            }
    } else {
        for (int64_t r = 0; r < k; ++r)
            for (int64_t c = 0; c < n / 8; ++c) {
                uint32_t word = 0;
                for (int i = 0; i < 8; ++i)
                    word |= ((uint32_t)codes[r * n + 8 * c + i] & 0xfu) << (4 * i);
                out[r * (n / 8) + c] = (int32_t)word;
            }
    }
}

/* Reconstruction SNR as the GPTQ page reports it:
 * 20*log10(||w|| / max(||w - deq||, 1e-12)); binary32 terms, binary64 sums. */
static double snr_from_sums(double sw, double se) {
    double nw = sqrt(sw), ne = sqrt(se);
    return 20.0 * log10(nw / fmax(ne, 1e-12));
}

/* quantize_sym / quantize_asym.  w is bf16 [n, k] (a torch Linear weight).
 * The page transposes to wt = w.float().t() ([k, n]) and views it as
 * [k/group, group, n]; the statistics run over the middle axis.
 *   sym : amax = max|x|, scale = max(amax / 8, 1e-9),
 *         code = clamp(round(x/scale) + 8, 0, 15), deq = (code - 8) * scale,
 *         qzeros = pack(all 7, along n)
 *   asym: scale = max(wmax - wmin, 1e-9) / 15, zp = clamp(round(-wmin/scale), 0, 15),
 *         code = clamp(round(x/scale) + zp, 0, 15), deq = (code - zp) * scale,
 *         qzeros = pack(zp, along n) -- the zero point itself, no "-1"
 * Outputs: qweight int32 [k/8, n], qzeros int32 [k/group, n/8], scales fp16
 * [k/group, n], g_idx int32 [k] = kk // group, snr_db (binary64, from the binary32
 * deq before the fp16 rounding of the scales).  Any output pointer may be NULL. */
/* quantize_sym / quantize_asym on a binary32 [n, k] weight: the page first
 * takes w.float(), so every input type reaches this arithmetic as binary32. */
void orc_gptq_quantize_f32(const float* w, int64_t n, int64_t k, int group, int sym,
                           int32_t* qweight, int32_t* qzeros, uint16_t* scales,
                           int32_t* g_idx, double* snr_db) {
    int64_t g = k / group;
    float* wt = (float*)malloc(sizeof(float) * (size_t)(k * n));
    int32_t* codes = (int32_t*)malloc(sizeof(int32_t) * (size_t)(k * n));
    float* deq = (float*)malloc(sizeof(float) * (size_t)(k * n));
    float* scale = (float*)malloc(sizeof(float) * (size_t)(g * n));
    int32_t* zp = (int32_t*)malloc(sizeof(int32_t) * (size_t)(g * n));

    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < k; ++c) wt[c * n + r] = w[r * k + c];

    for (int64_t gi = 0; gi < g; ++gi) {
        for (int64_t col = 0; col < n; ++col) {
            float s, z;
            if (sym) {
                float amax = 0.0f;
                for (int j = 0; j < group; ++j)
                    amax = fmaxf(amax, fabsf(wt[(gi * group + j) * n + col]));
                s = fmaxf(amax / 8.0f, 1e-9f);
                z = 8.0f;
            } else {
                float wmax = -INFINITY, wmin = INFINITY;
                for (int j = 0; j < group; ++j) {
                    float x = wt[(gi * group + j) * n + col];
                    wmax = fmaxf(wmax, x);
                    wmin = fminf(wmin, x);
                }
                s = fmaxf(wmax - wmin, 1e-9f) / 15.0f;
                z = clampf(rne(-wmin / s), 0.0f, 15.0f);
            }
            scale[gi * n + col] = s;
            zp[gi * n + col] = (int32_t)z;
            for (int j = 0; j < group; ++j) {
                int64_t idx = (gi * group + j) * n + col;
                float c = clampf(rne(wt[idx] / s) + z, 0.0f, 15.0f);
                codes[idx] = (int32_t)c;
                deq[idx] = (c - z) * s;
            }
        }
    }

    if (snr_db) {
        double sw = 0.0, se = 0.0;
        for (int64_t i = 0; i < k * n; ++i) {
            float x = wt[i], e = x - deq[i];
            sw += (double)(x * x);
            se += (double)(e * e);
        }
        *snr_db = snr_from_sums(sw, se);
    }
    if (qweight) orc_pack_int32(codes, k, n, 0, qweight);
    if (qzeros) {
        int32_t* zfill = (int32_t*)malloc(sizeof(int32_t) * (size_t)(g * n));
        for (int64_t i = 0; i < g * n; ++i) zfill[i] = sym ? 7 : zp[i];
        orc_pack_int32(zfill, g, n, 1, qzeros);
        free(zfill);
    }
    if (scales)
        for (int64_t i = 0; i < g * n; ++i) scales[i] = orc_f32_to_f16(scale[i]);
    if (g_idx)
        for (int64_t c = 0; c < k; ++c) g_idx[c] = (int32_t)(c / group);

    free(wt); free(codes); free(deq); free(scale); free(zp);
}

/* Dequantize stored GPTQ tensors (the rule the module docstring states for
 * uint4b8: w = (code - 8) * scale; with real zero points w = (code - zp) * scale;
 * the scale is the stored fp16 value).  Output binary32, layout [k, n] when
 * out_kn != 0 (the page's deq layout) else [n, k] (the original weight layout). */
/* The bf16 weight widened exactly to binary32, then the binary32 path. */
void orc_gptq_quantize(const uint16_t* w, int64_t n, int64_t k, int group, int sym,
                       int32_t* qweight, int32_t* qzeros, uint16_t* scales,
                       int32_t* g_idx, double* snr_db) {
    float* wf = (float*)malloc(sizeof(float) * (size_t)(k * n));
    for (int64_t i = 0; i < n * k; ++i) wf[i] = orc_bf16_to_f32(w[i]);
    orc_gptq_quantize_f32(wf, n, k, group, sym, qweight, qzeros, scales, g_idx, snr_db);
    free(wf);
}

void orc_gptq_dequantize(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                         int64_t n, int64_t k, int group, int sym, int out_kn, float* out) {
    for (int64_t kk = 0; kk < k; ++kk) {
        int64_t gi = kk / group;
        for (int64_t col = 0; col < n; ++col) {
            uint32_t word = (uint32_t)qweight[(kk / 8) * n + col];
            int code = (int)((word >> (4 * (kk % 8))) & 0xfu);
            int z;
            if (sym) z = 8;
            else {
                uint32_t zw = (uint32_t)qzeros[gi * (n / 8) + col / 8];
                z = (int)((zw >> (4 * (col % 8))) & 0xfu);
            }
            float s = orc_f16_to_f32(scales[gi * n + col]);
            float v = (float)(code - z) * s;
            if (out_kn) out[kk * n + col] = v;
            else out[col * k + kk] = v;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* [MX] quantize_dflash_mxfp4.py                                              */
/* ------------------------------------------------------------------------- */

/* e2m1 magnitudes in code order; the sign is bit 3 of the nibble. */
static const float E2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
#define MX_GROUP 32

/* floor(log2(a)) for finite a > 0, as the exact binary exponent. */
static int floor_log2(float a) {
    int e;
    (void)frexpf(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    return e - 1;
}

int orc_floor_log2(float a) { return floor_log2(a); }

/* One e2m1 code for a value already divided by the block scale:
 * sign from signbit(v); magnitude clamped to 6; nearest grid magnitude by
 * explicit distances, first minimum on equal distances; then the tie rule. */
int orc_e2m1_code(float v, int tie_mode) {
    int sign = signbit(v) ? 1 : 0;
    float mag = fminf(fabsf(v), 6.0f);
    float d[8];
    for (int i = 0; i < 8; ++i) d[i] = fabsf(mag - E2M1[i]);
    int code = 0;
    for (int i = 1; i < 8; ++i)
        if (d[i] < d[code]) code = i;
    int ties = 0;
    for (int i = 0; i < 8; ++i)
        if (d[i] == d[code]) ++ties;
    if (ties > 1) {
        if (tie_mode == ORC_TIE_PAGE_LITERAL) {
            code = (code / 2) * 2; /* the page's literal rewrite */
        } else if (code & 1) {
            code += 1; /* half-even: the tied pair is (code, code+1); take the even one */
        }
    }
    return code | (sign << 3);
}

/* quantize_mxfp4 on a binary32 [n, k] matrix, k % 32 == 0.
 * Per block of 32 along k: amax = max|x|; exp = floor(log2 amax) - 2 (0 when
 * amax == 0), clamped to [-127, 127]; v = x / 2^exp; code per orc_e2m1_code.
 * packed[n][j] = code[2j] | code[2j+1] << 4, e8m0[n][b] = exp + 127. */
void orc_mxfp4_quantize_f32(const float* w, int64_t n, int64_t k, int tie_mode,
                            uint8_t* packed, uint8_t* e8m0) {
    int64_t nb = k / MX_GROUP;
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* x = w + r * k + b * MX_GROUP;
            float amax = 0.0f;
            for (int j = 0; j < MX_GROUP; ++j) amax = fmaxf(amax, fabsf(x[j]));
            int ex = (amax > 0.0f) ? floor_log2(amax) - 2 : 0;
            if (ex < -127) ex = -127;
            if (ex > 127) ex = 127;
            float scale = ldexpf(1.0f, ex);
            int code[MX_GROUP];
            for (int j = 0; j < MX_GROUP; ++j) code[j] = orc_e2m1_code(x[j] / scale, tie_mode);
            for (int j = 0; j < MX_GROUP / 2; ++j)
                packed[r * (k / 2) + b * (MX_GROUP / 2) + j] =
                    (uint8_t)(code[2 * j] | (code[2 * j + 1] << 4));
            e8m0[r * nb + b] = (uint8_t)(ex + 127);
        }
    }
}

void orc_mxfp4_quantize(const uint16_t* w, int64_t n, int64_t k, int tie_mode,
                        uint8_t* packed, uint8_t* e8m0) {
    float* row = (float*)malloc(sizeof(float) * (size_t)k);
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t c = 0; c < k; ++c) row[c] = orc_bf16_to_f32(w[r * k + c]);
        orc_mxfp4_quantize_f32(row, 1, k, tie_mode, packed + r * (k / 2),
                               e8m0 + r * (k / MX_GROUP));
    }
    free(row);
}

/* dequantize_mxfp4: val = +-E2M1[code & 7] * 2^(e8m0 - 127), binary32 [n, k]. */
void orc_mxfp4_dequantize(const uint8_t* packed, const uint8_t* e8m0, int64_t n, int64_t k,
                          float* out) {
    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < k; ++c) {
            uint8_t byte = packed[r * (k / 2) + c / 2];
            int code = (c % 2 == 0) ? (byte & 0xf) : (byte >> 4);
            float mag = E2M1[code & 7];
            float val = (code & 8) ? -mag : mag;
            float scale = ldexpf(1.0f, (int)e8m0[r * (k / MX_GROUP) + c / MX_GROUP] - 127);
            out[r * k + c] = val * scale;
        }
}

/* search_scale, step 0: the per-alpha column scales.
 *   a_c = max(a, 1e-8); an = a_c / mean(a_c)
 *   t = clamp(an ^ alpha, 1e-2, 1e2); s = t / exp(mean(log t))
 * s_out is [n_alpha, k]; a_c_out (may be NULL) receives a_c. */
void orc_awq_prepare_scales(const float* a, int64_t k, const float* alphas, int n_alpha,
                            float* s_out, float* a_c_out) {
    float* a_c = (float*)malloc(sizeof(float) * (size_t)k);
    float* an = (float*)malloc(sizeof(float) * (size_t)k);
    double sum = 0.0;
    for (int64_t c = 0; c < k; ++c) {
        a_c[c] = fmaxf(a[c], 1e-8f);
        sum += (double)a_c[c];
    }
    float mean = (float)(sum / (double)k);
    for (int64_t c = 0; c < k; ++c) an[c] = a_c[c] / mean;
    for (int i = 0; i < n_alpha; ++i) {
        float* s = s_out + (int64_t)i * k;
        double lsum = 0.0;
        for (int64_t c = 0; c < k; ++c) {
            float t = (float)pow((double)an[c], (double)alphas[i]);
            t = clampf(t, 1e-2f, 1e2f);
            s[c] = t;
            lsum += (double)(float)log((double)t);
        }
        float lmean = (float)(lsum / (double)k);
        float gm = (float)exp((double)lmean);
        for (int64_t c = 0; c < k; ++c) s[c] = s[c] / gm;
    }
    if (a_c_out) memcpy(a_c_out, a_c, sizeof(float) * (size_t)k);
    free(a_c);
    free(an);
}

/* search_scale: AWQ alpha search against the diagonal surrogate
 * err(alpha) = sum((dequant(quant(W*s)) / s - W) * a_c)^2 over a strided row
 * subsample (rows 0, stride, 2*stride, ... with stride = max(1, n / max_rows),
 * first max_rows of them, when n > max_rows).  The first alpha with the strictly
 * smallest error wins.  Outputs: best_s [k], *best_idx, *best_alpha, errs [n_alpha]
 * (binary32 terms, binary64 sums). */
void orc_awq_search(const uint16_t* w, int64_t n, int64_t k, const float* a,
                    const float* alphas, int n_alpha, int max_rows, int tie_mode,
                    float* best_s, int32_t* best_idx, float* best_alpha, double* errs) {
    int64_t stride = 1, rows = n;
    if (n > max_rows) {
        stride = n / max_rows;
        if (stride < 1) stride = 1;
        rows = (n + stride - 1) / stride;
        if (rows > max_rows) rows = max_rows;
    }
    float* wsub = (float*)malloc(sizeof(float) * (size_t)(rows * k));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < k; ++c) wsub[r * k + c] = orc_bf16_to_f32(w[(r * stride) * k + c]);

    float* s_all = (float*)malloc(sizeof(float) * (size_t)(n_alpha * k));
    float* a_c = (float*)malloc(sizeof(float) * (size_t)k);
    orc_awq_prepare_scales(a, k, alphas, n_alpha, s_all, a_c);

    float* ws = (float*)malloc(sizeof(float) * (size_t)(rows * k));
    float* deq = (float*)malloc(sizeof(float) * (size_t)(rows * k));
    uint8_t* packed = (uint8_t*)malloc((size_t)(rows * k / 2));
    uint8_t* e8 = (uint8_t*)malloc((size_t)(rows * k / MX_GROUP));

    int bi = -1;
    double best = 0.0;
    for (int i = 0; i < n_alpha; ++i) {
        const float* s = s_all + (int64_t)i * k;
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < k; ++c) ws[r * k + c] = wsub[r * k + c] * s[c];
        orc_mxfp4_quantize_f32(ws, rows, k, tie_mode, packed, e8);
        orc_mxfp4_dequantize(packed, e8, rows, k, deq);
        double err = 0.0;
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < k; ++c) {
                float e = (deq[r * k + c] / s[c] - wsub[r * k + c]) * a_c[c];
                err += (double)(e * e);
            }
        if (errs) errs[i] = err;
        if (bi < 0 || err < best) { best = err; bi = i; }
    }
    if (best_s) memcpy(best_s, s_all + (int64_t)bi * k, sizeof(float) * (size_t)k);
    if (best_idx) *best_idx = bi;
    if (best_alpha) *best_alpha = alphas[bi];

    free(wsub); free(s_all); free(a_c); free(ws); free(deq); free(packed); free(e8);
}

/* Relative weight error as the MXFP4 page reports it: ||deq - w|| / ||w||,
 * and the GPTQ-style SNR of the same pair.  w is bf16 [n, k]; deq is binary32
 * (deq_bf16 == 0) or bf16, laid out [n, k] (deq_kn == 0) or [k, n]. */
void orc_quant_snr(const uint16_t* w, const void* deq, int deq_bf16, int deq_kn, int64_t n,
                   int64_t k, double* snr_db, double* rel_err) {
    double sw = 0.0, se = 0.0;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < k; ++c) {
            float x = orc_bf16_to_f32(w[r * k + c]);
            int64_t di = deq_kn ? c * n + r : r * k + c;
            float d = deq_bf16 ? orc_bf16_to_f32(((const uint16_t*)deq)[di]) : ((const float*)deq)[di];
            float e = x - d;
            sw += (double)(x * x);
            se += (double)(e * e);
        }
    if (snr_db) *snr_db = snr_from_sums(sw, se);
    if (rel_err) *rel_err = sqrt(se) / sqrt(sw);
}

/* The AWQ fold of quantize_dflash_mxfp4.py's main(): once search_scale has
 * chosen s, the weights are rewritten as (W.float() * s).to(bfloat16) (columns
 * of q/k/v, gate/up, the conv kernel projections, down), (norm.float() /
 * s).to(bfloat16) (the norm weights, a [1, k] case) and (up.float() /
 * s.unsqueeze(1)).to(bfloat16) (rows of up).  Each element: one binary32
 * multiply or IEEE division of the exact bf16 value by s, then one rounding to
 * bf16.  axis 0: s has k entries, one per column; axis 1: s has n entries, one
 * per row.  op 0: multiply; op 1: divide.  out may equal w. */
void orc_awq_fold(const uint16_t* w, int64_t n, int64_t k, const float* s, int axis, int op,
                  uint16_t* out) {
    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < k; ++c) {
            const float x = orc_bf16_to_f32(w[r * k + c]);
            const float sv = axis == 0 ? s[c] : s[r];
            const float y = op == 0 ? x * sv : x / sv;
            out[r * k + c] = orc_f32_to_bf16(y);
        }
}

/* ------------------------------------------------------------------------- */
/* [UX] uintx_quant.py                                                        */
/* ------------------------------------------------------------------------- */

int64_t orc_uintx_packed_bytes(int64_t numel, int nbits) {
    int64_t total = 0;
    for (int kb = 8; kb >= 1; kb /= 2)
        if (nbits & kb) {
            int vpb = 8 / kb;
            total += (numel + vpb - 1) / vpb;
        }
    return total;
}

/* pack_uintx / _pack_shard: the code bits are split into power-of-two shards,
 * widest first (8, 4, 2, 1 -- only those present in nbits); bits
 * [offset, offset + kb) of every code go to the kb-bit shard.  A kb-bit shard
 * holds vpb = 8/kb values per byte laid out as vpb contiguous chunks of
 * L = ceil(numel / vpb) values: byte i = sum_j chunk_j[i] << (j*kb), positions
 * past numel reading 0.  The shards are concatenated in that order. */
void orc_uintx_pack(const uint8_t* codes, int64_t numel, int nbits, uint8_t* out) {
    int64_t pos = 0;
    int offset = 0;
    for (int kb = 8; kb >= 1; kb /= 2) {
        if (!(nbits & kb)) continue;
        int vpb = 8 / kb;
        int64_t len = (numel + vpb - 1) / vpb;
        unsigned mask = (1u << kb) - 1u;
        for (int64_t i = 0; i < len; ++i) {
            unsigned byte = 0;
            for (int j = 0; j < vpb; ++j) {
                int64_t e = (int64_t)j * len + i;
                unsigned v = 0;
                if (e < numel) v = (kb == nbits) ? codes[e] : ((unsigned)codes[e] >> offset) & mask;
                byte |= v << (j * kb);
            }
            out[pos + i] = (uint8_t)byte;
        }
        pos += len;
        offset += kb;
    }
}

/* unpack_uintx / _unpack_shard: the inverse of orc_uintx_pack. */
void orc_uintx_unpack(const uint8_t* packed, int64_t numel, int nbits, uint8_t* codes) {
    memset(codes, 0, (size_t)numel);
    int64_t pos = 0;
    int offset = 0;
    for (int kb = 8; kb >= 1; kb /= 2) {
        if (!(nbits & kb)) continue;
        int vpb = 8 / kb;
        int64_t len = (numel + vpb - 1) / vpb;
        unsigned mask = (1u << kb) - 1u;
        for (int64_t e = 0; e < numel; ++e) {
            int64_t j = e / len, i = e % len;
            unsigned v = ((unsigned)packed[pos + i] >> (j * kb)) & mask;
            codes[e] = (uint8_t)(codes[e] | (v << offset));
        }
        pos += len;
        offset += kb;
    }
}

/* UIntXQuantizer._quantize_impl: affine, asymmetric, preserve_zero, per group of
 * `group` values along in_features, every step in bf16:
 *   mn, mx = group min, max; mn' = min(mn, 0); mx' = max(mx, 0)
 *   scale = (mx' - mn') / (qmax - qmin); scale = max(scale, fp32 eps)
 *   zp    = clamp(qmin - round(mn' / scale), qmin, qmax) -> int
 *   q     = clamp(round(w * (1.0 / scale)) + zp, qmin, qmax) -> uint8
 * then pack_uintx of the flattened row-major codes.  scale_out holds the bf16
 * scales [n, k/group], zp_out the uint8 zero points, codes_out (may be NULL) the
 * unpacked codes. */
/* uintx in the weight's own dtype (uintx_quant.py works in the weight dtype):
 * dt = 0 binary32, 1 bf16, 2 binary16.  Every op is the binary32 op on the
 * operands, rounded once to dt (identity for binary32). */
static float r_dt(float x, int dt) {
    if (dt == 1) return bf(x);
    if (dt == 2) return orc_f16_to_f32(orc_f32_to_f16(x));
    return x;
}
static float load_dt(const void* w, int64_t i, int dt) {
    if (dt == 1) return orc_bf16_to_f32(((const uint16_t*)w)[i]);
    if (dt == 2) return orc_f16_to_f32(((const uint16_t*)w)[i]);
    return ((const float*)w)[i];
}
static void store_dt(void* out, int64_t i, int dt, float v) {
    if (dt == 1) ((uint16_t*)out)[i] = orc_f32_to_bf16(v);
    else if (dt == 2) ((uint16_t*)out)[i] = orc_f32_to_f16(v);
    else ((float*)out)[i] = v;
}

/* UIntXQuantizer._quantize_impl + pack_uintx: per group of `group` values along
 * k, min/max extended to include 0, scale = (max_pos - min_neg) / qmax clamped
 * to float32 eps, zero point = clamp(qmin - round(min_neg / scale)), codes =
 * clamp(round(w * (1 / scale)) + zp); every op in dt. */
void orc_uintx_quantize_dt(const void* w, int dt, int64_t n, int64_t k, int nbits, int group,
                           uint8_t* packed, void* scale_out, uint8_t* zp_out, uint8_t* codes_out) {
    const int qmin = 0, qmax = (1 << nbits) - 1;
    const float eps = 0x1p-23f; /* torch.finfo(torch.float32).eps */
    int64_t groups = k / group;
    uint8_t* codes = (uint8_t*)malloc((size_t)(n * k));
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t gi = 0; gi < groups; ++gi) {
            const int64_t g0 = r * k + gi * group;
            float mn = INFINITY, mx = -INFINITY;
            for (int j = 0; j < group; ++j) {
                float x = load_dt(w, g0 + j, dt);
                mn = fminf(mn, x);
                mx = fmaxf(mx, x);
            }
            float mn_neg = fminf(mn, 0.0f), mx_pos = fmaxf(mx, 0.0f);
            float sc = r_dt(mx_pos - mn_neg, dt);
            sc = r_dt(sc / (float)(qmax - qmin), dt);
            sc = fmaxf(sc, eps); /* eps is exact in bf16, binary16 and binary32 */
            float ratio = r_dt(mn_neg / sc, dt);
            float zpf = r_dt((float)qmin - rne(ratio), dt);
            zpf = clampf(zpf, (float)qmin, (float)qmax);
            int zp = (int)zpf;
            float inv = r_dt(1.0f / sc, dt);
            for (int j = 0; j < group; ++j) {
                float x = load_dt(w, g0 + j, dt);
                float p = r_dt(x * inv, dt);
                float q = r_dt(rne(p) + (float)zp, dt);
                q = clampf(q, (float)qmin, (float)qmax);
                codes[g0 + j] = (uint8_t)q;
            }
            store_dt(scale_out, r * groups + gi, dt, sc);
            zp_out[r * groups + gi] = (uint8_t)zp;
        }
    }
    if (packed) orc_uintx_pack(codes, n * k, nbits, packed);
    if (codes_out) memcpy(codes_out, codes, (size_t)(n * k));
    free(codes);
}

void orc_uintx_quantize(const uint16_t* w, int64_t n, int64_t k, int nbits, int group,
                        uint8_t* packed, uint16_t* scale_out, uint8_t* zp_out,
                        uint8_t* codes_out) {
    orc_uintx_quantize_dt(w, 1, n, k, nbits, group, packed, scale_out, zp_out, codes_out);
}

/* _dequantize_native: (q - zp) then times the scale, both in dt. */
void orc_uintx_dequantize_dt(const uint8_t* packed, const void* scale, int dt, const uint8_t* zp,
                             int64_t n, int64_t k, int nbits, int group, void* out) {
    int64_t groups = k / group;
    uint8_t* codes = (uint8_t*)malloc((size_t)(n * k));
    orc_uintx_unpack(packed, n * k, nbits, codes);
    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < k; ++c) {
            int64_t gi = r * groups + c / group;
            float sc = load_dt(scale, gi, dt);
            float d = r_dt((float)codes[r * k + c] - (float)zp[gi], dt);
            d = r_dt(d * sc, dt);
            store_dt(out, r * k + c, dt, d);
        }
    free(codes);
}

void orc_uintx_dequantize(const uint8_t* packed, const uint16_t* scale, const uint8_t* zp,
                          int64_t n, int64_t k, int nbits, int group, uint16_t* out_bf16) {
    orc_uintx_dequantize_dt(packed, scale, 1, zp, n, k, nbits, group, out_bf16);
}
