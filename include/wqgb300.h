/*
 * wqgb300.h -- C ABI of libwqgb300.so: group-wise low-bit weight quantization
 * and its inverse on one NVIDIA GB300 (sm_103a).
 *
 * Formats (each restated from the page that defines it):
 *   GPTQ int4   -- export_gptq_cpu.py: pack_int32, quantize_sym, quantize_asym and
 *                  the module docstring (uint4b8: w = (code - 8) * scale).
 *   OCP MXFP4   -- quantize_dflash_mxfp4.py: E2M1 table, quantize_mxfp4,
 *                  dequantize_mxfp4, search_scale (AWQ alpha search).
 *   uintx       -- uintx_quant.py: module docstring, _pack_shard, pack_uintx,
 *                  unpack_uintx, UIntXQuantizer._quantize_impl, _dequantize_native.
 *   SNR / rel.  -- export_gptq_cpu.py quantize_* (snr) and the relative-error
 *                  report in quantize_dflash_mxfp4.py main().
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates or frees device memory.  Scratch space, where an operation
 *     needs it, is the caller's `workspace` of at least wq_workspace_bytes(...).
 *   - Matrices are dense row-major.  A weight is a torch Linear weight
 *     [n = out_features, k = in_features].  bf16 and fp16 values are passed as
 *     their 16-bit patterns (uint16_t).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     is asynchronous on that stream; results, including scalars such as snr_db,
 *     are written to device memory.
 *   - Return value: WQ_OK, or an argument error detected on the host before any
 *     launch (nothing is launched then), or WQ_ERR_CUDA when a launch failed
 *     (wq_last_cuda_error() gives the CUDA error string).  No exception crosses
 *     the ABI and nothing aborts the process.
 *   - n == 0 or k == 0 is a valid empty input: nothing is launched, WQ_OK.
 *   - Pointers to the main tensors must be 16-byte aligned (WQ_ERR_MISALIGNED
 *     otherwise); side tensors (scales, zero points, g_idx) need only their
 *     element alignment.
 *   - Inputs must be finite; results for NaN/Inf inputs are unspecified (the
 *     pages do not handle them either).
 *   - The library is safe to call from several host threads on different
 *     streams, provided their workspaces do not overlap.
 */
#ifndef WQGB300_H
#define WQGB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int wq_status;

#define WQ_OK 0
#define WQ_ERR_NULL_PTR 1
#define WQ_ERR_BAD_SHAPE 2
#define WQ_ERR_BAD_DTYPE 3
#define WQ_ERR_MISALIGNED 4
#define WQ_ERR_UNSUPPORTED 5
#define WQ_ERR_WORKSPACE_TOO_SMALL 6
#define WQ_ERR_CUDA 7
#define WQ_ERR_DEVICE_TIMEOUT 8 /* a bounded device-side wait ran out (see wq_device_status) */

/* Element types: outputs take F32 or BF16; weight inputs of gptq_quantize_ex
 * and mxfp4_quantize_ex also F16. */
#define WQ_DTYPE_F32 0
#define WQ_DTYPE_BF16 1
#define WQ_DTYPE_F16 2

/* Layout of a dequantized matrix. NK = [n, k] (the weight's own layout);
 * KN = [k, n] (the transposed layout the GPTQ page computes its deq in). */
#define WQ_LAYOUT_NK 0
#define WQ_LAYOUT_KN 1

/* MXFP4 rounding of exact e2m1 midpoints.
 * HALF_EVEN: the even e2m1 index of the two neighbours (0.25->0, 0.75->1,
 *   1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4) -- what the page's docstring,
 *   comment and quark config ("round_method": "half_even") state.
 * PAGE_LITERAL: the page's code as written, argmin (first of equal distances)
 *   then (argmin // 2) * 2 on ties: 0.75->0, 1.75->1, 3.5->2, others as above. */
#define WQ_TIE_HALF_EVEN 0
#define WQ_TIE_PAGE_LITERAL 1

/* Operations that take a workspace (first argument of wq_workspace_bytes). */
#define WQ_OP_GPTQ_QUANTIZE 0 /* arg = group; only needed when snr_db != NULL */
#define WQ_OP_QUANT_SNR 1     /* arg ignored */
#define WQ_OP_AWQ_SEARCH 2    /* arg = n_alpha */
#define WQ_OP_MXFP4_ERR 3     /* mxfp4_quantize_err; arg ignored */
#define WQ_OP_UINTX_ERR 4     /* uintx_quantize_err; arg = nbits (ignored) */

/* Human-readable name of a status code (static string). */
const char* wq_status_string(wq_status status);

/* Text of the CUDA error behind the last WQ_ERR_CUDA returned on this host
 * thread ("" if none). */
const char* wq_last_cuda_error(void);

/* Library version string. */
const char* wq_version(void);

/* Device-side status of the kernels that wait on hardware events (the GPTQ
 * quantize kernels wait on the mbarriers of their TMA loads; gptq_gemm also on
 * its dequant, MMA and epilogue hand-offs).  Every such wait
 * is bounded: one that runs out (a load that never lands) makes the kernel skip
 * the rest of its work and record WQ_ERR_DEVICE_TIMEOUT in a per-device status
 * word; the outputs of that call are then incomplete.  This call reads the word
 * of the current device and clears it: WQ_OK when no wait ran out since the last
 * call, WQ_ERR_DEVICE_TIMEOUT otherwise, or WQ_ERR_CUDA if the read failed.  It
 * is synchronous (a device-to-host copy on the legacy default stream): call it
 * after the streams that ran the kernels have been synchronised. */
wq_status wq_device_status(void);

/* Diagnostic: the budget of a class of bounded device-side waits, for launches
 * made after this call, process-wide; returns the previous budget (0xFFFFFFFF
 * and no change for an unknown site).  Pure host state: needs no GPU.
 *   WQ_WAIT_GPTQ_STAGE  polls of each wait of gptq_quantize_sym / _asym (bf16
 *                       weights) on the mbarrier of a TMA load; default 2^22.
 *   WQ_WAIT_GEMM_MMA    slices of 64 polls of each wait of the MMA-issuing
 *                       thread of gptq_gemm / uintx_gemm; default 512.
 * The defaults are far beyond any latency.  A budget of 0 makes every such wait
 * give up at once, which runs the kernel's timeout path without any fault: it
 * stops its work, lets the copies and MMAs it already issued complete (those
 * drains keep their own budgets), frees what it holds and records
 * WQ_ERR_DEVICE_TIMEOUT for wq_device_status; the outputs of that call are then
 * incomplete.  Meant for testing that path; restore the returned value after. */
#define WQ_WAIT_GPTQ_STAGE 0
#define WQ_WAIT_GEMM_MMA 1
unsigned wq_set_wait_budget(int site, unsigned budget);

/* Bytes of workspace `op` needs for an [n, k] weight (0 if none).  Pure host
 * arithmetic: needs no GPU. */
size_t wq_workspace_bytes(int op, int64_t n, int64_t k, int arg);

/* ---------------------------------------------------------------- GPTQ int4
 * gptq_quantize_sym  (export_gptq_cpu.py, quantize_sym)
 * gptq_quantize_asym (export_gptq_cpu.py, quantize_asym)
 *
 * In:  w        bf16 [n, k], 16-byte aligned.
 *      group    group size along k: 32, 64, 128 (the page's default) or 256;
 *               k % group == 0, n % 8 == 0 (qzeros packs 8 columns per int32).
 * Out: qweight  int32 [k/8, n]: word (r, c) holds the codes of w[c][8r .. 8r+7],
 *               code of w[c][8r+i] in bits 4i..4i+3 (low nibble first).
 *      qzeros   int32 [k/group, n/8] (may be NULL): sym stores 7 in every nibble
 *               (the classic zp - 1 convention); asym packs the zero point zp
 *               itself of columns 8c'..8c'+7, low nibble first (no "-1").
 *      scales   fp16 [k/group, n] (bit patterns), round-to-nearest-even of the
 *               binary32 scale.
 *      g_idx    int32 [k] = kk / group (may be NULL).
 *      snr_db   (may be NULL) one double: 20*log10(||w|| / max(||w - deq||, 1e-12))
 *               over the whole tensor, deq = (code - zp) * binary32 scale.  Needs
 *               workspace >= wq_workspace_bytes(WQ_OP_GPTQ_QUANTIZE, n, k, group).
 * Math per (group g, column c), binary32 IEEE, round half to even:
 *   sym : scale = max(amax / 8, 1e-9), code = clamp(round(x / scale) + 8, 0, 15)
 *   asym: scale = max(wmax - wmin, 1e-9) / 15, zp = clamp(round(-wmin/scale), 0, 15),
 *         code = clamp(round(x / scale) + zp, 0, 15)
 * Bit-exact with a true IEEE division (the kernel uses a correctly rounded
 * reciprocal plus one FMA correction step).  n and k must be below 2^31 (the
 * kernel loads w through a TMA tensor map with 32-bit coordinates).  Device
 * status: see wq_device_status. */
wq_status gptq_quantize_sym(const uint16_t* w, int64_t n, int64_t k, int group, int32_t* qweight,
                            int32_t* qzeros, uint16_t* scales, int32_t* g_idx, double* snr_db,
                            void* workspace, size_t workspace_bytes, void* stream);
wq_status gptq_quantize_asym(const uint16_t* w, int64_t n, int64_t k, int group, int32_t* qweight,
                             int32_t* qzeros, uint16_t* scales, int32_t* g_idx, double* snr_db,
                             void* workspace, size_t workspace_bytes, void* stream);

/* gptq_quantize_ex (export_gptq_cpu.py quantize_sym / quantize_asym, which start
 * from w.float()) -- the same outputs, workspace and rules as gptq_quantize_sym /
 * _asym (sym selects), for a weight of type w_dtype: WQ_DTYPE_BF16 calls those
 * entry points; WQ_DTYPE_F16 and WQ_DTYPE_F32 take the binary32 arithmetic on
 * the exactly widened values (IEEE divisions, round half to even, the SNR from
 * binary32 squares with compensated sums).  w 16-byte aligned; other inputs
 * WQ_ERR_BAD_DTYPE. */
wq_status gptq_quantize_ex(const void* w, int w_dtype, int64_t n, int64_t k, int group, int sym,
                           int32_t* qweight, int32_t* qzeros, uint16_t* scales, int32_t* g_idx,
                           double* snr_db, void* workspace, size_t workspace_bytes, void* stream);

/* gptq_dequantize (export_gptq_cpu.py module docstring: uint4b8 w = (code-8)*scale;
 * with real zero points w = (code - zp) * scale).
 * In:  qweight, qzeros (ignored when sym != 0, may be NULL then), scales as
 *      produced above; sym selects the rule.
 * Out: out  [n, k] (out_layout WQ_LAYOUT_NK) or [k, n] (WQ_LAYOUT_KN), element
 *      type out_dtype (WQ_DTYPE_F32: exact; WQ_DTYPE_BF16: round to nearest even
 *      of the exact value), 16-byte aligned. */
wq_status gptq_dequantize(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                          int64_t n, int64_t k, int group, int sym, int out_dtype, int out_layout,
                          void* out, void* stream);

/* ---------------------------------------------------------------- OCP MXFP4
 * mxfp4_quantize (quantize_dflash_mxfp4.py, quantize_mxfp4)
 * In:  w bf16 [n, k], k % 32 == 0, 16-byte aligned; tie_mode WQ_TIE_*.
 * Out: packed  u8 [n, k/2]: byte j = code[2j] | code[2j+1] << 4, code = sign << 3 |
 *              e2m1 magnitude index (0, .5, 1, 1.5, 2, 3, 4, 6).
 *      e8m0    u8 [n, k/32] = exp + 127, exp = clamp(floor(log2 amax) - 2, -127,
 *              127) (exp = 0 for an all-zero block).  floor(log2) is the exact
 *              binary exponent.
 * Each value v = w / 2^exp, magnitude clamped at 6, nearest grid magnitude,
 * sign = signbit(v) (so -0.0 codes as 8). */
wq_status mxfp4_quantize(const uint16_t* w, int64_t n, int64_t k, int tie_mode, uint8_t* packed,
                         uint8_t* e8m0, void* stream);

/* mxfp4_quantize_err (quantize_dflash_mxfp4.py: quantize_mxfp4, then main()'s
 * relative-error report of the quantized target, rel = ||deq - w|| / ||w|| with
 * deq as dequantize_mxfp4 returns it) -- mxfp4_quantize plus the reconstruction
 * error of the same pass: the kernel decodes its own codes on-chip, so w is read
 * once and no dequantized tensor is written.
 * In/Out: as mxfp4_quantize (bf16 w), and
 *      snr_db, rel_err  one double each on the device (either may be NULL; both
 *               NULL is plain mxfp4_quantize): over the whole tensor, Sw = sum w^2,
 *               Se = sum (w - deq)^2 with binary32 terms, snr_db = 20*log10(
 *               sqrt(Sw) / max(sqrt(Se), 1e-12)), rel_err = sqrt(Se) / sqrt(Sw);
 *               the same definitions as quant_snr, within 1e-4 relative of
 *               binary64 sums of the same terms.
 *      workspace  >= wq_workspace_bytes(WQ_OP_MXFP4_ERR, n, k, 0), 16-byte
 *               aligned; calls that overlap on the GPU need separate workspaces.
 * n == 0 or k == 0 launches nothing and leaves snr_db / rel_err unwritten. */
wq_status mxfp4_quantize_err(const uint16_t* w, int64_t n, int64_t k, int tie_mode, uint8_t* packed,
                             uint8_t* e8m0, double* snr_db, double* rel_err, void* workspace,
                             size_t workspace_bytes, void* stream);

/* mxfp4_quantize_ex (quantize_dflash_mxfp4.py quantize_mxfp4, which starts from
 * w.float()) -- as mxfp4_quantize for a weight of type w_dtype (WQ_DTYPE_BF16
 * calls it; WQ_DTYPE_F16 / WQ_DTYPE_F32: the block exponent from the binary32
 * amax, the values scaled by the exact power of two and rounded to e2m1 by the
 * tie mode).  w and packed 16-byte aligned. */
wq_status mxfp4_quantize_ex(const void* w, int w_dtype, int64_t n, int64_t k, int tie_mode,
                            uint8_t* packed, uint8_t* e8m0, void* stream);

/* mxfp4_dequantize (quantize_dflash_mxfp4.py, dequantize_mxfp4)
 * out[n][c] = +-E2M1[code & 7] * 2^(e8m0 - 127) as binary32 (WQ_DTYPE_F32) or bf16
 * (WQ_DTYPE_BF16; exact, the value has at most 2 significant bits).  e8m0 = 255
 * gives inf (or NaN for a zero code), as 2^128 does in binary32.  out 16-byte
 * aligned. */
wq_status mxfp4_dequantize(const uint8_t* packed, const uint8_t* e8m0, int64_t n, int64_t k,
                           int out_dtype, void* out, void* stream);

/* awq_search (quantize_dflash_mxfp4.py, search_scale)
 * In:  W bf16 [n, k] (k % 32 == 0); a binary32 [k] per-channel mean |x| (device);
 *      alphas: n_alpha (1..16) binary32 values on the HOST; max_rows (>= 1) rows
 *      kept by the strided subsample (rows 0, s, 2s, ... with s = max(1, n /
 *      max_rows), first max_rows of them, when n > max_rows); tie_mode as above.
 * Out (device): best_s binary32 [k]; best_idx int32 [1]; best_alpha binary32 [1];
 *      errs double [n_alpha]: err(alpha) = sum(((deq(quant(W*s))/s) - W) * a_c)^2
 *      with a_c = max(a, 1e-8), s = t / exp(mean(log t)), t = clamp((a_c /
 *      mean(a_c))^alpha, 1e-2, 1e2).  The first alpha with the strictly smallest
 *      error wins.  Scale preparation: binary64 sums rounded once to binary32,
 *      pow/log/exp in binary64 rounded once to binary32.
 * workspace >= wq_workspace_bytes(WQ_OP_AWQ_SEARCH, n, k, n_alpha). */
wq_status awq_search(const uint16_t* w, int64_t n, int64_t k, const float* a,
                     const float* alphas_host, int n_alpha, int max_rows, int tie_mode,
                     float* best_s, int32_t* best_idx, float* best_alpha, double* errs,
                     void* workspace, size_t workspace_bytes, void* stream);

/* awq_search_static_scratch -- awq_search without a caller workspace.
 * The paper has no counterpart: this is a convenience of this library for
 * callers that cannot allocate device memory when they run the search (code
 * inside another component's memory pool, framework plug-ins that must not
 * allocate on their threads, paths that must not risk the device-wide
 * synchronisation an allocation can cause).
 * Same arguments and results as awq_search, minus workspace/workspace_bytes.
 * Scratch: a fixed 2,883,840-byte array inside the library (held by every GPU
 * that loads the library until the process exits), enough for k <= 16384 and
 * n_alpha <= 16.  Larger k returns WQ_ERR_BAD_SHAPE and n_alpha outside 1..16
 * WQ_ERR_UNSUPPORTED (as awq_search), before any launch.  The first call in a
 * device's CUDA context (with that device current) looks the array's device
 * address up once; make that first call before any stream capture.  The address
 * is cached per context, so a call after a context reset (cudaDeviceReset) looks
 * it up again.  `stream` must belong to the current device (WQ_ERR_UNSUPPORTED
 * otherwise).  Every call shares the array: calls that overlap on the GPU race
 * and must be serialised by the caller.  Calls no allocation routine. */
wq_status awq_search_static_scratch(const uint16_t* w, int64_t n, int64_t k, const float* a,
                                    const float* alphas_host, int n_alpha, int max_rows,
                                    int tie_mode, float* best_s, int32_t* best_idx,
                                    float* best_alpha, double* errs, void* stream);

/* awq_fold (quantize_dflash_mxfp4.py, main(): the fold after search_scale --
 * norm weights / s, conv kernel projections, q/k/v, gate/up and down columns
 * * s, up's rows / down's s).
 * In:  w    bf16 [n, k] (a norm weight is the case n = 1), 16-byte aligned; k % 8 == 0.
 *      s    binary32 device array: k entries (axis WQ_FOLD_COLUMNS, 16-byte
 *           aligned) or n entries (axis WQ_FOLD_ROWS).
 *      op   WQ_FOLD_MUL or WQ_FOLD_DIV.
 * Out: out  bf16 [n, k], 16-byte aligned; may be w itself (in-place fold).
 * Math per element: bf16(binary32(w op s)), op a binary32 multiply or IEEE
 * division, each rounded to nearest even -- the page's (W.float() * s).to(
 * torch.bfloat16) with its two roundings; overflow gives inf as the page's
 * cast does.  s is meant to be finite and nonzero (NaN bit patterns are not
 * specified). */
/* gptq_linear (export_gptq_cpu.py module docstring: the exported checkpoint is
 * served by a W4A16 uint4b8 layer) -- the consumer of the GPTQ tensors for
 * decode batches: y = x deq(W)^T without materialising deq.
 * In:  x        bf16 [m, k], 16-byte aligned, 1 <= m <= 8 (WQ_ERR_UNSUPPORTED above).
 *      qweight, qzeros, scales as produced by gptq_quantize_*; group 32, 64,
 *               128 or 256; sym selects the rule (qzeros may be NULL for sym);
 *               qweight 16-byte aligned.
 * Out: out      [m, n], binary32 (WQ_DTYPE_F32) or bf16 (WQ_DTYPE_BF16: the
 *               binary32 result rounded to nearest even).
 *      workspace >= gptq_linear_workspace_bytes(m, n), 256-byte aligned,
 *               ZEROED ONCE before its first use (cudaMemset); every completed
 *               call leaves its arrival counters at zero again, so no reset is
 *               needed between calls (zero it again after a call that failed).
 *               Calls that overlap on the GPU need separate workspaces.
 * Math: deq = (code - zp) * fp16 scale (exact in binary32); the products
 * x * (code - zp) (exact) are summed in binary32 over runs of at most 64 input
 * channels of one group, each run sum is multiplied by the group's scale and
 * added in binary32; K-slices are added in a fixed order.  Every product passes
 * through at most k + 1 roundings, so the result is within (k + 2) * 2^-24 *
 * sum_k |x * deq| of the exact value, and it is the same from run to run.
 * k == 0 writes zeros. */
size_t gptq_linear_workspace_bytes(int64_t m, int64_t n);
wq_status gptq_linear(const uint16_t* x, int64_t m, const int32_t* qweight, const int32_t* qzeros,
                      const uint16_t* scales, int64_t n, int64_t k, int group, int sym,
                      int out_dtype, void* out, void* workspace, size_t workspace_bytes,
                      void* stream);

/* gptq_gemm (export_gptq_cpu.py module docstring: the W4A16 uint4b8 layer that
 * serves the checkpoint, here for prefill batches) -- y = x deq(W)^T on the
 * tensor cores (tcgen05), any m >= 1, without materialising deq.
 * In:  x        bf16 [m, k], 16-byte aligned.
 *      qweight  i32 [k/8, n], 16-byte aligned; qzeros i32 [k/group, n/8] (may be
 *               NULL for sym); scales fp16 [k/group, n]; all as produced by
 *               gptq_quantize_*; group 32, 64, 128 or 256; n % 8 == 0.
 * Out: out      [m, n], binary32 (WQ_DTYPE_F32) or bf16 (WQ_DTYPE_BF16: the
 *               binary32 result rounded to nearest even); no workspace.
 * Math: the tensor cores multiply x by the integers (code - zp), exact in bf16,
 * so each product is exact; each group's products are summed in binary32 by
 * the MMA, and the group sums are folded in group order as y = fma(P_g,
 * scale_g, y).  The MMA's internal additions are not documented as
 * round-to-nearest, so the bound allows one binary32 ulp for each of them:
 * |y - exact| <= (k + 2) * 2^-23 * sum_k |x * deq|; the result is the same from
 * run to run.  k == 0 writes zeros.
 * Device errors: a device-side wait that runs out records WQ_ERR_DEVICE_TIMEOUT
 * for wq_device_status; out is then unspecified. */
wq_status gptq_gemm(const uint16_t* x, int64_t m, const int32_t* qweight, const int32_t* qzeros,
                    const uint16_t* scales, int64_t n, int64_t k, int group, int sym, int out_dtype,
                    void* out, void* stream);

/* uintx_gemm (uintx_quant.py, UIntXQuantizer.forward: the weight is rebuilt by
 * _dequantize_native in bf16, then F.linear) -- y = x deq(W)^T on the tensor
 * cores (tcgen05), any m >= 1, without materialising deq.
 * In:  x       bf16 [m, k], 16-byte aligned; k % 64 == 0 (WQ_ERR_UNSUPPORTED
 *              otherwise: the shard reads need 8-element alignment).
 *      packed, scale (bf16 [n, k/group]), zp (u8 [n, k/group]) as produced by
 *              uintx_quantize with nbits 2..7 and group 32, 64, 128 or 256;
 *              packed 16-byte aligned.
 * Out: out     [m, n], binary32 or bf16 (the binary32 result rounded to nearest
 *              even); no workspace.
 * Math: deq = the page's bf16 values ((q - zp) in bf16, times the bf16 scale,
 * rounded once), exactly as uintx_dequantize writes them; the tensor cores
 * multiply x by them (exact products) and add all k products in binary32
 * (addition rounding not documented as round-to-nearest, so the bound allows
 * one ulp per addition): |y - x deq^T| <= (k + 2) * 2^-23 * sum_k |x * deq|;
 * the same bits from run to run.  k == 0 writes zeros.  Device errors: as
 * gptq_gemm. */
wq_status uintx_gemm(const uint16_t* x, int64_t m, const uint8_t* packed, const uint16_t* scale,
                     const uint8_t* zp, int64_t n, int64_t k, int nbits, int group, int out_dtype,
                     void* out, void* stream);

/* mxfp4_linear (quantize_dflash_mxfp4.py: the drafter's linears are served in
 * MXFP4; deq as dequantize_mxfp4) -- the consumer for decode batches:
 * y = x deq(W)^T without materialising deq.  No workspace.
 * In:  x       bf16 [m, k], 16-byte aligned, 1 <= m <= 8; k % 32 == 0.
 *      packed  u8 [n, k/2] and e8m0 u8 [n, k/32] as produced by mxfp4_quantize
 *              (packed 16-byte aligned).
 * Out: out     [m, n] binary32 or bf16 (the binary32 result rounded to nearest even).
 * Math: per 8 weights the products x * (+-e2m1 value) are exact and summed in
 * binary32, multiplied by 2^(e8m0 - 127) and added in binary32; the sums over
 * lanes and warps run in a fixed order, so the result is the same from run to
 * run and within (k + 2) * 2^-24 * sum_k |x * deq| of the exact value while no
 * block scale leaves the normal binary32 range (E8M0 bytes below 24 add at most
 * 2^-149 per block of absolute error; 255 gives inf as dequantize_mxfp4 does). */
wq_status mxfp4_linear(const uint16_t* x, int64_t m, const uint8_t* packed, const uint8_t* e8m0,
                       int64_t n, int64_t k, int out_dtype, void* out, void* stream);

#define WQ_FOLD_COLUMNS 0
#define WQ_FOLD_ROWS 1
#define WQ_FOLD_MUL 0
#define WQ_FOLD_DIV 1
wq_status awq_fold(const uint16_t* w, int64_t n, int64_t k, const float* s, int axis, int op,
                   uint16_t* out, void* stream);

/* ---------------------------------------------------------------- uintx
 * uintx_packed_bytes: size of the packed buffer for numel codes of nbits bits:
 * the sum over the power-of-two shards k in {4, 2, 1} present in nbits of
 * ceil(numel / (8/k)).  Pure host arithmetic. */
int64_t uintx_packed_bytes(int64_t numel, int nbits);

/* uintx_quantize (uintx_quant.py, UIntXQuantizer._quantize_impl + pack_uintx)
 * In:  w bf16 [n, k]; nbits in 2..7 (8 -> WQ_ERR_UNSUPPORTED, as the page's
 *      can_quantize refuses uint8); group (the page's default 64; any multiple of
 *      8 that divides k is accepted, 64 takes the single-pass kernel when
 *      (n*k) % 512 == 0); w, packed 16-byte aligned.
 * Out: packed u8 [uintx_packed_bytes(n*k, nbits)]: shards widest first; a k-bit
 *      shard holds 8/k values per byte as 8/k contiguous chunks of
 *      ceil(numel/(8/k)) values (chunk j in bits j*k .. j*k+k-1).
 *      scale bf16 [n, k/group] (the page stores it as the u8 byte view of bf16);
 *      zp u8 [n, k/group].
 * Arithmetic in bf16: each step is the binary32 operation on bf16 operands,
 * rounded once to bf16 (divisions are IEEE; "1.0 / scale" is a bf16 reciprocal):
 *   scale = max((max(mx,0) - min(mn,0)) / qmax, 2^-23), zp = clamp(-round(min(mn,0)
 *   / scale), 0, qmax), q = clamp(round(w * (1/scale)) + zp, 0, qmax). */
wq_status uintx_quantize(const uint16_t* w, int64_t n, int64_t k, int nbits, int group,
                         uint8_t* packed, uint16_t* scale, uint8_t* zp, void* stream);

/* uintx_quantize_err (uintx_quant.py: _quantize_impl + pack_uintx, and the
 * reconstruction error of the weight that _dequantize_native rebuilds; the same
 * SNR / relative-error definitions as export_gptq_cpu.py quantize_* and
 * quantize_dflash_mxfp4.py main()) -- uintx_quantize plus the error of the same
 * pass, deq = bf16(bf16(q - zp) * scale) formed on-chip from the codes.
 * In/Out: as uintx_quantize (bf16 w), and snr_db, rel_err (device doubles,
 * either may be NULL; both NULL is plain uintx_quantize) as mxfp4_quantize_err;
 * workspace >= wq_workspace_bytes(WQ_OP_UINTX_ERR, n, k, nbits), 16-byte aligned.
 * n == 0 or k == 0 launches nothing and leaves snr_db / rel_err unwritten. */
wq_status uintx_quantize_err(const uint16_t* w, int64_t n, int64_t k, int nbits, int group,
                             uint8_t* packed, uint16_t* scale, uint8_t* zp, double* snr_db,
                             double* rel_err, void* workspace, size_t workspace_bytes, void* stream);

/* uintx_dequantize (uintx_quant.py, unpack_uintx + _dequantize_native)
 * out = bf16(bf16(q - zp) * scale), as bf16 (WQ_DTYPE_BF16) or its exact binary32
 * widening (WQ_DTYPE_F32, what dequantize() returns).  out [n, k], 16-byte
 * aligned. */
wq_status uintx_dequantize(const uint8_t* packed, const uint16_t* scale, const uint8_t* zp,
                           int64_t n, int64_t k, int nbits, int group, int out_dtype, void* out,
                           void* stream);

/* uintx_quantize_ex / uintx_dequantize_ex (uintx_quant.py works in the weight's
 * own dtype) -- uintx_quantize / uintx_dequantize for a weight of type w_dtype:
 * WQ_DTYPE_BF16 calls those entry points; WQ_DTYPE_F16 and WQ_DTYPE_F32 do every
 * op in that type (the binary32 op rounded once to fp16; fp32 ops as they are).
 * scale has the weight's type ([n, k/group]); the dequantized output too.  The
 * group is any multiple of 8 that divides k.  w, scale and out need their
 * element alignment only.  Results are unspecified where 1/scale overflows the
 * type (groups of fp16 values spanning less than about 15 * 2^-16). */
wq_status uintx_quantize_ex(const void* w, int w_dtype, int64_t n, int64_t k, int nbits, int group,
                            uint8_t* packed, void* scale, uint8_t* zp, void* stream);
wq_status uintx_dequantize_ex(const uint8_t* packed, const void* scale, int w_dtype, const uint8_t* zp,
                              int64_t n, int64_t k, int nbits, int group, void* out, void* stream);

/* ---------------------------------------------------------------- SNR
 * quant_snr (export_gptq_cpu.py quantize_* snr; quantize_dflash_mxfp4.py main()
 * relative error): over the whole tensor, Sw = sum w^2, Se = sum (w - deq)^2 with
 * binary32 terms and binary64 sums;
 *   snr_db = 20*log10(sqrt(Sw) / max(sqrt(Se), 1e-12)), rel_err = sqrt(Se)/sqrt(Sw).
 * In:  w bf16 [n, k]; deq of dtype deq_dtype (WQ_DTYPE_F32 | WQ_DTYPE_BF16) in
 *      layout deq_layout (WQ_LAYOUT_NK [n, k] | WQ_LAYOUT_KN [k, n]); both
 *      16-byte aligned.
 * Out: snr_db, rel_err: one double each on the device (either may be NULL).
 * workspace >= wq_workspace_bytes(WQ_OP_QUANT_SNR, n, k, 0). */
wq_status quant_snr(const uint16_t* w, const void* deq, int deq_dtype, int deq_layout, int64_t n,
                    int64_t k, double* snr_db, double* rel_err, void* workspace,
                    size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WQGB300_H */
