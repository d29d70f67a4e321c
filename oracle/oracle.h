/*
 * oracle.h -- interface of the CPU oracle (test infrastructure only).
 *
 * Private to oracle/: the CUDA library neither includes nor links it.  All
 * pointers are host pointers; all matrices are dense row-major.  bf16 and fp16
 * values travel as their 16-bit patterns (uint16_t).  See oracle.c for the
 * algorithms and the page passages they restate.
 */
#ifndef WQ_ORACLE_H
#define WQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_TIE_HALF_EVEN 0
#define ORC_TIE_PAGE_LITERAL 1

float orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float x);
float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float x);
int orc_floor_log2(float a);
int orc_e2m1_code(float v, int tie_mode);

void orc_pack_int32(const int32_t* codes, int64_t k, int64_t n, int dim, int32_t* out);
void orc_gptq_quantize_f32(const float* w, int64_t n, int64_t k, int group, int sym,
                           int32_t* qweight, int32_t* qzeros, uint16_t* scales,
                           int32_t* g_idx, double* snr_db);
void orc_gptq_quantize(const uint16_t* w, int64_t n, int64_t k, int group, int sym,
                       int32_t* qweight, int32_t* qzeros, uint16_t* scales, int32_t* g_idx,
                       double* snr_db);
void orc_gptq_dequantize(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                         int64_t n, int64_t k, int group, int sym, int out_kn, float* out);

void orc_mxfp4_quantize_f32(const float* w, int64_t n, int64_t k, int tie_mode, uint8_t* packed,
                            uint8_t* e8m0);
void orc_mxfp4_quantize(const uint16_t* w, int64_t n, int64_t k, int tie_mode, uint8_t* packed,
                        uint8_t* e8m0);
void orc_mxfp4_dequantize(const uint8_t* packed, const uint8_t* e8m0, int64_t n, int64_t k,
                          float* out);
void orc_awq_prepare_scales(const float* a, int64_t k, const float* alphas, int n_alpha,
                            float* s_out, float* a_c_out);
void orc_awq_search(const uint16_t* w, int64_t n, int64_t k, const float* a, const float* alphas,
                    int n_alpha, int max_rows, int tie_mode, float* best_s, int32_t* best_idx,
                    float* best_alpha, double* errs);
void orc_quant_snr(const uint16_t* w, const void* deq, int deq_bf16, int deq_kn, int64_t n,
                   int64_t k, double* snr_db, double* rel_err);
void orc_awq_fold(const uint16_t* w, int64_t n, int64_t k, const float* s, int axis, int op,
                  uint16_t* out);

int64_t orc_uintx_packed_bytes(int64_t numel, int nbits);
void orc_uintx_pack(const uint8_t* codes, int64_t numel, int nbits, uint8_t* out);
void orc_uintx_unpack(const uint8_t* packed, int64_t numel, int nbits, uint8_t* codes);
void orc_uintx_quantize_dt(const void* w, int dt, int64_t n, int64_t k, int nbits, int group,
                           uint8_t* packed, void* scale_out, uint8_t* zp_out, uint8_t* codes_out);
void orc_uintx_dequantize_dt(const uint8_t* packed, const void* scale, int dt, const uint8_t* zp,
                             int64_t n, int64_t k, int nbits, int group, void* out);
void orc_uintx_quantize(const uint16_t* w, int64_t n, int64_t k, int nbits, int group,
                        uint8_t* packed, uint16_t* scale_out, uint8_t* zp_out, uint8_t* codes_out);
void orc_uintx_dequantize(const uint8_t* packed, const uint16_t* scale, const uint8_t* zp,
                          int64_t n, int64_t k, int nbits, int group, uint16_t* out_bf16);

#ifdef __cplusplus
}
#endif

#endif /* WQ_ORACLE_H */
