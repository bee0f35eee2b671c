/*
 * smla_oracle.h -- the CPU oracle's own interface (test infrastructure).
 * Nothing outside tests/, __graft_entry__.smoke() and bench.py's CPU leg uses
 * it; the CUDA library has its own, unrelated, header.
 */
#ifndef SMLA_ORACLE_H
#define SMLA_ORACLE_H

#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* One decode problem, all arrays in host memory.
 * q:       E4M3 bytes, element (t, h, d) at t*q_stride_token + h*q_stride_head + d.
 * pool[i]: pool_rows[i] rows of head_dim E4M3 bytes each, rows contiguous.
 * indices: int32 (t, c) at t*idx_stride_token + c; -1 marks a hole.
 * lens:    int32 [tokens], active count per token (clamped to [0, width]).
 * sinks:   float [heads] or NULL. */
typedef struct smla_oracle_problem {
    int32_t tokens, heads, width, head_dim, num_pools, pool_split;
    const uint8_t* q;
    int64_t q_stride_token, q_stride_head;
    const uint8_t* pool[2];
    int64_t pool_rows[2];
    const int32_t* indices;
    int64_t idx_stride_token;
    const int32_t* lens;
    const float* sinks;
    double bmm1_scale, bmm2_scale, k_scale;
} smla_oracle_problem;

enum {
    SMLA_ORACLE_NO_P_ROUNDING = 1, /* keep P unrounded (no E4M3 step) */
    SMLA_ORACLE_EXACT = 2,         /* no FP32 roundings anywhere */
    SMLA_ORACLE_P_UP = 4,          /* round P * (1 + 2^-16) to E4M3 (the upper code of the tie window) */
    SMLA_ORACLE_P_DOWN = 8         /* round P * (1 - 2^-16) to E4M3 (the lower code) */
};

double smla_oracle_e4m3_to_double(uint8_t byte);
uint8_t smla_oracle_e4m3_from_float(float value);
uint16_t smla_oracle_bf16_from_float(float value);
float smla_oracle_bf16_to_float(uint16_t bits);

/* The plain definition: out[512] (double) and the base-2 LSE of (t, h). */
int smla_oracle_fp64(const smla_oracle_problem* p, int t, int h, double* out, double* lse2);

/* The E4M3-P datapath on `splits` splits of `chunk`-column chunks: out_value
 * (pre-BF16 value, double), out_bf16 (bits), the base-2 LSE and tie_out[512],
 * the most that P codes within a relative 2^-16 of a rounding midpoint can
 * move each output value by taking their other code; any may be NULL. */
int smla_oracle_emulate(const smla_oracle_problem* p, int t, int h, int splits, int chunk,
                        int flags, double* out_value, uint16_t* out_bf16, double* lse2_out,
                        double* tie_out);

int smla_oracle_fp64_all(const smla_oracle_problem* p, double* out, double* lse2, int threads);
int smla_oracle_fp64_pairs(const smla_oracle_problem* p, const int32_t* tokens,
                           const int32_t* heads, int n, double* out, double* lse2, int threads);
int smla_oracle_emulate_pairs(const smla_oracle_problem* p, const int32_t* tokens,
                              const int32_t* heads, int n, int splits, int chunk, int flags,
                              double* out_value, uint16_t* out_bf16, double* lse2, double* tie,
                              int threads);
int smla_oracle_max_threads(void);

/* LSE merge of partial sets (the DCP owner's merge).
 * parts: BF16 bits, element (s, t, h, j) at s*part_stride_source +
 *        t*part_stride_token + h*part_stride_head + j, j < 512.
 * lses:  float, (s, t, h) at s*lse_stride_source + t*lse_stride_token + h
 *        (base 2; not finite = empty source).
 * lens:  int32 [tokens] or NULL; a token of count <= 0 merges to zeros. */
typedef struct smla_oracle_merge_problem {
    int32_t sources, tokens, heads;
    const uint16_t* parts;
    int64_t part_stride_source, part_stride_token, part_stride_head;
    const float* lses;
    int64_t lse_stride_source, lse_stride_token;
    const int32_t* lens;
} smla_oracle_merge_problem;

/* The merge in double of `sources` rows [sources][512] with base-2 LSEs. */
int smla_oracle_merge_f64(int sources, const double* rows, const double* lses, double* out, double* lse2);
int smla_oracle_merge(const smla_oracle_merge_problem* m, int t, int h, double* out_value,
                      uint16_t* out_bf16, double* lse2_out);
int smla_oracle_merge_pairs(const smla_oracle_merge_problem* m, const int32_t* tokens,
                            const int32_t* heads, int n, double* out_value, uint16_t* out_bf16,
                            double* lse2, int threads);

/* MXFP4 quantisation of the indexer query (one token, head_dim 128). */
uint8_t smla_oracle_e2m1_from_float(float value);
double smla_oracle_e2m1_to_double(uint8_t code);
int smla_oracle_mxfp4_q_quant(int heads, int padded, const float* q, const float* weights, float weight_scale,
                              uint8_t* packed, int32_t* scale, float* w_out);

/* Value projection and sigmoid gate after the merge: latent BF16 [T][H][512],
 * w_uv BF16 [H][512][128], gate BF16 [T][H * 128], lens [T] or NULL; outputs
 * [T][H * 128] (value before the final rounding, and BF16 bits). */
int smla_oracle_value_gate(int tokens, int heads, const uint16_t* latent, const uint16_t* w_uv,
                           const uint16_t* gate, const int32_t* lens, double* out_value, uint16_t* out_bf16);

#ifdef __cplusplus
}
#endif
#endif
