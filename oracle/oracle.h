/* oracle.h -- C interface of the CPU oracle (test infrastructure only; see oracle.c). */
#ifndef BRE_ORACLE_H
#define BRE_ORACLE_H
#include <stdint.h>

#define OR_FMT_Q2_K 1
#define OR_FMT_Q8_0 2

float or_f16_to_f32(uint16_t h);
float or_bf16_to_f32(uint16_t b);
uint16_t or_bf16_rne(float f);
uint16_t or_bf16_rne_f64(double x);
float or_e4m3_to_f32(uint8_t b);
float or_e8m0_to_f32(uint8_t e);
float or_sigmoid(float z);

void or_dequant_q2k(const uint8_t *blk, int64_t nblk, float *out);
void or_dequant_q8_0(const uint8_t *blk, int64_t nblk, float *out);

void or_engram_gather(const uint8_t *const *tables, const int64_t *n_rows, int n_tables,
                      const int64_t *ids, int T, int H, uint16_t *out, int32_t *err);

void or_route(const uint16_t *x, const float *wr, const float *bias, int T, int d, int E, int k,
              int32_t *ids, float *w, float *z_out, float *s_out);

float or_sqrt_softplus(float z);
void or_route_ex(const uint16_t *x, const float *wr, const float *bias, int T, int d, int E, int k,
                 int score_fn, const float *vbias, const uint8_t *media, const int32_t *tid2eid,
                 const int32_t *tok, int vocab, int32_t *ids, float *w, int32_t *err);

void or_permute(const int32_t *ids, int T, int k, int E, int32_t *offsets, int32_t *perm,
                int32_t *inv, int32_t *active, int32_t *n_active, int32_t *err);

void or_expert_ffn(int fmt, const uint8_t *gate, const uint8_t *up, const uint8_t *down, int d, int F,
                   const uint16_t *xs, int n, double *y);

int or_moe_layer(const uint16_t *x, int T, int d, int E, int k, int F, const float *wr,
                 const float *bias, const uint8_t *const *gate_e, const uint8_t *const *up_e,
                 const uint8_t *const *down_e, const uint8_t *sh_gate, const uint8_t *sh_up,
                 const uint8_t *sh_down, int F_shared, uint16_t *out, double *out_f64,
                 int32_t *ids_out, float *w_out);

void or_residual(const uint16_t *x, const uint16_t *moe, int T, int d, float scale, uint16_t *x_new);
void or_rmsnorm(const uint16_t *x, int T, int d, float eps, uint16_t *u);

void or_engram_kv(const uint16_t *rows, const uint16_t *w, int T, int K, int N, double *kv);
void or_engram_gate(const double *kv, uint16_t *resid, const float *qn, const float *kn, const uint8_t *mask,
                    int T, int W, double eps, double *gate_out);

#endif
