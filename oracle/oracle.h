/* oracle.h -- declarations of the CPU oracle (TEST INFRASTRUCTURE ONLY).
 * Private to oracle/; nothing outside tests may include or link it. */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>

/* FP8 weights: every projection matrix as E4M3 codes [rows][K] and one
   float scale per output row (w ~ e4m3(code) * scale); the embedding used for
   the token lookup and the norms stay bf16. */
typedef struct {
  const uint8_t *const *wq, *const *wk, *const *wv, *const *wo, *const *w_gate, *const *w_up,
      *const *w_down; /* L pointers each */
  const float *const *sq, *const *sk, *const *sv, *const *so, *const *s_gate, *const *s_up,
      *const *s_down; /* L pointers each */
  const uint8_t *lm;  /* [V][H]: the LM head (the embedding's codes when tied) */
  const float *s_lm;  /* [V] */
} or_q8;

typedef struct {
  int L, H, nq, nkv, d, F, V;
  double eps, theta;
  const uint16_t *embed;      /* [V][H] */
  const uint16_t *final_norm; /* [H] */
  const uint16_t *lm_head;    /* [V][H], NULL when tied to embed */
  const uint16_t *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo,
      *const *mlp_norm, *const *w_gate, *const *w_up, *const *w_down; /* L pointers each */
  const or_q8 *q8;            /* NULL: the bf16 projections above */
} or_model;

typedef struct {
  int L, H, nq, nkv, d, F, V, B;
} or_shape;

double or_bf16_to_double(uint16_t h);
uint16_t or_bf16_rne(double v);
void or_rmsnorm(int n, const double *x, const uint16_t *g, double eps, double *y);
void or_matvec(int M, int K, const uint16_t *W, const double *x, double *y);
double or_e4m3_to_double(uint8_t c);
uint8_t or_e4m3_rne(double v);
void or_quantize_rows(int M, int K, const uint16_t *W, uint8_t *Q, float *scale);
void or_matvec_q8(int M, int K, const uint8_t *Q, const float *scale, const double *x,
                  double *y);
void or_rope(int d, double pos, double theta, double *z);
double or_silu(double z);
void or_attention(int d, int n, const double *q, const uint16_t *K, const uint16_t *V, double *o);
int or_argmax(int n, const double *v);
int or_decode_step(const or_model *m, int B, int max_ctx, uint16_t *kc, uint16_t *vc,
                   const int32_t *tokens, const int32_t *positions, double *logits);

int or_replay(const void *table, int n_instr, int n_counters, const or_shape *s, int S,
              const uint32_t *list_off, const uint32_t *list_idx, uint32_t *inc_out, char *msg,
              int msg_len);
int or_simulate(const void *table, int n_instr, int n_counters, int S, int fifo_depth,
                uint64_t seed, int trials, const uint32_t *list_off, const uint32_t *list_idx,
                const uint32_t *att_first, int n_att, int att_count, char *msg, int msg_len);
long or_explore(const void *table, int n_instr, int n_counters, int fifo_depth, long max_states,
                char *msg, int msg_len);
int or_redeal(const void *table, int n_instr, const or_shape *s, int attn_chunk,
              const int32_t *positions, const uint32_t *list_idx, int n_list,
              uint32_t *exec_idx, char *msg, int msg_len);
#endif
