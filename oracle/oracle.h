/*
 * CPU oracle for one decode step of the parallel-layer MoE model.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this library.  It shares no
 * code, header, table or helper with the CUDA path; the two meet only through
 * the seeded synthetic inputs.
 *
 * Source of the definition: "Inside the megakernel serving engine for North
 * Mini Code" — §Where the speedup comes from (parallel transformer layers:
 * attention and MoE read the same normalised input and are rejoined by a
 * residual add + RMSNorm), §Tasks (the decode graph: QKV with RoPE, attention
 * over a paged KV cache, O-proj, router, top-k, expert gate/up with
 * SiLU-and-multiply, expert down, weighted combine of each token's expert
 * outputs, LM head).  All arithmetic is fp64 on BF16 inputs.
 */
#ifndef PMD_ORACLE_H
#define PMD_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Where the decode step stores a BF16 copy of an activation.  The K/V that a
 * step appends to the cache are always BF16 (the cache is BF16).  Each flag
 * adds one more rounding point; 0 is the pure definition. */
enum {
  ORC_BF16_X = 1,     /* normalised input of each layer and of the LM head  */
  ORC_BF16_Q = 2,     /* query after RoPE                                    */
  ORC_BF16_ATTN = 4,  /* attention output entering O-proj                    */
  ORC_BF16_A = 8      /* expert hidden SiLU(g)*u entering the down projection */
};

typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim;
  int n_experts, top_k, moe_inter, vocab, page_size, num_pages;
  double rope_theta, rms_eps;
} orc_dims;

/* Optional 8-bit routed-expert weights.  Format: the OCP 8-bit floating
 * point specification's E4M3 (1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 = subnormal m/8 * 2^-6; no infinities,
 * S.1111.111 is NaN), one fp32 scale per output row: the weight is
 * scale[row] * e4m3(q[row][col]).  Layouts: q_gate, q_up [E][I][H] and
 * q_down [E][H][I] bytes; s_gate, s_up [E][I] and s_down [E][H] fp32; each a
 * per-layer pointer array. */
typedef struct {
  const uint8_t* const* q_gate;
  const uint8_t* const* q_up;
  const uint8_t* const* q_down;
  const float* const* s_gate;
  const float* const* s_up;
  const float* const* s_down;
} orc_fp8_experts;

/* BF16 weights as raw uint16 bit patterns, row-major.
 * Per-layer pointers: attn_norm [H]; w_qkv [(hq+2hkv)*d][H] (q heads, k heads,
 * v heads); w_o [H][hq*d]; w_router [E][H]; w_gate, w_up [E][I][H];
 * w_down [E][H][I]; k_pool, v_pool [num_pages][hkv][page_size][d]. */
typedef struct {
  const uint16_t* embed;      /* [V][H] */
  const uint16_t* lm_head;    /* [V][H] */
  const uint16_t* final_norm; /* [H]    */
  const uint16_t* const* attn_norm;
  const uint16_t* const* w_qkv;
  const uint16_t* const* w_o;
  const uint16_t* const* w_router;
  const uint16_t* const* w_gate;
  const uint16_t* const* w_up;
  const uint16_t* const* w_down;
  uint16_t* const* k_pool;
  uint16_t* const* v_pool;
  const orc_fp8_experts* fp8;  /* NULL: the experts use w_gate / w_up / w_down   */
} orc_model;

/* Optional per-layer record of intermediate values; any pointer may be NULL. */
typedef struct {
  double* h_in;      /* [L+1][B][H] residual entering layer l; [L] = after the last */
  double* x;         /* [L][B][H]      normalised layer input                      */
  double* q;         /* [L][B][hq*d]   query after RoPE                            */
  double* attn;      /* [L][B][hq*d]   attention output                            */
  double* attn_proj; /* [L][B][H]      O-proj output                               */
  double* router;    /* [L][B][E]      router logits                               */
  int32_t* idx;      /* [L][B][k]      selected experts, best first                */
  double* w;         /* [L][B][k]      renormalised routing weights                */
  double* gap;       /* [L][B]         r_(k) - r_(k+1) of the fp32 logits          */
  double* moe;       /* [L][B][H]      weighted expert sum                         */
  double* xf;        /* [B][H]         final normalised state                      */
} orc_trace;

enum { ORC_OK = 0, ORC_ERR_ARG = -1, ORC_ERR_PAGE = -2, ORC_ERR_NOMEM = -3 };

/* ---- building blocks (each pinned separately by the tests) ---- */
double orc_bf16_to_double(uint16_t b);
uint16_t orc_double_to_bf16(double x);           /* via fp32, round to nearest even */
double orc_round_bf16(double x);
void orc_rmsnorm(int n, const double* h, const uint16_t* gain, double eps, double* out);
void orc_rope(int d, double* v, long pos, double theta);
void orc_matvec(int rows, int cols, const uint16_t* w, int nvec, const double* x,
                double* y);
double orc_e4m3_to_double(uint8_t b);
/* y[r] = sum_c (scale[r] * e4m3(q[r][c])) * x[c], summed as orc_matvec sums */
void orc_matvec_e4m3(int rows, int cols, const uint8_t* q, const float* scale, const double* x,
                     double* y);
int orc_paged_attention(const orc_dims* dm, const uint16_t* k_pool, const uint16_t* v_pool,
                        const int32_t* page_table, int n_keys, int kv_head,
                        const double* q, double* out);
void orc_route(int n_experts, int top_k, const double* logits, int32_t* idx, double* w,
               double* gap);
void orc_moe(const orc_dims* dm, const orc_model* m, int layer, const double* x, int n_sel,
             const int32_t* idx, const double* w, unsigned flags, double* out);

/* ---- one decode step for a batch ----
 * tokens [B]; seq_lens [B] = tokens already cached (the new token lands at
 * position seq_lens[b]); page_tables [B][max_pages].  Writes the new K/V into
 * the model's pools, the logits [B][V] and, if trace != NULL, the trace. */
int orc_decode_step(const orc_dims* dm, const orc_model* m, int batch, const int32_t* tokens,
                    const int32_t* seq_lens, const int32_t* page_tables, int max_pages,
                    unsigned flags, double* logits, orc_trace* trace);

/* orc_decode_step with routing imposed where force_mask [L][B] is non-zero:
 * token b of layer l then uses the experts force_idx [L][B][k] (instead of its
 * own top-k), its weights renormalised over them.  Both NULL = orc_decode_step.
 * For comparing with an implementation that decided a near tie (a k-th /
 * (k+1)-th router gap within its rounding) the other way. */
int orc_decode_step_forced(const orc_dims* dm, const orc_model* m, int batch, const int32_t* tokens,
                           const int32_t* seq_lens, const int32_t* page_tables, int max_pages,
                           unsigned flags, const int32_t* force_idx, const uint8_t* force_mask,
                           double* logits, orc_trace* trace);

/* Subset of the step used to time the oracle on a bounded sample: runs layers
 * [l0, l1) on the residual h [B][H] in place (no embedding, no LM head). */
int orc_run_layers(const orc_dims* dm, const orc_model* m, int l0, int l1, int batch,
                   const int32_t* seq_lens, const int32_t* page_tables, int max_pages,
                   unsigned flags, double* h);

void orc_set_threads(int n);
int orc_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif
