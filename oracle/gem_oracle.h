/*
 * gem_oracle.h — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar C11 reference of one decoder-layer step of a Qwen3 /
 * Gemma-4-style model with Q4_0 weights, accumulated in fp64.  It exists to check the
 * CUDA library; only the tests, the package smoke check and the benchmark's CPU
 * baseline may call it.  It shares no code, header, table or helper with the CUDA
 * library, and it includes nothing from it.
 *
 * Sources (page title, section):
 *   [GEM]  "gem" engine research record, "Verified model facts" (Q4_0 layout,
 *          Gemma 4 31B geometry, full-attention V from the K projection with
 *          unweighted RMS normalisation), "Native Metal diagnostic: buffer
 *          ownership" (Q4_0 matvec, weighted RMSNorm, NeoX RoPE, scalar C checks).
 *   [GELO] "GELO LLM generation", section 02 (QK-norm, GQA, sliding window,
 *          p-RoPE), section 04 (Qwen3 table), section 05 (apply_qk_norm,
 *          cached attention with n_kv = n_cache + 1).
 *
 * Readings where the pages are silent are listed beside each function.
 */
#ifndef GEM_ORACLE_H
#define GEM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE-754 binary16 bit pattern -> double (exact). */
double gem_oracle_half_to_double(uint16_t h);
/* double -> binary32 (round to nearest even) -> binary16 (round to nearest even). */
uint16_t gem_oracle_double_to_half_via_f32(double v);

/* Dequantise rows [0, N) of a Q4_0 matrix (N rows x K/32 blocks x 18 bytes). */
void gem_oracle_q4_0_dequant(const uint8_t *W, int64_t N, int64_t K, double *out);

/* y[b][n] = sum_k deq(W)[n][k] * x[b][k] (+ residual[b][n]); fp32 x, fp64 y. */
int gem_oracle_q4_0_gemv_f32(const uint8_t *W, int64_t N, int64_t K, const float *x,
                             int64_t ldx, int B, const float *residual, int64_t ldr,
                             double *y, int64_t ldy);
/* Same on fp64 activations (used inside the layer step). */
int gem_oracle_q4_0_gemv_f64(const uint8_t *W, int64_t N, int64_t K, const double *x,
                             int64_t ldx, int B, double *y, int64_t ldy);

/* out = x / sqrt(mean(x^2) + eps) * gamma   (gamma NULL = unweighted). */
void gem_oracle_rmsnorm(const double *x, int64_t n, const float *gamma, double eps,
                        double *out);

/* NeoX rotation of the first rope_dim dims of v at position pos, base theta. */
void gem_oracle_rope_neox(double *v, int d, int rope_dim, double pos, double theta);

/* Grouped-query decode attention for one sequence.
 *   q: [n_q][d] fp64; caches: binary16 bits [n_kv][cap][d]; out: [n_q][d].
 *   Attended positions: full (window == 0): 0..pos; sliding: max(0,pos-window+1)..pos.
 *   Slot of position j: j (full) or j mod window (sliding).
 *   probs (nullable): [n_q][T] softmax weights in position order. */
int gem_oracle_gqa_attention(const double *q, const uint16_t *k_cache,
                             const uint16_t *v_cache, int n_q, int n_kv, int d,
                             int64_t cap, int64_t pos, int window, double scale,
                             double *out, double *probs);

double gem_oracle_silu(double g);
double gem_oracle_gelu_tanh(double g);

/* One decoder layer step. */
typedef struct {
    int64_t H, n_q, n_kv, d, F;
    double eps, theta, scale;
    int rope_dim, window, act; /* act: 0 SiLU, 1 GELU (tanh form) */
    int qk_norm, v_from_k, post_norms;
    const uint8_t *w_qkv, *w_o, *w_gate, *w_up, *w_down;
    const float *g_attn, *g_ffn, *g_q, *g_k, *g_post_attn, *g_post_ffn;
    int compact_kv; /* full-attention layer with V from K: the cache keeps V only (k_cache may be
                       NULL); attention rebuilds K_j = RoPE_j(V_j * g_k) */
} gem_oracle_layer;

/* x_in: [B][H] fp32; caches: [B][n_kv][cap][d] binary16 (the new row is written);
 * pos: [B]; x_out: [B][H] fp64.  Optional stage outputs (nullable, fp64):
 *   qkv_out [B][n_qkv] (after norm/RoPE of q and k), attn_out [B][n_q*d],
 *   h_out [B][H] (after the attention residual). */
int gem_oracle_decode_layer(const gem_oracle_layer *L, int B, const float *x_in,
                            uint16_t *k_cache, uint16_t *v_cache, int64_t cap,
                            const int32_t *pos, double *x_out, double *qkv_out,
                            double *attn_out, double *h_out);

/* Same step with fp64 input (stacking layers inside the oracle). */
int gem_oracle_decode_layer_f64(const gem_oracle_layer *L, int B, const double *x_in,
                                uint16_t *k_cache, uint16_t *v_cache, int64_t cap,
                                const int32_t *pos, double *x_out, double *qkv_out,
                                double *attn_out, double *h_out);

/* The step with two extra, optional arguments (nullable):
 *   kvnew_out [B][2][n_kv][d]: the new K (index 0) and V (index 1) rows before rounding.
 *   flip      [B][2][n_kv][d]: where non-zero, the appended binary16 code is the other
 *             neighbour of the binary32 value (the one round-to-nearest-even did not pick);
 *             a value that is exactly representable keeps its code.  This evaluates the
 *             step for the other valid outcome of a rounding decision that lies within
 *             the arithmetic's precision of a binary16 midpoint. */
int gem_oracle_decode_layer_ex(const gem_oracle_layer *L, int B, const double *x_in,
                               uint16_t *k_cache, uint16_t *v_cache, int64_t cap,
                               const int32_t *pos, double *x_out, double *qkv_out,
                               double *attn_out, double *h_out, double *kvnew_out,
                               const int8_t *flip);

/* The binary16 neighbour of fp32(v) on the other side from round-to-nearest-even
 * (equal to the RNE code when fp32(v) is exactly representable). */
uint16_t gem_oracle_other_half_via_f32(double v);

/* Attention over a compact full-attention cache (V rows only): K_j = RoPE_j(V16_j * gamma_k)
 * rebuilt in fp64, then softmax(scale q.K) V as gem_oracle_gqa_attention (window 0). */
int gem_oracle_gqa_attention_compact(const double *q, const uint16_t *v_cache, const float *gamma_k,
                                     int n_q, int n_kv, int d, int64_t cap, int64_t pos,
                                     int rope_dim, double theta, double scale, double *out);

/* Index of the largest value; ties go to the lowest index. */
int64_t gem_oracle_argmax(const double *v, int64_t n);

/* The k largest entries, largest first (ties: lowest index; NaN after every number, by
 * index); returns 0, or 1 for k outside 1..n.  idx, val: [k]. */
int gem_oracle_topk(const double *v, int64_t n, int k, int64_t *idx, double *val);

/* Q8_0: 34-byte blocks (binary16 scale, 32 int8 codes), weight = q * d. */
void gem_oracle_q8_0_dequant(const uint8_t *W, int64_t N, int64_t K, double *out);
int gem_oracle_q8_0_gemv_f64(const uint8_t *W, int64_t N, int64_t K, const double *x,
                             int64_t ldx, int B, double *y, int64_t ldy);

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int gem_oracle_num_threads(void);
void gem_oracle_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
