/*
 * CPU oracle for the batch-invariant transformer forward step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code; only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Every function is the plain definition of one step of a Llama-style decoder
 * step, written as serial loops in binary32 (`float`), compiled with
 * -ffp-contract=off so that no multiply-add is fused; logprobs and the seeded
 * sampler are written in float64 (the sampler's decision is the pages').  Values that the GPU
 * stores in bf16 are rounded to bf16 (round to nearest even) at exactly those
 * storage points when `round_bf16` is non-zero; with it zero the oracle is a
 * pure fp32 computation (used by the float64 brute-force pin).
 *
 * Sources (page title, section):
 *   "Lockstep" — "The fix": every reduction has one fixed order.
 *   "Batch invariance and reproducible inference" — "Non-associativity,
 *     concretely" (binary32 round-to-nearest-even sums); "1 · Split-K and
 *     segmented attention reductions" (split-KV partials and their merge);
 *     "temperature=0 means deterministic" (greedy argmax over the logits).
 *
 * All arrays are row-major, dense, caller-owned.  bf16 tensors are passed as
 * float arrays holding bf16-representable values.  Functions return 0 on
 * success and a negative code on invalid arguments; they never abort.
 */
#ifndef ORC_ORACLE_H
#define ORC_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- binary32 / bf16 primitives ------------------------------------- */
float orc_bf16_round(float x);                              /* RNE to bf16, NaN stays NaN */
void  orc_bf16_round_array(const float* in, float* out, int64_t n);
float orc_sum_serial(const float* x, int64_t n);            /* ((x0+x1)+x2)+... */
float orc_sum_pairwise(const float* x, int64_t n);          /* recursive halving tree */

/* ---- row operations --------------------------------------------------- */
/* y[r,i] = round?( (x[r,i] * rinv_r) * gamma[i] ), rinv_r = 1/sqrt(sum_i x^2 / d + eps) */
int orc_rmsnorm(const float* x, const float* gamma, float* y,
                int64_t rows, int32_t d, float eps, int round_bf16);

/* C[m,n] = sum_k A[m,k] * W[n,k], one serial fp32 loop over k per element */
int orc_matmul(const float* A, const float* W, float* C,
               int64_t M, int32_t N, int32_t K);

/* p[j] = exp(s[j]-max) / sum_j exp(s[j]-max) */
int orc_softmax(const float* s, float* p, int32_t n);

/* h = round?( silu(g) * u ), silu(g) = g / (1 + exp(-g)) */
int orc_swiglu(const float* g, const float* u, float* h, int64_t n, int round_bf16);

/* lowest index of the maximum; NaN counts as larger than every number */
int32_t orc_argmax(const float* x, int32_t n);
int orc_argmax_rows(const float* x, int32_t* out, int64_t rows, int32_t n);

/* ---- logprobs and seeded sampling ---------------------------------------
 * "The weaker guarantees, which are usually enough" (per-request sampling
 * determinism: Gumbel noise from murmur_hash32(seed, position, column) in
 * float64) and "Mathematically equivalent is not bitwise equivalent"
 * (logprobs from a log_softmax kernel, never log(softmax)). */

/* lp[r,j] = x[r,j] - m_r - log(sum_i exp(x[r,i] - m_r)), m_r = max_i x[r,i]; in float64 */
int orc_log_softmax_rows(const float* x, double* lp, int64_t rows, int32_t n);

/* MurmurHash3, x86 32-bit variant, of len bytes with a 32-bit seed */
uint32_t orc_murmur3_32(const uint8_t* key, int32_t len, uint32_t seed);

/* Gumbel-max draw of one row at temperature t > 0, all in float64:
 *   h_j = murmur3_32(le32(pos) || le32(j), seed), u_j = (h_j + 0.5) / 2^32,
 *   g_j = -log(-log(u_j)), token = argmax_j (x_j / t + g_j)
 * ties to the lowest index, a NaN score larger than every number.  A row with
 * t <= 0 (or NaN) is decoded greedily (orc_argmax).
 * Parity unpinned in one detail: the byte layout of the hash key (position
 * first, then column) is a reading.  The pages name the hash's inputs but
 * print no hash or token that would fix their order. */
int32_t orc_sample_gumbel(const float* x, int32_t n, uint32_t seed, int32_t pos, float t);
int orc_sample_gumbel_rows(const float* x, const uint32_t* seeds, const int32_t* pos, const float* t,
                           int32_t* out, int64_t rows, int32_t n);

/* ---- rotary embedding (rotate-half) ------------------------------------ */
/* cos/sin tables [n_pos, Dh/2]: angle = pos * theta^(-2i/Dh) in float64, then
 * cos and sin in float64 rounded to float. */
int orc_rope_table(float* cos_t, float* sin_t, int32_t n_pos, int32_t Dh, double theta);
/* rotates n_vec vectors of length Dh in place; vector v sits at position pos[v] */
int orc_rope_apply(float* x, const int32_t* pos, int64_t n_vec, int32_t Dh,
                   const float* cos_t, const float* sin_t, int32_t n_pos);

/* ---- attention ---------------------------------------------------------- */
/* One query head against n_keys keys (rows of length Dh, stride `kv_stride`
 * floats between consecutive keys): s_j = (q . k_j) * scale, p = softmax(s),
 * out[d] = sum_j p_j v_j[d].  Textbook form, no splits. */
int orc_attention_head(const float* q, const float* k, const float* v,
                       int32_t n_keys, int64_t kv_stride, int32_t Dh,
                       float scale, float* out);

/* Same quantity through fixed key chunks of `chunk` keys: per chunk the max m,
 * the sum l of exp(s-m) and the unnormalised output o; chunks are then merged
 * in ascending order (M = max m_j; L = sum l_j e^(m_j-M); O = sum o_j e^(m_j-M);
 * out = O / L).  Used only to check that splitting does not change the value
 * beyond rounding. */
int orc_attention_head_split(const float* q, const float* k, const float* v,
                             int32_t n_keys, int64_t kv_stride, int32_t Dh,
                             float scale, int32_t chunk, float* out);

/* ---- one decoder layer over a ragged batch ----------------------------- */
typedef struct {
    int32_t d;          /* hidden size */
    int32_t H;          /* query heads */
    int32_t Hkv;        /* key/value heads; head h reads kv head h / (H/Hkv) */
    int32_t Dh;         /* head dim */
    int32_t F;          /* ffn width */
    float   eps;        /* RMSNorm epsilon */
    double  rope_theta; /* RoPE base */
    int32_t round_bf16; /* 1: round at the bf16 storage points; 0: pure fp32 */
} orc_dims;

typedef struct {
    const float* gamma_attn; /* [d] */
    const float* w_qkv;      /* [(H+2Hkv)*Dh, d]: q rows, then k rows, then v rows */
    const float* w_o;        /* [d, H*Dh] */
    const float* gamma_ffn;  /* [d] */
    const float* w_gate;     /* [F, d] */
    const float* w_up;       /* [F, d] */
    const float* w_down;     /* [d, F] */
} orc_layer_weights;

/* Request i owns query tokens [cu_q[i], cu_q[i+1]) at positions pos0[i] + t.
 * Its keys/values live in k_pool/v_pool rows kv_row0[i] + position, each row
 * [Hkv, Dh]; positions < pos0[i] hold its history, the layer writes rows for
 * its new tokens.  x_in/x_out are the residual stream [T, d]; attn_out (may be
 * NULL) receives the attention output [T, H*Dh] before it is rounded. */
int orc_layer_forward(const orc_dims* dims, const orc_layer_weights* w,
                      int32_t B, const int32_t* cu_q, const int32_t* pos0,
                      const int64_t* kv_row0, float* k_pool, float* v_pool,
                      const float* x_in, float* x_out, float* attn_out);

/* Final RMSNorm of the selected rows, the LM head in fp32 and greedy argmax.
 * rows[r] indexes x; logits [R, V]; tokens [R] (may be NULL). */
int orc_lm_head(const orc_dims* dims, const float* gamma_final, const float* w_lm,
                int32_t V, const float* x, const int32_t* rows, int32_t R,
                float* logits, int32_t* tokens);

/* Embedding gather: x[t] = E[ids[t]] */
int orc_embed(const float* E, int32_t V, int32_t d, const int32_t* ids, int64_t T, float* x);

/* Number of OpenMP threads the oracle uses (1 if built without OpenMP). */
int orc_num_threads(void);
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
