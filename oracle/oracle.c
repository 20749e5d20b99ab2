/*
 * CPU oracle for the batch-invariant transformer forward step.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the bench's
 * CPU-baseline leg; never by the product path.  Shares no code with the CUDA
 * library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math [-fopenmp] -fPIC -shared
 *
 * Each function is a plain definition written as serial binary32 loops (see
 * oracle.h for the page and section each follows).  OpenMP, when present, only
 * splits independent rows, (token, head) pairs or output elements across
 * threads; every individual sum is one serial loop, so the result does not
 * depend on the thread count.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* binary32 / bf16 primitives                                                */
/* ------------------------------------------------------------------------ */

/* bf16 keeps the top 16 bits of a binary32.  Round to nearest, ties to even:
 * add 0x7fff plus the lowest kept bit, then truncate.  NaNs are kept NaN by
 * forcing a quiet-NaN mantissa bit. */
float orc_bf16_round(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) {
        u = (u | 0x00400000u) & 0xffff0000u;
    } else {
        uint32_t keep_lsb = (u >> 16) & 1u;
        u = (u + 0x7fffu + keep_lsb) & 0xffff0000u;
    }
    float r;
    memcpy(&r, &u, sizeof r);
    return r;
}

void orc_bf16_round_array(const float* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(in[i]);
}

static float maybe_round(float x, int round_bf16) {
    return round_bf16 ? orc_bf16_round(x) : x;
}

/* "Batch invariance and reproducible inference", "Non-associativity,
 * concretely": the serial order adds left to right. */
float orc_sum_serial(const float* x, int64_t n) {
    float acc = 0.0f;
    if (n <= 0) return acc;
    acc = x[0];
    for (int64_t i = 1; i < n; ++i) acc = acc + x[i];
    return acc;
}

/* Pairwise order: sum each half, then add the two halves (for n = 4 this is
 * (x0 + x1) + (x2 + x3)). */
float orc_sum_pairwise(const float* x, int64_t n) {
    if (n <= 0) return 0.0f;
    if (n == 1) return x[0];
    int64_t h = n / 2;
    float a = orc_sum_pairwise(x, h);
    float b = orc_sum_pairwise(x + h, n - h);
    return a + b;
}

/* ------------------------------------------------------------------------ */
/* Row operations                                                            */
/* ------------------------------------------------------------------------ */

int orc_rmsnorm(const float* x, const float* gamma, float* y,
                int64_t rows, int32_t d, float eps, int round_bf16) {
    if (!x || !gamma || !y || rows < 0 || d <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * (int64_t)d;
        float* yr = y + r * (int64_t)d;
        float ss = 0.0f;
        for (int32_t i = 0; i < d; ++i) ss = ss + xr[i] * xr[i];
        float mean = ss / (float)d;
        float rinv = 1.0f / sqrtf(mean + eps);
        for (int32_t i = 0; i < d; ++i) {
            float v = (xr[i] * rinv) * gamma[i];
            yr[i] = maybe_round(v, round_bf16);
        }
    }
    return 0;
}

int orc_matmul(const float* A, const float* W, float* C,
               int64_t M, int32_t N, int32_t K) {
    if (!A || !W || !C || M < 0 || N < 0 || K < 0) return -1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int32_t n = 0; n < N; ++n) {
            const float* a = A + m * (int64_t)K;
            const float* w = W + (int64_t)n * K;
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) acc = acc + a[k] * w[k];
            C[m * (int64_t)N + n] = acc;
        }
    }
    return 0;
}

int orc_softmax(const float* s, float* p, int32_t n) {
    if (!s || !p || n <= 0) return -1;
    float m = s[0];
    for (int32_t j = 1; j < n; ++j) if (s[j] > m) m = s[j];
    float z = 0.0f;
    for (int32_t j = 0; j < n; ++j) {
        p[j] = expf(s[j] - m);
        z = z + p[j];
    }
    for (int32_t j = 0; j < n; ++j) p[j] = p[j] / z;
    return 0;
}

int orc_swiglu(const float* g, const float* u, float* h, int64_t n, int round_bf16) {
    if (!g || !u || !h || n < 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float silu = g[i] / (1.0f + expf(-g[i]));
        h[i] = maybe_round(silu * u[i], round_bf16);
    }
    return 0;
}

/* "temperature=0 means deterministic": greedy decoding is an argmax.  Ties go
 * to the lowest index; a NaN is larger than any number, and the first NaN
 * wins among NaNs. */
int32_t orc_argmax(const float* x, int32_t n) {
    if (!x || n <= 0) return -1;
    int32_t best = 0;
    for (int32_t j = 1; j < n; ++j) {
        float b = x[best], c = x[j];
        int b_nan = isnan(b), c_nan = isnan(c);
        if (b_nan) break;               /* first NaN already holds */
        if (c_nan || c > b) best = j;
    }
    return best;
}

int orc_argmax_rows(const float* x, int32_t* out, int64_t rows, int32_t n) {
    if (!x || !out || rows < 0 || n <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) out[r] = orc_argmax(x + r * (int64_t)n, n);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Logprobs and seeded sampling                                               */
/* ------------------------------------------------------------------------ */

/* "Mathematically equivalent is not bitwise equivalent": logprobs are the
 * log_softmax of the logits.  The definition, row by row, in float64. */
int orc_log_softmax_rows(const float* x, double* lp, int64_t rows, int32_t n) {
    if (!x || !lp || rows < 0 || n <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * (int64_t)n;
        double m = (double)xr[0];
        for (int32_t j = 1; j < n; ++j) if ((double)xr[j] > m) m = (double)xr[j];
        double z = 0.0;
        for (int32_t j = 0; j < n; ++j) z += exp((double)xr[j] - m);
        const double lz = log(z);
        for (int32_t j = 0; j < n; ++j) lp[r * (int64_t)n + j] = ((double)xr[j] - m) - lz;
    }
    return 0;
}

static uint32_t rotl32(uint32_t v, int r) { return (v << r) | (v >> (32 - r)); }

/* MurmurHash3_x86_32 (Austin Appleby's public-domain hash): 4-byte blocks
 * read little-endian, each scrambled and mixed into h; the 1-3 tail bytes
 * scrambled into h; then the length and the final avalanche. */
uint32_t orc_murmur3_32(const uint8_t* key, int32_t len, uint32_t seed) {
    const uint32_t c1 = 0xcc9e2d51u, c2 = 0x1b873593u;
    uint32_t h = seed;
    const int32_t nblocks = len / 4;
    for (int32_t i = 0; i < nblocks; ++i) {
        uint32_t k = (uint32_t)key[4 * i] | ((uint32_t)key[4 * i + 1] << 8) | ((uint32_t)key[4 * i + 2] << 16) |
                     ((uint32_t)key[4 * i + 3] << 24);
        k *= c1;
        k = rotl32(k, 15);
        k *= c2;
        h ^= k;
        h = rotl32(h, 13);
        h = h * 5u + 0xe6546b64u;
    }
    const uint8_t* tail = key + 4 * nblocks;
    uint32_t k = 0;
    switch (len & 3) {
        case 3: k ^= (uint32_t)tail[2] << 16; /* fall through */
        case 2: k ^= (uint32_t)tail[1] << 8;  /* fall through */
        case 1:
            k ^= (uint32_t)tail[0];
            k *= c1;
            k = rotl32(k, 15);
            k *= c2;
            h ^= k;
    }
    h ^= (uint32_t)len;
    h ^= h >> 16;
    h *= 0x85ebca6bu;
    h ^= h >> 13;
    h *= 0xc2b2ae35u;
    h ^= h >> 16;
    return h;
}

/* "The weaker guarantees, which are usually enough": a request's draws come
 * from its own seed, position and the column, not from a global stream. */
int32_t orc_sample_gumbel(const float* x, int32_t n, uint32_t seed, int32_t pos, float t) {
    if (!x || n <= 0) return -1;
    if (!(t > 0.0f)) return orc_argmax(x, n); /* temperature 0 (or not positive): greedy */
    int32_t best = -1;
    double best_s = 0.0;
    for (int32_t j = 0; j < n; ++j) {
        uint8_t key[8];
        const uint32_t p = (uint32_t)pos, c = (uint32_t)j;
        for (int b = 0; b < 4; ++b) {
            key[b] = (uint8_t)(p >> (8 * b));
            key[4 + b] = (uint8_t)(c >> (8 * b));
        }
        const uint32_t h = orc_murmur3_32(key, 8, seed);
        const double u = ((double)h + 0.5) / 4294967296.0;
        const double g = -log(-log(u));
        const double sc = (double)x[j] / (double)t + g;
        if (best < 0) {
            best = j;
            best_s = sc;
            continue;
        }
        if (isnan(best_s)) break; /* first NaN already holds */
        if (isnan(sc) || sc > best_s) {
            best = j;
            best_s = sc;
        }
    }
    return best;
}

int orc_sample_gumbel_rows(const float* x, const uint32_t* seeds, const int32_t* pos, const float* t,
                           int32_t* out, int64_t rows, int32_t n) {
    if (!x || !seeds || !pos || !t || !out || rows < 0 || n <= 0) return -1;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t r = 0; r < rows; ++r) {
        out[r] = orc_sample_gumbel(x + r * (int64_t)n, n, seeds[r], pos[r], t[r]);
        bad |= out[r] < 0;
    }
    return bad ? -2 : 0;
}

/* ------------------------------------------------------------------------ */
/* Rotary embedding                                                          */
/* ------------------------------------------------------------------------ */

int orc_rope_table(float* cos_t, float* sin_t, int32_t n_pos, int32_t Dh, double theta) {
    if (!cos_t || !sin_t || n_pos < 0 || Dh <= 0 || (Dh & 1)) return -1;
    int32_t half = Dh / 2;
    for (int32_t i = 0; i < half; ++i) {
        double inv_freq = pow(theta, -(double)(2 * i) / (double)Dh);
        for (int32_t p = 0; p < n_pos; ++p) {
            double ang = (double)p * inv_freq;
            cos_t[(int64_t)p * half + i] = (float)cos(ang);
            sin_t[(int64_t)p * half + i] = (float)sin(ang);
        }
    }
    return 0;
}

/* Rotate-half pairing: element i pairs with element i + Dh/2. */
int orc_rope_apply(float* x, const int32_t* pos, int64_t n_vec, int32_t Dh,
                   const float* cos_t, const float* sin_t, int32_t n_pos) {
    if (!x || !pos || !cos_t || !sin_t || Dh <= 0 || (Dh & 1)) return -1;
    int32_t half = Dh / 2;
    for (int64_t v = 0; v < n_vec; ++v) {
        int32_t p = pos[v];
        if (p < 0 || p >= n_pos) return -2;
        float* xv = x + v * (int64_t)Dh;
        const float* c = cos_t + (int64_t)p * half;
        const float* s = sin_t + (int64_t)p * half;
        for (int32_t i = 0; i < half; ++i) {
            float x0 = xv[i], x1 = xv[i + half];
            float a = x0 * c[i];
            float b = x1 * s[i];
            float e = x1 * c[i];
            float f = x0 * s[i];
            xv[i] = a - b;
            xv[i + half] = e + f;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                 */
/* ------------------------------------------------------------------------ */

static float dot_serial(const float* a, const float* b, int32_t n) {
    float acc = 0.0f;
    for (int32_t i = 0; i < n; ++i) acc = acc + a[i] * b[i];
    return acc;
}

int orc_attention_head(const float* q, const float* k, const float* v,
                       int32_t n_keys, int64_t kv_stride, int32_t Dh,
                       float scale, float* out) {
    if (!q || !k || !v || !out || n_keys <= 0 || Dh <= 0) return -1;
    float* s = (float*)malloc(sizeof(float) * (size_t)n_keys * 2);
    if (!s) return -3;
    float* p = s + n_keys;
    for (int32_t j = 0; j < n_keys; ++j)
        s[j] = dot_serial(q, k + (int64_t)j * kv_stride, Dh) * scale;
    orc_softmax(s, p, n_keys);
    for (int32_t d = 0; d < Dh; ++d) {
        float acc = 0.0f;
        for (int32_t j = 0; j < n_keys; ++j) acc = acc + p[j] * v[(int64_t)j * kv_stride + d];
        out[d] = acc;
    }
    free(s);
    return 0;
}

/* "Batch invariance and reproducible inference", "1 · Split-K and segmented
 * attention reductions": the key axis is cut into chunks whose fp32 partials
 * are merged.  Here the chunk boundaries are multiples of `chunk` from key 0. */
int orc_attention_head_split(const float* q, const float* k, const float* v,
                             int32_t n_keys, int64_t kv_stride, int32_t Dh,
                             float scale, int32_t chunk, float* out) {
    if (!q || !k || !v || !out || n_keys <= 0 || Dh <= 0 || chunk <= 0) return -1;
    int32_t n_chunks = (n_keys + chunk - 1) / chunk;
    float* m = (float*)malloc(sizeof(float) * (size_t)n_chunks * (2 + Dh));
    float* s = (float*)malloc(sizeof(float) * (size_t)chunk);
    if (!m || !s) { free(m); free(s); return -3; }
    float* l = m + n_chunks;
    float* o = l + n_chunks;
    for (int32_t c = 0; c < n_chunks; ++c) {
        int32_t j0 = c * chunk;
        int32_t n = n_keys - j0 < chunk ? n_keys - j0 : chunk;
        for (int32_t j = 0; j < n; ++j)
            s[j] = dot_serial(q, k + (int64_t)(j0 + j) * kv_stride, Dh) * scale;
        float mc = s[0];
        for (int32_t j = 1; j < n; ++j) if (s[j] > mc) mc = s[j];
        float lc = 0.0f;
        for (int32_t j = 0; j < n; ++j) { s[j] = expf(s[j] - mc); lc = lc + s[j]; }
        for (int32_t d = 0; d < Dh; ++d) {
            float acc = 0.0f;
            for (int32_t j = 0; j < n; ++j) acc = acc + s[j] * v[(int64_t)(j0 + j) * kv_stride + d];
            o[(int64_t)c * Dh + d] = acc;
        }
        m[c] = mc;
        l[c] = lc;
    }
    float M = m[0];
    for (int32_t c = 1; c < n_chunks; ++c) if (m[c] > M) M = m[c];
    float L = 0.0f;
    for (int32_t c = 0; c < n_chunks; ++c) L = L + l[c] * expf(m[c] - M);
    for (int32_t d = 0; d < Dh; ++d) {
        float O = 0.0f;
        for (int32_t c = 0; c < n_chunks; ++c) O = O + o[(int64_t)c * Dh + d] * expf(m[c] - M);
        out[d] = O / L;
    }
    free(m);
    free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* One decoder layer                                                         */
/* ------------------------------------------------------------------------ */

int orc_layer_forward(const orc_dims* dims, const orc_layer_weights* w,
                      int32_t B, const int32_t* cu_q, const int32_t* pos0,
                      const int64_t* kv_row0, float* k_pool, float* v_pool,
                      const float* x_in, float* x_out, float* attn_out) {
    if (!dims || !w || !cu_q || !pos0 || !kv_row0 || !k_pool || !v_pool || !x_in || !x_out)
        return -1;
    const int32_t d = dims->d, H = dims->H, Hkv = dims->Hkv, Dh = dims->Dh, F = dims->F;
    const int rb = dims->round_bf16;
    if (d <= 0 || H <= 0 || Hkv <= 0 || Dh <= 0 || F <= 0 || H % Hkv != 0 || B < 0) return -1;
    const int64_t T = cu_q[B];
    const int32_t NQKV = (H + 2 * Hkv) * Dh;
    const int32_t group = H / Hkv;
    const float scale = 1.0f / sqrtf((float)Dh);

    int32_t max_pos = 0;
    for (int32_t i = 0; i < B; ++i) {
        int32_t end = pos0[i] + (cu_q[i + 1] - cu_q[i]);
        if (end > max_pos) max_pos = end;
    }

    float* y    = (float*)malloc(sizeof(float) * (size_t)(T * d + 1));
    float* qkv  = (float*)malloc(sizeof(float) * (size_t)(T * NQKV + 1));
    float* att  = (float*)malloc(sizeof(float) * (size_t)(T * H * Dh + 1));
    float* tmp  = (float*)malloc(sizeof(float) * (size_t)(T * d + 1));
    float* g    = (float*)malloc(sizeof(float) * (size_t)(T * F + 1));
    float* u    = (float*)malloc(sizeof(float) * (size_t)(T * F + 1));
    float* cos_t = (float*)malloc(sizeof(float) * (size_t)(max_pos * (Dh / 2) + 1));
    float* sin_t = (float*)malloc(sizeof(float) * (size_t)(max_pos * (Dh / 2) + 1));
    int32_t* tok_pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T + 1));
    int32_t* tok_req = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T + 1));
    int rc = 0;
    if (!y || !qkv || !att || !tmp || !g || !u || !cos_t || !sin_t || !tok_pos || !tok_req) {
        rc = -3;
        goto done;
    }
    for (int32_t i = 0; i < B; ++i)
        for (int32_t t = cu_q[i]; t < cu_q[i + 1]; ++t) {
            tok_req[t] = i;
            tok_pos[t] = pos0[i] + (t - cu_q[i]);
        }
    orc_rope_table(cos_t, sin_t, max_pos, Dh, dims->rope_theta);

    /* 1. pre-attention RMSNorm (stored bf16) */
    orc_rmsnorm(x_in, w->gamma_attn, y, T, d, dims->eps, rb);
    /* 2. q, k, v projections in fp32 */
    orc_matmul(y, w->w_qkv, qkv, T, NQKV, d);
    /* 3. RoPE on q and k, then bf16 storage of q, k, v; k and v go to the pool */
    for (int64_t t = 0; t < T; ++t) {
        float* row = qkv + t * NQKV;
        int32_t p = tok_pos[t];
        for (int32_t h = 0; h < H + Hkv; ++h)
            orc_rope_apply(row + (int64_t)h * Dh, &p, 1, Dh, cos_t, sin_t, max_pos);
        for (int32_t j = 0; j < NQKV; ++j) row[j] = maybe_round(row[j], rb);
        int64_t kv_row = kv_row0[tok_req[t]] + p;
        memcpy(k_pool + kv_row * Hkv * Dh, row + (int64_t)H * Dh, sizeof(float) * (size_t)Hkv * Dh);
        memcpy(v_pool + kv_row * Hkv * Dh, row + (int64_t)(H + Hkv) * Dh, sizeof(float) * (size_t)Hkv * Dh);
    }
    /* 4. causal attention: the query at position p sees keys 0..p of its own request */
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) {
            int32_t p = tok_pos[t];
            int32_t kvh = h / group;
            int64_t base = (kv_row0[tok_req[t]] * Hkv + kvh) * (int64_t)Dh;
            orc_attention_head(qkv + t * NQKV + (int64_t)h * Dh, k_pool + base, v_pool + base,
                               p + 1, (int64_t)Hkv * Dh, Dh, scale, att + (t * H + h) * (int64_t)Dh);
        }
    }
    if (attn_out) memcpy(attn_out, att, sizeof(float) * (size_t)(T * H * Dh));
    for (int64_t j = 0; j < T * H * Dh; ++j) att[j] = maybe_round(att[j], rb);
    /* 5. output projection plus residual, stored bf16 */
    orc_matmul(att, w->w_o, tmp, T, d, H * Dh);
    for (int64_t j = 0; j < T * d; ++j) x_out[j] = maybe_round(x_in[j] + tmp[j], rb);
    /* 6. pre-FFN RMSNorm */
    orc_rmsnorm(x_out, w->gamma_ffn, y, T, d, dims->eps, rb);
    /* 7. gate and up projections, SwiGLU stored bf16 */
    orc_matmul(y, w->w_gate, g, T, F, d);
    orc_matmul(y, w->w_up, u, T, F, d);
    orc_swiglu(g, u, g, T * F, rb);
    /* 8. down projection plus residual, stored bf16 */
    orc_matmul(g, w->w_down, tmp, T, d, F);
    for (int64_t j = 0; j < T * d; ++j) x_out[j] = maybe_round(x_out[j] + tmp[j], rb);

done:
    free(y); free(qkv); free(att); free(tmp); free(g); free(u);
    free(cos_t); free(sin_t); free(tok_pos); free(tok_req);
    return rc;
}

int orc_lm_head(const orc_dims* dims, const float* gamma_final, const float* w_lm,
                int32_t V, const float* x, const int32_t* rows, int32_t R,
                float* logits, int32_t* tokens) {
    if (!dims || !gamma_final || !w_lm || !x || !rows || !logits || V <= 0 || R < 0) return -1;
    const int32_t d = dims->d;
    float* xr = (float*)malloc(sizeof(float) * (size_t)R * d + 1);
    float* y = (float*)malloc(sizeof(float) * (size_t)R * d + 1);
    if (!xr || !y) { free(xr); free(y); return -3; }
    for (int32_t r = 0; r < R; ++r) memcpy(xr + (int64_t)r * d, x + (int64_t)rows[r] * d, sizeof(float) * (size_t)d);
    orc_rmsnorm(xr, gamma_final, y, R, d, dims->eps, dims->round_bf16);
    orc_matmul(y, w_lm, logits, R, V, d);
    if (tokens) orc_argmax_rows(logits, tokens, R, V);
    free(xr);
    free(y);
    return 0;
}

int orc_embed(const float* E, int32_t V, int32_t d, const int32_t* ids, int64_t T, float* x) {
    if (!E || !ids || !x || V <= 0 || d <= 0 || T < 0) return -1;
    for (int64_t t = 0; t < T; ++t) {
        if (ids[t] < 0 || ids[t] >= V) return -2;
        memcpy(x + t * d, E + (int64_t)ids[t] * d, sizeof(float) * (size_t)d);
    }
    return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
