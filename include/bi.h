/*
 * bi.h — C ABI of the batch-invariant transformer forward step for one GB300
 * (sm_103a).
 *
 * Invariant-mode contract ("Lockstep", "The fix" and "Proving it"): for any
 * request, its rows of every output (logits, tokens, hidden states) are
 * bit-identical whatever the other rows of the batch are, whatever their order,
 * and however its own prompt was cut into prefill chunks.  Every reduction runs
 * in one fixed order with split points that depend on the request alone:
 *   - RMSNorm: one warp per row, lane-serial over 16-byte chunks, then a fixed
 *     xor-butterfly;
 *   - GEMM: tcgen05 MMAs (the two-SM pair form with M = 256 or, for at most
 *     64 rows, 128, or the single-SM form with M = 128; N = the tile width,
 *     128 or 256; all give every element the same bits), bf16 in, fp32
 *     accumulate in TMEM, one K tile (64), K loop in ascending order, no
 *     split-K, whatever M is;
 *   - attention: keys cut into chunks of BI_KV_CHUNK positions aligned to key 0
 *     ("Batch invariance and reproducible inference", "1 · Split-K and
 *     segmented attention reductions"), fp32 partials merged in ascending chunk
 *     order, the same arithmetic for decode and prefill;
 *   - argmax: lowest index among the maxima, NaN larger than any number.
 * BI_VARIANT mode ("From batch size to reduction tree") lets the attention
 * split count follow occupancy (the batch size) and the GEMM split K over an
 * fp32 workspace when few output tiles are available: it is the fast path and
 * the negative control, and its results depend on the batch.
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented DEVICE are device pointers owned by the
 *     caller; HOST pointers are read during the call only.  The library keeps
 *     no pointer after a call returns except those handed to bi_model_create
 *     (borrowed until bi_model_destroy).
 *   - bf16 tensors are arrays of bi_bf16 (the 16-bit bf16 bit pattern).
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous.  No call allocates device memory except
 *     bi_model_create (its RoPE table).  Workspaces are caller-owned, sized by
 *     the *_workspace_size functions, 16-byte aligned (as cudaMalloc's are),
 *     and only the call they are passed to may use them until that call's
 *     work has finished on the stream.
 *   - Argument validation happens before any launch: on failure nothing is
 *     launched or written, the call returns a bi_status other than BI_OK and
 *     bi_last_error() describes it.
 *   - Faults found on the device (a page index outside the pool, a bounded
 *     wait that ran out, a token id outside the vocabulary) are written as a
 *     nonzero code into the caller's `dev_status` word (DEVICE int32; the first
 *     fault wins) and the kernels skip the offending access.
 *     bi_check_status() synchronises the stream and turns the word into a
 *     bi_status.  No kernel traps, asserts or waits without a bound.
 */
#ifndef BI_H
#define BI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t bi_bf16;   /* bf16 bit pattern */
typedef void* bi_stream;    /* cudaStream_t */

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID = 1,      /* null pointer, misaligned pointer, bad enum */
    BI_ERR_SHAPE = 2,        /* sizes outside what the kernels support */
    BI_ERR_UNSUPPORTED = 3,  /* a combination with no invariant path */
    BI_ERR_CUDA = 4,         /* a CUDA runtime call failed */
    BI_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out */
    BI_ERR_DEVICE = 6,       /* a device-side check failed (index out of range) */
    BI_ERR_WORKSPACE = 7     /* workspace too small */
} bi_status;

typedef enum { BI_INVARIANT = 0, BI_VARIANT = 1 } bi_mode;
typedef enum { BI_BF16 = 0, BI_F32 = 1 } bi_dtype;
typedef enum {
    BI_EP_NONE = 0,      /* C = acc */
    BI_EP_RESIDUAL = 1,  /* C = bf16(acc + residual); C may alias residual */
    BI_EP_SWIGLU = 2     /* gate/up interleaved in groups of 32 rows: C[:, N/2] = bf16(silu(g) * u) */
} bi_epilogue;

/* Fixed constants of the method (never functions of a batch). */
#define BI_KV_CHUNK 256      /* attention key chunk (positions) */
#define BI_PAGE 16           /* KV page (positions) */
#define BI_GEMM_BLOCK_M 128  /* accumulator rows per CTA (a pair MMA spans two CTAs: M = 256) */
#define BI_GEMM_UMMA_N 128  /* MMA N */
#define BI_GEMM_BLOCK_K 64   /* K tile */
#define BI_SWIGLU_GROUP 32   /* gate/up interleave group (rows) */

/* Device status codes written into dev_status. */
#define BI_DEV_OK 0
#define BI_DEV_TIMEOUT_PRODUCER 0x101
#define BI_DEV_TIMEOUT_MMA 0x102
#define BI_DEV_TIMEOUT_EPILOGUE 0x103
#define BI_DEV_TIMEOUT_DRAIN 0x104
#define BI_DEV_TIMEOUT_ATTENTION 0x105  /* a K/V copy into an attention CTA did not land in time */
#define BI_DEV_PAIR_TMEM 0x106  /* the two CTAs of a GEMM pair were given different tensor-memory columns */
#define BI_DEV_BAD_PAGE 0x201
#define BI_DEV_BAD_POSITION 0x202
#define BI_DEV_BAD_TOKEN 0x203
#define BI_DEV_BAD_LOGIT_ROWS 0x204  /* a replayed step's device logit rows are not the 0..R-1 its capture fused on */

/* ---- diagnostics -------------------------------------------------------- */

/* Thread-local message describing the last failed call on this thread. */
const char* bi_last_error(void);
/* ABI version of this library. */
int32_t bi_version(void);
/* Synchronises `stream`, reads the DEVICE word *dev_status and maps it:
 * 0 -> BI_OK, timeout codes -> BI_ERR_TIMEOUT, others -> BI_ERR_DEVICE. */
bi_status bi_check_status(const int32_t* dev_status, bi_stream stream);
/* Enqueues a write of 0 to the DEVICE word *dev_status. */
bi_status bi_reset_status(int32_t* dev_status, bi_stream stream);

/* ---- RMSNorm ("Lockstep", "The fix"; row reduction in one fixed order) ---
 * y[r, i] = bf16( (x[r, i] * rinv_r) * gamma[i] ),
 * rinv_r  = 1 / sqrt( (sum_i x[r, i]^2) / d + eps ),
 * the sum in fp32: each lane of a warp adds the squares of its 16-byte chunks
 * (8 elements, chunk c goes to lane c % 32) in ascending order, then the 32
 * lane sums meet in an xor-butterfly (16, 8, 4, 2, 1).
 * x, y: DEVICE [rows, d] row-major (may alias); gamma: DEVICE [d].
 * Requires d % 8 == 0 and 16-byte aligned pointers. */
bi_status bi_rmsnorm(const bi_bf16* x, const bi_bf16* gamma, bi_bf16* y,
                     int64_t rows, int32_t d, float eps, bi_stream stream);

/* ---- GEMM ("Batch invariance and reproducible inference", "2 · Cross-block
 * accumulation" and "3 · Kernel selection changing with shape") -------------
 * C[m, n] = sum_k A[m, k] * W[n, k] with fp32 accumulation, then the epilogue.
 * A: DEVICE [M, K] bf16 row-major; W: DEVICE [N, K] bf16 row-major (the
 * nn.Linear layout); C: DEVICE [M, N] (or [M, N/2] for BI_EP_SWIGLU) in c_dtype
 * (BI_EP_RESIDUAL and BI_EP_SWIGLU need BI_BF16); residual: DEVICE [M, N] bf16
 * for BI_EP_RESIDUAL, else NULL.
 * BI_INVARIANT: every element's K sum, for every M, runs in ascending 64-wide K
 * tiles through 16-deep MMAs into one TMEM accumulator; only data movement
 * (the MMA form and tile width, TMA box, ring depth) may follow M.
 * BI_VARIANT: when the output has fewer tiles than SMs, K is split over CTAs
 * into an fp32 workspace and the partials are added in split order.
 * Requires K % 64 == 0, N % 128 == 0, M >= 0, 16-byte aligned pointers.
 * ws: DEVICE scratch of at least bi_gemm_workspace_size(M, N, K, mode) bytes
 * (0 in invariant mode; may then be NULL). */
size_t bi_gemm_workspace_size(int64_t M, int32_t N, int32_t K, bi_mode mode);
bi_status bi_gemm(const bi_bf16* A, const bi_bf16* W, void* C, bi_dtype c_dtype,
                  const bi_bf16* residual, bi_epilogue ep,
                  int64_t M, int32_t N, int32_t K, bi_mode mode,
                  void* ws, size_t ws_bytes, int32_t* dev_status, bi_stream stream);

/* bi_gemm's failure-detection check (for tests; the pages have no
 * counterpart).  Runs bi_gemm (BI_INVARIANT, no epilogue) with two changes:
 * every bounded wait of the kernel gives up after wait_limit_ns (1 ms to 2 s),
 * and the copies of ring stage skip_stage (counted in issue order from 0, in
 * every CTA of a pair; -1: none) are never issued.  The MMA issuer's wait for
 * that stage then runs out: the kernel writes BI_DEV_TIMEOUT_MMA into
 * dev_status (DEVICE, required), every role stops, the copies and products
 * in flight are drained, tensor memory is freed and the kernel returns; C
 * holds no defined values.  Nothing faults or waits without a bound, and the
 * stream stays usable. */
bi_status bi_gemm_wait_test(const bi_bf16* A, const bi_bf16* W, void* C, bi_dtype c_dtype, int64_t M,
                            int32_t N, int32_t K, uint64_t wait_limit_ns, int32_t skip_stage,
                            int32_t* dev_status, bi_stream stream);

/* Packs logical gate [F, d] and up [F, d] weights into the interleaved [2F, d]
 * layout BI_EP_SWIGLU reads: rows 64j..64j+31 = gate rows 32j..32j+31, rows
 * 64j+32..64j+63 = up rows 32j..32j+31.  All DEVICE; F % 32 == 0. */
bi_status bi_pack_gate_up(const bi_bf16* w_gate, const bi_bf16* w_up, bi_bf16* w_gu,
                          int32_t F, int32_t d, bi_stream stream);

/* ---- RoPE + KV append ----------------------------------------------------
 * qkv: DEVICE [T, (H + 2*Hkv) * Dh] fp32 (q heads, then k heads, then v heads).
 * Token t sits at position tok_pos[t] of request tok_req[t] (DEVICE [T] each).
 * q and k are rotated (rotate-half: element i pairs with i + Dh/2; angle
 * pos * theta^(-2i/Dh), cos/sin tabulated in float64 and rounded to fp32:
 * rope_cos/rope_sin DEVICE [max_pos, Dh/2]), then q goes to q_out (DEVICE
 * [T, H, Dh] bf16) and k, v to the paged caches.
 * KV cache layout (per layer): DEVICE [num_pages, Hkv, BI_PAGE, Dh] bf16;
 * position p of request r lives in page page_table[r * max_pages + p / 16],
 * slot p % 16.  page_table: DEVICE [*, max_pages] int32. */
bi_status bi_rope_kv_append(const float* qkv, const int32_t* tok_req, const int32_t* tok_pos,
                            const float* rope_cos, const float* rope_sin, int32_t max_pos,
                            bi_bf16* q_out, bi_bf16* k_cache, bi_bf16* v_cache,
                            const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                            int32_t T, int32_t H, int32_t Hkv, int32_t Dh,
                            int32_t* dev_status, bi_stream stream);

/* Host helper: fills HOST cos/sin tables [n_pos, Dh/2] (float64 angles and
 * cos/sin rounded to fp32). */
bi_status bi_rope_table(float* cos_out, float* sin_out, int32_t n_pos, int32_t Dh, double theta);

/* ---- Attention ("Lockstep", "The fix": split points from the request;
 * "Batch invariance and reproducible inference", "1 · Split-K and segmented
 * attention reductions") -----------------------------------------------------
 * For query head h (kv head h / (H/Hkv)) of a token at position p: keys
 * 0..p of its request, cut into chunks [256j, min(256j + 256, p + 1)).  Per
 * chunk, in fp32: s_j = (k_j . q) * scale, the dot product on the tensor
 * cores (bf16 products, fp32 accumulation over 16-deep steps of the head dim
 * in ascending order); m = max_j s_j; p_j = exp(s_j - m); l = sum_j p_j in a
 * fixed tree (per thread t of 128 the serial sum over j = t, t + 128, then an
 * xor-butterfly over each warp's 32 lanes, then the 4 warps in order);
 * o = sum_j p_j v_j on the tensor cores with p_j split into bf16 hi and lo
 * parts, 16-key steps in ascending order.  Chunks merge in ascending order:
 * state (M, L, O) starts at chunk 0; each next chunk gives M' = max(M, m),
 * L' = L e^(M-M') + l e^(m-M'), O' = O e^(M-M') + o e^(m-M'); the output is
 * O / L.  Decode and prefill run the same per-chunk arithmetic and the same
 * merge, so a position's output has the same bits from either.
 * Supported: Dh in {64, 128}, H / Hkv in {1, 2, 4, 8}.
 *
 * bi_decode_attention: one query per request at position seq_lens[i] - 1
 * (its K/V already appended).  q: DEVICE [B, H, Dh] bf16; out: DEVICE
 * [B, H, Dh] in out_dtype; seq_lens: DEVICE [B]; max_seq_len: HOST bound on
 * seq_lens (sizes the grid; larger values are reported as BI_DEV_BAD_POSITION).
 * BI_VARIANT: the split count follows the occupancy rule of "From batch size
 * to reduction tree" with num_seq = B, device_core_count = the SM count,
 * block_h = min(16, H/Hkv), max_kv_splits = 16 and kv_chunk_size_1 = 256:
 *   cores2  = int(cores * max(log2(max_s / 64), 1)),
 *   splits2 = min(ceil(cores2 / (B * ceil(H / block_h))), 16),
 *   chunk2  = ceil(max_s / splits2),
 *   n_i     = max(ceil(s_i / 256), ceil(s_i / chunk2)),
 * and request i's keys are cut into pieces of ceil(s_i / n_i) positions from
 * key 0; so the pieces depend on the batch.  max_s = max_seq_len.
 * ws: DEVICE scratch of bi_decode_attention_workspace_size bytes.
 * scale <= 0 (or NaN) selects the default fl32(1 / fl32(sqrt(Dh))). */
size_t bi_decode_attention_workspace_size(int32_t B, int32_t H, int32_t Dh, int32_t max_seq_len,
                                          bi_mode mode);
bi_status bi_decode_attention(const bi_bf16* q, const bi_bf16* k_cache, const bi_bf16* v_cache,
                              const int32_t* page_table, const int32_t* seq_lens,
                              void* out, bi_dtype out_dtype,
                              int32_t B, int32_t H, int32_t Hkv, int32_t Dh,
                              int32_t max_pages, int32_t num_pages, int32_t max_seq_len,
                              float scale, bi_mode mode, void* ws, size_t ws_bytes,
                              int32_t* dev_status, bi_stream stream);

/* bi_decode_attention_noalloc: bi_decode_attention for callers that cannot
 * allocate device memory where they run it (an allocator that forbids new
 * allocations once serving has started, a host that only hands over input
 * and output pointers).  There is no counterpart on the pages; it is a
 * packaging of the same kernels.  The split partials live in one static
 * device array of 16 MiB (16777216 bytes) that every GPU loading this
 * library holds until the process exits; the
 * call allocates nothing and computes exactly what bi_decode_attention
 * computes.  A batch whose partials need more
 * (B * H * splits * (Dh + 2) * 4 bytes, splits = ceil(max_seq_len / 256) in
 * invariant mode) is rejected with BI_ERR_WORKSPACE before any launch.
 * The first call on each device (and the first after a device reset, which
 * gives the array a new address) looks up the array's device address; make
 * that first call before any stream capture.  All calls share the one array:
 * calls whose work overlaps on the GPU race and corrupt each other's
 * partials, so keep them ordered (one stream, or events).  Nothing in the
 * array needs to start at zero: each call writes every partial it reads.
 * scale <= 0 (or NaN) selects the default, as in bi_decode_attention. */
bi_status bi_decode_attention_noalloc(const bi_bf16* q, const bi_bf16* k_cache, const bi_bf16* v_cache,
                                      const int32_t* page_table, const int32_t* seq_lens,
                                      void* out, bi_dtype out_dtype,
                                      int32_t B, int32_t H, int32_t Hkv, int32_t Dh,
                                      int32_t max_pages, int32_t num_pages, int32_t max_seq_len,
                                      float scale, bi_mode mode, int32_t* dev_status, bi_stream stream);

/* bi_prefill_attention: causal attention for ragged query blocks.  Request i
 * owns queries [cu_q[i], cu_q[i+1]) at positions q_pos0[i] + t (cu_q: DEVICE
 * [B+1], q_pos0: DEVICE [B]); its K/V for positions 0..q_pos0[i]+q_len-1 must
 * already be in the cache.  q: DEVICE [T, H, Dh] bf16; out: DEVICE [T, H, Dh].
 * max_seq_len: HOST upper bound on q_pos0[i] + q_len_i (0 < max_seq_len <=
 * max_pages * 16).
 * BI_INVARIANT: the same per-(query, chunk) arithmetic and merge as
 * bi_decode_attention, so a token gets the same bits from either call and
 * from any cutting of its prompt into calls ("Batch invariance and
 * reproducible inference", "Mathematically equivalent is not bitwise
 * equivalent": prefill and decode must reduce alike).  The products run on
 * tcgen05 tensor cores with the accumulators in tensor memory; no workspace
 * (ws may be NULL).
 * BI_VARIANT: every query's keys are cut by the occupancy rule documented at
 * bi_decode_attention, with num_seq = B and max_s = max_seq_len, and the
 * pieces merged in order: the split then depends on the batch (the negative
 * control).  Its fp32 partials live in ws.
 * ws: DEVICE scratch of bi_prefill_attention_workspace_size bytes, 16-byte
 * aligned.  scale <= 0 (or NaN) selects the default fl32(1 / fl32(sqrt(Dh))). */
size_t bi_prefill_attention_workspace_size(int32_t T, int32_t H, int32_t Dh, int32_t max_seq_len, bi_mode mode);
bi_status bi_prefill_attention(const bi_bf16* q, const int32_t* cu_q, const int32_t* q_pos0,
                               const bi_bf16* k_cache, const bi_bf16* v_cache,
                               const int32_t* page_table, void* out, bi_dtype out_dtype,
                               int32_t B, int32_t T, int32_t H, int32_t Hkv, int32_t Dh,
                               int32_t max_pages, int32_t num_pages, int32_t max_seq_len, float scale,
                               bi_mode mode, void* ws, size_t ws_bytes,
                               int32_t* dev_status, bi_stream stream);

/* ---- Greedy argmax ("Batch invariance and reproducible inference",
 * "temperature=0 means deterministic") --------------------------------------
 * out[r] = lowest index of the maximum of logits[r, :]; a NaN is larger than
 * any number (the first NaN wins).  logits DEVICE [R, V] fp32; out DEVICE [R]. */
bi_status bi_argmax(const float* logits, int32_t* out, int32_t R, int32_t V, bi_stream stream);

/* ---- Logprobs ("Batch invariance and reproducible inference", "Mathematically
 * equivalent is not bitwise equivalent": logprobs come from one log_softmax
 * kernel, never log(softmax); "The replacement kernels are deliberately dull":
 * no reduction whose order follows the batch) ------------------------------
 * logprobs[r, j] = (logits[r, j] - m_r) - log(z_r), m_r = max_j logits[r, j],
 * z_r = sum_j exp(logits[r, j] - m_r), fp32, summed in one fixed order that
 * depends on V alone (segments of 4096 columns, each reduced in a fixed tree,
 * merged in segment order): a row's logprobs are bitwise the same whatever
 * rows share the call.  A NaN logit makes its row NaN.  logits and logprobs
 * DEVICE [R, V] fp32 (may not overlap); ws DEVICE scratch of
 * bi_log_softmax_workspace_size(R, V) bytes, 16-byte aligned. */
size_t bi_log_softmax_workspace_size(int32_t R, int32_t V);
bi_status bi_log_softmax(const float* logits, float* logprobs, int32_t R, int32_t V,
                         void* ws, size_t ws_bytes, bi_stream stream);

/* ---- Seeded sampling ("Batch invariance and reproducible inference", "The
 * weaker guarantees, which are usually enough": Gumbel noise from
 * murmur_hash32(seed, position, column) in float64) -------------------------
 * tokens[r] = argmax_j (logits[r, j] / t_r + g_j) in float64, where
 *   h_j = MurmurHash3_x86_32(le32(positions[r]) || le32(j), seeds[r]),
 *   u_j = (h_j + 0.5) / 2^32,  g_j = -log(-log(u_j)),  t_r = temperatures[r];
 * ties go to the lowest index and a NaN score beats every number.  A row with
 * t_r <= 0 (or NaN) takes the greedy argmax of its logits (as bi_argmax).  A
 * row's token depends only on its logits, seed, position and temperature.
 * logits DEVICE [R, V] fp32; seeds DEVICE [R] uint32; positions DEVICE [R]
 * int32; temperatures DEVICE [R] fp32; tokens DEVICE [R] int32; ws DEVICE
 * scratch of bi_sample_workspace_size(R, V) bytes, 16-byte aligned. */
size_t bi_sample_workspace_size(int32_t R, int32_t V);
bi_status bi_sample(const float* logits, const uint32_t* seeds, const int32_t* positions,
                    const float* temperatures, int32_t* tokens, int32_t R, int32_t V,
                    void* ws, size_t ws_bytes, bi_stream stream);

/* ---- Embedding gather -----------------------------------------------------
 * x[t] = E[ids[t]]; E DEVICE [V, d] bf16, ids DEVICE [T], x DEVICE [T, d].
 * Requires d % 8 == 0.  Out-of-range ids report BI_DEV_BAD_TOKEN and write 0. */
bi_status bi_embed(const bi_bf16* E, const int32_t* ids, bi_bf16* x, int32_t T, int32_t V,
                   int32_t d, int32_t* dev_status, bi_stream stream);

/* ---- Model and forward step ------------------------------------------------ */
typedef struct {
    int32_t d, H, Hkv, Dh, F, V, n_layers;
    float eps;          /* RMSNorm epsilon */
    double rope_theta;  /* RoPE base */
    int32_t max_pos;    /* positions the RoPE table covers */
} bi_model_config;

/* Weights: DEVICE bf16 pointers, borrowed (must outlive the model).  The
 * per-layer members are HOST arrays of n_layers DEVICE pointers (copied). */
typedef struct {
    const bi_bf16* embed;               /* [V, d] */
    const bi_bf16* gamma_final;         /* [d] */
    const bi_bf16* w_lm;                /* [V, d] */
    const bi_bf16* const* gamma_attn;   /* [d] */
    const bi_bf16* const* w_qkv;        /* [(H + 2*Hkv) * Dh, d] q, k, v rows */
    const bi_bf16* const* w_o;          /* [d, H * Dh] */
    const bi_bf16* const* gamma_ffn;    /* [d] */
    const bi_bf16* const* w_gu;         /* [2F, d] packed by bi_pack_gate_up */
    const bi_bf16* const* w_down;       /* [d, F] */
} bi_model_weights;

/* Per-layer paged KV pools: HOST arrays of n_layers DEVICE pointers, each
 * [num_pages, Hkv, BI_PAGE, Dh] bf16 (read during the call only). */
typedef struct {
    bi_bf16* const* k;
    bi_bf16* const* v;
    int32_t num_pages;
} bi_kv_cache;

/* One ragged step.  Request i contributes q_len[i] >= 1 new tokens at
 * positions pos0[i] .. pos0[i] + q_len[i] - 1; its context after the step is
 * pos0[i] + q_len[i] positions (its earlier positions already in the cache).
 * Requests' tokens are concatenated in order (T = sum q_len). */
typedef struct {
    int32_t B;
    const int32_t* q_len;       /* HOST [B] */
    const int32_t* pos0;        /* HOST [B] */
    const int32_t* token_ids;   /* DEVICE [T] */
    const int32_t* page_table;  /* DEVICE [B, max_pages] */
    int32_t max_pages;
    int32_t R;                  /* rows that need logits */
    const int32_t* logit_rows;  /* HOST [R] token indices in 0..T-1 */
    /* DEVICE [3T + R] or NULL.  NULL: the step derives its per-token metadata
     * from q_len, pos0 and logit_rows and hands it to its first kernel as a
     * launch parameter (3T + R <= 1024: every decode step of up to 256
     * tokens), or copies it host to device through a pinned staging buffer
     * (larger steps).  Non-NULL: the caller has written it on the
     * device: [request of token t, T][position of token t, T][tokens with
     * q_len 1 in token order, nd][the other tokens in order, T - nd][logit
     * rows, R].  The step then reads no host memory after the call and calls
     * nothing that synchronises, so it can be captured in a CUDA graph
     * (programmatic dependent launch and cluster launches are captured as
     * graph edges and nodes) and replayed with new contents of meta,
     * token_ids and page_table.  q_len, pos0 and logit_rows still give the
     * shapes (T, nd, R) and bounds: a replayed position must not exceed the
     * captured pos0[i] + q_len[i] - 1 of its request slot (the attention split
     * count and workspace were sized from it); larger positions are reported
     * as BI_DEV_BAD_POSITION.  When logit_rows is 0..R-1 with R <= 8, the
     * final RMSNorm runs inside the LM head on the first R rows of the
     * residual stream (bit for bit the norm kernel's output), so the logit
     * rows in meta must then be 0..R-1 too: any other list is reported as
     * BI_DEV_BAD_LOGIT_ROWS (the logits then belong to rows 0..R-1). */
    const int32_t* meta;
} bi_batch;

typedef struct bi_model bi_model;

/* bi_model_create ("Lockstep", "The fix": the engine whose output for a
 * request does not depend on its batch; the decoder's steps are the plain
 * Llama-style layer the forward step below lists).  Checks the shapes the
 * kernels support (d, V and (H + 2 Hkv) Dh multiples of 128; F and H Dh
 * multiples of 64; Dh in {64, 128}; H / Hkv in {1, 2, 4, 8}), borrows the
 * weight pointers, copies the per-layer pointer arrays and allocates the
 * model's device buffers: the RoPE cos and sin tables for max_pos positions
 * (bi_rope_table's values).  Returns BI_ERR_SHAPE, BI_ERR_UNSUPPORTED or
 * BI_ERR_INVALID without allocating on a bad config, BI_ERR_CUDA if the tables
 * cannot be allocated.  *out is owned by the caller until bi_model_destroy,
 * which frees the tables and the step's pinned staging buffers (NULL is
 * accepted). */
bi_status bi_model_create(const bi_model_config* cfg, const bi_model_weights* w, bi_model** out);
void bi_model_destroy(bi_model* m);

/* Workspace for bi_forward_step ("The fix": every intermediate of the step has
 * a fixed place, so no allocation happens while a step runs) with at most
 * max_T tokens, max_B requests, max_R logit rows and contexts up to max_seq
 * positions.  Covers both modes (the batch-variant mode's split partials
 * included).  0 on a bad argument. */
size_t bi_forward_workspace_size(const bi_model_config* cfg, int32_t max_T, int32_t max_B,
                                 int32_t max_R, int32_t max_seq);

/* bi_forward_step ("Lockstep", "The fix" and "Proving it": one step of a
 * ragged batch whose rows for a request are bit-identical whatever else the
 * batch holds, whatever the order of its requests and however a prompt was
 * cut into prefill chunks; the harness that checks this replays steps under
 * every schedule it enumerates and compares the bits with the solo run).
 * Embedding -> n_layers x (RMSNorm, QKV GEMM, RoPE + KV append, attention,
 * O GEMM + residual, RMSNorm, gate/up GEMM + SwiGLU, down GEMM + residual) ->
 * final RMSNorm of the logit rows -> LM head (fp32) -> greedy argmax (taken in
 * the LM head's epilogue: the same tokens as bi_argmax of the logits).
 * logits_out: DEVICE [R, V] fp32 or NULL (then no logits are stored when
 * tokens_out is given); tokens_out: DEVICE [R] or NULL; hidden_out: DEVICE
 * [T, d] bf16 residual stream after the last layer, or NULL.  ws: DEVICE
 * scratch of bi_forward_workspace_size bytes, 16-byte aligned.
 * Copies the step's small metadata (token positions and lists) host to device
 * on `stream`.  The step's first kernel waits for all earlier work on
 * `stream`; the weights must not be written by work still in flight on other
 * streams while a step runs. */
bi_status bi_forward_step(bi_model* m, const bi_batch* batch, const bi_kv_cache* kv,
                          float* logits_out, int32_t* tokens_out, bi_bf16* hidden_out,
                          bi_mode mode, void* ws, size_t ws_bytes, int32_t* dev_status,
                          bi_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* BI_H */
