// C ABI of libbi: argument validation, the model object and the forward step.
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace bi {

static thread_local std::string g_err;

void set_error(const std::string& msg) { g_err = msg; }

bi_status fail(bi_status s, const std::string& msg) {
    g_err = msg;
    return s;
}

bi_status cuda_fail(cudaError_t e, const char* what) {
    g_err = std::string(what) + ": " + cudaGetErrorString(e);
    return BI_ERR_CUDA;
}

int num_sms() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
    });
    return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static size_t align_up(size_t v, size_t a = 256) { return (v + a - 1) / a * a; }

// The attention scale fl32(1 / fl32(sqrt(Dh))) unless the caller gives a positive one.
float default_scale(float scale, int32_t Dh) {
    return scale > 0.0f ? scale : 1.0f / sqrtf(static_cast<float>(Dh));
}

}  // namespace bi

using namespace bi;

// ===========================================================================
// Diagnostics
// ===========================================================================
extern "C" const char* bi_last_error(void) { return g_err.c_str(); }

extern "C" int32_t bi_version(void) { return 1; }

extern "C" bi_status bi_check_status(const int32_t* dev_status, bi_stream stream) {
    if (!dev_status) return fail(BI_ERR_INVALID, "bi_check_status: null status");
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost,
                                    static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bi_check_status");
    if (v == 0) return BI_OK;
    char buf[96];
    snprintf(buf, sizeof buf, "device status 0x%x", v);
    if (v >= BI_DEV_TIMEOUT_PRODUCER && v <= BI_DEV_TIMEOUT_ATTENTION) return fail(BI_ERR_TIMEOUT, buf);
    if (v == BI_DEV_PAIR_TMEM) return fail(BI_ERR_CUDA, buf);
    return fail(BI_ERR_DEVICE, buf);
}

extern "C" bi_status bi_reset_status(int32_t* dev_status, bi_stream stream) {
    if (!dev_status) return fail(BI_ERR_INVALID, "bi_reset_status: null status");
    cudaError_t e = cudaMemsetAsync(dev_status, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_reset_status");
}

// ===========================================================================
// Kernels
// ===========================================================================
extern "C" bi_status bi_rmsnorm(const bi_bf16* x, const bi_bf16* gamma, bi_bf16* y, int64_t rows, int32_t d,
                                float eps, bi_stream stream) {
    if (rows < 0 || d <= 0 || d % 8 != 0) return fail(BI_ERR_SHAPE, "bi_rmsnorm: need rows >= 0, d % 8 == 0");
    if (rows == 0) return BI_OK;
    if (!x || !gamma || !y) return fail(BI_ERR_INVALID, "bi_rmsnorm: null pointer");
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(y))
        return fail(BI_ERR_INVALID, "bi_rmsnorm: pointers must be 16-byte aligned");
    if (rows > (static_cast<int64_t>(1) << 34)) return fail(BI_ERR_SHAPE, "bi_rmsnorm: too many rows");
    cudaError_t e = launch_rmsnorm(x, gamma, y, rows, d, eps, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_rmsnorm launch");
}

static bi_status check_gemm_args(const bi_bf16* A, const bi_bf16* W, void* C, bi_dtype c_dtype,
                                 const bi_bf16* residual, bi_epilogue ep, int64_t M, int32_t N, int32_t K,
                                 bi_mode mode) {
    if (M < 0 || N <= 0 || K <= 0) return fail(BI_ERR_SHAPE, "bi_gemm: need M >= 0, N > 0, K > 0");
    if (K % BI_GEMM_BLOCK_K != 0 || N % BI_GEMM_UMMA_N != 0)
        return fail(BI_ERR_SHAPE, "bi_gemm: need K % 64 == 0 and N % 128 == 0");
    if (M > 0x7fffffffLL) return fail(BI_ERR_SHAPE, "bi_gemm: M too large");
    if (mode != BI_INVARIANT && mode != BI_VARIANT) return fail(BI_ERR_INVALID, "bi_gemm: bad mode");
    if (c_dtype != BI_BF16 && c_dtype != BI_F32) return fail(BI_ERR_INVALID, "bi_gemm: bad dtype");
    if (ep != BI_EP_NONE && ep != BI_EP_RESIDUAL && ep != BI_EP_SWIGLU) return fail(BI_ERR_INVALID, "bi_gemm: bad epilogue");
    if (ep != BI_EP_NONE && c_dtype != BI_BF16) return fail(BI_ERR_UNSUPPORTED, "bi_gemm: fused epilogues write bf16");
    if (M == 0) return BI_OK;
    if (!A || !W || !C) return fail(BI_ERR_INVALID, "bi_gemm: null pointer");
    if (ep == BI_EP_RESIDUAL && !residual) return fail(BI_ERR_INVALID, "bi_gemm: residual epilogue needs residual");
    if (!aligned16(A) || !aligned16(W) || !aligned16(C) || (residual && !aligned16(residual)))
        return fail(BI_ERR_INVALID, "bi_gemm: pointers must be 16-byte aligned");
    return BI_OK;
}

extern "C" size_t bi_gemm_workspace_size(int64_t M, int32_t N, int32_t K, bi_mode mode) {
    if (M <= 0 || N <= 0 || K <= 0 || K % BI_GEMM_BLOCK_K || N % BI_GEMM_UMMA_N) return 0;
    return gemm_ws_bytes(M, N, K, mode);
}

extern "C" bi_status bi_gemm(const bi_bf16* A, const bi_bf16* W, void* C, bi_dtype c_dtype, const bi_bf16* residual,
                             bi_epilogue ep, int64_t M, int32_t N, int32_t K, bi_mode mode, void* ws,
                             size_t ws_bytes, int32_t* dev_status, bi_stream stream) {
    bi_status st = check_gemm_args(A, W, C, c_dtype, residual, ep, M, N, K, mode);
    if (st != BI_OK || M == 0) return st;
    return run_gemm(A, W, C, c_dtype, residual, ep, M, N, K, mode, ws, ws_bytes, dev_status,
                    static_cast<cudaStream_t>(stream));
}

extern "C" bi_status bi_gemm_wait_test(const bi_bf16* A, const bi_bf16* W, void* C, bi_dtype c_dtype, int64_t M,
                                       int32_t N, int32_t K, uint64_t wait_limit_ns, int32_t skip_stage,
                                       int32_t* dev_status, bi_stream stream) {
    bi_status st = check_gemm_args(A, W, C, c_dtype, nullptr, BI_EP_NONE, M, N, K, BI_INVARIANT);
    if (st != BI_OK || M == 0) return st;
    if (!dev_status) return fail(BI_ERR_INVALID, "bi_gemm_wait_test: needs dev_status");
    if (wait_limit_ns < 1000000ull || wait_limit_ns > kWaitLimitNs)
        return fail(BI_ERR_INVALID, "bi_gemm_wait_test: wait limit outside [1 ms, 2 s]");
    const GemmWaitTest wt{wait_limit_ns, skip_stage};
    return run_gemm(A, W, C, c_dtype, nullptr, BI_EP_NONE, M, N, K, BI_INVARIANT, nullptr, 0, dev_status,
                    static_cast<cudaStream_t>(stream), false, nullptr, nullptr, &wt);
}

extern "C" bi_status bi_pack_gate_up(const bi_bf16* w_gate, const bi_bf16* w_up, bi_bf16* w_gu, int32_t F,
                                     int32_t d, bi_stream stream) {
    if (F <= 0 || d <= 0 || F % BI_SWIGLU_GROUP || d % 8) return fail(BI_ERR_SHAPE, "bi_pack_gate_up: need F % 32 == 0, d % 8 == 0");
    if (!w_gate || !w_up || !w_gu) return fail(BI_ERR_INVALID, "bi_pack_gate_up: null pointer");
    if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_gu)) return fail(BI_ERR_INVALID, "bi_pack_gate_up: alignment");
    cudaError_t e = launch_pack_gate_up(w_gate, w_up, w_gu, F, d, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_pack_gate_up launch");
}

extern "C" bi_status bi_rope_table(float* cos_out, float* sin_out, int32_t n_pos, int32_t Dh, double theta) {
    if (!cos_out || !sin_out) return fail(BI_ERR_INVALID, "bi_rope_table: null pointer");
    if (n_pos < 0 || Dh <= 0 || Dh % 2) return fail(BI_ERR_SHAPE, "bi_rope_table: bad shape");
    const int32_t half = Dh / 2;
    for (int32_t i = 0; i < half; ++i) {
        const double inv_freq = pow(theta, -static_cast<double>(2 * i) / static_cast<double>(Dh));
        for (int32_t p = 0; p < n_pos; ++p) {
            const double ang = static_cast<double>(p) * inv_freq;
            cos_out[static_cast<int64_t>(p) * half + i] = static_cast<float>(cos(ang));
            sin_out[static_cast<int64_t>(p) * half + i] = static_cast<float>(sin(ang));
        }
    }
    return BI_OK;
}

extern "C" bi_status bi_rope_kv_append(const float* qkv, const int32_t* tok_req, const int32_t* tok_pos,
                                       const float* rope_cos, const float* rope_sin, int32_t max_pos, bi_bf16* q_out,
                                       bi_bf16* k_cache, bi_bf16* v_cache, const int32_t* page_table,
                                       int32_t max_pages, int32_t num_pages, int32_t T, int32_t H, int32_t Hkv,
                                       int32_t Dh, int32_t* dev_status, bi_stream stream) {
    if (T < 0 || H <= 0 || Hkv <= 0 || Dh <= 0 || Dh % 2 || max_pages <= 0 || num_pages <= 0 || max_pos <= 0)
        return fail(BI_ERR_SHAPE, "bi_rope_kv_append: bad shape");
    if (T == 0) return BI_OK;
    if (!qkv || !tok_req || !tok_pos || !rope_cos || !rope_sin || !q_out || !k_cache || !v_cache || !page_table)
        return fail(BI_ERR_INVALID, "bi_rope_kv_append: null pointer");
    cudaError_t e = launch_rope_kv_append(qkv, tok_req, tok_pos, rope_cos, rope_sin, max_pos, q_out, k_cache, v_cache,
                                          page_table, max_pages, num_pages, T, H, Hkv, Dh, dev_status,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_rope_kv_append launch");
}

static bi_status check_attn(const void* q, const void* kc, const void* vc, const void* pt, const void* out,
                            bi_dtype out_dtype, int32_t H, int32_t Hkv, int32_t Dh, int32_t max_pages,
                            int32_t num_pages) {
    if (!attention_supported(H, Hkv, Dh))
        return fail(BI_ERR_UNSUPPORTED, "attention: need Dh in {64,128} and H/Hkv in {1,2,4,8}");
    if (max_pages <= 0 || num_pages <= 0) return fail(BI_ERR_SHAPE, "attention: need max_pages, num_pages > 0");
    if (out_dtype != BI_BF16 && out_dtype != BI_F32) return fail(BI_ERR_INVALID, "attention: bad dtype");
    if (!q || !kc || !vc || !pt || !out) return fail(BI_ERR_INVALID, "attention: null pointer");
    if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(out))
        return fail(BI_ERR_INVALID, "attention: pointers must be 16-byte aligned");
    return BI_OK;
}

extern "C" size_t bi_decode_attention_workspace_size(int32_t B, int32_t H, int32_t Dh, int32_t max_seq_len,
                                                     bi_mode mode) {
    if (B <= 0 || H <= 0 || Dh <= 0) return 0;
    int32_t splits = invariant_max_splits(max_seq_len);
    if (mode == BI_VARIANT) splits = std::max(splits, 16);
    return decode_ws_bytes(B, H, Dh, splits);
}

extern "C" bi_status bi_decode_attention(const bi_bf16* q, const bi_bf16* k_cache, const bi_bf16* v_cache,
                                         const int32_t* page_table, const int32_t* seq_lens, void* out,
                                         bi_dtype out_dtype, int32_t B, int32_t H, int32_t Hkv, int32_t Dh,
                                         int32_t max_pages, int32_t num_pages, int32_t max_seq_len, float scale,
                                         bi_mode mode, void* ws, size_t ws_bytes, int32_t* dev_status,
                                         bi_stream stream) {
    if (B < 0) return fail(BI_ERR_SHAPE, "bi_decode_attention: B < 0");
    if (B == 0) return BI_OK;
    bi_status st = check_attn(q, k_cache, v_cache, page_table, out, out_dtype, H, Hkv, Dh, max_pages, num_pages);
    if (st != BI_OK) return st;
    if (!seq_lens) return fail(BI_ERR_INVALID, "bi_decode_attention: null seq_lens");
    if (max_seq_len <= 0 || max_seq_len > max_pages * BI_PAGE)
        return fail(BI_ERR_SHAPE, "bi_decode_attention: need 0 < max_seq_len <= max_pages * 16");
    if (mode != BI_INVARIANT && mode != BI_VARIANT) return fail(BI_ERR_INVALID, "bi_decode_attention: bad mode");
    int32_t max_splits = invariant_max_splits(max_seq_len), chunk2 = 0;
    if (mode == BI_VARIANT) variant_split_plan(B, H, Hkv, max_seq_len, &chunk2, &max_splits);
    const size_t need = decode_ws_bytes(B, H, Dh, max_splits);
    if (!ws || ws_bytes < need) return fail(BI_ERR_WORKSPACE, "bi_decode_attention: workspace too small");
    if (!aligned16(ws)) return fail(BI_ERR_INVALID, "bi_decode_attention: workspace must be 16-byte aligned");
    float* ws_o = static_cast<float*>(ws);
    float* ws_ml = ws_o + static_cast<size_t>(B) * H * max_splits * Dh;
    AttnGeom g{q, k_cache, v_cache, page_table, out, out_dtype == BI_F32, H, Hkv, Dh, max_pages, num_pages,
               default_scale(scale, Dh), dev_status};
    EntryMap em{0, seq_lens, nullptr, nullptr, B};
    cudaError_t e = launch_decode_attention(g, em, B, max_splits, chunk2, ws_o, ws_ml, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_decode_attention launch");
}

extern "C" size_t bi_prefill_attention_workspace_size(int32_t T, int32_t H, int32_t Dh, int32_t max_seq_len,
                                                      bi_mode mode) {
    if (T <= 0 || H <= 0 || Dh <= 0 || mode != BI_VARIANT) return 0;
    // the occupancy rule never cuts a context into more than max(ceil(s / 256), 16) pieces
    return decode_ws_bytes(T, H, Dh, std::max(invariant_max_splits(max_seq_len), 16));
}

extern "C" bi_status bi_prefill_attention(const bi_bf16* q, const int32_t* cu_q, const int32_t* q_pos0,
                                          const bi_bf16* k_cache, const bi_bf16* v_cache, const int32_t* page_table,
                                          void* out, bi_dtype out_dtype, int32_t B, int32_t T, int32_t H,
                                          int32_t Hkv, int32_t Dh, int32_t max_pages, int32_t num_pages,
                                          int32_t max_seq_len, float scale, bi_mode mode, void* ws,
                                          size_t ws_bytes, int32_t* dev_status, bi_stream stream) {
    if (B < 0 || T < 0) return fail(BI_ERR_SHAPE, "bi_prefill_attention: negative size");
    if (B == 0 || T == 0) return BI_OK;
    bi_status st = check_attn(q, k_cache, v_cache, page_table, out, out_dtype, H, Hkv, Dh, max_pages, num_pages);
    if (st != BI_OK) return st;
    if (!cu_q || !q_pos0) return fail(BI_ERR_INVALID, "bi_prefill_attention: null cu_q / q_pos0");
    if (max_seq_len <= 0 || max_seq_len > max_pages * BI_PAGE)
        return fail(BI_ERR_SHAPE, "bi_prefill_attention: need 0 < max_seq_len <= max_pages * 16");
    if (mode != BI_INVARIANT && mode != BI_VARIANT) return fail(BI_ERR_INVALID, "bi_prefill_attention: bad mode");
    AttnGeom g{q, k_cache, v_cache, page_table, out, out_dtype == BI_F32, H, Hkv, Dh, max_pages, num_pages,
               default_scale(scale, Dh), dev_status};
    EntryMap em{2, cu_q, q_pos0, nullptr, B};
    cudaError_t e;
    if (mode == BI_INVARIANT) {
        e = launch_prefill_attention(g, em, T, T, static_cast<cudaStream_t>(stream));
    } else {
        // every query as a decode entry whose pieces follow the occupancy rule of this batch
        int32_t max_splits = 0, chunk2 = 0;
        variant_split_plan(B, H, Hkv, max_seq_len, &chunk2, &max_splits);
        const size_t need = decode_ws_bytes(T, H, Dh, max_splits);
        if (!ws || ws_bytes < need) return fail(BI_ERR_WORKSPACE, "bi_prefill_attention: workspace too small");
        if (!aligned16(ws)) return fail(BI_ERR_INVALID, "bi_prefill_attention: workspace must be 16-byte aligned");
        float* ws_o = static_cast<float*>(ws);
        float* ws_ml = ws_o + static_cast<size_t>(T) * H * max_splits * Dh;
        e = launch_decode_attention(g, em, T, max_splits, chunk2, ws_o, ws_ml, static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_prefill_attention launch");
}

extern "C" bi_status bi_argmax(const float* logits, int32_t* out, int32_t R, int32_t V, bi_stream stream) {
    if (R < 0 || V <= 0) return fail(BI_ERR_SHAPE, "bi_argmax: need R >= 0, V > 0");
    if (R == 0) return BI_OK;
    if (!logits || !out) return fail(BI_ERR_INVALID, "bi_argmax: null pointer");
    cudaError_t e = launch_argmax(logits, out, R, V, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_argmax launch");
}

extern "C" size_t bi_log_softmax_workspace_size(int32_t R, int32_t V) { return log_softmax_ws_bytes(R, V); }

extern "C" bi_status bi_log_softmax(const float* logits, float* logprobs, int32_t R, int32_t V, void* ws,
                                    size_t ws_bytes, bi_stream stream) {
    if (R < 0 || V <= 0) return fail(BI_ERR_SHAPE, "bi_log_softmax: need R >= 0, V > 0");
    if (R == 0) return BI_OK;
    if (!logits || !logprobs) return fail(BI_ERR_INVALID, "bi_log_softmax: null pointer");
    const char* a = reinterpret_cast<const char*>(logits);
    const char* b = reinterpret_cast<const char*>(logprobs);
    const size_t n = static_cast<size_t>(R) * V * sizeof(float);
    if (a < b + n && b < a + n) return fail(BI_ERR_INVALID, "bi_log_softmax: logits and logprobs overlap");
    if (!ws || ws_bytes < log_softmax_ws_bytes(R, V) || !aligned16(ws))
        return fail(BI_ERR_WORKSPACE, "bi_log_softmax: workspace too small or not 16-byte aligned");
    cudaError_t e = launch_log_softmax(logits, logprobs, R, V, ws, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_log_softmax launch");
}

extern "C" size_t bi_sample_workspace_size(int32_t R, int32_t V) { return sample_ws_bytes(R, V); }

extern "C" bi_status bi_sample(const float* logits, const uint32_t* seeds, const int32_t* positions,
                               const float* temperatures, int32_t* tokens, int32_t R, int32_t V, void* ws,
                               size_t ws_bytes, bi_stream stream) {
    if (R < 0 || V <= 0) return fail(BI_ERR_SHAPE, "bi_sample: need R >= 0, V > 0");
    if (R == 0) return BI_OK;
    if (!logits || !seeds || !positions || !temperatures || !tokens) return fail(BI_ERR_INVALID, "bi_sample: null pointer");
    if (!ws || ws_bytes < sample_ws_bytes(R, V) || !aligned16(ws))
        return fail(BI_ERR_WORKSPACE, "bi_sample: workspace too small or not 16-byte aligned");
    cudaError_t e = launch_sample(logits, seeds, positions, temperatures, tokens, R, V, ws,
                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_sample launch");
}

extern "C" bi_status bi_embed(const bi_bf16* E, const int32_t* ids, bi_bf16* x, int32_t T, int32_t V, int32_t d,
                              int32_t* dev_status, bi_stream stream) {
    if (T < 0 || V <= 0 || d <= 0 || d % 8) return fail(BI_ERR_SHAPE, "bi_embed: need d % 8 == 0");
    if (T == 0) return BI_OK;
    if (!E || !ids || !x) return fail(BI_ERR_INVALID, "bi_embed: null pointer");
    if (!aligned16(E) || !aligned16(x)) return fail(BI_ERR_INVALID, "bi_embed: alignment");
    cudaError_t e = launch_embed(E, ids, x, T, V, d, dev_status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_embed launch");
}

// ===========================================================================
// Model and forward step
// ===========================================================================
struct bi_model {
    bi_model_config cfg;
    const bi_bf16* embed;
    const bi_bf16* gamma_final;
    const bi_bf16* w_lm;
    std::vector<const bi_bf16*> gamma_attn, w_qkv, w_o, gamma_ffn, w_gu, w_down;
    float* rope_cos = nullptr;  // device [max_pos, Dh/2]
    float* rope_sin = nullptr;
    // pinned staging for the per-step metadata, double-buffered
    int32_t* stage[2] = {nullptr, nullptr};
    size_t stage_cap[2] = {0, 0};
    cudaEvent_t stage_done[2] = {nullptr, nullptr};
    int stage_next = 0;
};

extern "C" bi_status bi_model_create(const bi_model_config* cfg, const bi_model_weights* w, bi_model** out) {
    if (!cfg || !w || !out) return fail(BI_ERR_INVALID, "bi_model_create: null pointer");
    *out = nullptr;
    const bi_model_config& c = *cfg;
    if (c.d <= 0 || c.H <= 0 || c.Hkv <= 0 || c.Dh <= 0 || c.F <= 0 || c.V <= 0 || c.n_layers <= 0 || c.max_pos <= 0)
        return fail(BI_ERR_SHAPE, "bi_model_create: nonpositive dimension");
    constexpr int n_mult = BI_GEMM_UMMA_N;
    if (c.d % n_mult || c.F % 64 || c.V % n_mult || ((c.H + 2 * c.Hkv) * c.Dh) % n_mult || (c.H * c.Dh) % 64 ||
        c.F % 64)
        return fail(BI_ERR_SHAPE, "bi_model_create: GEMM widths must be multiples of 128 (K multiples of 64)");
    if (!attention_supported(c.H, c.Hkv, c.Dh)) return fail(BI_ERR_UNSUPPORTED, "bi_model_create: attention shape");
    if (!w->embed || !w->gamma_final || !w->w_lm || !w->gamma_attn || !w->w_qkv || !w->w_o || !w->gamma_ffn ||
        !w->w_gu || !w->w_down)
        return fail(BI_ERR_INVALID, "bi_model_create: null weight pointer");
    for (int l = 0; l < c.n_layers; ++l)
        if (!w->gamma_attn[l] || !w->w_qkv[l] || !w->w_o[l] || !w->gamma_ffn[l] || !w->w_gu[l] || !w->w_down[l])
            return fail(BI_ERR_INVALID, "bi_model_create: null layer weight");
    bi_model* m = new bi_model();
    m->cfg = c;
    m->embed = w->embed;
    m->gamma_final = w->gamma_final;
    m->w_lm = w->w_lm;
    m->gamma_attn.assign(w->gamma_attn, w->gamma_attn + c.n_layers);
    m->w_qkv.assign(w->w_qkv, w->w_qkv + c.n_layers);
    m->w_o.assign(w->w_o, w->w_o + c.n_layers);
    m->gamma_ffn.assign(w->gamma_ffn, w->gamma_ffn + c.n_layers);
    m->w_gu.assign(w->w_gu, w->w_gu + c.n_layers);
    m->w_down.assign(w->w_down, w->w_down + c.n_layers);
    const size_t n = static_cast<size_t>(c.max_pos) * (c.Dh / 2);
    std::vector<float> hc(n), hs(n);
    bi_rope_table(hc.data(), hs.data(), c.max_pos, c.Dh, c.rope_theta);
    cudaError_t e = cudaMalloc(&m->rope_cos, n * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&m->rope_sin, n * sizeof(float));
    if (e == cudaSuccess) e = cudaMemcpy(m->rope_cos, hc.data(), n * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(m->rope_sin, hs.data(), n * sizeof(float), cudaMemcpyHostToDevice);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&m->stage_done[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        bi_model_destroy(m);
        return cuda_fail(e, "bi_model_create");
    }
    *out = m;
    return BI_OK;
}

extern "C" void bi_model_destroy(bi_model* m) {
    if (!m) return;
    for (int i = 0; i < 2; ++i) {
        if (m->stage_done[i]) {
            cudaEventSynchronize(m->stage_done[i]);
            cudaEventDestroy(m->stage_done[i]);
        }
        if (m->stage[i]) cudaFreeHost(m->stage[i]);
    }
    cudaFree(m->rope_cos);
    cudaFree(m->rope_sin);
    delete m;
}

namespace {

struct FwdLayout {
    size_t x, y, qkv, q, attn, h, yr, logits, am_keys, am_counter, meta, dec_ws, gemm_ws, total;
    int32_t dec_splits;
};

FwdLayout fwd_layout(const bi_model_config& c, int32_t T, int32_t B, int32_t R, int32_t max_seq) {
    FwdLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes);
        return o;
    };
    const size_t nqkv = static_cast<size_t>(c.H + 2 * c.Hkv) * c.Dh;
    L.x = take(static_cast<size_t>(T) * c.d * 2);
    L.y = take(static_cast<size_t>(T) * c.d * 2);
    L.qkv = take(static_cast<size_t>(T) * nqkv * 4);
    L.q = take(static_cast<size_t>(T) * c.H * c.Dh * 2);
    L.attn = take(static_cast<size_t>(T) * c.H * c.Dh * 2);
    L.h = take(static_cast<size_t>(T) * c.F * 2);
    L.yr = take(static_cast<size_t>(R) * c.d * 2);
    L.logits = take(static_cast<size_t>(R) * c.V * 4);
    L.am_keys = take(static_cast<size_t>(R) * 8);
    L.am_counter = take(16);
    L.meta = take((static_cast<size_t>(T) * 4 + R + 16) * 4);
    L.dec_splits = std::max(invariant_max_splits(max_seq), 16);
    L.dec_ws = take(decode_ws_bytes(B, c.H, c.Dh, L.dec_splits));
    L.gemm_ws = take(static_cast<size_t>(num_sms()) * BI_GEMM_BLOCK_M * BI_GEMM_UMMA_N * 4 + 4096);
    L.total = off + 256;
    return L;
}

}  // namespace

extern "C" size_t bi_forward_workspace_size(const bi_model_config* cfg, int32_t max_T, int32_t max_B, int32_t max_R,
                                            int32_t max_seq) {
    if (!cfg || max_T <= 0 || max_B <= 0 || max_R < 0 || max_seq <= 0) return 0;
    return fwd_layout(*cfg, max_T, max_B, max_R, max_seq).total;
}

#define BI_TRY(expr)                        \
    do {                                    \
        bi_status st_ = (expr);             \
        if (st_ != BI_OK) return st_;       \
    } while (0)
#define BI_TRY_CUDA(expr, what)                          \
    do {                                                 \
        cudaError_t ce_ = (expr);                        \
        if (ce_ != cudaSuccess) return cuda_fail(ce_, what); \
    } while (0)

extern "C" bi_status bi_forward_step(bi_model* m, const bi_batch* batch, const bi_kv_cache* kv, float* logits_out,
                                     int32_t* tokens_out, bi_bf16* hidden_out, bi_mode mode, void* ws,
                                     size_t ws_bytes, int32_t* dev_status, bi_stream stream) {
    if (!m || !batch || !kv) return fail(BI_ERR_INVALID, "bi_forward_step: null pointer");
    if (mode != BI_INVARIANT && mode != BI_VARIANT) return fail(BI_ERR_INVALID, "bi_forward_step: bad mode");
    const bi_model_config& c = m->cfg;
    const bi_batch& b = *batch;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (b.B < 0 || b.R < 0) return fail(BI_ERR_SHAPE, "bi_forward_step: negative B or R");
    if (b.B == 0) return BI_OK;
    if (!b.q_len || !b.pos0 || !b.token_ids || !b.page_table || b.max_pages <= 0 || (b.R > 0 && !b.logit_rows))
        return fail(BI_ERR_INVALID, "bi_forward_step: incomplete batch");
    if (!kv->k || !kv->v || kv->num_pages <= 0) return fail(BI_ERR_INVALID, "bi_forward_step: incomplete kv cache");
    for (int l = 0; l < c.n_layers; ++l)
        if (!kv->k[l] || !kv->v[l]) return fail(BI_ERR_INVALID, "bi_forward_step: null kv layer");

    // ---- host metadata ----
    int64_t T64 = 0;
    int32_t max_seq = 0, max_seq_dec = 0, nd = 0;
    for (int32_t i = 0; i < b.B; ++i) {
        if (b.q_len[i] < 1 || b.pos0[i] < 0) return fail(BI_ERR_SHAPE, "bi_forward_step: need q_len >= 1, pos0 >= 0");
        const int64_t end = static_cast<int64_t>(b.pos0[i]) + b.q_len[i];
        if (end > c.max_pos) return fail(BI_ERR_SHAPE, "bi_forward_step: position beyond the RoPE table");
        if (end > static_cast<int64_t>(b.max_pages) * BI_PAGE)
            return fail(BI_ERR_SHAPE, "bi_forward_step: context beyond max_pages * 16");
        T64 += b.q_len[i];
        max_seq = std::max<int32_t>(max_seq, static_cast<int32_t>(end));
        if (b.q_len[i] == 1) {
            ++nd;
            max_seq_dec = std::max<int32_t>(max_seq_dec, static_cast<int32_t>(end));
        }
    }
    if (T64 > 0x3fffffff) return fail(BI_ERR_SHAPE, "bi_forward_step: too many tokens");
    const int32_t T = static_cast<int32_t>(T64);
    for (int32_t r = 0; r < b.R; ++r)
        if (b.logit_rows[r] < 0 || b.logit_rows[r] >= T) return fail(BI_ERR_SHAPE, "bi_forward_step: logit row out of range");
    const FwdLayout L = fwd_layout(c, T, b.B, b.R, max_seq);
    if (!ws || ws_bytes < L.total) return fail(BI_ERR_WORKSPACE, "bi_forward_step: workspace too small");
    if (!aligned16(ws)) return fail(BI_ERR_INVALID, "bi_forward_step: workspace must be 16-byte aligned");
    if (!dev_status) return fail(BI_ERR_INVALID, "bi_forward_step: null dev_status");

    // pinned staging: [tok_req T][tok_pos T][dec_list nd][pre_list T-nd][logit_rows R]
    const size_t meta_n = static_cast<size_t>(T) * 3 + b.R;
    char* base = static_cast<char*>(ws);
    const int32_t* d_meta = b.meta;
    // host metadata of a small step travels as the first kernel's parameter (no copy ahead of it)
    StepMeta param_meta;
    const bool meta_in_param = d_meta == nullptr && meta_n <= static_cast<size_t>(kStepMetaMax);
    if (d_meta == nullptr) {
        // the step derives the metadata on the host: into the first kernel's parameter, or (larger steps)
        // through pinned staging and a copy
        int32_t* hm = param_meta.v;
        int slot = 0;
        if (!meta_in_param) {
            slot = m->stage_next;
            m->stage_next ^= 1;
            BI_TRY_CUDA(cudaEventSynchronize(m->stage_done[slot]), "bi_forward_step: staging event");
            if (m->stage_cap[slot] < meta_n) {
                if (m->stage[slot]) cudaFreeHost(m->stage[slot]);
                m->stage[slot] = nullptr;
                m->stage_cap[slot] = 0;
                const size_t cap = std::max<size_t>(meta_n * 2, 4096);
                BI_TRY_CUDA(cudaHostAlloc(&m->stage[slot], cap * sizeof(int32_t), cudaHostAllocDefault),
                            "cudaHostAlloc");
                m->stage_cap[slot] = cap;
            }
            hm = m->stage[slot];
        }
        int32_t* h_req = hm;
        int32_t* h_pos = hm + T;
        int32_t* h_dec = hm + 2 * static_cast<size_t>(T);
        int32_t* h_pre = h_dec + nd;
        int32_t* h_rows = hm + 3 * static_cast<size_t>(T);
        {
            int32_t t = 0, di = 0, pi = 0;
            for (int32_t i = 0; i < b.B; ++i)
                for (int32_t j = 0; j < b.q_len[i]; ++j, ++t) {
                    h_req[t] = i;
                    h_pos[t] = b.pos0[i] + j;
                    if (b.q_len[i] == 1) h_dec[di++] = t; else h_pre[pi++] = t;
                }
            std::memcpy(h_rows, b.logit_rows, sizeof(int32_t) * b.R);
        }
        int32_t* d_stage = reinterpret_cast<int32_t*>(base + L.meta);
        if (meta_in_param) {
            param_meta.n = static_cast<int32_t>(meta_n);
        } else {
            BI_TRY_CUDA(cudaMemcpyAsync(d_stage, hm, meta_n * sizeof(int32_t), cudaMemcpyHostToDevice, s),
                        "metadata copy");
            BI_TRY_CUDA(cudaEventRecord(m->stage_done[slot], s), "cudaEventRecord");
        }
        d_meta = d_stage;
    }
    const int32_t* d_req = d_meta;
    const int32_t* d_pos = d_meta + T;
    const int32_t* d_dec = d_meta + 2 * static_cast<size_t>(T);
    const int32_t* d_pre = d_dec + nd;
    const int32_t* d_rows = d_meta + 3 * static_cast<size_t>(T);

    bi_bf16* x = reinterpret_cast<bi_bf16*>(base + L.x);
    bi_bf16* y = reinterpret_cast<bi_bf16*>(base + L.y);
    float* qkv = reinterpret_cast<float*>(base + L.qkv);
    bi_bf16* q = reinterpret_cast<bi_bf16*>(base + L.q);
    bi_bf16* attn = reinterpret_cast<bi_bf16*>(base + L.attn);
    bi_bf16* h = reinterpret_cast<bi_bf16*>(base + L.h);
    float* dec_o = reinterpret_cast<float*>(base + L.dec_ws);
    void* gws = base + L.gemm_ws;
    const size_t gws_bytes = static_cast<size_t>(num_sms()) * BI_GEMM_BLOCK_M * BI_GEMM_UMMA_N * 4 + 4096;
    const int32_t nqkv = (c.H + 2 * c.Hkv) * c.Dh;
    const float scale = default_scale(0.0f, c.Dh);

    int32_t dec_splits = invariant_max_splits(max_seq_dec), chunk2 = 0;
    if (mode == BI_VARIANT) variant_split_plan(b.B, c.H, c.Hkv, max_seq, &chunk2, &dec_splits);
    if (dec_splits > L.dec_splits) return fail(BI_ERR_SHAPE, "bi_forward_step: split plan exceeds workspace");
    float* dec_ml = dec_o + static_cast<size_t>(std::max(nd, 1)) * c.H * dec_splits * c.Dh;

    // greedy tokens come straight out of the LM head's epilogue unless the
    // batch-variant plan splits its K (then the argmax reads stored logits)
    const bool lm_head = b.R > 0 && (logits_out || tokens_out);
    const bool fuse = lm_head && tokens_out != nullptr && gemm_plan(b.R, c.V, c.d, mode).splits == 1;
    ArgmaxFuse am{reinterpret_cast<unsigned long long*>(base + L.am_keys), tokens_out,
                  reinterpret_cast<unsigned int*>(base + L.am_counter)};
    // With few tokens the RMSNorms run inside the GEMMs that consume them (their A writers apply the norm
    // kernel's arithmetic), which saves a launch and a round trip of y per norm; a row's bits are the same
    // either way.  The gate/up GEMM streams the most weight per row of A, and above 4 rows its writers'
    // per-stage pass shows on the step (8 rows: 348 against 337 us), so it takes the norm only up to 4 rows.
    constexpr int64_t kNormInGateUpMaxRows = 4;
    const bool norm_in_qkv = gemm_can_fuse_norm(T, nqkv, c.d, mode);
    const bool norm_in_gu = T <= kNormInGateUpMaxRows && gemm_can_fuse_norm(T, 2 * c.F, c.d, mode);
    // (the LM head's rows are x's first R rows when every request contributes its one decode token)
    bool rows_leading = true;
    for (int32_t i = 0; i < b.R && rows_leading; ++i) rows_leading = b.logit_rows[i] == i;
    const bool norm_in_lm = lm_head && rows_leading && gemm_can_fuse_norm(b.R, c.V, c.d, mode);

    // The step's first kernel waits for all earlier work on the stream; every
    // later kernel of the step starts after it, so weights (never written
    // within a step) may be fetched before each kernel's dependency wait.
    // the embedding gather and the first norm in one kernel (it also writes the residual stream x, and
    // initialises the fused argmax's keys)
    BI_TRY_CUDA(launch_embed_rmsnorm(m->embed, b.token_ids, c.V, m->gamma_attn[0], x, y, T, c.d, c.eps, dev_status,
                                     s, fuse ? &am : nullptr, b.R, meta_in_param ? &param_meta : nullptr,
                                     meta_in_param ? const_cast<int32_t*>(d_meta) : nullptr),
                "embed + rmsnorm");
    for (int l = 0; l < c.n_layers; ++l) {
        // layer 0's norm ran with the embedding gather; later layers' in their QKV GEMM when it takes few rows
        const NormFuse qkv_norm{x, m->gamma_attn[l], nullptr, c.eps};
        const NormFuse* qn = l > 0 && norm_in_qkv ? &qkv_norm : nullptr;
        if (l > 0 && qn == nullptr) BI_TRY_CUDA(launch_rmsnorm(x, m->gamma_attn[l], y, T, c.d, c.eps, s), "rmsnorm");
        if (gemm_can_fuse_rope(T, nqkv, c.d, mode, c.Dh)) {
            // RoPE and the K/V append run in the QKV GEMM's epilogue (no fp32 qkv round trip)
            const RopeFuse rf{d_req, d_pos, m->rope_cos, m->rope_sin, reinterpret_cast<uint16_t*>(q),
                              reinterpret_cast<uint16_t*>(kv->k[l]), reinterpret_cast<uint16_t*>(kv->v[l]),
                              b.page_table, c.max_pos, b.max_pages, kv->num_pages, c.H, c.Hkv, c.Dh};
            BI_TRY(run_gemm(y, m->w_qkv[l], nullptr, BI_F32, nullptr, BI_EP_NONE, T, nqkv, c.d, mode, gws,
                            gws_bytes, dev_status, s, true, nullptr, &rf, nullptr, qn));
        } else {
            BI_TRY(run_gemm(y, m->w_qkv[l], qkv, BI_F32, nullptr, BI_EP_NONE, T, nqkv, c.d, mode, gws, gws_bytes,
                            dev_status, s, true, nullptr, nullptr, nullptr, qn));
            BI_TRY_CUDA(launch_rope_kv_append(qkv, d_req, d_pos, m->rope_cos, m->rope_sin, c.max_pos, q, kv->k[l],
                                              kv->v[l], b.page_table, b.max_pages, kv->num_pages, T, c.H, c.Hkv,
                                              c.Dh, dev_status, s),
                        "rope_kv_append");
        }
        AttnGeom g{q, kv->k[l], kv->v[l], b.page_table, attn, 0, c.H, c.Hkv, c.Dh, b.max_pages, kv->num_pages,
                   scale, dev_status};
        if (nd > 0) {
            EntryMap em{1, d_dec, d_req, d_pos, b.B};
            // a decode entry's only new key (its last position) was appended just before
            BI_TRY_CUDA(launch_decode_attention(g, em, nd, dec_splits, chunk2, dec_o, dec_ml, s, /*early_kv=*/true),
                        "decode attention");
        }
        if (T - nd > 0) {
            EntryMap em{1, d_pre, d_req, d_pos, b.B};
            BI_TRY_CUDA(launch_prefill_attention(g, em, T - nd, T, s), "prefill attention");
        }
        BI_TRY(run_gemm(attn, m->w_o[l], x, BI_BF16, x, BI_EP_RESIDUAL, T, c.d, c.H * c.Dh, mode, gws, gws_bytes,
                        dev_status, s, true));
        const NormFuse ffn_norm{x, m->gamma_ffn[l], nullptr, c.eps};
        if (!norm_in_gu) BI_TRY_CUDA(launch_rmsnorm(x, m->gamma_ffn[l], y, T, c.d, c.eps, s), "rmsnorm");
        BI_TRY(run_gemm(y, m->w_gu[l], h, BI_BF16, nullptr, BI_EP_SWIGLU, T, 2 * c.F, c.d, mode, gws, gws_bytes,
                        dev_status, s, true, nullptr, nullptr, nullptr, norm_in_gu ? &ffn_norm : nullptr));
        BI_TRY(run_gemm(h, m->w_down[l], x, BI_BF16, x, BI_EP_RESIDUAL, T, c.d, c.F, mode, gws, gws_bytes,
                        dev_status, s, true));
    }
    if (hidden_out)
        BI_TRY_CUDA(cudaMemcpyAsync(hidden_out, x, static_cast<size_t>(T) * c.d * 2, cudaMemcpyDeviceToDevice, s),
                    "hidden copy");
    if (lm_head) {
        bi_bf16* yr = reinterpret_cast<bi_bf16*>(base + L.yr);
        float* logits = logits_out ? logits_out : fuse ? nullptr : reinterpret_cast<float*>(base + L.logits);
        // the final norm of the logit rows (gathered by d_rows), in the LM head when it has few rows; there it
        // reads x's first R rows, and d_rows (which a replayed graph may have changed) is checked against them
        const NormFuse final_norm{x, m->gamma_final, d_rows, c.eps};
        if (!norm_in_lm)
            BI_TRY_CUDA(launch_rmsnorm(x, m->gamma_final, yr, b.R, c.d, c.eps, s, d_rows), "final rmsnorm");
        BI_TRY(run_gemm(yr, m->w_lm, logits, BI_F32, nullptr, BI_EP_NONE, b.R, c.V, c.d, mode, gws, gws_bytes,
                        dev_status, s, true, fuse ? &am : nullptr, nullptr, nullptr,
                        norm_in_lm ? &final_norm : nullptr));
        if (tokens_out && !fuse) BI_TRY_CUDA(launch_argmax(logits, tokens_out, b.R, c.V, s), "argmax");
    }
    return BI_OK;
}
