// Host-side declarations shared by the translation units of libbi.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/bi.h"

namespace bi {

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous kernel in the stream drains, and synchronises with it through
// griddepcontrol.wait (pdl_wait in common.cuh), which every kernel of this
// library executes before touching shared global data.
template <typename... P, typename... A>
inline cudaError_t launch_k(bool pdl, void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            A&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              A&&... args) {
    return launch_k(true, kernel, grid, block, smem, s, static_cast<A&&>(args)...);
}

// As launch_pdl, in clusters of two CTAs along x (grid.x even): the CTA pairs
// of the tensor-core GEMM.
template <typename... P, typename... A>
inline cudaError_t launch_pair_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                   A&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// thread-local error message (api.cu)
void set_error(const std::string& msg);
bi_status fail(bi_status s, const std::string& msg);
bi_status cuda_fail(cudaError_t e, const char* what);
int num_sms();
// the attention scale: the caller's when positive, else fl32(1 / fl32(sqrt(Dh)))
float default_scale(float scale, int32_t Dh);

// ---- elementwise / row kernels (k_rows.cu) ----
// Greedy argmax fused into an fp32 GEMM epilogue: keys[rows] (set to
// kArgmaxKeyNone and counter to 0 before the GEMM) receive each row's winning
// key; the last CTA writes tokens[row] and resets the counter.
struct ArgmaxFuse {
    unsigned long long* keys;
    int32_t* tokens;
    unsigned int* counter;
};

// RoPE + KV append fused into the QKV GEMM's epilogue (the arithmetic of
// rope_append_kernel on the fp32 accumulator instead of a stored fp32 qkv):
// GEMM row t is token t; its columns are q heads, then k heads, then v heads.
struct RopeFuse {
    const int32_t* tok_req;
    const int32_t* tok_pos;
    const float* rc;
    const float* rs;
    uint16_t* q_out;
    uint16_t* kc;
    uint16_t* vc;
    const int32_t* page_table;
    int32_t max_pos, max_pages, num_pages, H, Hkv, Dh;
};

// rows: output rows; src_rows (device, optional): output row r normalises input row src_rows[r];
// am (optional): initialise its keys[0, rows) and counter for a fused argmax that follows
cudaError_t launch_rmsnorm(const bi_bf16* x, const bi_bf16* gamma, bi_bf16* y, int64_t rows,
                           int32_t d, float eps, cudaStream_t s, const int32_t* src_rows = nullptr,
                           const ArgmaxFuse* am = nullptr);
// RMSNorm fused into a GEMM's A operand (few rows): A row r = bf16((x[r] * rinv) * gamma)
// for x's first M rows, rinv from x[r]'s sum of squares in the RMSNorm kernel's order, so
// the GEMM reads exactly the bits the RMSNorm kernel would have written.  rows (device,
// optional): the rows the caller means; where rows[r] != r the kernel reports
// BI_DEV_BAD_LOGIT_ROWS (a replayed step whose rows no longer lead).
struct NormFuse {
    const bi_bf16* x;
    const bi_bf16* gamma;
    const int32_t* rows;
    float eps;
};
// after_all: launch without programmatic serialisation, so the kernel (and
// every kernel chained after it) starts only once all earlier work on the
// stream has finished.
// A forward step's per-token metadata small enough to travel as a kernel parameter (3T + R values: every
// decode step of up to 256 tokens), so that a step with host metadata needs no host-to-device copy ahead of its
// first kernel.
constexpr int kStepMetaMax = 1024;
struct StepMeta {
    int32_t n;
    int32_t v[kStepMetaMax];
};
// x[t] = E[ids[t]] and y[t] = rmsnorm(x[t]) in one kernel (the norm's arithmetic), waiting for all earlier work;
// with meta, the kernel first writes meta->v[0 .. n) to meta_out for the kernels after it
cudaError_t launch_embed_rmsnorm(const bi_bf16* E, const int32_t* ids, int32_t V, const bi_bf16* gamma, bi_bf16* x,
                                 bi_bf16* y, int32_t T, int32_t d, float eps, int32_t* status, cudaStream_t s,
                                 const ArgmaxFuse* am = nullptr, int64_t am_rows = 0, const StepMeta* meta = nullptr,
                                 int32_t* meta_out = nullptr);
cudaError_t launch_embed(const bi_bf16* E, const int32_t* ids, bi_bf16* x, int32_t T, int32_t V,
                         int32_t d, int32_t* status, cudaStream_t s, bool after_all = false);
cudaError_t launch_rope_kv_append(const float* qkv, const int32_t* tok_req, const int32_t* tok_pos,
                                  const float* rc, const float* rs, int32_t max_pos, bi_bf16* q_out,
                                  bi_bf16* kc, bi_bf16* vc, const int32_t* page_table,
                                  int32_t max_pages, int32_t num_pages, int32_t T, int32_t H,
                                  int32_t Hkv, int32_t Dh, int32_t* status, cudaStream_t s);
cudaError_t launch_argmax(const float* logits, int32_t* out, int32_t R, int32_t V, cudaStream_t s);

// ---- logprobs and seeded sampling (k_logits.cu) ----
size_t log_softmax_ws_bytes(int32_t R, int32_t V);
cudaError_t launch_log_softmax(const float* logits, float* out, int32_t R, int32_t V, void* ws, cudaStream_t s);
size_t sample_ws_bytes(int32_t R, int32_t V);
cudaError_t launch_sample(const float* logits, const uint32_t* seeds, const int32_t* positions, const float* temps,
                          int32_t* tokens, int32_t R, int32_t V, void* ws, cudaStream_t s);
cudaError_t launch_pack_gate_up(const bi_bf16* g, const bi_bf16* u, bi_bf16* gu, int32_t F,
                                int32_t d, cudaStream_t s);

// ---- attention (k_attention.cu) ----
// How a work entry e maps to (query/output row t, request r, position p).
struct EntryMap {
    int32_t kind;            // 0: decode by request, 1: token list, 2: ragged cu_q
    const int32_t* a;        // kind 0: seq_lens[B]; kind 1: list[n]; kind 2: cu_q[B+1]
    const int32_t* b;        // kind 1: tok_req[T];  kind 2: q_pos0[B]
    const int32_t* c;        // kind 1: tok_pos[T]
    int32_t nreq;            // kind 2: B
};

struct AttnGeom {
    const bi_bf16* q;        // [rows, H, Dh]
    const bi_bf16* kc;       // [num_pages, Hkv, 16, Dh]
    const bi_bf16* vc;
    const int32_t* page_table;
    void* out;               // [rows, H, Dh]
    int32_t out_f32;
    int32_t H, Hkv, Dh, max_pages, num_pages;
    float scale;
    int32_t* status;
};

// split size: 0 -> fixed BI_KV_CHUNK chunks; >0 -> variant rule with chunk2
size_t decode_ws_bytes(int32_t n_entries, int32_t H, int32_t Dh, int32_t max_splits);
int32_t invariant_max_splits(int32_t max_seq);
// variant occupancy rule: fills chunk2 and the bound on splits per request
void variant_split_plan(int32_t B, int32_t H, int32_t Hkv, int32_t max_seq, int32_t* chunk2,
                        int32_t* max_splits);
// early_kv: the caller guarantees that of each entry's keys only the last
// position was written since the kernels before this one in the stream began
// (the forward step's decode entries); chunks before it then request their
// K/V copies before the dependency wait.
cudaError_t launch_decode_attention(const AttnGeom& g, const EntryMap& em, int32_t n_entries,
                                    int32_t max_splits, int32_t variant_chunk2, float* ws_o,
                                    float* ws_ml, cudaStream_t s, bool early_kv = false);
// q_rows: rows of g.q (every token index an entry names is below it)
cudaError_t launch_prefill_attention(const AttnGeom& g, const EntryMap& em, int32_t n_entries, int32_t q_rows,
                                     cudaStream_t s);
bool attention_supported(int32_t H, int32_t Hkv, int32_t Dh);

// Tensor map over a paged K or V cache [num_pages, Hkv, 16, Dh] seen as rows
// of Dh bf16 (row (page * Hkv + head) * 16 + slot), boxes of 16 rows x 64
// elements with the 128-byte swizzle (k_gemm.cu owns the driver entry point).
bool encode_kv_map(CUtensorMap* map, const bi_bf16* cache, int64_t num_pages, int32_t Hkv, int32_t Dh);
// Tensor map over queries q [rows, H, Dh] seen as three dimensions (Dh, H,
// rows): a box of 64 elements x G heads x 128/G tokens brings the 128
// (token, head) rows of one GQA group of consecutive tokens, each row's 64
// elements as 128 bytes with the 128-byte swizzle.
bool encode_q_map(CUtensorMap* map, const bi_bf16* q, int64_t rows, int32_t H, int32_t Dh, int32_t G);

// ---- GEMM (k_gemm.cu) ----
struct GemmPlan {
    int32_t splits;          // 1 = invariant path
};
GemmPlan gemm_plan(int64_t M, int32_t N, int32_t K, bi_mode mode);
size_t gemm_ws_bytes(int64_t M, int32_t N, int32_t K, bi_mode mode);
// weights_settled: no kernel that may still be running when this one starts
// writes W (true inside bi_forward_step, whose first kernel waits for all
// earlier work on the stream), so W may be fetched before the dependency wait.
// am (optional, fp32 output, no epilogue, plan without split-K): fused greedy
// argmax over each row's N outputs; C may then be null (outputs not stored).
// The GEMM's failure-detection check: every bounded wait gives up after
// wait_ns, and the copies of ring stage skip_stage (in issue order, in every
// CTA of a pair) are withheld, so the MMA issuer's wait for them runs out.
struct GemmWaitTest {
    uint64_t wait_ns;
    int32_t skip_stage;
};
bi_status run_gemm(const bi_bf16* A, const bi_bf16* W, void* C, bi_dtype c_dtype,
                   const bi_bf16* residual, bi_epilogue ep, int64_t M, int32_t N, int32_t K,
                   bi_mode mode, void* ws, size_t ws_bytes, int32_t* status, cudaStream_t s,
                   bool weights_settled = false, const ArgmaxFuse* am = nullptr,
                   const RopeFuse* rope = nullptr, const GemmWaitTest* wait_test = nullptr,
                   const NormFuse* norm = nullptr);
// whether run_gemm can take its A operand through a fused RMSNorm (norm) for this shape and mode
bool gemm_can_fuse_norm(int64_t M, int32_t N, int32_t K, bi_mode mode);
// whether run_gemm can fuse RoPE + KV append for this shape and mode
bool gemm_can_fuse_rope(int64_t M, int32_t N, int32_t K, bi_mode mode, int32_t Dh);

}  // namespace bi
