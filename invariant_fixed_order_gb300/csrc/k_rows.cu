// Row-wise kernels: RMSNorm (optionally of gathered rows), embedding gather,
// RoPE + paged KV append, greedy argmax, gate/up packing.
#include "common.cuh"
#include "internal.h"

namespace bi {

// ---------------------------------------------------------------------------
// RMSNorm: one warp per row ("Lockstep", "The fix": one fixed reduction order).
// Lane l owns 16-byte chunks l, l+32, l+64, ... and adds their squares in
// ascending element order with fused multiply-adds; the 32 lane sums then meet
// in an xor-butterfly (16, 8, 4, 2, 1).  Addition is commutative, so every
// lane ends with the same bits and the order depends on d only.
//
// A lane issues all loads of a block of CPL chunks (and of their gains)
// before it uses any, so a row costs one memory latency rather than one per
// chunk; when the row fits one block (d <= 256 * CPL) it stays in registers
// for the second pass.  Blocking changes when values arrive, not the order in
// which they are added.
// ---------------------------------------------------------------------------
constexpr int kNormWarps = 4;

// kEmbed: the row is the embedding row E[ids[row]] (the step's first norm);
// the warp also writes it to x_out, the residual stream (an id outside the
// vocabulary reports BI_DEV_BAD_TOKEN and reads as zeros, as embed_kernel).
template <int CPL, bool kEmbed>
__device__ __forceinline__ void rmsnorm_rows(const uint4* x, const uint4* __restrict__ gamma, uint4* y, int64_t rows,
                                             int32_t d8, float eps, float fd, const int32_t* __restrict__ src_rows,
                                             unsigned long long* am_keys, unsigned int* am_counter, int64_t am_rows,
                                             const int32_t* __restrict__ ids, int32_t V, uint4* x_out,
                                             int32_t* status) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kNormWarps + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;  // uniform per warp
    if (am_keys != nullptr && lane == 0 && row < am_rows) {  // a fused argmax later in the stream
        am_keys[row] = kArgmaxKeyNone;
        if (row == 0) *am_counter = 0u;
    }
    const uint4* xr;
    bool zero = false;
    if constexpr (kEmbed) {
        const int32_t id = ids[row];
        zero = !(id >= 0 && id < V);
        if (zero && lane == 0) report(status, BI_DEV_BAD_TOKEN);
        xr = x + static_cast<int64_t>(zero ? 0 : id) * d8;
    } else {
        const int64_t src = src_rows != nullptr ? static_cast<int64_t>(src_rows[row]) : row;
        xr = x + src * d8;
    }
    uint4* yr = y + row * d8;
    constexpr int kBlock = 32 * CPL;
    uint4 v[CPL], g[CPL];
    auto load_block = [&](int base, bool with_gamma) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = base + lane + 32 * i;
            if (c < d8) {
                v[i] = zero ? make_uint4(0, 0, 0, 0) : xr[c];
                if (with_gamma) g[i] = gamma[c];
            }
        }
    };
    auto store_block = [&](int base, float rinv) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = base + lane + 32 * i;
            if (c < d8) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                const uint32_t gw[4] = {g[i].x, g[i].y, g[i].z, g[i].w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = __fmul_rn(__fmul_rn(bf16_lo(w[e]), rinv), bf16_lo(gw[e]));
                    const float b = __fmul_rn(__fmul_rn(bf16_hi(w[e]), rinv), bf16_hi(gw[e]));
                    o[e] = pack_bf16x2(a, b);
                }
                yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    };
    const bool cached = d8 <= kBlock;
    float ss = 0.0f;
    for (int base = 0; base < d8; base += kBlock) {
        load_block(base, cached);
        if constexpr (kEmbed) {
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = base + lane + 32 * i;
                if (c < d8) x_out[row * d8 + c] = v[i];
            }
        }
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            if (base + lane + 32 * i < d8) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = bf16_lo(w[e]);
                    ss = __fmaf_rn(a, a, ss);
                    const float b = bf16_hi(w[e]);
                    ss = __fmaf_rn(b, b, ss);
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    const float mean = __fdiv_rn(ss, fd);
    const float rinv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
    if (cached) {
        store_block(0, rinv);
    } else {
        for (int base = 0; base < d8; base += kBlock) {
            load_block(base, true);
            store_block(base, rinv);
        }
    }
}

template <int CPL, bool kEmbed>
__global__ void __launch_bounds__(kNormWarps * 32)
rmsnorm_kernel(const uint4* x, const uint4* __restrict__ gamma, uint4* y, int64_t rows, int32_t d8, float eps,
               float fd, const int32_t* __restrict__ src_rows, unsigned long long* am_keys, unsigned int* am_counter,
               int64_t am_rows, const int32_t* __restrict__ ids, int32_t V, uint4* x_out, int32_t* status) {
    pdl_trigger();
    pdl_wait();
    rmsnorm_rows<CPL, kEmbed>(x, gamma, y, rows, d8, eps, fd, src_rows, am_keys, am_counter, am_rows, ids, V, x_out,
                              status);
}

// The step's first kernel with its per-token metadata as a parameter: every thread first copies its share of
// the values to meta_out (read by the step's later kernels after their dependency wait), then the embedding
// gather and the norm as rmsnorm_kernel<CPL, true>.
template <int CPL>
__global__ void __launch_bounds__(kNormWarps * 32)
embed_rmsnorm_meta_kernel(const __grid_constant__ StepMeta meta, int32_t* meta_out, const uint4* x,
                          const uint4* __restrict__ gamma, uint4* y, int64_t rows, int32_t d8, float eps, float fd,
                          unsigned long long* am_keys, unsigned int* am_counter, int64_t am_rows,
                          const int32_t* __restrict__ ids, int32_t V, uint4* x_out, int32_t* status) {
    pdl_trigger();
    pdl_wait();
    for (int32_t i = static_cast<int32_t>(blockIdx.x * blockDim.x + threadIdx.x); i < meta.n;
         i += static_cast<int32_t>(gridDim.x * blockDim.x))
        meta_out[i] = meta.v[i];
    rmsnorm_rows<CPL, true>(x, gamma, y, rows, d8, eps, fd, nullptr, am_keys, am_counter, am_rows, ids, V, x_out,
                            status);
}

template <bool kEmbed>
static cudaError_t launch_rmsnorm_t(bool pdl, const bi_bf16* x, const bi_bf16* gamma, bi_bf16* y, int64_t rows,
                                    int32_t d, float eps, cudaStream_t s, const int32_t* src_rows,
                                    const ArgmaxFuse* am, int64_t am_rows, const int32_t* ids, int32_t V,
                                    bi_bf16* x_out, int32_t* status) {
    if (rows <= 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((rows + kNormWarps - 1) / kNormWarps));
    const dim3 block(kNormWarps * 32);
    const int32_t d8 = d / 8;
    auto go = [&](auto kernel) {
        return launch_k(pdl, kernel, grid, block, 0, s, reinterpret_cast<const uint4*>(x),
                        reinterpret_cast<const uint4*>(gamma), reinterpret_cast<uint4*>(y), rows, d8, eps,
                        static_cast<float>(d), src_rows, am ? am->keys : nullptr, am ? am->counter : nullptr, am_rows,
                        ids, V, reinterpret_cast<uint4*>(x_out), status);
    };
    if (d8 <= 32) return go(rmsnorm_kernel<1, kEmbed>);
    if (d8 <= 64) return go(rmsnorm_kernel<2, kEmbed>);
    if (d8 <= 128) return go(rmsnorm_kernel<4, kEmbed>);
    if (d8 <= 256) return go(rmsnorm_kernel<8, kEmbed>);
    return go(rmsnorm_kernel<16, kEmbed>);
}

cudaError_t launch_rmsnorm(const bi_bf16* x, const bi_bf16* gamma, bi_bf16* y, int64_t rows, int32_t d, float eps,
                           cudaStream_t s, const int32_t* src_rows, const ArgmaxFuse* am) {
    return launch_rmsnorm_t<false>(true, x, gamma, y, rows, d, eps, s, src_rows, am, rows, nullptr, 0, nullptr,
                                   nullptr);
}

cudaError_t launch_embed_rmsnorm(const bi_bf16* E, const int32_t* ids, int32_t V, const bi_bf16* gamma, bi_bf16* x,
                                 bi_bf16* y, int32_t T, int32_t d, float eps, int32_t* status, cudaStream_t s,
                                 const ArgmaxFuse* am, int64_t am_rows, const StepMeta* meta, int32_t* meta_out) {
    // the step's first kernel: launched without programmatic serialisation, so it waits for all earlier work;
    // it also initialises the keys of the step's fused greedy argmax (rows < am_rows <= T)
    if (meta == nullptr)
        return launch_rmsnorm_t<true>(false, E, gamma, y, T, d, eps, s, nullptr, am, am_rows, ids, V, x, status);
    if (T <= 0 || meta_out == nullptr || meta->n < 0 || meta->n > kStepMetaMax) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>((T + kNormWarps - 1) / kNormWarps));
    const dim3 block(kNormWarps * 32);
    const int32_t d8 = d / 8;
    auto go = [&](auto kernel) {
        return launch_k(false, kernel, grid, block, 0, s, *meta, meta_out, reinterpret_cast<const uint4*>(E),
                        reinterpret_cast<const uint4*>(gamma), reinterpret_cast<uint4*>(y), static_cast<int64_t>(T),
                        d8, eps, static_cast<float>(d), am ? am->keys : nullptr, am ? am->counter : nullptr, am_rows,
                        ids, V, reinterpret_cast<uint4*>(x), status);
    };
    if (d8 <= 32) return go(embed_rmsnorm_meta_kernel<1>);
    if (d8 <= 64) return go(embed_rmsnorm_meta_kernel<2>);
    if (d8 <= 128) return go(embed_rmsnorm_meta_kernel<4>);
    if (d8 <= 256) return go(embed_rmsnorm_meta_kernel<8>);
    return go(embed_rmsnorm_meta_kernel<16>);
}

// ---------------------------------------------------------------------------
// Embedding gather: x[t] = E[ids[t]].
// ---------------------------------------------------------------------------
__global__ void embed_kernel(const uint4* __restrict__ E, const int32_t* __restrict__ ids,
                             uint4* __restrict__ x, int32_t V, int32_t d8, int32_t* status) {
    pdl_trigger();
    pdl_wait();
    const int32_t t = blockIdx.x;
    const int32_t id = ids[t];
    const bool ok = id >= 0 && id < V;
    if (!ok && threadIdx.x == 0) report(status, BI_DEV_BAD_TOKEN);
    for (int c = threadIdx.x; c < d8; c += blockDim.x)
        x[static_cast<int64_t>(t) * d8 + c] = ok ? E[static_cast<int64_t>(id) * d8 + c] : make_uint4(0, 0, 0, 0);
}

cudaError_t launch_embed(const bi_bf16* E, const int32_t* ids, bi_bf16* x, int32_t T, int32_t V,
                         int32_t d, int32_t* status, cudaStream_t s, bool after_all) {
    if (T <= 0) return cudaSuccess;
    return launch_k(!after_all, embed_kernel, dim3(T), dim3(128), 0, s, reinterpret_cast<const uint4*>(E), ids,
                    reinterpret_cast<uint4*>(x), V, d / 8, status);
}

// ---------------------------------------------------------------------------
// RoPE (rotate-half) + KV append.  q and k heads are rotated in fp32 from the
// fp32 projection, each output rounded once to bf16:
//   out[i]        = x[i] * cos - x[i + Dh/2] * sin
//   out[i + Dh/2] = x[i + Dh/2] * cos + x[i] * sin
// (each product rounded, then the sum: no fused multiply-add).
// ---------------------------------------------------------------------------
// One thread per rotated pair: grid (T, ceil((H + 2 Hkv) * Dh/2 / 128)).
constexpr int kRopeThreads = 128;

__global__ void __launch_bounds__(kRopeThreads)
rope_append_kernel(const float* __restrict__ qkv, const int32_t* __restrict__ tok_req,
                   const int32_t* __restrict__ tok_pos, const float* __restrict__ rc,
                   const float* __restrict__ rs, int32_t max_pos, uint16_t* __restrict__ q_out,
                   uint16_t* __restrict__ kc, uint16_t* __restrict__ vc,
                   const int32_t* __restrict__ page_table, int32_t max_pages, int32_t num_pages,
                   int32_t H, int32_t Hkv, int32_t Dh, int32_t* status) {
    pdl_trigger();
    pdl_wait();
    const int32_t t = blockIdx.x;
    const int32_t half = Dh / 2;
    const int32_t w = static_cast<int32_t>(blockIdx.y) * kRopeThreads + threadIdx.x;
    if (w >= (H + 2 * Hkv) * half) return;
    const bool reporter = blockIdx.y == 0 && threadIdx.x == 0;
    const int32_t pos = tok_pos[t];
    const int32_t req = tok_req[t];
    bool ok = pos >= 0 && pos < max_pos && (pos / BI_PAGE) < max_pages;
    int32_t page = 0;
    if (ok) {
        page = page_table[static_cast<int64_t>(req) * max_pages + pos / BI_PAGE];
        if (page < 0 || page >= num_pages) {
            if (reporter) report(status, BI_DEV_BAD_PAGE);
            ok = false;
        }
    } else if (reporter) {
        report(status, BI_DEV_BAD_POSITION);
    }
    const int32_t slot = pos & (BI_PAGE - 1);
    const int32_t head = w / half;
    const int32_t i = w - head * half;
    const float* row = qkv + static_cast<int64_t>(t) * ((H + 2 * Hkv) * Dh);
    const float x0 = row[head * Dh + i];
    const float x1 = row[head * Dh + i + half];
    float r0, r1;
    if (head < H + Hkv) {
        const float c = ok ? rc[static_cast<int64_t>(pos) * half + i] : 1.0f;
        const float sn = ok ? rs[static_cast<int64_t>(pos) * half + i] : 0.0f;
        r0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn));
        r1 = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, sn));
    } else {
        r0 = x0;
        r1 = x1;
    }
    const uint16_t b0 = f32_to_bf16(r0), b1 = f32_to_bf16(r1);
    if (head < H) {
        uint16_t* qo = q_out + (static_cast<int64_t>(t) * H + head) * Dh;
        qo[i] = b0;
        qo[i + half] = b1;
    } else if (ok) {
        const bool is_k = head < H + Hkv;
        const int32_t g = is_k ? head - H : head - H - Hkv;
        uint16_t* dst = (is_k ? kc : vc) + ((static_cast<int64_t>(page) * Hkv + g) * BI_PAGE + slot) * Dh;
        dst[i] = b0;
        dst[i + half] = b1;
    }
}

cudaError_t launch_rope_kv_append(const float* qkv, const int32_t* tok_req, const int32_t* tok_pos,
                                  const float* rc, const float* rs, int32_t max_pos, bi_bf16* q_out,
                                  bi_bf16* kc, bi_bf16* vc, const int32_t* page_table,
                                  int32_t max_pages, int32_t num_pages, int32_t T, int32_t H,
                                  int32_t Hkv, int32_t Dh, int32_t* status, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int32_t work = (H + 2 * Hkv) * (Dh / 2);
    const dim3 grid(T, (work + kRopeThreads - 1) / kRopeThreads);
    return launch_pdl(rope_append_kernel, grid, dim3(kRopeThreads), 0, s, qkv, tok_req, tok_pos, rc, rs, max_pos,
                      q_out, kc, vc, page_table, max_pages, num_pages, H, Hkv, Dh, status);
}

// ---------------------------------------------------------------------------
// Greedy argmax ("temperature=0 means deterministic").  (value, index) pairs
// are totally ordered: a NaN beats every number, a larger number beats a
// smaller one, and between equals (or two NaNs) the lower index wins.  The
// winner of a totally ordered set does not depend on the reduction order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool beats(float a, int32_t ia, float b, int32_t ib) {
    const bool an = isnan(a), bn = isnan(b);
    if (an != bn) return an;
    if (!an && a != b) return a > b;
    return ia < ib;
}

constexpr int kArgmaxThreads = 1024;
constexpr int kArgmaxUnroll = 8;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kArgmaxThreads)
argmax_kernel(const float* __restrict__ logits, int32_t* __restrict__ out, int32_t V, int32_t nv) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sv[kArgmaxThreads / 32];
    __shared__ int32_t si[kArgmaxThreads / 32];
    const float* row = logits + static_cast<int64_t>(blockIdx.x) * V;
    float bv = -INFINITY;
    int32_t bi = 0x7fffffff;
    // nv > 0: the row is read as nv aligned float4s, then the V - 4 nv tail
    const float4* row4 = reinterpret_cast<const float4*>(row);
    for (int32_t base = 0; base < nv; base += kArgmaxUnroll * kArgmaxThreads) {
        float4 a[kArgmaxUnroll];
#pragma unroll
        for (int u = 0; u < kArgmaxUnroll; ++u) {
            const int32_t q = base + u * kArgmaxThreads + static_cast<int32_t>(threadIdx.x);
            if (q < nv) a[u] = row4[q];
        }
#pragma unroll
        for (int u = 0; u < kArgmaxUnroll; ++u) {
            const int32_t q = base + u * kArgmaxThreads + static_cast<int32_t>(threadIdx.x);
            if (q < nv) {
                const float v4[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (beats(v4[e], 4 * q + e, bv, bi)) { bv = v4[e]; bi = 4 * q + e; }
            }
        }
    }
    for (int32_t j = 4 * nv + static_cast<int32_t>(threadIdx.x); j < V; j += kArgmaxThreads) {
        const float v = row[j];
        if (beats(v, j, bv, bi)) { bv = v; bi = j; }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (beats(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
    __syncthreads();
    if (warp == 0) {
        bv = sv[lane];
        bi = si[lane];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (beats(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) out[blockIdx.x] = bi;
    }
}

cudaError_t launch_argmax(const float* logits, int32_t* out, int32_t R, int32_t V, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    // every row starts 16-byte aligned when the base is and V % 4 == 0
    const bool vec = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && V % 4 == 0;
    return launch_pdl(argmax_kernel, dim3(R), dim3(kArgmaxThreads), 0, s, logits, out, V, vec ? V / 4 : 0);
}

// ---------------------------------------------------------------------------
// Gate/up interleave (a plain copy).
// ---------------------------------------------------------------------------
__global__ void pack_gate_up_kernel(const uint4* __restrict__ g, const uint4* __restrict__ u,
                                    uint4* __restrict__ gu, int32_t d8) {
    pdl_trigger();
    pdl_wait();
    const int32_t r = blockIdx.x;  // output row in [0, 2F)
    const int32_t j = r / (2 * BI_SWIGLU_GROUP), w = r % (2 * BI_SWIGLU_GROUP);
    const uint4* src = (w < BI_SWIGLU_GROUP ? g : u) +
                       static_cast<int64_t>(j * BI_SWIGLU_GROUP + (w % BI_SWIGLU_GROUP)) * d8;
    for (int c = threadIdx.x; c < d8; c += blockDim.x) gu[static_cast<int64_t>(r) * d8 + c] = src[c];
}

cudaError_t launch_pack_gate_up(const bi_bf16* g, const bi_bf16* u, bi_bf16* gu, int32_t F,
                                int32_t d, cudaStream_t s) {
    if (F <= 0) return cudaSuccess;
    return launch_pdl(pack_gate_up_kernel, dim3(2 * F), dim3(256), 0, s, reinterpret_cast<const uint4*>(g),
                      reinterpret_cast<const uint4*>(u), reinterpret_cast<uint4*>(gu), d / 8);
}

}  // namespace bi
