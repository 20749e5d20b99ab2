// Logprobs and seeded sampling over rows of fp32 logits.
//
// "Mathematically equivalent is not bitwise equivalent": logprobs come from
// one log_softmax kernel pair, whichever step (prefill rescoring or decode)
// produced the logits.  A row is cut into segments of kSeg columns (a
// function of V alone); each segment's max and sum of exponentials are
// reduced in one fixed order, and the segments' partials are merged in
// segment order, so a row's logprobs are bitwise the same whatever other rows
// share the launch ("The replacement kernels are deliberately dull": no
// reduction whose order follows the batch).
//
// "The weaker guarantees, which are usually enough": a request's draw depends
// only on its own seed, its position and the column: Gumbel noise from
// MurmurHash3 (x86, 32-bit) of (position, column) under the request's seed,
// in float64, and the token is the argmax of logit / temperature + noise.
// The argmax is a total order (a NaN beats every number, ties go to the
// lowest index), so segments of a row may be searched by separate CTAs and
// combined in any order without changing the winner.  float64 is slow on
// this GPU, so every score is first computed in fp32 with a proven error
// bound; only the columns whose fp32 score lies within the bounds of their
// segment's best fp32 score can be that segment's float64 winner, and only
// they are scored in float64.  The token is the float64 argmax exactly.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace bi {

constexpr int kSeg = 4096;            // columns per segment (log_softmax and sampling)
constexpr int kSegThreads = 256;
constexpr int kPerThread = kSeg / kSegThreads;  // 16 columns per thread: j = seg * kSeg + tid + 256 k

int32_t logit_segments(int32_t V) { return (V + kSeg - 1) / kSeg; }

// ---------------------------------------------------------------------------
// log_softmax: lp_j = (x_j - m) - log(z), m = max_j x_j, z = sum_j exp(x_j - m)
// Pass 1 (one CTA per segment s): m_s = max over the segment, z_s = sum of
// exp(x_j - m_s) in a fixed order: each thread's 16 columns in ascending k,
// an xor butterfly inside each warp, the 8 warps' sums in warp order (a
// segment without a finite maximum contributes z_s = 0).  Pass 2: every CTA
// of the row merges the row's partials in segment order, m = max_s m_s,
// z = sum_s z_s * exp(m_s - m), and writes its segment's logprobs.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSegThreads)
log_softmax_partial_kernel(const float* __restrict__ x, int32_t V, int32_t nseg, float2* __restrict__ part) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[kSegThreads / 32];
    __shared__ float bc;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    const int32_t seg = blockIdx.x, r = blockIdx.y;
    const float* xr = x + static_cast<int64_t>(r) * V;
    float v[kPerThread];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int32_t j = seg * kSeg + tid + kSegThreads * k;
        v[k] = j < V ? xr[j] : -INFINITY;
        mx = fmaxf(mx, v[k]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (tid == 0) {
        float m = red[0];
        for (int w = 1; w < kSegThreads / 32; ++w) m = fmaxf(m, red[w]);
        bc = m;
    }
    __syncthreads();
    const float m = bc;
    float z = 0.0f;
    if (m != -INFINITY) {
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int32_t j = seg * kSeg + tid + kSegThreads * k;
            if (j < V) z = __fadd_rn(z, expf(__fsub_rn(v[k], m)));
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, off));
    __syncthreads();  // red[] is reused
    if (lane == 0) red[warp] = z;
    __syncthreads();
    if (tid == 0) {
        float t = red[0];
        for (int w = 1; w < kSegThreads / 32; ++w) t = __fadd_rn(t, red[w]);
        part[static_cast<int64_t>(r) * nseg + seg] = make_float2(m, t);
    }
}

__global__ void __launch_bounds__(kSegThreads)
log_softmax_write_kernel(const float* __restrict__ x, int32_t V, int32_t nseg, const float2* __restrict__ part,
                         float* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    __shared__ float2 ml;
    const int tid = threadIdx.x;
    const int32_t seg = blockIdx.x, r = blockIdx.y;
    if (tid == 0) {
        const float2* pr = part + static_cast<int64_t>(r) * nseg;
        float m = pr[0].x;
        for (int32_t q = 1; q < nseg; ++q) m = fmaxf(m, pr[q].x);
        float z = 0.0f;
        for (int32_t q = 0; q < nseg; ++q) z = __fadd_rn(z, __fmul_rn(pr[q].y, expf(__fsub_rn(pr[q].x, m))));
        ml = make_float2(m, logf(z));
    }
    __syncthreads();
    const float m = ml.x, lz = ml.y;
    const float* xr = x + static_cast<int64_t>(r) * V;
    float* orow = out + static_cast<int64_t>(r) * V;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int32_t j = seg * kSeg + tid + kSegThreads * k;
        if (j < V) orow[j] = __fsub_rn(__fsub_rn(xr[j], m), lz);
    }
}

size_t log_softmax_ws_bytes(int32_t R, int32_t V) {
    if (R <= 0 || V <= 0) return 0;
    return static_cast<size_t>(R) * logit_segments(V) * sizeof(float2) + 256;
}

cudaError_t launch_log_softmax(const float* logits, float* out, int32_t R, int32_t V, void* ws, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    const int32_t nseg = logit_segments(V);
    float2* part = static_cast<float2*>(ws);
    cudaError_t e = launch_pdl(log_softmax_partial_kernel, dim3(nseg, R), dim3(kSegThreads), 0, s, logits, V, nseg,
                               part);
    if (e != cudaSuccess) return e;
    return launch_pdl(log_softmax_write_kernel, dim3(nseg, R), dim3(kSegThreads), 0, s, logits, V, nseg,
                      static_cast<const float2*>(part), out);
}

// ---------------------------------------------------------------------------
// Seeded Gumbel-max sampling
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t rotl32(uint32_t v, int r) { return (v << r) | (v >> (32 - r)); }

// MurmurHash3_x86_32 of the 8-byte key le32(pos) || le32(col): two 4-byte
// blocks, no tail, length 8, then the final avalanche.
__device__ __forceinline__ uint32_t murmur3_pos_col(uint32_t pos, uint32_t col, uint32_t seed) {
    constexpr uint32_t c1 = 0xcc9e2d51u, c2 = 0x1b873593u;
    uint32_t h = seed;
    uint32_t k = pos * c1;
    k = rotl32(k, 15) * c2;
    h ^= k;
    h = rotl32(h, 13) * 5u + 0xe6546b64u;
    k = col * c1;
    k = rotl32(k, 15) * c2;
    h ^= k;
    h = rotl32(h, 13) * 5u + 0xe6546b64u;
    h ^= 8u;
    h ^= h >> 16;
    h *= 0x85ebca6bu;
    h ^= h >> 13;
    h *= 0xc2b2ae35u;
    h ^= h >> 16;
    return h;
}

// (score a, index ia) beats (b, ib) in the sampling total order.
__device__ __forceinline__ bool beats(double a, int32_t ia, double b, int32_t ib) {
    const bool an = isnan(a), bn = isnan(b);
    if (an || bn) return an && (!bn || ia < ib);
    return a > b || (a == b && ia < ib);
}

// The float64 score of column j (the definition): x_j / t + g_j, or x_j for
// a greedy row.
__device__ __forceinline__ double score64(float x, double td, bool greedy, uint32_t h) {
    if (greedy) return static_cast<double>(x);
    const double u = (static_cast<double>(h) + 0.5) * 0x1p-32;  // exact: (0, 1)
    return __dadd_rn(__ddiv_rn(static_cast<double>(x), td), -log(-log(u)));
}

// fp32 estimate of score64 and the bound on their difference.  With
// u = (h + 0.5) / 2^32: w = -log(u) from u itself when u < 1/2 (w >= ln 2),
// else from 1 - u = (2^32 - 1 - h + 0.5) / 2^32 through log1pf, so neither
// loses digits to cancellation; the arguments carry a relative error of at
// most 2^-23 (two roundings).  __logf is within 2^-21.41 absolute on [0.5, 2]
// and 3 ulp elsewhere, log1pf within 1 ulp: |w32 - w| / w < 9e-6 and
// |g32 - g| < 1e-5 over the whole range of g ([-3.14, 22.9], its ends at
// h = 0 and h = 2^32 - 1).  x * (1/t) and the sum add 3 * 2^-24 of
// |x / t| and of |s|.  delta(s) = 1e-4 + 1e-6 (|s| + 48) covers all of it
// with a margin of five or more (|x / t| <= |s| + 24).  A greedy row is exact
// in fp32 (delta = 0).
__device__ __forceinline__ float score32(float x, float rt, bool greedy, uint32_t h) {
    if (greedy) return x;
    float w;
    if (h < 0x80000000u) {
        const float u = __fmul_rn(__fadd_rn(static_cast<float>(h), 0.5f), 0x1p-32f);
        w = -__logf(u);
    } else {
        const float v = __fmul_rn(__fadd_rn(static_cast<float>(0xffffffffu - h), 0.5f), 0x1p-32f);
        w = -log1pf(-v);
    }
    return __fadd_rn(__fmul_rn(x, rt), -__logf(w));
}
__device__ __forceinline__ float score_bound(float s, bool greedy) {
    return greedy ? 0.0f : __fadd_rn(1e-4f, __fmul_rn(1e-6f, __fadd_rn(fabsf(s), 48.0f)));
}

// grid (segments, rows): the float64 winner of one segment of a row.  Every
// column's fp32 score is kept in registers; with M the segment's best fp32
// score (reached at column k), the segment's float64 winner w satisfies
// s32_w + delta_w >= s64_w >= s64_k >= M - delta(M), so only such columns
// (and any non-finite score or maximum: a NaN beats every number, an
// overflow leaves no bound) are scored in float64.  The row's winner is the
// float64 winner of its own segment, so the merge below is exact.
__global__ void __launch_bounds__(kSegThreads)
sample_segment_kernel(const float* __restrict__ x, const uint32_t* __restrict__ seeds,
                      const int32_t* __restrict__ positions, const float* __restrict__ temps, int32_t V,
                      int32_t nseg, double* __restrict__ ws_score, int32_t* __restrict__ ws_idx) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[kSegThreads / 32];
    __shared__ float s_thr;
    __shared__ double s_sc[kSegThreads / 32];
    __shared__ int32_t s_ix[kSegThreads / 32];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    const int32_t seg = blockIdx.x, r = blockIdx.y;
    const float* xr = x + static_cast<int64_t>(r) * V;
    const float t = temps[r];
    const bool greedy = !(t > 0.0f);  // temperature 0 (or not positive): the greedy argmax of the logits
    const float rt = greedy ? 1.0f : __frcp_rn(t);
    const double td = static_cast<double>(t);
    const uint32_t seed = seeds[r], pos = static_cast<uint32_t>(positions[r]);
    float s32[kPerThread];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int32_t j = seg * kSeg + tid + kSegThreads * k;
        s32[k] = -INFINITY;
        if (j < V) {
            const uint32_t h = greedy ? 0u : murmur3_pos_col(pos, static_cast<uint32_t>(j), seed);
            s32[k] = score32(xr[j], rt, greedy, h);
            mx = fmaxf(mx, s32[k]);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (tid == 0) {
        float m = red[0];
        for (int w = 1; w < kSegThreads / 32; ++w) m = fmaxf(m, red[w]);
        s_thr = isfinite(m) ? __fsub_rn(m, score_bound(m, greedy)) : -INFINITY;
    }
    __syncthreads();
    const float thr = s_thr;
    double best = 0.0;
    int32_t bi = -1;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int32_t j = seg * kSeg + tid + kSegThreads * k;
        if (j < V) {
            const bool cand = !isfinite(s32[k]) || !(thr > -INFINITY) ||
                              __fadd_rn(s32[k], score_bound(s32[k], greedy)) >= thr;
            if (cand) {
                const uint32_t h = greedy ? 0u : murmur3_pos_col(pos, static_cast<uint32_t>(j), seed);
                const double sc = score64(xr[j], td, greedy, h);
                if (bi < 0 || beats(sc, j, best, bi)) {
                    best = sc;
                    bi = j;
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const double os = __shfl_xor_sync(0xffffffffu, best, off);
        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi >= 0 && (bi < 0 || beats(os, oi, best, bi))) {
            best = os;
            bi = oi;
        }
    }
    if (lane == 0) {
        s_sc[warp] = best;
        s_ix[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kSegThreads / 32; ++w)
            if (s_ix[w] >= 0 && (bi < 0 || beats(s_sc[w], s_ix[w], best, bi))) {
                best = s_sc[w];
                bi = s_ix[w];
            }
        ws_score[static_cast<int64_t>(r) * nseg + seg] = best;
        ws_idx[static_cast<int64_t>(r) * nseg + seg] = bi;
    }
}

// grid (rows), one warp: the winner over a row's segments.
__global__ void __launch_bounds__(32)
sample_merge_kernel(const double* __restrict__ ws_score, const int32_t* __restrict__ ws_idx, int32_t nseg,
                    int32_t* __restrict__ tokens) {
    pdl_trigger();
    pdl_wait();
    const int32_t r = blockIdx.x;
    const int lane = threadIdx.x;
    double best = 0.0;
    int32_t bi = -1;
    for (int32_t sg = lane; sg < nseg; sg += 32) {
        const double sc = ws_score[static_cast<int64_t>(r) * nseg + sg];
        const int32_t ix = ws_idx[static_cast<int64_t>(r) * nseg + sg];
        if (ix >= 0 && (bi < 0 || beats(sc, ix, best, bi))) {
            best = sc;
            bi = ix;
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const double os = __shfl_xor_sync(0xffffffffu, best, off);
        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi >= 0 && (bi < 0 || beats(os, oi, best, bi))) {
            best = os;
            bi = oi;
        }
    }
    if (lane == 0) tokens[r] = bi;
}

size_t sample_ws_bytes(int32_t R, int32_t V) {
    if (R <= 0 || V <= 0) return 0;
    const size_t n = static_cast<size_t>(R) * logit_segments(V);
    return n * (sizeof(double) + sizeof(int32_t)) + 256;
}

cudaError_t launch_sample(const float* logits, const uint32_t* seeds, const int32_t* positions, const float* temps,
                          int32_t* tokens, int32_t R, int32_t V, void* ws, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    const int32_t nseg = logit_segments(V);
    const size_t n = static_cast<size_t>(R) * nseg;
    double* ws_score = static_cast<double*>(ws);
    int32_t* ws_idx = reinterpret_cast<int32_t*>(ws_score + n);
    cudaError_t e = launch_pdl(sample_segment_kernel, dim3(nseg, R), dim3(kSegThreads), 0, s, logits, seeds,
                               positions, temps, V, nseg, ws_score, ws_idx);
    if (e != cudaSuccess) return e;
    return launch_pdl(sample_merge_kernel, dim3(R), dim3(32), 0, s, static_cast<const double*>(ws_score),
                      static_cast<const int32_t*>(ws_idx), nseg, tokens);
}

}  // namespace bi
