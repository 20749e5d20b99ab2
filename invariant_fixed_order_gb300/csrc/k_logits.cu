// Logprobs and seeded sampling over rows of fp32 logits.
//
// "Mathematically equivalent is not bitwise equivalent": logprobs come from
// one log_softmax kernel, whichever step (prefill rescoring or decode)
// produced the logits.  The kernel runs one CTA per row and reduces the row
// in one fixed order that depends on V alone ("The replacement kernels are
// deliberately dull": a block per row, no cross-block reduction), so a row's
// logprobs are bitwise the same whatever other rows share the launch.
//
// "The weaker guarantees, which are usually enough": a request's draw depends
// only on its own seed, its position and the column: Gumbel noise from
// MurmurHash3 (x86, 32-bit) of (position, column) under the request's seed,
// in float64, and the token is the argmax of logit / temperature + noise.
// The argmax is a total order (a NaN beats every number, ties go to the
// lowest index), so segments of a row may be searched by separate CTAs and
// combined in any order without changing the winner.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace bi {

constexpr int kLsThreads = 512;
constexpr int kLsWarps = kLsThreads / 32;
constexpr int kSampleSeg = 4096;     // columns per sampling CTA
constexpr int kSampleThreads = 256;

// ---------------------------------------------------------------------------
// log_softmax: lp_j = (x_j - m) - log(z), m = max_j x_j, z = sum_j exp(x_j - m)
// Fixed order of z: thread t sums its columns serially in ascending order
// (vector path: float4 q = t + 512 i, its 4 lanes in order; scalar path:
// column t + 512 i), then an xor butterfly inside each warp, then the warps'
// sums in warp order.
// ---------------------------------------------------------------------------
template <bool kVec4>
__global__ void __launch_bounds__(kLsThreads)
log_softmax_kernel(const float* __restrict__ x, float* __restrict__ out, int32_t V) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[kLsWarps];
    __shared__ float bc;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    const float* xr = x + static_cast<int64_t>(blockIdx.x) * V;
    float* orow = out + static_cast<int64_t>(blockIdx.x) * V;
    const int32_t nq = kVec4 ? V / 4 : V;

    // max (order-free; NaN never wins fmaxf, but reaches z below and makes the row NaN)
    float mx = -INFINITY;
    for (int32_t q = tid; q < nq; q += kLsThreads) {
        if constexpr (kVec4) {
            const float4 v = reinterpret_cast<const float4*>(xr)[q];
            mx = fmaxf(mx, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
        } else {
            mx = fmaxf(mx, xr[q]);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (tid == 0) {
        float m = red[0];
        for (int w = 1; w < kLsWarps; ++w) m = fmaxf(m, red[w]);
        bc = m;
    }
    __syncthreads();
    const float m = bc;

    // z in the fixed order above
    float z = 0.0f;
    for (int32_t q = tid; q < nq; q += kLsThreads) {
        if constexpr (kVec4) {
            const float4 v = reinterpret_cast<const float4*>(xr)[q];
            z = __fadd_rn(z, expf(__fsub_rn(v.x, m)));
            z = __fadd_rn(z, expf(__fsub_rn(v.y, m)));
            z = __fadd_rn(z, expf(__fsub_rn(v.z, m)));
            z = __fadd_rn(z, expf(__fsub_rn(v.w, m)));
        } else {
            z = __fadd_rn(z, expf(__fsub_rn(xr[q], m)));
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, off));
    __syncthreads();  // red[] is reused
    if (lane == 0) red[warp] = z;
    __syncthreads();
    if (tid == 0) {
        float s = red[0];
        for (int w = 1; w < kLsWarps; ++w) s = __fadd_rn(s, red[w]);
        bc = logf(s);
    }
    __syncthreads();
    const float lz = bc;

    for (int32_t q = tid; q < nq; q += kLsThreads) {
        if constexpr (kVec4) {
            const float4 v = reinterpret_cast<const float4*>(xr)[q];
            reinterpret_cast<float4*>(orow)[q] =
                make_float4(__fsub_rn(__fsub_rn(v.x, m), lz), __fsub_rn(__fsub_rn(v.y, m), lz),
                            __fsub_rn(__fsub_rn(v.z, m), lz), __fsub_rn(__fsub_rn(v.w, m), lz));
        } else {
            orow[q] = __fsub_rn(__fsub_rn(xr[q], m), lz);
        }
    }
}

cudaError_t launch_log_softmax(const float* logits, float* out, int32_t R, int32_t V, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    const bool vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    if (vec) return launch_pdl(log_softmax_kernel<true>, dim3(R), dim3(kLsThreads), 0, s, logits, out, V);
    return launch_pdl(log_softmax_kernel<false>, dim3(R), dim3(kLsThreads), 0, s, logits, out, V);
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

// grid (segments, rows): the best (score, column) of one row's segment.
__global__ void __launch_bounds__(kSampleThreads)
sample_segment_kernel(const float* __restrict__ x, const uint32_t* __restrict__ seeds,
                      const int32_t* __restrict__ positions, const float* __restrict__ temps, int32_t V,
                      int32_t nseg, double* __restrict__ ws_score, int32_t* __restrict__ ws_idx) {
    pdl_trigger();
    pdl_wait();
    __shared__ double s_sc[kSampleThreads / 32];
    __shared__ int32_t s_ix[kSampleThreads / 32];
    const int32_t seg = blockIdx.x, r = blockIdx.y;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    const float* xr = x + static_cast<int64_t>(r) * V;
    const float t = temps[r];
    const bool greedy = !(t > 0.0f);  // temperature 0 (or not positive): the greedy argmax of the logits
    const double td = static_cast<double>(t);
    const uint32_t seed = seeds[r], pos = static_cast<uint32_t>(positions[r]);
    const int32_t j0 = seg * kSampleSeg, j1 = min(V, j0 + kSampleSeg);
    double best = 0.0;
    int32_t bi = -1;
    for (int32_t j = j0 + tid; j < j1; j += kSampleThreads) {
        double sc = static_cast<double>(xr[j]);
        if (!greedy) {
            const uint32_t h = murmur3_pos_col(pos, static_cast<uint32_t>(j), seed);
            const double u = (static_cast<double>(h) + 0.5) * 0x1p-32;  // exact: (0, 1)
            const double g = -log(-log(u));
            sc = __dadd_rn(__ddiv_rn(sc, td), g);
        }
        if (bi < 0 || beats(sc, j, best, bi)) {
            best = sc;
            bi = j;
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
        for (int w = 1; w < kSampleThreads / 32; ++w)
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

int32_t sample_segments(int32_t V) { return (V + kSampleSeg - 1) / kSampleSeg; }

size_t sample_ws_bytes(int32_t R, int32_t V) {
    if (R <= 0 || V <= 0) return 0;
    const size_t n = static_cast<size_t>(R) * sample_segments(V);
    return n * sizeof(double) + n * sizeof(int32_t) + 256;
}

cudaError_t launch_sample(const float* logits, const uint32_t* seeds, const int32_t* positions, const float* temps,
                          int32_t* tokens, int32_t R, int32_t V, void* ws, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    const int32_t nseg = sample_segments(V);
    double* ws_score = static_cast<double*>(ws);
    int32_t* ws_idx = reinterpret_cast<int32_t*>(ws_score + static_cast<size_t>(R) * nseg);
    cudaError_t e = launch_pdl(sample_segment_kernel, dim3(nseg, R), dim3(kSampleThreads), 0, s, logits, seeds,
                               positions, temps, V, nseg, ws_score, ws_idx);
    if (e != cudaSuccess) return e;
    return launch_pdl(sample_merge_kernel, dim3(R), dim3(32), 0, s, static_cast<const double*>(ws_score),
                      static_cast<const int32_t*>(ws_idx), nseg, tokens);
}

}  // namespace bi
