// Paged split-KV attention ("Lockstep", "The fix": the split points come from
// the request, not the batch; "Batch invariance and reproducible inference",
// "1 · Split-K and segmented attention reductions": the split count is
// ceil(seq_len / tile), a function of the request's own length).
//
// One device function computes the fp32 partial (m, l, o) of G query heads
// (one GQA group) of one query against one chunk of keys.  Decode runs it in
// one CTA per (query, kv head, chunk) and merges the partials in a second
// kernel; prefill runs it chunk after chunk in one CTA per (query, kv head)
// and folds as it goes.  Both use the same chunk boundaries (multiples of
// BI_KV_CHUNK from key 0), the same partial and the same fold, so a token's
// output has the same bits whichever path, batch or prefill chunking
// produced it.  Every floating-point step below is an explicit round-to-
// nearest intrinsic so the compiler cannot fuse or reorder it differently in
// the two kernels.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace bi {

constexpr int kAttnThreads = 128;
constexpr int kMaxChunkPages = BI_KV_CHUNK / BI_PAGE + 1;  // a variant piece may straddle one more page
constexpr int kSub = 64;                                   // keys per staged sub-chunk
constexpr int kRing = 4;                                   // staged sub-chunks in flight

template <int G, int DH>
struct AttnSmem {
    uint16_t ring[kRing][kSub][DH];  // K or V rows of one sub-chunk per stage
    float q[G][DH];
    float p[G][BI_KV_CHUNK];         // scores, then exp(score - m)
    float m[G];
    float l[G];
    int32_t pages[kMaxChunkPages];
};

template <int G, int DH>
struct AttnShape {
    static constexpr int kSlots = G * DH / 2;  // (head, dim pair) outputs
    static constexpr int kSlotsPerThread = (kSlots + kAttnThreads - 1) / kAttnThreads;
    static constexpr int kPieces = DH / 64;    // 16-byte pieces per lane per key (8 lanes per key)
};

struct Entry {
    int32_t t, r, p;
};

__device__ __forceinline__ Entry get_entry(const EntryMap& em, int32_t e) {
    Entry x;
    if (em.kind == 0) {
        x.t = e;
        x.r = e;
        x.p = em.a[e] - 1;
    } else if (em.kind == 1) {
        x.t = em.a[e];
        x.r = em.b[x.t];
        x.p = em.c[x.t];
    } else {
        int lo = 0, hi = em.nreq - 1;  // last request whose first token is <= e
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (em.a[mid] <= e) lo = mid; else hi = mid - 1;
        }
        x.t = e;
        x.r = lo;
        x.p = em.b[lo] + (e - em.a[lo]);
    }
    return x;
}

// Piece size of the batch-variant occupancy rule (kv_chunk_size_1 = 256).
__host__ __device__ __forceinline__ int32_t variant_piece(int32_t s, int32_t chunk2) {
    const int32_t n1 = (s + BI_KV_CHUNK - 1) / BI_KV_CHUNK;
    const int32_t n2 = (s + chunk2 - 1) / chunk2;
    const int32_t n = n1 > n2 ? n1 : n2;
    return (s + n - 1) / n;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Loads the G query heads of token t (bf16) into shared memory as fp32.
template <int G, int DH>
__device__ __forceinline__ void load_q(AttnSmem<G, DH>& sm, const uint16_t* q, int32_t t, int32_t H,
                                       int32_t g) {
    const uint16_t* src = q + (static_cast<int64_t>(t) * H + static_cast<int64_t>(g) * G) * DH;
    for (int i = threadIdx.x; i < G * DH; i += kAttnThreads) sm.q[i / DH][i % DH] = bf16_to_f32(src[i]);
}

// Partial of keys [k0, k0 + n) (1 <= n <= BI_KV_CHUNK) for the G heads whose
// fp32 queries sit in sm.q.  On return sm.m / sm.l hold each head's max score
// and sum of exp(score - max); o[i][0..1] holds the thread's output slot i
// (head = slot / (DH/2), dims 2*(slot % (DH/2)) + {0, 1}).
//   score_j = (q . k_j) * scale: lane s (of the 8 lanes of key j) adds
//             q[d] k_j[d] with fused multiply-adds over d = 64u + 8s .. 64u +
//             8s + 7 for u = 0, 1, ... in that order, then the 8 lane sums meet
//             in an xor-butterfly (4, 2, 1);
//   m = max_j score_j;  l = sum_j exp(score_j - m), o = sum_j exp(score_j - m)
//             v_j, both serial in j.
// K and V rows stream through a ring of kRing shared-memory stages of kSub
// keys each (cp.async), K sub-chunks first, then V sub-chunks.
template <int G, int DH>
__device__ __forceinline__ void chunk_partial(AttnSmem<G, DH>& sm, const uint16_t* __restrict__ kc,
                                              const uint16_t* __restrict__ vc, const int32_t* page_row,
                                              int32_t g, int32_t Hkv, int32_t k0, int32_t n, float scale,
                                              int32_t max_pages, int32_t num_pages, int32_t* status,
                                              float (&o)[AttnShape<G, DH>::kSlotsPerThread][2]) {
    using S = AttnShape<G, DH>;
    constexpr int kVecPerRow = DH / 8;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    const int32_t lp0 = k0 / BI_PAGE;
    const int32_t np = (k0 + n - 1) / BI_PAGE - lp0 + 1;
    if (tid < np) {
        const int32_t lp = lp0 + tid;
        int32_t pg = lp < max_pages ? page_row[lp] : -1;
        if (pg < 0 || pg >= num_pages) {
            report(status, BI_DEV_BAD_PAGE);
            pg = 0;
        }
        sm.pages[tid] = pg;
    }
    __syncthreads();

    const int ns = (n + kSub - 1) / kSub;  // sub-chunks of K, then as many of V
    auto issue = [&](int t) {
        if (t < 2 * ns) {
            const bool is_v = t >= ns;
            const int sc = is_v ? t - ns : t;
            const int32_t j0 = sc * kSub;
            const int32_t nk = min(kSub, n - j0);
            const uint16_t* base = is_v ? vc : kc;
            uint16_t(*dst)[DH] = sm.ring[t % kRing];
            for (int gi = tid; gi < nk * kVecPerRow; gi += kAttnThreads) {
                const int32_t jl = gi / kVecPerRow, part = gi % kVecPerRow;
                const int32_t kp = k0 + j0 + jl;
                const int32_t pg = sm.pages[kp / BI_PAGE - lp0];
                cp_async16(&dst[jl][part * 8],
                           base + ((static_cast<int64_t>(pg) * Hkv + g) * BI_PAGE + (kp & (BI_PAGE - 1))) * DH + part * 8);
            }
        }
        cp_async_commit();  // possibly empty: keeps one group per sub-chunk slot
    };
#pragma unroll
    for (int t = 0; t < kRing; ++t) issue(t);

    const int kk = lane >> 3, sub = lane & 7;
    float qr[G][S::kPieces * 8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int u = 0; u < S::kPieces; ++u)
#pragma unroll
            for (int d = 0; d < 8; ++d) qr[h][u * 8 + d] = sm.q[h][u * 64 + sub * 8 + d];

    float oacc[S::kSlotsPerThread][2];
    float lacc[S::kSlotsPerThread];
#pragma unroll
    for (int si = 0; si < S::kSlotsPerThread; ++si) {
        oacc[si][0] = oacc[si][1] = 0.0f;
        lacc[si] = 0.0f;
    }

    for (int t = 0; t < 2 * ns; ++t) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory");
        __syncthreads();
        const uint16_t(*buf)[DH] = sm.ring[t % kRing];
        if (t < ns) {
            // scores of this sub-chunk's keys: warp w takes keys it*16 + w*4 + lane/8
            const int32_t j0 = t * kSub;
            const int32_t nk = min(kSub, n - j0);
            for (int it = 0; it < (nk + 15) / 16; ++it) {
                const int32_t jl = it * 16 + warp * 4 + kk;
                const bool valid = jl < nk;
                float acc[G];
#pragma unroll
                for (int h = 0; h < G; ++h) acc[h] = 0.0f;
                if (valid) {
#pragma unroll
                    for (int u = 0; u < S::kPieces; ++u) {
                        const uint4 kv = *reinterpret_cast<const uint4*>(&buf[jl][u * 64 + sub * 8]);
                        const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float k_lo = bf16_lo(w[e]), k_hi = bf16_hi(w[e]);
#pragma unroll
                            for (int h = 0; h < G; ++h) {
                                acc[h] = __fmaf_rn(qr[h][u * 8 + 2 * e], k_lo, acc[h]);
                                acc[h] = __fmaf_rn(qr[h][u * 8 + 2 * e + 1], k_hi, acc[h]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    acc[h] = __fadd_rn(acc[h], __shfl_xor_sync(0xffffffffu, acc[h], 4));
                    acc[h] = __fadd_rn(acc[h], __shfl_xor_sync(0xffffffffu, acc[h], 2));
                    acc[h] = __fadd_rn(acc[h], __shfl_xor_sync(0xffffffffu, acc[h], 1));
                }
                if (valid && sub == 0) {
#pragma unroll
                    for (int h = 0; h < G; ++h) sm.p[h][j0 + jl] = __fmul_rn(acc[h], scale);
                }
            }
            if (t == ns - 1) {
                __syncthreads();
                // per head: m = max score (exact, order-free), p = exp(score - m)
                for (int h = warp; h < G; h += kAttnThreads / 32) {
                    float mx = -INFINITY;
                    for (int jl = lane; jl < n; jl += 32) mx = fmaxf(mx, sm.p[h][jl]);
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    for (int jl = lane; jl < n; jl += 32) sm.p[h][jl] = expf(__fsub_rn(sm.p[h][jl], mx));
                    if (lane == 0) sm.m[h] = mx;
                }
            }
        } else {
            // o and l over this sub-chunk's keys, continuing the serial key order
            const int32_t j0 = (t - ns) * kSub;
            const int32_t nk = min(kSub, n - j0);
#pragma unroll
            for (int si = 0; si < S::kSlotsPerThread; ++si) {
                const int slot = tid + si * kAttnThreads;
                if (slot < S::kSlots) {
                    const int h = slot / (DH / 2), dp = slot % (DH / 2);
                    const float* ph = sm.p[h] + j0;
                    float o0 = oacc[si][0], o1 = oacc[si][1], l = lacc[si];
                    for (int jl = 0; jl < nk; ++jl) {
                        const float pv = ph[jl];
                        const uint32_t vv = *reinterpret_cast<const uint32_t*>(&buf[jl][2 * dp]);
                        o0 = __fmaf_rn(pv, bf16_lo(vv), o0);
                        o1 = __fmaf_rn(pv, bf16_hi(vv), o1);
                        l = __fadd_rn(l, pv);
                    }
                    oacc[si][0] = o0;
                    oacc[si][1] = o1;
                    lacc[si] = l;
                }
            }
        }
        __syncthreads();
        issue(t + kRing);
    }
    cp_async_wait_all();
#pragma unroll
    for (int si = 0; si < S::kSlotsPerThread; ++si) {
        const int slot = tid + si * kAttnThreads;
        if (slot < S::kSlots && slot % (DH / 2) == 0) sm.l[slot / (DH / 2)] = lacc[si];
        o[si][0] = oacc[si][0];
        o[si][1] = oacc[si][1];
    }
    __syncthreads();
}

// Ascending-order merge step of two partials (M, L, O) and (m, l, o).
__device__ __forceinline__ void fold_step(float& M, float& L, float& O0, float& O1, float m, float l,
                                          float o0, float o1) {
    const float Mn = fmaxf(M, m);
    const float a = expf(__fsub_rn(M, Mn));
    const float b = expf(__fsub_rn(m, Mn));
    L = __fadd_rn(__fmul_rn(L, a), __fmul_rn(l, b));
    O0 = __fadd_rn(__fmul_rn(O0, a), __fmul_rn(o0, b));
    O1 = __fadd_rn(__fmul_rn(O1, a), __fmul_rn(o1, b));
    M = Mn;
}

__device__ __forceinline__ void store_out2(void* out, int32_t out_f32, int64_t idx, float a, float b) {
    if (out_f32) {
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(out) + idx) = make_float2(a, b);
    } else {
        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(out) + idx) = pack_bf16x2(a, b);
    }
}

// Number of pieces and piece size for a context of s positions.
__device__ __forceinline__ void pieces(int32_t s, int32_t chunk2, int32_t& size, int32_t& count) {
    size = chunk2 > 0 ? variant_piece(s, chunk2) : BI_KV_CHUNK;
    count = (s + size - 1) / size;
}

// ---------------------------------------------------------------------------
// Decode: grid (entries, Hkv, max_splits).
// ---------------------------------------------------------------------------
template <int G, int DH>
__global__ void __launch_bounds__(kAttnThreads)
decode_split_kernel(AttnGeom geo, EntryMap em, int32_t max_splits, int32_t chunk2, float* __restrict__ ws_o,
                    float* __restrict__ ws_ml) {
    using S = AttnShape<G, DH>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AttnSmem<G, DH>& sm = *reinterpret_cast<AttnSmem<G, DH>*>(smem_raw);
    const int32_t e = blockIdx.x, g = blockIdx.y, split = blockIdx.z;
    const Entry en = get_entry(em, e);
    const int32_t s = en.p + 1;
    int32_t size, count;
    pieces(s > 0 ? s : 1, chunk2, size, count);
    const bool ok = en.p >= 0 && (s + BI_PAGE - 1) / BI_PAGE <= geo.max_pages && count <= max_splits;
    if (!ok) {
        if (split == 0 && g == 0 && threadIdx.x == 0) report(geo.status, BI_DEV_BAD_POSITION);
        return;
    }
    if (split >= count) return;
    const int32_t k0 = split * size;
    const int32_t n = min(size, s - k0);
    load_q<G, DH>(sm, reinterpret_cast<const uint16_t*>(geo.q), en.t, geo.H, g);
    __syncthreads();
    float o[S::kSlotsPerThread][2];
    chunk_partial<G, DH>(sm, reinterpret_cast<const uint16_t*>(geo.kc), reinterpret_cast<const uint16_t*>(geo.vc),
                         geo.page_table + static_cast<int64_t>(en.r) * geo.max_pages, g, geo.Hkv, k0, n,
                         geo.scale, geo.max_pages, geo.num_pages, geo.status, o);
#pragma unroll
    for (int si = 0; si < S::kSlotsPerThread; ++si) {
        const int slot = threadIdx.x + si * kAttnThreads;
        if (slot < S::kSlots) {
            const int h = slot / (DH / 2), dp = slot % (DH / 2);
            const int64_t row = (static_cast<int64_t>(e) * geo.H + g * G + h) * max_splits + split;
            *reinterpret_cast<float2*>(ws_o + row * DH + 2 * dp) = make_float2(o[si][0], o[si][1]);
            if (dp == 0) *reinterpret_cast<float2*>(ws_ml + row * 2) = make_float2(sm.m[h], sm.l[h]);
        }
    }
}

// Merge: grid (entries, H), DH/2 threads, each one dim pair; serial over splits.
template <int DH>
__global__ void __launch_bounds__(DH / 2)
decode_merge_kernel(AttnGeom geo, EntryMap em, int32_t max_splits, int32_t chunk2, const float* __restrict__ ws_o,
                    const float* __restrict__ ws_ml) {
    const int32_t e = blockIdx.x, h = blockIdx.y, dp = threadIdx.x;
    const Entry en = get_entry(em, e);
    const int32_t s = en.p + 1;
    int32_t size, count;
    pieces(s > 0 ? s : 1, chunk2, size, count);
    const int64_t oidx = (static_cast<int64_t>(en.t) * geo.H + h) * DH + 2 * dp;
    const bool ok = en.p >= 0 && (s + BI_PAGE - 1) / BI_PAGE <= geo.max_pages && count <= max_splits;
    if (!ok) {
        store_out2(geo.out, geo.out_f32, oidx, 0.0f, 0.0f);
        return;
    }
    const int64_t row0 = (static_cast<int64_t>(e) * geo.H + h) * max_splits;
    float M = ws_ml[row0 * 2], L = ws_ml[row0 * 2 + 1];
    float O0 = ws_o[row0 * DH + 2 * dp], O1 = ws_o[row0 * DH + 2 * dp + 1];
    for (int32_t j = 1; j < count; ++j) {
        const int64_t r = row0 + j;
        fold_step(M, L, O0, O1, ws_ml[r * 2], ws_ml[r * 2 + 1], ws_o[r * DH + 2 * dp], ws_o[r * DH + 2 * dp + 1]);
    }
    store_out2(geo.out, geo.out_f32, oidx, __fdiv_rn(O0, L), __fdiv_rn(O1, L));
}

// ---------------------------------------------------------------------------
// Prefill: grid (entries, Hkv); each CTA walks its query's chunks in order.
// ---------------------------------------------------------------------------
template <int G, int DH>
__global__ void __launch_bounds__(kAttnThreads)
prefill_kernel(AttnGeom geo, EntryMap em) {
    using S = AttnShape<G, DH>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AttnSmem<G, DH>& sm = *reinterpret_cast<AttnSmem<G, DH>*>(smem_raw);
    const int32_t e = blockIdx.x, g = blockIdx.y;
    const Entry en = get_entry(em, e);
    const int32_t s = en.p + 1;
    const bool ok = en.p >= 0 && (s + BI_PAGE - 1) / BI_PAGE <= geo.max_pages;
    if (!ok) {
        if (threadIdx.x == 0) report(geo.status, BI_DEV_BAD_POSITION);
#pragma unroll
        for (int si = 0; si < S::kSlotsPerThread; ++si) {
            const int slot = threadIdx.x + si * kAttnThreads;
            if (slot < S::kSlots) {
                const int h = slot / (DH / 2), dp = slot % (DH / 2);
                store_out2(geo.out, geo.out_f32, (static_cast<int64_t>(en.t) * geo.H + g * G + h) * DH + 2 * dp, 0.f, 0.f);
            }
        }
        return;
    }
    load_q<G, DH>(sm, reinterpret_cast<const uint16_t*>(geo.q), en.t, geo.H, g);
    __syncthreads();
    float M[S::kSlotsPerThread], L[S::kSlotsPerThread], O[S::kSlotsPerThread][2];
    const int32_t count = (s + BI_KV_CHUNK - 1) / BI_KV_CHUNK;
    const int32_t* page_row = geo.page_table + static_cast<int64_t>(en.r) * geo.max_pages;
    for (int32_t j = 0; j < count; ++j) {
        const int32_t k0 = j * BI_KV_CHUNK;
        const int32_t n = min(BI_KV_CHUNK, s - k0);
        float o[S::kSlotsPerThread][2];
        chunk_partial<G, DH>(sm, reinterpret_cast<const uint16_t*>(geo.kc), reinterpret_cast<const uint16_t*>(geo.vc),
                             page_row, g, geo.Hkv, k0, n, geo.scale, geo.max_pages, geo.num_pages, geo.status, o);
#pragma unroll
        for (int si = 0; si < S::kSlotsPerThread; ++si) {
            const int slot = threadIdx.x + si * kAttnThreads;
            const int h = slot < S::kSlots ? slot / (DH / 2) : 0;
            const float m = sm.m[h], l = sm.l[h];
            if (j == 0) {
                M[si] = m;
                L[si] = l;
                O[si][0] = o[si][0];
                O[si][1] = o[si][1];
            } else {
                fold_step(M[si], L[si], O[si][0], O[si][1], m, l, o[si][0], o[si][1]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int si = 0; si < S::kSlotsPerThread; ++si) {
        const int slot = threadIdx.x + si * kAttnThreads;
        if (slot < S::kSlots) {
            const int h = slot / (DH / 2), dp = slot % (DH / 2);
            store_out2(geo.out, geo.out_f32, (static_cast<int64_t>(en.t) * geo.H + g * G + h) * DH + 2 * dp,
                       __fdiv_rn(O[si][0], L[si]), __fdiv_rn(O[si][1], L[si]));
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
bool attention_supported(int32_t H, int32_t Hkv, int32_t Dh) {
    if (H <= 0 || Hkv <= 0 || H % Hkv != 0) return false;
    const int32_t G = H / Hkv;
    return (Dh == 64 || Dh == 128) && (G == 1 || G == 2 || G == 4 || G == 8);
}

int32_t invariant_max_splits(int32_t max_seq) {
    return max_seq <= 0 ? 1 : (max_seq + BI_KV_CHUNK - 1) / BI_KV_CHUNK;
}

void variant_split_plan(int32_t B, int32_t H, int32_t Hkv, int32_t max_seq, int32_t* chunk2,
                        int32_t* max_splits) {
    if (max_seq < 1) max_seq = 1;
    const float ext_seq_len = static_cast<float>(max_seq) / 64.0f;
    const float lg = log2f(ext_seq_len);
    const int32_t cores2 = static_cast<int32_t>(static_cast<float>(num_sms()) * (lg > 1.0f ? lg : 1.0f));
    const int32_t group = H / Hkv;
    const int32_t block_h = group < 16 ? group : 16;
    const int32_t token_grid = (B > 0 ? B : 1) * ((H + block_h - 1) / block_h);
    int32_t splits2 = (cores2 + token_grid - 1) / token_grid;
    if (splits2 > 16) splits2 = 16;
    if (splits2 < 1) splits2 = 1;
    const int32_t c2 = (max_seq + splits2 - 1) / splits2;
    *chunk2 = c2;
    const int32_t n1 = (max_seq + BI_KV_CHUNK - 1) / BI_KV_CHUNK;
    const int32_t n2 = (max_seq + c2 - 1) / c2;
    *max_splits = n1 > n2 ? n1 : n2;
}

size_t decode_ws_bytes(int32_t n_entries, int32_t H, int32_t Dh, int32_t max_splits) {
    const size_t rows = static_cast<size_t>(n_entries) * H * max_splits;
    return rows * (Dh + 2) * sizeof(float) + 256;
}

template <int G, int DH>
static cudaError_t launch_decode_t(const AttnGeom& g, const EntryMap& em, int32_t n, int32_t max_splits,
                                   int32_t chunk2, float* ws_o, float* ws_ml, cudaStream_t s) {
    const size_t smem = sizeof(AttnSmem<G, DH>);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<G, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(n, g.Hkv, max_splits);
    decode_split_kernel<G, DH><<<grid, kAttnThreads, smem, s>>>(g, em, max_splits, chunk2, ws_o, ws_ml);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_merge_kernel<DH><<<dim3(n, g.H), DH / 2, 0, s>>>(g, em, max_splits, chunk2, ws_o, ws_ml);
    return cudaGetLastError();
}

template <int G, int DH>
static cudaError_t launch_prefill_t(const AttnGeom& g, const EntryMap& em, int32_t n, cudaStream_t s) {
    const size_t smem = sizeof(AttnSmem<G, DH>);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<G, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    prefill_kernel<G, DH><<<dim3(n, g.Hkv), kAttnThreads, smem, s>>>(g, em);
    return cudaGetLastError();
}

#define BI_ATTN_DISPATCH(FN, ...)                                              \
    do {                                                                       \
        const int32_t G_ = g.H / g.Hkv;                                        \
        if (g.Dh == 128) {                                                     \
            if (G_ == 1) return FN<1, 128>(__VA_ARGS__);                       \
            if (G_ == 2) return FN<2, 128>(__VA_ARGS__);                       \
            if (G_ == 4) return FN<4, 128>(__VA_ARGS__);                       \
            if (G_ == 8) return FN<8, 128>(__VA_ARGS__);                       \
        } else if (g.Dh == 64) {                                               \
            if (G_ == 1) return FN<1, 64>(__VA_ARGS__);                        \
            if (G_ == 2) return FN<2, 64>(__VA_ARGS__);                        \
            if (G_ == 4) return FN<4, 64>(__VA_ARGS__);                        \
            if (G_ == 8) return FN<8, 64>(__VA_ARGS__);                        \
        }                                                                      \
        return cudaErrorInvalidValue;                                          \
    } while (0)

cudaError_t launch_decode_attention(const AttnGeom& g, const EntryMap& em, int32_t n_entries,
                                    int32_t max_splits, int32_t variant_chunk2, float* ws_o, float* ws_ml,
                                    cudaStream_t s) {
    if (n_entries <= 0) return cudaSuccess;
    BI_ATTN_DISPATCH(launch_decode_t, g, em, n_entries, max_splits, variant_chunk2, ws_o, ws_ml, s);
}

cudaError_t launch_prefill_attention(const AttnGeom& g, const EntryMap& em, int32_t n_entries, cudaStream_t s) {
    if (n_entries <= 0) return cudaSuccess;
    BI_ATTN_DISPATCH(launch_prefill_t, g, em, n_entries, s);
}

}  // namespace bi
