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

#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace bi {

constexpr int kAttnThreads = 128;
constexpr int kWarps = kAttnThreads / 32;
constexpr int kMaxChunkPages = BI_KV_CHUNK / BI_PAGE + 1;  // a variant piece may straddle one more page
constexpr int kSub = 64;                                   // keys per staged sub-chunk
constexpr int kRing = 2;  // staged sub-chunks in flight (a shallow ring fits 6 CTAs per SM)

template <int G, int DH>
struct AttnShape {
    static_assert(G >= 1 && G <= 8, "a GQA group fills at most the 8 rows a0/a2 of an m16n8k16 tile");
    static constexpr int kKSteps = DH / 16;           // 16-deep MMA steps over the head dim
    static constexpr int kDimsPerWarp = DH / kWarps;  // PV: output dims per warp
    static constexpr int kNB = kDimsPerWarp / 8;      // PV: 8-wide n-blocks per warp
};

template <int G, int DH>
struct AttnSmem {
    uint16_t ring[kRing][kSub][DH];  // K or V rows; 16-byte chunk c of row r sits at chunk c ^ (r & 7)
    float p[G][BI_KV_CHUNK];         // scores, then exp(score - m)
    float red[kWarps][G];            // per-warp partial sums of l
    float m[G];
    float l[G];
    int32_t pages[kMaxChunkPages];
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

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// d += A(16x16, rows 8..15 zero) * B(16x8), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_rows8(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    const uint32_t z = 0;
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(z), "r"(a2), "r"(z), "r"(b0), "r"(b1));
}
// Byte offset of (row, 16-byte chunk c) in a swizzled ring stage.
template <int DH>
__device__ __forceinline__ uint32_t ring_off(int row, int c) {
    return static_cast<uint32_t>(row * DH * 2 + ((c ^ (row & 7)) << 4));
}

// Query fragments of the GQA group: row h of the MMA's A operand is head h of
// the group (rows >= G and 8..15 are zero); qa[ks] = {a0, a2} of 16-deep step ks.
template <int G, int DH>
__device__ __forceinline__ void load_q_frags(const uint16_t* q, int32_t t, int32_t H, int32_t g,
                                             uint32_t (&qa)[DH / 16][2]) {
    const int lane = threadIdx.x & 31, h = lane >> 2, c = 2 * (lane & 3);
    const uint16_t* src = q + (static_cast<int64_t>(t) * H + static_cast<int64_t>(g) * G + h) * DH;
#pragma unroll
    for (int ks = 0; ks < DH / 16; ++ks) {
        qa[ks][0] = h < G ? *reinterpret_cast<const uint32_t*>(src + ks * 16 + c) : 0u;
        qa[ks][1] = h < G ? *reinterpret_cast<const uint32_t*>(src + ks * 16 + 8 + c) : 0u;
    }
}

// Partial of keys [k0, k0 + n) (1 <= n <= BI_KV_CHUNK) for the G heads of
// one GQA group.  On return sm.m / sm.l hold each head's max score and sum of
// exp(score - max), and a thread with h = lane/4 < G holds in o[nb][0..1] the
// unnormalised output of head h at dims 32w + 8nb + 2(lane%4) + {0,1} (w =
// warp; DH/4 dims per warp).  The arithmetic, fixed for a given (n, G, DH):
//   score_j = (q . k_j) * scale: q and k_j in bf16 multiplied on the tensor
//             cores (m16n8k16, fp32 accumulate) over the head dim in 16-deep
//             steps in ascending order, then one fp32 multiply by scale;
//   m = max_j score_j;   p_j = exp(score_j - m);
//   l = sum over the 4 warps in order of (xor-butterfly over the 32 lanes of
//       (lane-serial sum of p_j over j = 32w + lane + 128i, i ascending));
//   o = sum_j p_j v_j on the tensor cores: p_j split into bf16 hi = bf16(p_j)
//       and lo = bf16(p_j - hi), for each 16-key step in ascending order the
//       hi product then the lo product accumulated in fp32.
// K and V rows stream through a ring of kRing shared-memory stages of kSub
// keys each (cp.async), K sub-chunks first, then V sub-chunks.
template <int G, int DH>
__device__ __forceinline__ void chunk_partial(AttnSmem<G, DH>& sm, const uint16_t* __restrict__ kc,
                                              const uint16_t* __restrict__ vc, const int32_t* page_row,
                                              int32_t g, int32_t Hkv, int32_t k0, int32_t n, float scale,
                                              int32_t max_pages, int32_t num_pages, int32_t* status,
                                              const uint32_t (&qa)[DH / 16][2],
                                              float (&o)[AttnShape<G, DH>::kNB][2]) {
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
    const int part = tid % kVecPerRow;     // this thread's 16-byte column of every row it copies
    auto issue = [&](int t) {
        if (t < 2 * ns) {
            const bool is_v = t >= ns;
            const int32_t j0 = (is_v ? t - ns : t) * kSub;
            const int32_t nk = min(kSub, n - j0);
            const uint16_t* base = (is_v ? vc : kc) + static_cast<int64_t>(g) * BI_PAGE * DH + part * 8;
            unsigned char* dst = reinterpret_cast<unsigned char*>(sm.ring[t % kRing]);
            for (int jl = tid / kVecPerRow; jl < nk; jl += kAttnThreads / kVecPerRow) {
                const int32_t kp = k0 + j0 + jl;
                const int64_t pg = sm.pages[kp / BI_PAGE - lp0];
                cp_async16(dst + ring_off<DH>(jl, part), base + (pg * Hkv * BI_PAGE + (kp & (BI_PAGE - 1))) * DH);
            }
            if (is_v) {
                // V rows past the last key up to the 16-key step boundary are read by
                // the MMA with p = 0: make them zero rather than stale
                const int32_t pad_end = min(kSub, (nk + 15) & ~15);
                for (int jl = nk + tid / kVecPerRow; jl < pad_end; jl += kAttnThreads / kVecPerRow)
                    *reinterpret_cast<uint4*>(dst + ring_off<DH>(jl, part)) = make_uint4(0, 0, 0, 0);
            }
        }
        cp_async_commit();  // possibly empty: keeps one group per sub-chunk slot
    };
#pragma unroll
    for (int t = 0; t < kRing; ++t) issue(t);

    const int hrow = lane >> 2, cq = 2 * (lane & 3);
    float oacc[S::kNB][4];
#pragma unroll
    for (int nb = 0; nb < S::kNB; ++nb) oacc[nb][0] = oacc[nb][1] = oacc[nb][2] = oacc[nb][3] = 0.0f;

    for (int t = 0; t < 2 * ns; ++t) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory");
        __syncthreads();
        const uint32_t buf = smem_u32(sm.ring[t % kRing]);
        if (t < ns) {
            // scores: warp w takes keys 16w .. 16w+15 of the sub-chunk, 8 per MMA n-block
            const int32_t j0 = t * kSub;
            const int32_t nk = min(kSub, n - j0);
#pragma unroll
            for (int nb2 = 0; nb2 < 2; ++nb2) {
                const int n0 = warp * 16 + nb2 * 8;
                if (n0 >= nk) break;
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int ks = 0; ks < S::kKSteps; ks += 2) {
                    uint32_t r[4];
                    ldsm_x4(buf + ring_off<DH>(n0 + (lane & 7), 2 * ks + (lane >> 3)), r);
                    mma_rows8(acc, qa[ks][0], qa[ks][1], r[0], r[1]);
                    mma_rows8(acc, qa[ks + 1][0], qa[ks + 1][1], r[2], r[3]);
                }
                if (hrow < G) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int key = n0 + cq + c;
                        if (key < nk) sm.p[hrow][j0 + key] = __fmul_rn(acc[c], scale);
                    }
                }
            }
            if (t == ns - 1) {
                __syncthreads();
                // m: exact max per head (order-free)
                for (int h = warp; h < G; h += kWarps) {
                    float mx = -INFINITY;
                    for (int j = lane; j < n; j += 32) mx = fmaxf(mx, sm.p[h][j]);
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    if (lane == 0) sm.m[h] = mx;
                }
                __syncthreads();
                // p = exp(score - m) and the fixed-tree sum l
                float ls[G];
#pragma unroll
                for (int h = 0; h < G; ++h) ls[h] = 0.0f;
                for (int j = tid; j < n; j += kAttnThreads) {
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float pv = expf(__fsub_rn(sm.p[h][j], sm.m[h]));
                        sm.p[h][j] = pv;
                        ls[h] = __fadd_rn(ls[h], pv);
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        ls[h] = __fadd_rn(ls[h], __shfl_xor_sync(0xffffffffu, ls[h], off));
                    if (lane == 0) sm.red[warp][h] = ls[h];
                }
                __syncthreads();
                if (tid < G) {
                    float l = sm.red[0][tid];
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) l = __fadd_rn(l, sm.red[w][tid]);
                    sm.l[tid] = l;
                }
            }
        } else {
            // PV: warp w owns dims DH/4 * w .. ; 16-key steps in ascending order
            const int32_t j0 = (t - ns) * kSub;
            const int32_t nk = min(kSub, n - j0);
            const int c0 = warp * S::kDimsPerWarp / 8;  // first 16-byte chunk of this warp's dims
            for (int kk = 0; kk < nk; kk += 16) {
                float pv[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int key = kk + cq + (x & 1) + (x >> 1) * 8;
                    pv[x] = (hrow < G && key < nk) ? sm.p[hrow][j0 + key] : 0.0f;
                }
                uint32_t hi[2], lo[2];
#pragma unroll
                for (int y = 0; y < 2; ++y) {
                    const float h0 = __uint_as_float(static_cast<uint32_t>(f32_to_bf16(pv[2 * y])) << 16);
                    const float h1 = __uint_as_float(static_cast<uint32_t>(f32_to_bf16(pv[2 * y + 1])) << 16);
                    hi[y] = pack_bf16x2(h0, h1);
                    lo[y] = pack_bf16x2(__fsub_rn(pv[2 * y], h0), __fsub_rn(pv[2 * y + 1], h1));
                }
#pragma unroll
                for (int nb = 0; nb < S::kNB; nb += 2) {
                    uint32_t r[4];
                    const int i = lane >> 3;
                    ldsm_x4_trans(buf + ring_off<DH>(kk + (i & 1) * 8 + (lane & 7), c0 + nb + (i >> 1)), r);
                    mma_rows8(oacc[nb], hi[0], hi[1], r[0], r[1]);
                    mma_rows8(oacc[nb], lo[0], lo[1], r[0], r[1]);
                    mma_rows8(oacc[nb + 1], hi[0], hi[1], r[2], r[3]);
                    mma_rows8(oacc[nb + 1], lo[0], lo[1], r[2], r[3]);
                }
            }
        }
        __syncthreads();
        issue(t + kRing);
    }
    cp_async_wait_all();
#pragma unroll
    for (int nb = 0; nb < S::kNB; ++nb) {
        o[nb][0] = oacc[nb][0];
        o[nb][1] = oacc[nb][1];
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
    pdl_trigger();
    pdl_wait();
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
    uint32_t qa[DH / 16][2];
    load_q_frags<G, DH>(reinterpret_cast<const uint16_t*>(geo.q), en.t, geo.H, g, qa);
    float o[S::kNB][2];
    chunk_partial<G, DH>(sm, reinterpret_cast<const uint16_t*>(geo.kc), reinterpret_cast<const uint16_t*>(geo.vc),
                         geo.page_table + static_cast<int64_t>(en.r) * geo.max_pages, g, geo.Hkv, k0, n,
                         geo.scale, geo.max_pages, geo.num_pages, geo.status, qa, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x / 32, h = lane >> 2;
    if (h < G) {
        const int64_t row = (static_cast<int64_t>(e) * geo.H + g * G + h) * max_splits + split;
#pragma unroll
        for (int nb = 0; nb < S::kNB; ++nb) {
            const int d = warp * S::kDimsPerWarp + nb * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2*>(ws_o + row * DH + d) = make_float2(o[nb][0], o[nb][1]);
        }
        if (warp == 0 && (lane & 3) == 0) *reinterpret_cast<float2*>(ws_ml + row * 2) = make_float2(sm.m[h], sm.l[h]);
    }
}

// Merge: grid (entries, H), DH/2 threads, each one dim pair; the fold runs
// over splits in ascending order, its inputs fetched kMergeBatch splits at a
// time so the loads of a batch are in flight together.
constexpr int kMergeBatch = 8;

template <int DH>
__global__ void __launch_bounds__(DH / 2)
decode_merge_kernel(AttnGeom geo, EntryMap em, int32_t max_splits, int32_t chunk2, const float* __restrict__ ws_o,
                    const float* __restrict__ ws_ml) {
    pdl_trigger();
    pdl_wait();
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
    float M = 0.0f, L = 0.0f, O0 = 0.0f, O1 = 0.0f;
    for (int32_t j0 = 0; j0 < count; j0 += kMergeBatch) {
        float2 ml[kMergeBatch], o[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            const int64_t r = row0 + j0 + u;
            if (j0 + u < count) {
                ml[u] = *reinterpret_cast<const float2*>(ws_ml + r * 2);
                o[u] = *reinterpret_cast<const float2*>(ws_o + r * DH + 2 * dp);
            }
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            if (j0 + u >= count) break;
            if (j0 + u == 0) {
                M = ml[u].x;
                L = ml[u].y;
                O0 = o[u].x;
                O1 = o[u].y;
            } else {
                fold_step(M, L, O0, O1, ml[u].x, ml[u].y, o[u].x, o[u].y);
            }
        }
    }
    store_out2(geo.out, geo.out_f32, oidx, __fdiv_rn(O0, L), __fdiv_rn(O1, L));
}

// ---------------------------------------------------------------------------
// Prefill: grid (entries, Hkv); each CTA walks its query's chunks in order.
// ---------------------------------------------------------------------------
template <int G, int DH>
__global__ void __launch_bounds__(kAttnThreads)
prefill_kernel(AttnGeom geo, EntryMap em) {
    pdl_trigger();
    pdl_wait();
    using S = AttnShape<G, DH>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AttnSmem<G, DH>& sm = *reinterpret_cast<AttnSmem<G, DH>*>(smem_raw);
    const int32_t e = blockIdx.x, g = blockIdx.y;
    const Entry en = get_entry(em, e);
    const int32_t s = en.p + 1;
    const bool ok = en.p >= 0 && (s + BI_PAGE - 1) / BI_PAGE <= geo.max_pages;
    const int lane = threadIdx.x & 31, warp = threadIdx.x / 32, h = lane >> 2;
    if (!ok) {
        if (threadIdx.x == 0) report(geo.status, BI_DEV_BAD_POSITION);
        if (h < G)
            for (int nb = 0; nb < S::kNB; ++nb)
                store_out2(geo.out, geo.out_f32,
                           (static_cast<int64_t>(en.t) * geo.H + g * G + h) * DH + warp * S::kDimsPerWarp + nb * 8 +
                               2 * (lane & 3),
                           0.f, 0.f);
        return;
    }
    uint32_t qa[DH / 16][2];
    load_q_frags<G, DH>(reinterpret_cast<const uint16_t*>(geo.q), en.t, geo.H, g, qa);
    const int hh = h < G ? h : 0;
    float M = 0.0f, L = 0.0f, O[S::kNB][2];
    const int32_t count = (s + BI_KV_CHUNK - 1) / BI_KV_CHUNK;
    const int32_t* page_row = geo.page_table + static_cast<int64_t>(en.r) * geo.max_pages;
    for (int32_t j = 0; j < count; ++j) {
        const int32_t k0 = j * BI_KV_CHUNK;
        const int32_t n = min(BI_KV_CHUNK, s - k0);
        float o[S::kNB][2];
        chunk_partial<G, DH>(sm, reinterpret_cast<const uint16_t*>(geo.kc), reinterpret_cast<const uint16_t*>(geo.vc),
                             page_row, g, geo.Hkv, k0, n, geo.scale, geo.max_pages, geo.num_pages, geo.status, qa, o);
        const float m = sm.m[hh], l = sm.l[hh];
        if (j == 0) {
            M = m;
            L = l;
#pragma unroll
            for (int nb = 0; nb < S::kNB; ++nb) {
                O[nb][0] = o[nb][0];
                O[nb][1] = o[nb][1];
            }
        } else {
            // the same fold as the decode merge, one dim pair at a time
            const float M0 = M, L0 = L;
#pragma unroll
            for (int nb = 0; nb < S::kNB; ++nb) {
                float Mx = M0, Lx = L0;
                fold_step(Mx, Lx, O[nb][0], O[nb][1], m, l, o[nb][0], o[nb][1]);
                M = Mx;
                L = Lx;
            }
        }
        __syncthreads();
    }
    if (h < G) {
#pragma unroll
        for (int nb = 0; nb < S::kNB; ++nb)
            store_out2(geo.out, geo.out_f32,
                       (static_cast<int64_t>(en.t) * geo.H + g * G + h) * DH + warp * S::kDimsPerWarp + nb * 8 +
                           2 * (lane & 3),
                       __fdiv_rn(O[nb][0], L), __fdiv_rn(O[nb][1], L));
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
    cudaError_t e = launch_pdl(decode_split_kernel<G, DH>, grid, dim3(kAttnThreads), smem, s, g, em, max_splits,
                               chunk2, ws_o, ws_ml);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_merge_kernel<DH>, dim3(n, g.H), dim3(DH / 2), 0, s, g, em, max_splits, chunk2,
                      static_cast<const float*>(ws_o), static_cast<const float*>(ws_ml));
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
    return launch_pdl(prefill_kernel<G, DH>, dim3(n, g.Hkv), dim3(kAttnThreads), smem, s, g, em);
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

// ===========================================================================
// Allocation-free decode attention.
//
// Some callers cannot allocate device memory at the point where they run
// decode attention: code running under an allocator that forbids new
// allocations once serving has started, callers that own no memory pool of
// their own, or hosts that only hand this library plain input and output
// pointers.  bi_decode_attention_noalloc serves them with the same kernels as
// bi_decode_attention, its fp32 split partials living in one statically sized
// device array below instead of a caller workspace.
// ===========================================================================

namespace bi {

// Scratch for the split partials of bi_decode_attention_noalloc.  Every GPU
// that loads this library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up once
// per device (the host-side symbol is only a stand-in, never a device address).
bi_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "bi_decode_attention_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(BI_ERR_UNSUPPORTED, "bi_decode_attention_noalloc: device index");
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "bi_decode_attention_noalloc: cudaGetSymbolAddress");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return BI_OK;
}
}  // namespace

}  // namespace bi

extern "C" bi_status bi_decode_attention_noalloc(const bi_bf16* q, const bi_bf16* k_cache, const bi_bf16* v_cache,
                                                 const int32_t* page_table, const int32_t* seq_lens, void* out,
                                                 bi_dtype out_dtype, int32_t B, int32_t H, int32_t Hkv, int32_t Dh,
                                                 int32_t max_pages, int32_t num_pages, int32_t max_seq_len,
                                                 float scale, bi_mode mode, int32_t* dev_status, bi_stream stream) {
    using namespace bi;
    if (B < 0) return fail(BI_ERR_SHAPE, "bi_decode_attention_noalloc: B < 0");
    if (B == 0) return BI_OK;
    if (!attention_supported(H, Hkv, Dh))
        return fail(BI_ERR_UNSUPPORTED, "bi_decode_attention_noalloc: need Dh in {64,128} and H/Hkv in {1,2,4,8}");
    if (max_pages <= 0 || num_pages <= 0) return fail(BI_ERR_SHAPE, "bi_decode_attention_noalloc: need max_pages, num_pages > 0");
    if (out_dtype != BI_BF16 && out_dtype != BI_F32) return fail(BI_ERR_INVALID, "bi_decode_attention_noalloc: bad dtype");
    if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !out)
        return fail(BI_ERR_INVALID, "bi_decode_attention_noalloc: null pointer");
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return fail(BI_ERR_INVALID, "bi_decode_attention_noalloc: pointers must be 16-byte aligned");
    if (max_seq_len <= 0 || max_seq_len > max_pages * BI_PAGE)
        return fail(BI_ERR_SHAPE, "bi_decode_attention_noalloc: need 0 < max_seq_len <= max_pages * 16");
    if (mode != BI_INVARIANT && mode != BI_VARIANT) return fail(BI_ERR_INVALID, "bi_decode_attention_noalloc: bad mode");
    int32_t max_splits = invariant_max_splits(max_seq_len), chunk2 = 0;
    if (mode == BI_VARIANT) variant_split_plan(B, H, Hkv, max_seq_len, &chunk2, &max_splits);
    const size_t need = decode_ws_bytes(B, H, Dh, max_splits);
    if (need > kNoAllocScratchBytes)
        return fail(BI_ERR_WORKSPACE,
                    "bi_decode_attention_noalloc: this batch needs " + std::to_string(need) +
                        " bytes of split partials, more than the " + std::to_string(kNoAllocScratchBytes) +
                        "-byte static scratch; use bi_decode_attention with a workspace");
    void* scratch = nullptr;
    bi_status st = noalloc_scratch(&scratch);
    if (st != BI_OK) return st;
    // every partial the merge reads is written earlier in this call: nothing in
    // the scratch has to start at zero
    float* ws_o = static_cast<float*>(scratch);
    float* ws_ml = ws_o + static_cast<size_t>(B) * H * max_splits * Dh;
    AttnGeom g{q, k_cache, v_cache, page_table, out, out_dtype == BI_F32, H, Hkv, Dh, max_pages, num_pages, scale,
               dev_status};
    EntryMap em{0, seq_lens, nullptr, nullptr, B};
    cudaError_t e = launch_decode_attention(g, em, B, max_splits, chunk2, ws_o, ws_ml, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_decode_attention_noalloc launch");
}
