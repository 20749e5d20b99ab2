// Paged split-KV attention ("Lockstep", "The fix": the split points come from
// the request, not the batch; "Batch invariance and reproducible inference",
// "1 · Split-K and segmented attention reductions": the split count is
// ceil(seq_len / tile), a function of the request's own length).
//
// Decode: one device function computes the fp32 partial (m, l, o) of one
// chunk of keys for the G heads of one GQA group of one query, in one CTA per
// (query, kv head, chunk); a second kernel merges the partials in ascending
// chunk order.  Prefill (prefill_tc.cuh) runs the same per-chunk arithmetic on
// the tcgen05 tensor cores for 128 (token, head) rows at a time and folds the
// chunks in order as it goes.  Both use the same chunk boundaries (multiples
// of BI_KV_CHUNK from key 0), the same per-row partial and the same fold, so
// a token's output has the same bits whichever path, batch or prefill
// chunking produced it.  Every floating-point step outside the MMAs is an
// explicit round-to-nearest intrinsic so the compiler cannot fuse or reorder
// it differently in the two kernels.
#include <math.h>

#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace bi {

constexpr int kAttnThreads = 128;
constexpr int kWarps = kAttnThreads / 32;
constexpr int kMaxChunkPages = BI_KV_CHUNK / BI_PAGE + 1;  // a variant piece may straddle one more page
constexpr int kSub = 64;  // keys per staged sub-chunk
// Staged sub-chunks in flight: a shallow ring (2) fits six CTAs per SM and
// serves many CTAs; a decode grid that fits the GPU in one wave at three
// CTAs per SM takes a deep one (4: all K sub-chunks of a chunk at once), so a
// CTA's copies overlap instead of queueing behind each other.
constexpr int kRing = 2;
constexpr int kDeepRing = 4;
// Row strides chosen for conflict-free shared-memory access patterns of the
// MMA fragments: scores (fp32), the bf16 hi/lo parts of p, staged outputs.
constexpr int kPStride = BI_KV_CHUNK + 4;
constexpr int kHStride = BI_KV_CHUNK + 8;

// The MMAs are transposed with respect to the usual attention tiling: the 16
// rows of an m16n8k16 tile are keys (scores) or head dims (PV), and its 8
// columns are (query token, head) pairs, token-major: NT tokens of one
// request sharing every K/V load.  A decode CTA has one token (NT = 1), so its
// columns are the G heads of one GQA group.
template <int G, int DH, int NT>
struct AttnShape {
    static_assert(G >= 1 && G <= 8 && NT >= 1, "unsupported group");
    static constexpr int kCols = NT * G;            // live columns
    static constexpr int kNB = (kCols + 7) / 8;     // 8-wide column blocks
    static constexpr int kKSteps = DH / 16;         // 16-deep MMA steps over the head dim
    static constexpr int kDimsPerWarp = DH / kWarps;
    static constexpr int kMT = kDimsPerWarp / 16;   // PV: 16-dim row tiles per warp
    static_assert(kMT >= 1, "head dim too small");
};

// Scores (fp32; after PV, the outputs being stored) and the bf16 hi = bf16(p)
// and lo = bf16(p - hi) parts of p that the PV MMAs read.  With few columns
// (decode) the two share storage, which keeps a CTA small enough for six per
// SM; with many they are separate, which keeps registers down.
template <int C, bool kShared>
struct ScoreStore;
template <int C>
struct ScoreStore<C, true> {
    union {
        float p[C][kPStride];
        uint16_t ph[2][C][kHStride];
    };
};
template <int C>
struct ScoreStore<C, false> {
    float p[C][kPStride];
    uint16_t ph[2][C][kHStride];
};

// A ring stage holds kSub keys of K or V in the layout a 128-byte-swizzled TMA
// box writes: per 64-element half of the head dim, kSub rows of 128 bytes, the
// 16-byte chunk c of row r at chunk c ^ (r & 7).  The ring comes first so a
// 1024-byte aligned dynamic shared memory base keeps every stage aligned.
template <int G, int DH, int NT, int RING = kRing>
struct AttnSmem {
    using S = AttnShape<G, DH, NT>;
    static constexpr bool kSharedScores = S::kCols <= 8;
    static constexpr int kStages = RING;
    uint8_t ring[RING][kSub * DH * 2];
    ScoreStore<S::kCols, kSharedScores> sc;
    uint64_t full[RING];             // TMA completion per ring stage
    int32_t abort;                   // a copy did not land: issue no more
    float red[kWarps][S::kCols];     // per-warp partial sums of l
    float m[S::kCols];
    float l[S::kCols];
    int32_t ncol[S::kCols];          // keys of the current chunk each column attends to
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

// e^x of the attention softmax and its merge, as 2^(x * log2 e) on the
// special-function unit (ex2.approx, subnormal results flushed to zero: at
// most ~2^-22 relative error, plus |x| * 2^-24 from rounding the product).
// Every kernel whose results must agree bit for bit (decode's chunk partials
// and merge, prefill's chunk softmax and fold) calls this one function.
__device__ __forceinline__ float attn_exp(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(__fmul_rn(x, 1.44269504088896341f)));
    return y;
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
// d += A(16x16) * B(16x8), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Byte offset of (row, 16-byte chunk c) in a ring stage (layout above).
template <int DH>
__device__ __forceinline__ uint32_t ring_off(int row, int c) {
    return static_cast<uint32_t>((c >> 3) * (kSub * 128) + row * 128 + (((c & 7) ^ (row & 7)) << 4));
}

// One-time setup of a CTA's ring barriers (thread 0; a barrier must follow).
template <typename Sm>
__device__ __forceinline__ void ring_init(Sm& sm) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < Sm::kStages; ++s) ptx::mbar_init(&sm.full[s], 1);
        sm.abort = 0;
        ptx::fence_barrier_init();
    }
}

// Bounded wait for a ring stage's TMA copies (every thread waits).
__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    if (ptx::mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(a, parity)) return true;
        if ((i & 255u) == 0u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Query fragments as the B operand of the score MMAs: column c = nb*8 + lane/4
// is head c % G of the c / G-th token of the CTA (tok[] gives its row in q;
// -1 or c >= kCols: zero); qb[nb][ks] = {b0, b1} of 16-deep step ks.
template <int G, int DH, int NT>
__device__ __forceinline__ void load_q_cols(const uint16_t* q, const int32_t (&tok)[NT], int32_t H, int32_t g,
                                            uint32_t (&qb)[AttnShape<G, DH, NT>::kNB][DH / 16][2]) {
    using S = AttnShape<G, DH, NT>;
    const int lane = threadIdx.x & 31, c8 = lane >> 2, k2 = 2 * (lane & 3);
#pragma unroll
    for (int nb = 0; nb < S::kNB; ++nb) {
        const int c = nb * 8 + c8;
        const int32_t t = c < S::kCols ? tok[c / G] : -1;
        const uint16_t* src = q + (static_cast<int64_t>(t) * H + static_cast<int64_t>(g) * G + c % G) * DH;
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
            qb[nb][ks][0] = t >= 0 ? *reinterpret_cast<const uint32_t*>(src + ks * 16 + k2) : 0u;
            qb[nb][ks][1] = t >= 0 ? *reinterpret_cast<const uint32_t*>(src + ks * 16 + 8 + k2) : 0u;
        }
    }
}

// Partial of keys [k0, k0 + n_max) (1 <= n_max <= BI_KV_CHUNK) for every
// column; column c attends to the first sm.ncol[c] of them (set by the caller
// before a barrier; 0 = none).  On return sm.m / sm.l hold each column's max
// score and sum of exp(score - max), and oacc[mt][nb] holds, in the m16n8
// accumulator layout, the unnormalised output of columns nb*8 + 2(lane%4)
// + {0,1} at head dims 32w + 16mt + lane/4 + {0, 8} (w = warp; DH/4 dims per
// warp).  The arithmetic of one column, fixed for a given number of keys:
//   score_j = (k_j . q) * scale: bf16 products on the tensor cores (m16n8k16,
//             fp32 accumulate) over the head dim in 16-deep steps in
//             ascending order, then one fp32 multiply by scale;
//   m = max_j score_j;   p_j = exp(score_j - m);
//   l = sum over the 4 warps in order of (xor-butterfly over the 32 lanes of
//       (lane-serial sum of p_j over j = 32w + lane + 128i, i ascending));
//   o = sum_j p_j v_j on the tensor cores: p_j split into bf16 hi = bf16(p_j)
//       and lo = bf16(p_j - hi), for each 16-key step in ascending order the
//       hi product then the lo product accumulated in fp32.
// A key a column does not attend to gets p = 0, which adds exact zeros, so a
// column's bits do not depend on the other columns of its CTA.  K and V rows
// stream through a ring of RING shared-memory stages of kSub keys each, K
// sub-chunks first, then V sub-chunks: as TMA boxes of one 16-key page of the
// KV head (two boxes per page at DH = 128) when the chunk starts on a page,
// else by cp.async into the same layout.  phase tracks the stages' mbarrier
// parities across calls.  ready() runs once the first stages are requested
// and before the query fragments qb are read (decode loads them there).
template <int G, int DH, int NT, int RING, typename Ready>
__device__ __forceinline__ void chunk_partial(AttnSmem<G, DH, NT, RING>& sm, const uint16_t* __restrict__ kc,
                                              const uint16_t* __restrict__ vc, const CUtensorMap* tmK,
                                              const CUtensorMap* tmV, uint32_t& phase, const int32_t* page_row,
                                              int32_t g, int32_t Hkv, int32_t k0, int32_t n_max, float scale,
                                              int32_t max_pages, int32_t num_pages, int32_t* status,
                                              uint32_t (&qb)[AttnShape<G, DH, NT>::kNB][DH / 16][2],
                                              float (&oacc)[AttnShape<G, DH, NT>::kMT][AttnShape<G, DH, NT>::kNB][4],
                                              Ready&& ready) {
    using S = AttnShape<G, DH, NT>;
    constexpr int kVecPerRow = DH / 8;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    const int c8 = lane >> 2, k2 = 2 * (lane & 3);
    const int32_t lp0 = k0 / BI_PAGE;
    const int32_t np = (k0 + n_max - 1) / BI_PAGE - lp0 + 1;
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

    const int ns = (n_max + kSub - 1) / kSub;  // sub-chunks of K, then as many of V
    const int part = tid % kVecPerRow;         // this thread's 16-byte column of every row it copies
    // TMA boxes start on a page; the ring must sit on a 1024-byte boundary for the swizzle
    const bool use_tma = (k0 & (BI_PAGE - 1)) == 0 && (smem_u32(&sm.ring[0][0]) & 1023u) == 0;
    constexpr int kHalves = DH / 64;
    // Stages with a TMA copy still to be waited for.  Every thread derives it
    // from the same values (sm.abort is only read after a barrier), so every
    // thread waits on the same stages and tracks the same barrier parities.
    uint32_t issued = 0;
    auto issue = [&](int t) {
        if (t < 2 * ns) {
            const bool is_v = t >= ns;
            const int32_t j0 = (is_v ? t - ns : t) * kSub;
            const int32_t nk = min(kSub, n_max - j0);
            uint8_t* dst = sm.ring[t % RING];
            if (use_tma) {
                if (sm.abort) return;
                issued |= 1u << (t % RING);
                if (tid == 0) {
                    const int npg = (nk + BI_PAGE - 1) / BI_PAGE;
                    const CUtensorMap* map = is_v ? tmV : tmK;
                    uint64_t* bar = &sm.full[t % RING];
                    ptx::fence_proxy_async_smem();  // earlier generic writes to the stage before the copy
                    ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(npg * kHalves * BI_PAGE * 128));
                    for (int i = 0; i < npg; ++i) {
                        const int32_t pg = sm.pages[(k0 + j0) / BI_PAGE - lp0 + i];
                        const int32_t y = (pg * Hkv + g) * BI_PAGE;
#pragma unroll
                        for (int h = 0; h < kHalves; ++h)
                            ptx::tma_load_2d(dst + h * (kSub * 128) + i * (BI_PAGE * 128), map, bar, h * 64, y);
                    }
                }
            } else {
                const uint16_t* base = (is_v ? vc : kc) + static_cast<int64_t>(g) * BI_PAGE * DH + part * 8;
                for (int jl = tid / kVecPerRow; jl < nk; jl += kAttnThreads / kVecPerRow) {
                    const int32_t kp = k0 + j0 + jl;
                    const int64_t pg = sm.pages[kp / BI_PAGE - lp0];
                    cp_async16(dst + ring_off<DH>(jl, part),
                               base + (pg * Hkv * BI_PAGE + (kp & (BI_PAGE - 1))) * DH);
                }
                // rows past the last key up to the 16-key step boundary are read by
                // the MMAs (K: scores never stored; V: times p = 0): zero, not stale
                const int32_t pad_end = min(kSub, (nk + 15) & ~15);
                for (int jl = nk + tid / kVecPerRow; jl < pad_end; jl += kAttnThreads / kVecPerRow)
                    *reinterpret_cast<uint4*>(dst + ring_off<DH>(jl, part)) = make_uint4(0, 0, 0, 0);
            }
        }
        if (!use_tma) cp_async_commit();  // possibly empty: keeps one group per sub-chunk slot
    };
#pragma unroll
    for (int t = 0; t < RING; ++t) issue(t);
    ready();

#pragma unroll
    for (int mt = 0; mt < S::kMT; ++mt)
#pragma unroll
        for (int nb = 0; nb < S::kNB; ++nb) oacc[mt][nb][0] = oacc[mt][nb][1] = oacc[mt][nb][2] = oacc[mt][nb][3] = 0.0f;

    int32_t ncol_r[S::kNB][2];  // keys of this thread's score columns
#pragma unroll
    for (int nb = 0; nb < S::kNB; ++nb)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int c = nb * 8 + k2 + x;
            ncol_r[nb][x] = c < S::kCols ? sm.ncol[c] : 0;
        }

    for (int t = 0; t < 2 * ns; ++t) {
        const int st = t % RING;
        bool padded = false;  // (uniform) rows of this stage were just zeroed by several threads
        if (use_tma) {
            if (issued & (1u << st)) {
                issued &= ~(1u << st);
                if (!wait_stage(&sm.full[st], (phase >> st) & 1u)) {
                    report(status, BI_DEV_TIMEOUT_ATTENTION);
                    sm.abort = 1;
                }
                phase ^= 1u << st;
                // a page box also brings the rows past the last key: in V they
                // meet p = 0 in the MMAs, so they must be zeros, not stale values
                const int32_t j0 = (t - ns) * kSub;
                const int32_t nk = min(kSub, n_max - j0);
                if (t >= ns && (nk & 15)) {
                    padded = true;
                    const int32_t pad_end = (nk + 15) & ~15;
                    for (int i = tid; i < (pad_end - nk) * kVecPerRow; i += kAttnThreads)
                        *reinterpret_cast<uint4*>(sm.ring[st] + ring_off<DH>(nk + i / kVecPerRow, i % kVecPerRow)) =
                            make_uint4(0, 0, 0, 0);
                    ptx::fence_proxy_async_smem();  // before the stage's next TMA write
                }
            }
        } else {
            asm volatile("cp.async.wait_group %0;" ::"n"(RING - 1) : "memory");
        }
        // a thread's own mbarrier wait makes a TMA stage visible to it; cp.async
        // stages and zero-padded rows need the CTA barrier
        if (!use_tma || padded) __syncthreads();
        const uint32_t buf = smem_u32(sm.ring[st]);
        if (t < ns) {
            // scores: warp w takes keys 16w .. 16w+15 of the sub-chunk as the MMA rows
            const int32_t j0 = t * kSub;
            const int32_t nk = min(kSub, n_max - j0);
            if (warp * 16 < nk) {
                float acc[S::kNB][4];
#pragma unroll
                for (int nb = 0; nb < S::kNB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;
#pragma unroll
                for (int ks = 0; ks < S::kKSteps; ++ks) {
                    uint32_t a[4];
                    ldsm_x4(buf + ring_off<DH>(warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4)), a);
#pragma unroll
                    for (int nb = 0; nb < S::kNB; ++nb) mma_16816(acc[nb], a, qb[nb][ks][0], qb[nb][ks][1]);
                }
#pragma unroll
                for (int nb = 0; nb < S::kNB; ++nb)
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const int c = nb * 8 + k2 + (x & 1);
                        const int32_t key = j0 + warp * 16 + c8 + (x >> 1) * 8;
                        if (c < S::kCols && key < n_max)
                            sm.sc.p[c][key] = key < ncol_r[nb][x & 1] ? __fmul_rn(acc[nb][x], scale) : -INFINITY;
                    }
            }
            if (t == ns - 1) {
                __syncthreads();
                // m: exact max per column (order-free); a column without keys gets 0
                for (int c = warp; c < S::kCols; c += kWarps) {
                    float mx = -INFINITY;
                    for (int j = lane; j < n_max; j += 32) mx = fmaxf(mx, sm.sc.p[c][j]);
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    if (lane == 0) sm.m[c] = sm.ncol[c] > 0 ? mx : 0.0f;
                }
                __syncthreads();
                // p = exp(score - m) (exp(-inf) = 0 for keys a column skips) and the fixed-tree sum l
                float ls[S::kCols];
#pragma unroll
                for (int c = 0; c < S::kCols; ++c) ls[c] = 0.0f;
                if constexpr (AttnSmem<G, DH, NT, RING>::kSharedScores) {
                    // the hi/lo parts overwrite the scores: each thread first takes
                    // all of its scores (j = tid + 128i) into registers
                    constexpr int kJ = BI_KV_CHUNK / kAttnThreads;
                    uint32_t hl[kJ][S::kCols];  // hi | lo << 16
#pragma unroll
                    for (int i = 0; i < kJ; ++i) {
                        const int j = tid + i * kAttnThreads;
                        if (j < n_max) {
#pragma unroll
                            for (int c = 0; c < S::kCols; ++c) {
                                const float pv = attn_exp(__fsub_rn(sm.sc.p[c][j], sm.m[c]));
                                const uint16_t hb = f32_to_bf16(pv);
                                const uint16_t lb = f32_to_bf16(__fsub_rn(pv, bf16_to_f32(hb)));
                                hl[i][c] = static_cast<uint32_t>(hb) | (static_cast<uint32_t>(lb) << 16);
                                ls[c] = __fadd_rn(ls[c], pv);
                            }
                        }
                    }
                    __syncthreads();
#pragma unroll
                    for (int i = 0; i < kJ; ++i) {
                        const int j = tid + i * kAttnThreads;
                        if (j < n_max) {
#pragma unroll
                            for (int c = 0; c < S::kCols; ++c) {
                                sm.sc.ph[0][c][j] = static_cast<uint16_t>(hl[i][c] & 0xffffu);
                                sm.sc.ph[1][c][j] = static_cast<uint16_t>(hl[i][c] >> 16);
                            }
                        }
                    }
                } else {
                    for (int j = tid; j < n_max; j += kAttnThreads) {
#pragma unroll
                        for (int c = 0; c < S::kCols; ++c) {
                            const float pv = attn_exp(__fsub_rn(sm.sc.p[c][j], sm.m[c]));
                            const uint16_t hb = f32_to_bf16(pv);
                            sm.sc.ph[0][c][j] = hb;
                            sm.sc.ph[1][c][j] = f32_to_bf16(__fsub_rn(pv, bf16_to_f32(hb)));
                            ls[c] = __fadd_rn(ls[c], pv);
                        }
                    }
                }
                // keys past n_max up to the 16-key step boundary enter PV with p = 0
                for (int j = n_max + tid; j < ((n_max + 15) & ~15); j += kAttnThreads)
#pragma unroll
                    for (int c = 0; c < S::kCols; ++c) sm.sc.ph[0][c][j] = sm.sc.ph[1][c][j] = 0;
#pragma unroll
                for (int c = 0; c < S::kCols; ++c) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        ls[c] = __fadd_rn(ls[c], __shfl_xor_sync(0xffffffffu, ls[c], off));
                    if (lane == 0) sm.red[warp][c] = ls[c];
                }
                __syncthreads();
                if (tid < S::kCols) {
                    float l = sm.red[0][tid];
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) l = __fadd_rn(l, sm.red[w][tid]);
                    sm.l[tid] = l;
                }
            }
        } else {
            // PV: warp w owns head dims DH/4 * w ..; 16-key steps in ascending order
            const int32_t j0 = (t - ns) * kSub;
            const int32_t nk = min(kSub, n_max - j0);
            for (int kk = 0; kk < nk; kk += 16) {
                uint32_t bh[S::kNB][2], bl[S::kNB][2];
#pragma unroll
                for (int nb = 0; nb < S::kNB; ++nb) {
                    const int c = nb * 8 + c8;
#pragma unroll
                    for (int y = 0; y < 2; ++y) {
                        const int32_t key = j0 + kk + k2 + 8 * y;
                        bh[nb][y] = c < S::kCols ? *reinterpret_cast<const uint32_t*>(&sm.sc.ph[0][c][key]) : 0u;
                        bl[nb][y] = c < S::kCols ? *reinterpret_cast<const uint32_t*>(&sm.sc.ph[1][c][key]) : 0u;
                    }
                }
#pragma unroll
                for (int mt = 0; mt < S::kMT; ++mt) {
                    uint32_t a[4];
                    const int c0 = (warp * S::kDimsPerWarp + mt * 16) / 8;
                    ldsm_x4_trans(buf + ring_off<DH>(kk + (lane & 7) + (lane >> 4) * 8, c0 + ((lane >> 3) & 1)), a);
#pragma unroll
                    for (int nb = 0; nb < S::kNB; ++nb) {
                        mma_16816(oacc[mt][nb], a, bh[nb][0], bh[nb][1]);
                        mma_16816(oacc[mt][nb], a, bl[nb][0], bl[nb][1]);
                    }
                }
            }
        }
        __syncthreads();
        issue(t + RING);
    }
    if (!use_tma) cp_async_wait_all();
    __syncthreads();
}

// Writes a thread's accumulator elements (oacc layout above), each through
// f(column, dim, value).
template <int G, int DH, int NT, typename F>
__device__ __forceinline__ void for_each_out(const float (&oacc)[AttnShape<G, DH, NT>::kMT][AttnShape<G, DH, NT>::kNB][4],
                                             F&& f) {
    using S = AttnShape<G, DH, NT>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
#pragma unroll
    for (int mt = 0; mt < S::kMT; ++mt)
#pragma unroll
        for (int nb = 0; nb < S::kNB; ++nb)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int c = nb * 8 + 2 * (lane & 3) + (x & 1);
                const int d = warp * S::kDimsPerWarp + mt * 16 + (lane >> 2) + (x >> 1) * 8;
                if (c < S::kCols) f(c, d, oacc[mt][nb][x]);
            }
}

// Ascending-order merge step of two partials (M, L, O) and (m, l, o).
__device__ __forceinline__ void fold_step(float& M, float& L, float& O0, float& O1, float m, float l,
                                          float o0, float o1) {
    const float Mn = fmaxf(M, m);
    const float a = attn_exp(__fsub_rn(M, Mn));
    const float b = attn_exp(__fsub_rn(m, Mn));
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
// Decode: grid (entries, Hkv, max_splits); one token, its G heads as columns.
// ---------------------------------------------------------------------------
template <int G, int DH, int RING>
__global__ void __launch_bounds__(kAttnThreads, 6)
decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnGeom geo,
                    EntryMap em, int32_t max_splits, int32_t chunk2, float* __restrict__ ws_o,
                    float* __restrict__ ws_ml, int32_t early_kv) {
    pdl_trigger();
    using S = AttnShape<G, DH, 1>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AttnSmem<G, DH, 1, RING>& sm = *reinterpret_cast<AttnSmem<G, DH, 1, RING>*>(smem_raw);
    // The entry map and the page table are written before the kernels that
    // precede this one in the stream start (host copies); q and this step's
    // keys are written by the kernel just before it.
    const int32_t e = blockIdx.x, g = blockIdx.y, split = blockIdx.z;
    const Entry en = get_entry(em, e);
    const int32_t s = en.p + 1;
    int32_t size, count;
    pieces(s > 0 ? s : 1, chunk2, size, count);
    const bool ok = en.p >= 0 && (s + BI_PAGE - 1) / BI_PAGE <= geo.max_pages && count <= max_splits;
    if (!ok || split >= count) {
        pdl_wait();
        if (!ok && split == 0 && g == 0 && threadIdx.x == 0) report(geo.status, BI_DEV_BAD_POSITION);
        return;
    }
    const int32_t k0 = split * size;
    const int32_t n = min(size, s - k0);
    // With early_kv the caller guarantees that only each request's last
    // position was written in this step: a chunk before it may then request
    // its K/V copies before the dependency wait.
    const bool settled = early_kv != 0 && k0 + n < s;
    if (!settled) pdl_wait();
    if (threadIdx.x < S::kCols) sm.ncol[threadIdx.x] = n;
    ring_init(sm);
    uint32_t phase = 0;
    const int32_t tok[1] = {en.t};
    uint32_t qb[S::kNB][DH / 16][2];
    float oacc[S::kMT][S::kNB][4];
    chunk_partial<G, DH, 1, RING>(
        sm, reinterpret_cast<const uint16_t*>(geo.kc), reinterpret_cast<const uint16_t*>(geo.vc), &tmK, &tmV, phase,
        geo.page_table + static_cast<int64_t>(en.r) * geo.max_pages, g, geo.Hkv, k0, n, geo.scale, geo.max_pages,
        geo.num_pages, geo.status, qb, oacc, [&] {
            if (settled) pdl_wait();
            load_q_cols<G, DH, 1>(reinterpret_cast<const uint16_t*>(geo.q), tok, geo.H, g, qb);
        });
    // stage the partials through the score buffer, then write whole rows
    constexpr int kOStride = DH + 4;
    float* stage = &sm.sc.p[0][0];  // [kCols][kOStride]
    for_each_out<G, DH, 1>(oacc, [&](int c, int d, float v) { stage[c * kOStride + d] = v; });
    __syncthreads();
    const int64_t row0 = (static_cast<int64_t>(e) * geo.H + static_cast<int64_t>(g) * G) * max_splits + split;
    for (int i = threadIdx.x; i < S::kCols * (DH / 4); i += kAttnThreads) {
        const int c = i / (DH / 4), d4 = i % (DH / 4);
        reinterpret_cast<float4*>(ws_o + (row0 + static_cast<int64_t>(c) * max_splits) * DH)[d4] =
            reinterpret_cast<const float4*>(stage + c * kOStride)[d4];
    }
    if (threadIdx.x < S::kCols) {
        const int c = threadIdx.x;
        *reinterpret_cast<float2*>(ws_ml + (row0 + static_cast<int64_t>(c) * max_splits) * 2) =
            make_float2(sm.m[c], sm.l[c]);
    }
}

// Merge: grid (entries, H), DH/2 threads, each one dim pair; the fold runs
// over splits in ascending order, its inputs fetched kMergeBatch splits at a
// time so the loads of a batch are in flight together.
constexpr int kMergeBatch = 32;

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
    const float rl = __frcp_rn(L);  // out = O * fl(1 / L) (prefill's output divides the same way)
    store_out2(geo.out, geo.out_f32, oidx, __fmul_rn(O0, rl), __fmul_rn(O1, rl));
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

template <int G, int DH, int RING>
static cudaError_t launch_decode_ring(const AttnGeom& g, const EntryMap& em, int32_t n, int32_t max_splits,
                                      int32_t chunk2, float* ws_o, float* ws_ml, bool early_kv, cudaStream_t s) {
    const size_t smem = sizeof(AttnSmem<G, DH, 1, RING>);
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [smem] {
        attr_err = cudaFuncSetAttribute(decode_split_kernel<G, DH, RING>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tmK, tmV;
    if (!encode_kv_map(&tmK, g.kc, g.num_pages, g.Hkv, DH) || !encode_kv_map(&tmV, g.vc, g.num_pages, g.Hkv, DH))
        return cudaErrorInvalidValue;
    dim3 grid(n, g.Hkv, max_splits);
    cudaError_t e = launch_pdl(decode_split_kernel<G, DH, RING>, grid, dim3(kAttnThreads), smem, s, tmK, tmV, g, em,
                               max_splits, chunk2, ws_o, ws_ml, static_cast<int32_t>(early_kv));
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_merge_kernel<DH>, dim3(n, g.H), dim3(DH / 2), 0, s, g, em, max_splits, chunk2,
                      static_cast<const float*>(ws_o), static_cast<const float*>(ws_ml));
}

template <int G, int DH>
static cudaError_t launch_decode_t(const AttnGeom& g, const EntryMap& em, int32_t n, int32_t max_splits,
                                   int32_t chunk2, float* ws_o, float* ws_ml, bool early_kv, cudaStream_t s) {
    // ring depth moves data only: the arithmetic of a chunk is the same for both
    const int64_t ctas = static_cast<int64_t>(n) * g.Hkv * max_splits;
    if (ctas <= 3ll * num_sms())
        return launch_decode_ring<G, DH, kDeepRing>(g, em, n, max_splits, chunk2, ws_o, ws_ml, early_kv, s);
    return launch_decode_ring<G, DH, kRing>(g, em, n, max_splits, chunk2, ws_o, ws_ml, early_kv, s);
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
                                    cudaStream_t s, bool early_kv) {
    if (n_entries <= 0) return cudaSuccess;
    BI_ATTN_DISPATCH(launch_decode_t, g, em, n_entries, max_splits, variant_chunk2, ws_o, ws_ml, early_kv, s);
}

}  // namespace bi

#include "prefill_tc.cuh"

namespace bi {

cudaError_t launch_prefill_attention(const AttnGeom& g, const EntryMap& em, int32_t n_entries, int32_t q_rows,
                                     cudaStream_t s) {
    if (n_entries <= 0) return cudaSuccess;
    BI_ATTN_DISPATCH(tc_prefill::launch_prefill_tc_t, g, em, n_entries, q_rows, s);
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
unsigned long long g_noalloc_ctx[kMaxDevices] = {};  // the context the address was taken in

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the context current on this thread (ids are never reused, so
// a context re-created after a device reset gets a new one); false when no
// context is current or the driver offers no such query.
bool current_ctx_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's context (the
// host-side symbol is only a stand-in, never a device address).  Looked up
// once per device and context: after a device reset the library's module is
// loaded again in a new context, the array gets a new address, and the next
// call looks it up anew.
bi_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "bi_decode_attention_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(BI_ERR_UNSUPPORTED, "bi_decode_attention_noalloc: device index");
    unsigned long long ctx = 0;
    const bool known = current_ctx_id(&ctx);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!known || g_noalloc_ptr[dev] == nullptr || g_noalloc_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "bi_decode_attention_noalloc: cudaGetSymbolAddress");
        // the lookup makes the device's primary context current if none was
        unsigned long long now = 0;
        g_noalloc_ptr[dev] = current_ctx_id(&now) ? p : nullptr;  // no id: look it up again next call
        g_noalloc_ctx[dev] = now;
        *out = p;
        return BI_OK;
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
    AttnGeom g{q, k_cache, v_cache, page_table, out, out_dtype == BI_F32, H, Hkv, Dh, max_pages, num_pages,
               default_scale(scale, Dh), dev_status};
    EntryMap em{0, seq_lens, nullptr, nullptr, B};
    cudaError_t e = launch_decode_attention(g, em, B, max_splits, chunk2, ws_o, ws_ml, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BI_OK : cuda_fail(e, "bi_decode_attention_noalloc launch");
}
