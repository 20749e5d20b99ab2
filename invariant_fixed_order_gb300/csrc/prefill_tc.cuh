// Causal prefill attention on the 5th-generation tensor cores (tcgen05),
// bitwise aligned with the decode routine of k_attention.cu.
//
// One CTA = 128 (query token, head) rows of one request and one KV head
// (128 / G consecutive tokens x the G heads of the group), 128 threads; thread
// t owns row t, which is also TMEM lane t.  Chunks of 256 keys from key 0,
// walked in order; per chunk:
//   S = Q K^T            tcgen05, M = 128 rows, N = 256 keys, K = Dh in 16-steps,
//                        A = Q (K-major SW128, loaded once), B = the chunk's K
//                        pages (K-major SW128, TMA page boxes) -> TMEM cols [0, 256)
//   softmax per row      thread-local: score = fl(acc * scale) or -inf past the
//                        row's keys; m = max; p = exp(score - m); hi = bf16(p),
//                        lo = bf16(p - hi); l summed in the decode routine's tree
//                        (lane-serial pairs j, j + 128; xor-butterfly over 32
//                        keys; the four 32-key groups in order); hi/lo packed
//                        into TMEM in place of the scores (A operand of PV)
//   o = P V              tcgen05, A = P (TMEM), B = the chunk's V pages read
//                        MN-major (dims contiguous), per 16-key step hi then lo,
//                        into a zeroed accumulator -> TMEM cols [256, 256 + Dh)
//   fold                 the decode merge's expressions into the running
//                        (M, L) in registers and O in TMEM cols [384, 384 + Dh)
// Outside the MMAs every step repeats the decode routine's arithmetic.  Inside
// them, a tcgen05 kind::f16 chain of 16-deep K steps gives the same fp32 bits
// as the decode routine's mma.sync m16n8k16 chain over the same steps, for
// either operand order and any N (measured on GB300 with random and
// subnormal-heavy bf16 data), so a token's output has the same bits from this
// kernel and from decode.
#pragma once

namespace bi {
namespace tc_prefill {

constexpr int kRows = 128;                 // rows per CTA = TMEM lanes = threads
constexpr int kThreads = 128;
constexpr int kChunk = BI_KV_CHUNK;        // 256 keys
constexpr int kKeyRegion = kChunk * 128;   // one 64-dim SW128 region of a chunk's K or V (32 KB)
constexpr int kQRegion = kRows * 128;      // one 64-dim SW128 region of Q (16 KB)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;              // scores, then p hi/lo in place
constexpr uint32_t kColO = 256;            // this chunk's o
constexpr uint32_t kColRun = 384;          // running O

// A bf16 pair packed into one 32-bit TMEM column of an A operand holds the
// even k in its low half (measured: the other order reproduces nothing).
constexpr bool kLowHalfEvenK = true;

template <int DH>
struct Smem {
    static constexpr int kRegions = DH / 64;
    uint8_t k[kRegions][kKeyRegion];       // 1024-aligned (first)
    uint8_t v[kRegions][kKeyRegion];
    uint8_t q[kRegions][kQRegion];
    uint64_t k_full, v_full, s_done, pv_done;
    uint32_t tmem_base;
    int32_t abort;
    int32_t pages[kChunk / BI_PAGE];
};

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled region.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Shared-memory descriptor, 128-byte swizzle, explicit leading / stride offsets.
__device__ __forceinline__ uint64_t desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, one CTA.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Each thread writes 16 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMEM address of column col of this thread's warp's lane quarter.
__device__ __forceinline__ uint32_t lane_addr(uint32_t base, uint32_t col) {
    return base + (static_cast<uint32_t>((threadIdx.x / 32) * 32) << 16) + col;
}

__device__ __forceinline__ uint32_t pack_pair(uint16_t even_k, uint16_t odd_k) {
    return kLowHalfEvenK ? (static_cast<uint32_t>(even_k) | (static_cast<uint32_t>(odd_k) << 16))
                         : (static_cast<uint32_t>(odd_k) | (static_cast<uint32_t>(even_k) << 16));
}

// Softmax of one chunk for this thread's row, in TMEM.  ncol = keys of the
// chunk the row attends to (0..256).  On return m, l are the row's partial and
// TMEM columns [16 g, 16 g + 16) hold key group g's p as the PV A operand:
// 8 packed hi pairs, then 8 packed lo pairs.
// n_max (the chunk's keys, the same in every thread) bounds the warp-collective
// TMEM reads; ncol masks this thread's row.
__device__ __forceinline__ void softmax_chunk(uint32_t tmem, int32_t n_max, int32_t ncol, float scale, float& m_out,
                                              float& l_out) {
    // m: exact max of the row's scores (order-free); a row without keys gets 0
    float mx = -INFINITY;
    for (int c0 = 0; c0 < n_max; c0 += 16) {
        uint32_t r[16];
        ptx::tmem_ld16(lane_addr(tmem, kColS + c0), r);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (c0 + j < ncol) mx = fmaxf(mx, __fmul_rn(__uint_as_float(r[j]), scale));
    }
    const float m = ncol > 0 ? mx : 0.0f;
    // p, its hi/lo parts, and l in the decode routine's tree: for each 32-key
    // group b (keys 32b + L and 32b + 128 + L), lane-serial pairs, then the
    // xor-butterfly 16, 8, 4, 2, 1 over L; the groups added in order
    float l = 0.0f;
#pragma unroll 1
    for (int b = 0; b < 4; ++b) {
        float u[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {       // keys 32b.. then 32b + 128..
#pragma unroll
            for (int q = 0; q < 2; ++q) {            // two 16-key groups of 32
                const int c0 = 32 * b + 128 * half + 16 * q;
                uint32_t r[16];
                ptx::tmem_ld16(lane_addr(tmem, kColS + c0), r);
                ptx::tmem_ld_wait();
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    float pv[2];
                    uint16_t hb[2], lb[2];
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const int key = c0 + j + x;
                        const float sc = key < ncol ? __fmul_rn(__uint_as_float(r[j + x]), scale) : -INFINITY;
                        pv[x] = expf(__fsub_rn(sc, m));
                        hb[x] = f32_to_bf16(pv[x]);
                        lb[x] = f32_to_bf16(__fsub_rn(pv[x], bf16_to_f32(hb[x])));
                        const int L = 16 * q + j + x;
                        u[L] = half == 0 ? __fadd_rn(0.0f, pv[x]) : __fadd_rn(u[L], pv[x]);
                    }
                    w[j / 2] = pack_pair(hb[0], hb[1]);
                    w[8 + j / 2] = pack_pair(lb[0], lb[1]);
                }
                tmem_st16(lane_addr(tmem, kColS + c0), w);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
            for (int L = 0; L < off; ++L) u[L] = __fadd_rn(u[L], u[L + off]);
        l = b == 0 ? u[0] : __fadd_rn(l, u[0]);
    }
    m_out = m;
    l_out = l;
}

// Zeroes Dh columns of this thread's lane from col.
template <int DH>
__device__ __forceinline__ void tmem_zero(uint32_t tmem, uint32_t col) {
    uint32_t z[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) z[j] = 0u;
#pragma unroll
    for (int c0 = 0; c0 < DH; c0 += 16) tmem_st16(lane_addr(tmem, col + c0), z);
}

// The decode merge's fold of this chunk's (m, l, o) into the running (M, L, O);
// the first chunk copies.  Every thread of the CTA calls it (the TMEM accesses
// are warp-collective; first is the same everywhere); a row that attends to no
// key of the chunk (active false) keeps its state.
template <int DH>
__device__ __forceinline__ void fold_chunk(uint32_t tmem, bool first, bool active, float m, float l, float& M,
                                           float& L) {
    float a = 1.0f, b = 1.0f;
    if (!active) {
    } else if (!first) {
        const float Mn = fmaxf(M, m);
        a = expf(__fsub_rn(M, Mn));
        b = expf(__fsub_rn(m, Mn));
        L = __fadd_rn(__fmul_rn(L, a), __fmul_rn(l, b));
        M = Mn;
    } else {
        M = m;
        L = l;
    }
#pragma unroll 1
    for (int c0 = 0; c0 < DH; c0 += 16) {
        uint32_t o[16], O[16];
        ptx::tmem_ld16(lane_addr(tmem, kColO + c0), o);
        if (!first) ptx::tmem_ld16(lane_addr(tmem, kColRun + c0), O);
        ptx::tmem_ld_wait();
        if (!first && active)
#pragma unroll
            for (int j = 0; j < 16; ++j)
                O[j] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(O[j]), a),
                                                 __fmul_rn(__uint_as_float(o[j]), b)));
        tmem_st16(lane_addr(tmem, kColRun + c0), first ? o : O);
    }
}

// V as the B operand of PV: rows are keys (128 B = 64 dims), regions of 64
// dims kKeyRegion apart, 8-key groups 1024 B apart.  For an MN-major operand
// with the 128-byte swizzle the descriptor's leading offset is the stride
// between 64-element regions along MN and the stride offset the one between
// 8-row groups along K (measured against the K-major form, bit for bit).
constexpr uint32_t kVLbo = kKeyRegion;
constexpr uint32_t kVSbo = 1024;

// Thread 0: TMA page boxes of keys [k0, k0 + n) of KV head g into a chunk
// buffer (one box per 16-key page and 64-dim region), counted on bar.
template <int DH>
__device__ __forceinline__ void issue_chunk(uint8_t (*dst)[kKeyRegion], const CUtensorMap* map, uint64_t* bar,
                                            const int32_t* page_row, int32_t k0, int32_t n, int32_t g,
                                            const AttnGeom& geo) {
    constexpr int kRegions = DH / 64;
    const int32_t np = (n + BI_PAGE - 1) / BI_PAGE;
    ptx::fence_proxy_async_smem();  // earlier generic writes to the buffer before the copies
    ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np * kRegions * BI_PAGE * 128));
    for (int i = 0; i < np; ++i) {
        const int32_t lp = k0 / BI_PAGE + i;
        int32_t pg = lp < geo.max_pages ? page_row[lp] : -1;
        if (pg < 0 || pg >= geo.num_pages) {
            report(geo.status, BI_DEV_BAD_PAGE);
            pg = 0;
        }
        const int32_t y = (pg * geo.Hkv + g) * BI_PAGE;
#pragma unroll
        for (int h = 0; h < kRegions; ++h) ptx::tma_load_2d(&dst[h][i * BI_PAGE * 128], map, bar, h * 64, y);
    }
}

// Every thread: bounded wait on bar's phase; the outcome is the same in every
// thread (a failure anywhere fails the block).
// The phase advances only on success, so a later drain waits on the same one.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t& phase, volatile int32_t* abort) {
    const bool ok = __syncthreads_or(!ptx::mbar_wait_bounded(bar, phase, abort)) == 0;
    if (ok) phase ^= 1u;
    return ok;
}

template <int G, int DH>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnGeom geo,
                  EntryMap em, int32_t n_entries) {
    pdl_trigger();
    pdl_wait();
    constexpr int NT = kRows / G;
    constexpr int kRegions = DH / 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem<DH>& sm = *reinterpret_cast<Smem<DH>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    const int32_t g = blockIdx.y;
    const int32_t e_begin = static_cast<int32_t>(blockIdx.x) * NT;
    const int32_t e_end = min(e_begin + NT, n_entries);
    __shared__ int32_t red[kThreads / 32];
    if (tid == 0) {
        sm.abort = 0;
        ptx::mbar_init(&sm.k_full, 1);
        ptx::mbar_init(&sm.v_full, 1);
        ptx::mbar_init(&sm.s_done, 1);
        ptx::mbar_init(&sm.pv_done, 1);
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc<1>(&sm.tmem_base, kTmemCols);
        ptx::tmem_relinquish<1>();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t idesc_s = ptx::idesc_bf16_f32(kRows, kChunk);
    const uint32_t idesc_pv = ptx::idesc_bf16_f32(kRows, DH) | (1u << 16);  // B (V) MN-major
    uint32_t ph_k = 0, ph_v = 0, ph_s = 0, ph_pv = 0;
    // outstanding asynchronous work, tracked alike in every thread
    bool k_pending = false, v_pending = false, s_pending = false, pv_pending = false;
    bool ok = true;

    for (int32_t e0 = e_begin; e0 < e_end && ok;) {
        // a run of consecutive entries of one request; this thread's row is
        // token e0 + tid / G, head tid % G
        const Entry first = get_entry(em, e0);
        const int32_t ti = tid / G;
        Entry en{-1, -1, -1};
        if (e0 + ti < e_end) en = get_entry(em, e0 + ti);
        const bool mine = e0 + ti < e_end && en.r == first.r;
        int32_t keys = 0;
        if (mine) {
            const int32_t s_len = en.p + 1;
            const bool valid = en.p >= 0 && (s_len + BI_PAGE - 1) / BI_PAGE <= geo.max_pages;
            if (!valid && tid % G == 0) report(geo.status, BI_DEV_BAD_POSITION);
            keys = valid ? s_len : 0;
        }
        const int32_t run_tokens = __syncthreads_count(mine && tid % G == 0);
        const int32_t wmax = __reduce_max_sync(0xffffffffu, keys);
        if (lane == 0) red[warp] = wmax;
        // Q rows, K-major with the 128-byte swizzle (rows outside the run: zeros)
        const uint16_t* qrow = reinterpret_cast<const uint16_t*>(geo.q) +
                               (static_cast<int64_t>(mine ? en.t : 0) * geo.H + static_cast<int64_t>(g) * G + tid % G) * DH;
#pragma unroll
        for (int c = 0; c < DH / 8; ++c) {
            const uint4 v = mine ? *reinterpret_cast<const uint4*>(qrow + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(&sm.q[c >> 3][sw128(tid, c)]) = v;
        }
        ptx::fence_proxy_async_smem();
        __syncthreads();
        int32_t s_max = red[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) s_max = max(s_max, red[w]);
        const int32_t count = (s_max + kChunk - 1) / kChunk;
        const int32_t* page_row = geo.page_table + static_cast<int64_t>(first.r) * geo.max_pages;
        if (tid == 0 && count > 0) {
            issue_chunk<DH>(sm.k, &tmK, &sm.k_full, page_row, 0, min(kChunk, s_max), g, geo);
            issue_chunk<DH>(sm.v, &tmV, &sm.v_full, page_row, 0, min(kChunk, s_max), g, geo);
        }
        k_pending = v_pending = count > 0;
        float M = 0.0f, L = 0.0f;
        for (int32_t j = 0; j < count && ok; ++j) {
            const int32_t k0 = j * kChunk;
            const int32_t n_max = min(kChunk, s_max - k0);
            const int32_t ncol = mine ? min(max(keys - k0, 0), kChunk) : 0;
            // S = Q K^T over the chunk's 256 key rows (rows past n_max are masked below)
            if (!(ok = wait_all(&sm.k_full, ph_k, &sm.abort))) break;
            k_pending = false;
            ptx::tc_fence_after();
            if (tid == 0) {
#pragma unroll
                for (int ks = 0; ks < DH / 16; ++ks) {
                    const uint32_t step = static_cast<uint32_t>((ks % 4) * 32);
                    ptx::tc_mma_f16<1>(tmem + kColS, desc(smem_u32(&sm.q[ks / 4][0]) + step, 16, 1024),
                                       desc(smem_u32(&sm.k[ks / 4][0]) + step, 16, 1024), idesc_s, ks > 0);
                }
                ptx::tc_commit<1>(&sm.s_done);
            }
            s_pending = true;
            if (!(ok = wait_all(&sm.s_done, ph_s, &sm.abort))) break;
            s_pending = false;
            ptx::tc_fence_after();
            // the K buffer is free: the next chunk's K pages
            if (tid == 0 && j + 1 < count)
                issue_chunk<DH>(sm.k, &tmK, &sm.k_full, page_row, k0 + kChunk, min(kChunk, s_max - k0 - kChunk), g,
                                geo);
            k_pending = j + 1 < count;
            float m, l;
            softmax_chunk(tmem, n_max, ncol, geo.scale, m, l);
            tmem_zero<DH>(tmem, kColO);
            if (!(ok = wait_all(&sm.v_full, ph_v, &sm.abort))) break;
            v_pending = false;
            // V rows past the last key up to the 16-key step meet p = 0 in the MMAs:
            // zeros, not whatever the page holds there
            if (n_max & 15) {
                const int pad = ((n_max + 15) & ~15) - n_max;
                for (int i = tid; i < pad * 8 * kRegions; i += kThreads) {
                    const int r = n_max + i / (8 * kRegions), rem = i % (8 * kRegions);
                    *reinterpret_cast<uint4*>(&sm.v[rem / 8][sw128(r, rem % 8)]) = make_uint4(0u, 0u, 0u, 0u);
                }
                ptx::fence_proxy_async_smem();
            }
            tmem_st_wait();
            ptx::tc_fence_before();
            __syncthreads();
            ptx::tc_fence_after();
            // o = P V: per 16-key step the hi part, then the lo part
            if (tid == 0) {
                const int steps = (n_max + 15) / 16;
                for (int ks = 0; ks < steps; ++ks) {
                    const uint64_t bd = desc(smem_u32(&sm.v[0][0]) + static_cast<uint32_t>(ks * 2048), kVLbo, kVSbo);
                    mma_ts(tmem + kColO, tmem + kColS + 16 * ks, bd, idesc_pv, 1u);
                    mma_ts(tmem + kColO, tmem + kColS + 16 * ks + 8, bd, idesc_pv, 1u);
                }
                ptx::tc_commit<1>(&sm.pv_done);
            }
            pv_pending = true;
            if (!(ok = wait_all(&sm.pv_done, ph_pv, &sm.abort))) break;
            pv_pending = false;
            ptx::tc_fence_after();
            // the V buffer is free: the next chunk's V pages
            if (tid == 0 && j + 1 < count)
                issue_chunk<DH>(sm.v, &tmV, &sm.v_full, page_row, k0 + kChunk, min(kChunk, s_max - k0 - kChunk), g,
                                geo);
            v_pending = j + 1 < count;
            fold_chunk<DH>(tmem, j == 0, ncol > 0, m, l, M, L);
            tmem_st_wait();
            ptx::tc_fence_before();
        }
        if (ok) {
            // out = O / L; a row without keys gets zeros
            ptx::tc_fence_after();
            const int64_t obase = (static_cast<int64_t>(mine ? en.t : 0) * geo.H + static_cast<int64_t>(g) * G + tid % G) * DH;
#pragma unroll 1
            for (int c0 = 0; c0 < DH; c0 += 16) {
                uint32_t O[16];
                ptx::tmem_ld16(lane_addr(tmem, kColRun + c0), O);
                ptx::tmem_ld_wait();
                if (mine)
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float a = keys > 0 && count > 0 ? __fdiv_rn(__uint_as_float(O[j]), L) : 0.0f;
                        const float b = keys > 0 && count > 0 ? __fdiv_rn(__uint_as_float(O[j + 1]), L) : 0.0f;
                        store_out2(geo.out, geo.out_f32, obase + c0 + j, a, b);
                    }
            }
        }
        ptx::tc_fence_before();
        __syncthreads();
        e0 += run_tokens;
    }

    if (!ok) {
        // a copy or an MMA did not complete in time: report, issue nothing more,
        // wait (bounded) for what is still in flight before the memory is freed
        if (tid == 0) report(geo.status, BI_DEV_TIMEOUT_ATTENTION);
        volatile int32_t none = 0;
        if (k_pending) wait_all(&sm.k_full, ph_k, &none);
        if (v_pending) wait_all(&sm.v_full, ph_v, &none);
        if (s_pending) wait_all(&sm.s_done, ph_s, &none);
        if (pv_pending) wait_all(&sm.pv_done, ph_pv, &none);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc<1>(tmem, kTmemCols);
}

template <int G, int DH>
cudaError_t launch_prefill_tc_t(const AttnGeom& g, const EntryMap& em, int32_t n, cudaStream_t s) {
    constexpr int NT = kRows / G;
    const size_t smem = sizeof(Smem<DH>) + 1024;  // + alignment of the base to 1024 bytes
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [smem] {
        attr_err = cudaFuncSetAttribute(prefill_tc_kernel<G, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tmK, tmV;
    if (!encode_kv_map(&tmK, g.kc, g.num_pages, g.Hkv, DH) || !encode_kv_map(&tmV, g.vc, g.num_pages, g.Hkv, DH))
        return cudaErrorInvalidValue;
    return launch_pdl(prefill_tc_kernel<G, DH>, dim3((n + NT - 1) / NT, g.Hkv), dim3(kThreads), smem, s, tmK, tmV,
                      g, em, n);
}

}  // namespace tc_prefill
}  // namespace bi
