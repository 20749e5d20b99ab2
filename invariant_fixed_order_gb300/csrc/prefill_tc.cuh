// Causal prefill attention on the 5th-generation tensor cores (tcgen05),
// bitwise aligned with the decode routine of k_attention.cu.
//
// One CTA = 128 (query token, head) rows of one request and one KV head
// (128 / G consecutive tokens x the G heads of the group).  Row r is tensor
// memory lane r; two threads share it (warps w and w + 4 reach the same lane
// quarter), each taking half of the row's keys and half of its head dims.
// Chunks of 256 keys from key 0 are walked in order; per chunk:
//   S = Q K^T            tcgen05, M = 128 rows, N = 256 keys, K = Dh in 16-deep
//                        steps; A = Q (K-major, 128-byte swizzle, one TMA box per
//                        64 dims and run of tokens), B = the chunk's keys (K-major,
//                        128-byte swizzle, gathered from their pages by 16-byte
//                        cp.async copies of every thread) -> TMEM columns [0, 256)
//   softmax per row      score = fl(acc * scale) (or -inf past the row's keys);
//                        m = max; p = exp(score - m); hi = bf16(p), lo =
//                        bf16(p - hi); l summed in the decode routine's tree:
//                        per 32-key group b the pairs (32b + i, 32b + 128 + i)
//                        added to 0 in that order, an xor-butterfly 16, 8, 4, 2,
//                        1 over i, then the four groups in order.  The thread of
//                        the lower half takes groups 0 and 1 (keys 0-63 and
//                        128-191), the other groups 2 and 3; the partial maxima
//                        and group sums meet in shared memory.  hi/lo pairs go
//                        back into TMEM in place of the scores, as the A operand
//                        of the next product
//   o = P V              tcgen05, A = P (TMEM), B = the chunk's values (gathered
//                        like K) read MN-major (head dims contiguous), per 16-key step the hi
//                        then the lo product, into an accumulator that starts
//                        at zero -> TMEM columns [256, 256 + Dh)
//   fold                 the decode merge's expressions into the running (M, L)
//                        in registers and O in TMEM columns [384, 384 + Dh)
// The next chunk's S product runs on the tensor cores while the fold runs;
// the next chunk's K and V copies fly during the softmax and the products.
// CTAs are persistent: a run's first copies fly while the previous run's
// output is written.
// Outside the MMAs every step repeats the decode routine's arithmetic.  Inside
// them, a tcgen05 kind::f16 chain of 16-deep K steps gives the same fp32 bits
// as the decode routine's mma.sync m16n8k16 chain over the same steps, for
// either operand order and any N (measured on GB300 with random and
// subnormal-heavy bf16 data), so a token's output has the same bits from this
// kernel and from decode.
#pragma once

#include <limits.h>

namespace bi {
namespace tc_prefill {

constexpr int kRows = 128;                 // rows per CTA = TMEM lanes
constexpr int kThreads = 256;              // two threads per row
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
static_assert(kLowHalfEvenK, "pack_p below writes the even key into the low half");

template <int DH>
struct Smem {
    static constexpr int kRegions = DH / 64;
    uint8_t k[kRegions][kKeyRegion];       // 1024-aligned (first)
    uint8_t v[kRegions][kKeyRegion];
    uint8_t q[kRegions][kQRegion];
    uint8_t stage[kRows * DH * 2];         // output staging: bf16 rows, or half of the fp32 dims
    uint64_t q_full, s_done, pv_done;
    uint32_t tmem_base;
    int32_t abort;
    float xmax[2][kRows];                  // each half's partial row maximum
    float xsum[2][kRows];                  // the upper half's group sums (groups 2 and 3)
    float xL[kRows];                       // the row's final L, for the upper half's output
    int32_t red_max[kThreads / 32];
    int32_t red_min[kThreads / 32];
    int32_t pg[4][kChunk / BI_PAGE];       // page-table entries of chunks c (slot c % 4), read ahead
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

// Each thread reads / writes 32 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// After tcgen05.wait::ld: ties each loaded register to that point, so no use
// of it can be scheduled before the wait (the load writes it asynchronously).
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Writes zeros into N consecutive columns of this thread's lane from taddr.
template <int N>
__device__ __forceinline__ void zero_cols(uint32_t taddr) {
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
    for (int c = 0; c < N; c += 16) tmem_st16(taddr + c, z);
}

// TMEM address of column col of this thread's lane quarter.
__device__ __forceinline__ uint32_t lane_addr(uint32_t base, uint32_t col) {
    return base + (static_cast<uint32_t>(((threadIdx.x / 32) & 3) * 32) << 16) + col;
}

// p of two consecutive keys (the even one first) as packed bf16 hi and lo
// pairs: hi = bf16(p) and lo = bf16(p - hi), rounded to nearest even as the
// decode routine rounds them.
__device__ __forceinline__ void pack_p(float p0, float p1, uint32_t& hi, uint32_t& lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);  // .x (low half) = p0
    hi = *reinterpret_cast<uint32_t*>(&h);
    const float r0 = __fsub_rn(p0, __uint_as_float(hi << 16));
    const float r1 = __fsub_rn(p1, __uint_as_float(hi & 0xffff0000u));
    __nv_bfloat162 l = __floats2bfloat162_rn(r0, r1);
    lo = *reinterpret_cast<uint32_t*>(&l);
}

// Softmax of one chunk for this thread's half of its row.  ncol = keys of the
// chunk the row attends to (0..256); n_max = the chunk's keys (the same in
// every thread, so the warp-collective TMEM accesses stay uniform).  kMask:
// some row of the CTA attends to fewer than all 256 keys of the chunk.  On
// return m is the row's maximum, and w01 (lower half) the sum of groups 0 and
// 1; the upper half has left groups 2 and 3 in xsum.  P sits in TMEM columns
// [16 c, 16 c + 16) for key group c of 16 keys: 8 packed hi pairs, then 8 lo.
// The maximum is taken over the raw dot products and scaled once: rounding
// is monotone and scale > 0, so max_j fl(s_j * scale) = fl(max_j s_j * scale).
// Reads one block of this thread's scores: keys ca .. ca + 15 and
// ca + 128 .. ca + 143 (ca = 32 (2 half + gi) + 16 q); columns at or past n_max
// are not read (zeros).  Completes at the next tcgen05.wait::ld.
__device__ __forceinline__ void load_block(uint32_t base, int half, int gi, int q, int32_t n_max, uint32_t (&ra)[16],
                                           uint32_t (&rb)[16]) {
    const int ca = 32 * (2 * half + gi) + 16 * q, cb = 128 + ca;
    if (ca < n_max) {
        ptx::tmem_ld16(base + ca, ra);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) ra[i] = 0u;
    }
    if (cb < n_max) {
        ptx::tmem_ld16(base + cb, rb);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) rb[i] = 0u;
    }
}

// p of one block (see load_block): P words back to TMEM in place of the
// scores, pair sums p_i + p_(i+128) into u (kFirst: u = the pair sums; else
// u += them, the butterfly's first level).
template <bool kMask, bool kFirst>
__device__ __forceinline__ void p_block(uint32_t base, int half, int gi, int q, int32_t n_max, int32_t ncol, float scale,
                                        float m, const uint32_t (&ra)[16], const uint32_t (&rb)[16], float (&u)[16]) {
    const int ca = 32 * (2 * half + gi) + 16 * q, cb = 128 + ca;
    uint32_t wa[16], wb[16];  // P words of keys ca .. ca + 15 and cb .. cb + 15
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        float pa[2], pb[2];
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int i = j + x;
            float sa = ca < n_max ? __fmul_rn(__uint_as_float(ra[i]), scale) : -INFINITY;
            float sb = cb < n_max ? __fmul_rn(__uint_as_float(rb[i]), scale) : -INFINITY;
            if (kMask) {
                if (ca + i >= ncol) sa = -INFINITY;
                if (cb + i >= ncol) sb = -INFINITY;
            }
            pa[x] = attn_exp(__fsub_rn(sa, m));
            pb[x] = attn_exp(__fsub_rn(sb, m));
            // decode adds both to 0; p >= 0 is never -0, so 0 + p = p exactly
            const float pair = __fadd_rn(pa[x], pb[x]);
            u[i] = kFirst ? pair : __fadd_rn(u[i], pair);
        }
        pack_p(pa[0], pa[1], wa[j / 2], wa[8 + j / 2]);
        pack_p(pb[0], pb[1], wb[j / 2], wb[8 + j / 2]);
    }
    if (ca < n_max) tmem_st16(base + ca, wa);
    if (cb < n_max) tmem_st16(base + cb, wb);
}

template <bool kMask, int DH>
__device__ __forceinline__ void softmax_half(Smem<DH>& sm, uint32_t tmem, int half, int row, int32_t n_max,
                                             int32_t ncol, float scale, float& m_out, float& w01) {
    const int c_lo = 64 * half, c_hi = 128 + 64 * half;  // this thread's key ranges (64 keys each)
    const uint32_t base = lane_addr(tmem, kColS);
    // pass 1: the row's maximum over its keys, 64 at a time
    float mx = -INFINITY;
#pragma unroll
    for (int rg = 0; rg < 2; ++rg) {
        const int c0 = rg == 0 ? c_lo : c_hi;
        if (c0 < n_max) {
            uint32_t r[64];
            tmem_ld32(base + c0, r);
            tmem_ld32(base + c0 + 32, r + 32);
            ptx::tmem_ld_wait();
            reg_fence<64>(r);
#pragma unroll
            for (int i = 0; i < 64; ++i)
                if (!kMask || c0 + i < ncol) mx = fmaxf(mx, __uint_as_float(r[i]));
        }
    }
    sm.xmax[half][row] = mx;
    __syncthreads();
    const float m = ncol > 0 ? __fmul_rn(fmaxf(sm.xmax[0][row], sm.xmax[1][row]), scale) : 0.0f;
    // pass 2: p, its hi/lo pairs and the group sums, 16 keys of each range at
    // a time; the next block's scores are read while this block is computed
    float w0 = 0.0f, w1 = 0.0f;
    uint32_t xa[16], xb[16], ya[16], yb[16];  // two blocks of scores: keys ca.. and cb..
    load_block(base, half, 0, 0, n_max, xa, xb);
#pragma unroll 1
    for (int gi = 0; gi < 2; ++gi) {
        float u[16];  // after the second block: the butterfly's first level (i, i + 16)
        ptx::tmem_ld_wait();
        reg_fence<16>(xa);
        reg_fence<16>(xb);
        load_block(base, half, gi, 1, n_max, ya, yb);
        p_block<kMask, true>(base, half, gi, 0, n_max, ncol, scale, m, xa, xb, u);
        ptx::tmem_ld_wait();
        reg_fence<16>(ya);
        reg_fence<16>(yb);
        if (gi == 0) load_block(base, half, 1, 0, n_max, xa, xb);
        p_block<kMask, false>(base, half, gi, 1, n_max, ncol, scale, m, ya, yb, u);
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1)
#pragma unroll
            for (int i = 0; i < off; ++i) u[i] = __fadd_rn(u[i], u[i + off]);
        if (gi == 0)
            w0 = u[0];
        else
            w1 = u[0];
    }
    m_out = m;
    if (half == 0) {
        w01 = __fadd_rn(w0, w1);
    } else {
        sm.xsum[0][row] = w0;
        sm.xsum[1][row] = w1;
        w01 = 0.0f;
    }
}

// V as the B operand of PV: rows are keys (128 B = 64 dims), regions of 64
// dims kKeyRegion apart, 8-key groups 1024 B apart.  For an MN-major operand
// with the 128-byte swizzle the descriptor's leading offset is the stride
// between 64-element regions along MN and the stride offset the one between
// 8-row groups along K (measured against the K-major form, bit for bit).
constexpr uint32_t kVLbo = kKeyRegion;
constexpr uint32_t kVSbo = 1024;

// Every thread: its share of the 16-byte copies (cp.async) that bring keys
// [k0, k0 + n) of KV head g into a chunk buffer, in the 128-byte-swizzled
// layout of a TMA page box (rows of 64 dims, regions of 64 dims kKeyRegion
// apart); committed as one group.  pages: the chunk's page-table entries (in
// shared memory, read ahead).  Sixteen consecutive threads copy one key's row,
// so each read is a contiguous 256-byte (DH = 128) run of its page.  Keys past
// n are not copied.
template <int DH>
__device__ __forceinline__ void load_chunk(uint8_t (*dst)[kKeyRegion], const uint16_t* __restrict__ cache,
                                           const int32_t* pages, int32_t k0, int32_t n, int32_t g,
                                           const AttnGeom& geo) {
    constexpr int kCPR = DH / 8;                 // 16-byte chunks per key row
    constexpr int kIters = kChunk * kCPR / kThreads;
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int i = static_cast<int>(threadIdx.x) + it * kThreads;
        const int key = i / kCPR, c = i % kCPR;
        if (key < n) {
            int32_t pg = pages[key / BI_PAGE];
            if (pg < 0 || pg >= geo.num_pages) {
                report(geo.status, BI_DEV_BAD_PAGE);
                pg = 0;
            }
            const uint16_t* src =
                cache + ((static_cast<int64_t>(pg) * geo.Hkv + g) * BI_PAGE + ((k0 + key) & (BI_PAGE - 1))) * DH + c * 8;
            cp_async16(&dst[c >> 3][sw128(key, c & 7)], src);
        }
    }
    cp_async_commit();
}

// Page-table entry lp of a request's row (raw; checked where it is used), or
// -1 past the row.
__device__ __forceinline__ int32_t read_page(const int32_t* page_row, int32_t lp, int32_t max_pages) {
    return lp < max_pages ? __ldg(page_row + lp) : -1;
}

// The copies of this thread's groups older than the newest `newer` are
// complete; after the barrier that follows, every thread's are, and the
// tensor cores may read them.
template <int kNewer>
__device__ __forceinline__ void copies_landed() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kNewer) : "memory");
    ptx::fence_proxy_async_smem();  // generic-proxy writes before the MMAs read them
}

// Every thread: bounded wait on bar's phase; the outcome is the same in every
// thread (a failure anywhere fails the block).  The phase advances only on
// success, so a later drain waits on the same one.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t& phase, volatile int32_t* abort) {
    const bool ok = __syncthreads_or(!ptx::mbar_wait_bounded(bar, phase, abort)) == 0;
    if (ok) phase ^= 1u;
    return ok;
}

// A finished run whose output is still in tensor memory (running O).
struct PendingOut {
    bool on;
    int32_t t0, tokens, g;  // first token, tokens of the run, KV head
};

// out = O / L of a finished run, staged through shared memory and written
// with 16-byte stores.  Every thread takes part: each writes its half of its
// row (a row without keys: zeros), then all copy whole rows out.  bf16 rows
// fit the stage at once, fp32 rows in two passes of half the dims.
template <int G, int DH>
__device__ __forceinline__ void write_out(Smem<DH>& sm, uint32_t tmem, const AttnGeom& geo, const PendingOut& po,
                                          int half, int row, bool has, float L_lower) {
    constexpr int kHalfDims = DH / 2;
    constexpr int kCPR = DH / 8;  // 16-byte chunks per stage row (DH * 2 bytes)
    const float L = half == 0 ? L_lower : sm.xL[row];
    const int passes = geo.out_f32 ? 2 : 1;
    const int esize = geo.out_f32 ? 4 : 2;
    for (int p = 0; p < passes; ++p) {
        if (!geo.out_f32 || half == p) {
#pragma unroll
            for (int c0 = 0; c0 < kHalfDims; c0 += 32) {
                uint32_t O[32];
                tmem_ld32(lane_addr(tmem, kColRun + half * kHalfDims + c0), O);
                ptx::tmem_ld_wait();
                reg_fence<32>(O);
                float val[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) val[x] = has ? __fdiv_rn(__uint_as_float(O[x]), L) : 0.0f;
                if (geo.out_f32) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int cc = c0 / 4 + c;
                        *reinterpret_cast<uint4*>(&sm.stage[row * DH * 2 + ((cc ^ (row % kCPR)) << 4)]) =
                            make_uint4(__float_as_uint(val[4 * c]), __float_as_uint(val[4 * c + 1]),
                                       __float_as_uint(val[4 * c + 2]), __float_as_uint(val[4 * c + 3]));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int cc = half * (kHalfDims / 8) + c0 / 8 + c;
                        *reinterpret_cast<uint4*>(&sm.stage[row * DH * 2 + ((cc ^ (row % kCPR)) << 4)]) =
                            make_uint4(pack_bf16x2(val[8 * c], val[8 * c + 1]),
                                       pack_bf16x2(val[8 * c + 2], val[8 * c + 3]),
                                       pack_bf16x2(val[8 * c + 4], val[8 * c + 5]),
                                       pack_bf16x2(val[8 * c + 6], val[8 * c + 7]));
                    }
                }
            }
        }
        __syncthreads();
        for (int k = threadIdx.x; k < kRows * kCPR; k += kThreads) {
            const int r = k / kCPR, c = k % kCPR;
            const int ti = r / G;
            if (ti < po.tokens) {
                const int64_t orow = static_cast<int64_t>(po.t0 + ti) * geo.H + static_cast<int64_t>(po.g) * G + r % G;
                char* dst = reinterpret_cast<char*>(geo.out) + (orow * DH) * esize + p * (DH / 2) * 4 + c * 16;
                *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&sm.stage[r * DH * 2 + ((c ^ (r % kCPR)) << 4)]);
            }
        }
        __syncthreads();
    }
}

// Persistent CTAs over tiles of (NT consecutive entries, one KV head); a
// tile's entries are walked as runs of one request each.
template <int G, int DH>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, AttnGeom geo, EntryMap em, int32_t n_entries) {
    pdl_trigger();
    pdl_wait();
    constexpr int NT = kRows / G;
    constexpr int kRegions = DH / 64;
    constexpr int kHalfDims = DH / 2;  // head dims of o and O per thread
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem<DH>& sm = *reinterpret_cast<Smem<DH>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    const int half = warp >> 2;                  // which half of the row's keys and dims
    const int row = 32 * (warp & 3) + lane;      // the row, = its TMEM lane
    const int32_t n_blocks = (n_entries + NT - 1) / NT;
    const int32_t n_tiles = n_blocks * geo.Hkv;
    if (tid == 0) {
        sm.abort = 0;
        ptx::prefetch_tmap(&tmQ);
        ptx::mbar_init(&sm.q_full, 1);
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
    const uint32_t col_o = kColO + half * kHalfDims, col_run = kColRun + half * kHalfDims;
    zero_cols<kHalfDims>(lane_addr(tmem, col_o));  // o starts at zero (and is zeroed after every fold)
    const uint16_t* kc = reinterpret_cast<const uint16_t*>(geo.kc);
    const uint16_t* vc = reinterpret_cast<const uint16_t*>(geo.vc);
    uint32_t ph_q = 0, ph_s = 0, ph_pv = 0;
    // outstanding asynchronous work, tracked alike in every thread (the K and V
    // copies are cp.async groups of each thread, waited for in commit order)
    bool q_pending = false, s_pending = false, pv_pending = false;
    bool ok = true;
    PendingOut po{false, 0, 0, 0};
    bool po_has = false;  // this thread's row of the pending run has keys
    float po_L = 0.0f;

    auto issue_s = [&]() {  // thread 0: S = Q K^T of the chunk in sm.k
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
            const uint32_t step = static_cast<uint32_t>((ks % 4) * 32);
            ptx::tc_mma_f16<1>(tmem + kColS, desc(smem_u32(&sm.q[ks / 4][0]) + step, 16, 1024),
                               desc(smem_u32(&sm.k[ks / 4][0]) + step, 16, 1024), idesc_s, ks > 0);
        }
        ptx::tc_commit<1>(&sm.s_done);
    };

    int32_t tile = blockIdx.x;
    int32_t e0 = 0, e_end = 0, g = 0;
    if (tile < n_tiles) {
        g = tile % geo.Hkv;
        e0 = (tile / geo.Hkv) * NT;
        e_end = min(e0 + NT, n_entries);
    }
    while (tile < n_tiles && ok) {
        // ---- a run of consecutive entries of one request: token first.t + row / G, head row % G ----
        const Entry first = get_entry(em, e0);
        const int32_t* page_row = geo.page_table + static_cast<int64_t>(first.r) * geo.max_pages;
        // the page-table entries of the run's first two chunks, in flight during the lookups below
        const int32_t pg_first = tid < 2 * (kChunk / BI_PAGE) ? read_page(page_row, tid, geo.max_pages) : 0;
        const int32_t ti = row / G;
        Entry en{-1, -1, -1};
        bool mine = false;
        if (e0 + ti < e_end) {
            if (em.kind == 2) {
                // entries are tokens; the request's tokens end at cu_q[r + 1]
                mine = e0 + ti < em.a[first.r + 1];
                en = Entry{e0 + ti, first.r, first.p + ti};
            } else {
                en = get_entry(em, e0 + ti);
                mine = en.r == first.r;
            }
        }
        int32_t keys = 0;
        if (mine) {
            const int32_t s_len = en.p + 1;
            // the queries are read as one box of consecutive tokens from first.t
            const bool valid = en.p >= 0 && (s_len + BI_PAGE - 1) / BI_PAGE <= geo.max_pages && en.t == first.t + ti;
            if (!valid && half == 0 && row % G == 0) report(geo.status, BI_DEV_BAD_POSITION);
            keys = valid ? s_len : 0;
        }
        const int32_t run_tokens = __syncthreads_count(mine && half == 0 && row % G == 0);
        const int32_t wmax = __reduce_max_sync(0xffffffffu, keys);
        const int32_t wmin = __reduce_min_sync(0xffffffffu, mine ? keys : INT_MAX);
        if (lane == 0) {
            sm.red_max[warp] = wmax;
            sm.red_min[warp] = wmin;
        }
        if (tid < 2 * (kChunk / BI_PAGE)) sm.pg[tid / (kChunk / BI_PAGE)][tid % (kChunk / BI_PAGE)] = pg_first;
        __syncthreads();
        int32_t s_max = sm.red_max[0], s_min = sm.red_min[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) {
            s_max = max(s_max, sm.red_max[w]);
            s_min = min(s_min, sm.red_min[w]);
        }
        const int32_t count = (s_max + kChunk - 1) / kChunk;
        // this run's queries and first chunk: the buffers are free (the last
        // products of the previous run have completed)
        if (count > 0) {
            if (tid == 0) {
                ptx::mbar_arrive_expect_tx(&sm.q_full, static_cast<uint32_t>(kRegions * kQRegion));
#pragma unroll
                for (int h = 0; h < kRegions; ++h)
                    ptx::tma_load_3d(&sm.q[h][0], &tmQ, &sm.q_full, h * 64, g * G, first.t, ptx::policy_evict_first());
            }
            load_chunk<DH>(sm.k, kc, sm.pg[0], 0, min(kChunk, s_max), g, geo);
            load_chunk<DH>(sm.v, vc, sm.pg[0], 0, min(kChunk, s_max), g, geo);
            q_pending = true;
        }
        // the previous run's output, while this run's first copies are in flight
        if (po.on) {
            write_out<G, DH>(sm, tmem, geo, po, half, row, po_has, po_L);
            po.on = false;
        }
        if (count > 0) {
            copies_landed<1>();  // K (V is the newer group)
            if (!(ok = wait_all(&sm.q_full, ph_q, &sm.abort))) break;
            q_pending = false;
            ptx::tc_fence_after();
            if (tid == 0) issue_s();
            s_pending = true;
        }
        float M = 0.0f, L = 0.0f;
        for (int32_t j = 0; j < count && ok; ++j) {
            const int32_t k0 = j * kChunk;
            const int32_t n_max = min(kChunk, s_max - k0);
            const int32_t ncol = mine ? min(max(keys - k0, 0), kChunk) : 0;
            const bool masked = k0 + kChunk > s_min;  // some row of the run stops inside this chunk
            if (!(ok = wait_all(&sm.s_done, ph_s, &sm.abort))) break;
            s_pending = false;
            ptx::tc_fence_after();
            // the K buffer is free: the next chunk's keys
            if (j + 1 < count)
                load_chunk<DH>(sm.k, kc, sm.pg[(j + 1) & 3], k0 + kChunk, min(kChunk, s_max - k0 - kChunk), g, geo);
            float m, w01;
            if (masked)
                softmax_half<true, DH>(sm, tmem, half, row, n_max, ncol, geo.scale, m, w01);
            else
                softmax_half<false, DH>(sm, tmem, half, row, n_max, ncol, geo.scale, m, w01);
            // this chunk's V (the next chunk's K, if requested, is the newer group)
            if (j + 1 < count)
                copies_landed<1>();
            else
                copies_landed<0>();
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
            // l in the decode routine's order: ((group 0 + group 1) + group 2) + group 3
            const float l = half == 0 ? __fadd_rn(__fadd_rn(w01, sm.xsum[0][row]), sm.xsum[1][row]) : 0.0f;
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
            // the V buffer is free: the next chunk's values; the S buffer is
            // free: the next chunk's scores while this chunk is folded
            // the page-table entries of chunk j + 2, stored after the fold
            const int32_t pg_ahead =
                tid < kChunk / BI_PAGE && j + 2 < count ? read_page(page_row, (j + 2) * (kChunk / BI_PAGE) + tid,
                                                                    geo.max_pages)
                                                        : 0;
            if (j + 1 < count) {
                load_chunk<DH>(sm.v, vc, sm.pg[(j + 1) & 3], k0 + kChunk, min(kChunk, s_max - k0 - kChunk), g, geo);
                copies_landed<1>();  // the next chunk's K (its V is the newer group)
                __syncthreads();
                ptx::tc_fence_after();
                if (tid == 0) issue_s();
                s_pending = true;
            }
            // the decode merge's fold; a row without keys in this chunk keeps its state
            const bool active = ncol > 0;
            float a = 1.0f, bw = 1.0f;
            if (active) {
                if (j == 0) {
                    M = m;
                    L = l;
                } else {
                    const float Mn = fmaxf(M, m);
                    a = attn_exp(__fsub_rn(M, Mn));
                    bw = attn_exp(__fsub_rn(m, Mn));
                    L = __fadd_rn(__fmul_rn(L, a), __fmul_rn(l, bw));
                    M = Mn;
                }
            }
#pragma unroll
            for (int c0 = 0; c0 < kHalfDims; c0 += 32) {
                uint32_t o[32], O[32];
                tmem_ld32(lane_addr(tmem, col_o + c0), o);
                if (j > 0) tmem_ld32(lane_addr(tmem, col_run + c0), O);
                ptx::tmem_ld_wait();
                reg_fence<32>(o);
                if (j > 0) {
                    reg_fence<32>(O);
                    if (active)
#pragma unroll
                        for (int x = 0; x < 32; ++x)
                            O[x] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(O[x]), a),
                                                             __fmul_rn(__uint_as_float(o[x]), bw)));
                    tmem_st32(lane_addr(tmem, col_run + c0), O);
                } else {
                    tmem_st32(lane_addr(tmem, col_run + c0), o);
                }
            }
            zero_cols<kHalfDims>(lane_addr(tmem, col_o));  // the next chunk's o starts at zero
            if (tid < kChunk / BI_PAGE && j + 2 < count) sm.pg[(j + 2) & 3][tid] = pg_ahead;
            tmem_st_wait();
            ptx::tc_fence_before();
        }
        if (!ok) break;
        // the run's output is written while the next run's first copies are in flight
        if (half == 0) sm.xL[row] = L;
        po = PendingOut{true, first.t, run_tokens, g};
        po_has = keys > 0 && count > 0;
        po_L = L;
        // the next run: the rest of this tile, else this CTA's next tile
        e0 += run_tokens;
        if (e0 >= e_end) {
            tile += gridDim.x;
            if (tile < n_tiles) {
                g = tile % geo.Hkv;
                e0 = (tile / geo.Hkv) * NT;
                e_end = min(e0 + NT, n_entries);
            }
        }
        __syncthreads();  // xL and the run's shared state before the next run reuses them
    }
    if (ok && po.on) write_out<G, DH>(sm, tmem, geo, po, half, row, po_has, po_L);

    if (!ok) {
        // a copy or an MMA did not complete in time: report, issue nothing more,
        // wait (bounded) for what is still in flight before the memory is freed
        if (tid == 0) report(geo.status, BI_DEV_TIMEOUT_ATTENTION);
        volatile int32_t none = 0;
        cp_async_wait_all();
        if (q_pending) wait_all(&sm.q_full, ph_q, &none);
        if (s_pending) wait_all(&sm.s_done, ph_s, &none);
        if (pv_pending) wait_all(&sm.pv_done, ph_pv, &none);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 0) ptx::tmem_dealloc<1>(tmem, kTmemCols);
}

template <int G, int DH>
cudaError_t launch_prefill_tc_t(const AttnGeom& g, const EntryMap& em, int32_t n, int32_t q_rows, cudaStream_t s) {
    constexpr int NT = kRows / G;
    const size_t smem = sizeof(Smem<DH>) + 1024;  // + alignment of the base to 1024 bytes
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [smem] {
        attr_err = cudaFuncSetAttribute(prefill_tc_kernel<G, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tmQ;
    if (!encode_q_map(&tmQ, g.q, q_rows, g.H, DH, G)) return cudaErrorInvalidValue;
    const int64_t tiles = static_cast<int64_t>((n + NT - 1) / NT) * g.Hkv;
    const int64_t ctas = std::min<int64_t>(tiles, num_sms());
    return launch_pdl(prefill_tc_kernel<G, DH>, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), smem, s, tmQ, g,
                      em, n);
}

}  // namespace tc_prefill
}  // namespace bi
