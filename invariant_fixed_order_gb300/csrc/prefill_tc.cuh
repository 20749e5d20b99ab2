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
constexpr int kConsumers = 256;            // two threads per row: warps 0-7 (warpgroups 0 and 1)
constexpr int kThreads = kConsumers + 128; // warpgroup 2: warp 8 produces, warps 9-11 only give registers back
// Registers per thread: the launch gives every thread kLaunchRegs; the
// producer warpgroup hands back down to kProducerRegs and the consumers take
// up kConsumerRegs, so 128 * kProducerRegs + 256 * kConsumerRegs must not
// exceed kThreads * kLaunchRegs (checked below) or the increase would wait
// forever.
constexpr int kLaunchRegs = 168;
constexpr int kProducerRegs = 56;
constexpr int kConsumerRegs = 224;
static_assert(128 * kProducerRegs + kConsumers * kConsumerRegs <= kThreads * kLaunchRegs,
              "register split exceeds what the launch provides");
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

// What the producer tells the consumers about a run: its tokens (-1: no
// more runs), first token, KV head, request, largest and smallest context of
// its rows, chunk count, and each row's context (0: no keys, or not in the run).
struct RunDesc {
    int32_t tokens, t0, g, r, s_max, s_min, count;
    int32_t keys[kRows];
};

template <int DH>
struct Smem {
    static constexpr int kRegions = DH / 64;
    uint8_t k[kRegions][kKeyRegion];       // 1024-aligned (first)
    uint8_t v[kRegions][kKeyRegion];
    uint8_t q[kRegions][kQRegion];
    uint8_t stage[kRows * DH * 2];         // output staging: bf16 rows, or half of the fp32 dims
    uint64_t q_full, k_full, v_full;       // producer -> consumers: copies landed
    uint64_t s_done, pv_done;              // products completed (also: K, V and Q buffers free)
    uint64_t pa_ready, pb_ready;           // consumers -> MMA thread: P of keys 0-127 / 128-255 written
    uint64_t drain;                        // the MMA thread's last commit
    uint64_t rd_full[2], rd_empty[2];      // run descriptors written / read
    uint32_t tmem_base;
    int32_t abort;
    float xmax[2][kRows];                  // each half's partial row maximum
    float xsum[2][kRows];                  // the upper half's group sums (groups 2 and 3)
    float xL[kRows];                       // the row's final L, for the upper half's output
    RunDesc rd[2];
};

// One arrival on a barrier of this CTA (release: the caller's earlier writes
// are visible to whoever completes a wait on the phase).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The consumer warps' own barrier (named barrier 1, 256 threads); the
// producer warp never takes part.
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool consumer_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

// Every bounded wait of this kernel: each try may suspend the thread for up to
// kHintNs (it resumes when the phase completes), so waiting warps take few
// issue slots from the softmax warps that share their schedulers.
constexpr uint32_t kHintNs = 20000;
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int32_t* abort) {
    return ptx::mbar_wait_bounded_hint(bar, parity, abort, kHintNs);
}
// Every thread of a warp: a bounded wait whose outcome is the same in the
// whole warp (a failure in one lane fails the warp), so the warp-collective
// tensor-memory accesses that follow stay uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort) {
    return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort));
}

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

// Packed fp32 pairs (the f32x2 instructions): each lane is one IEEE
// round-to-nearest operation, so the results are the bits of the scalar
// __fadd_rn / __fsub_rn / __fmul_rn the decode routine uses (checked on GB300
// against the scalar instructions).  Only additions, subtractions and
// products whose result does not feed an addition use them: packed, the sum
// of two products by per-row constants did not reproduce the scalar bits on
// GB300, so the fold stays scalar.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "add.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "sub.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "mul.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// p of two consecutive keys (the even one first) as packed bf16 hi and lo
// pairs: hi = bf16(p) and lo = bf16(p - hi), rounded to nearest even as the
// decode routine rounds them.
__device__ __forceinline__ void pack_p(float p0, float p1, uint32_t& hi, uint32_t& lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);  // .x (low half) = p0
    hi = *reinterpret_cast<uint32_t*>(&h);
    const float2 r = sub2(make_float2(p0, p1), make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u)));
    __nv_bfloat162 l = __floats2bfloat162_rn(r.x, r.y);
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
// Reads 16 of this thread's scores, keys c0 .. c0 + 15 (columns at or past
// n_max: zeros, not read).  Completes at the next tcgen05.wait::ld.
__device__ __forceinline__ void load16(uint32_t base, int c0, int32_t n_max, uint32_t (&r)[16]) {
    if (c0 < n_max) {
        ptx::tmem_ld16(base + c0, r);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = 0u;
    }
}

// p of keys c0 .. c0 + 15 into p[off ..], and their P words back to TMEM in
// place of the scores (8 packed hi pairs, then 8 lo pairs).
template <bool kMask>
__device__ __forceinline__ void p_block16(uint32_t base, int c0, int32_t n_max, int32_t ncol, float scale, float m,
                                          const uint32_t (&r)[16], float (&p)[64], int off) {
    // score = fl(acc * scale) (or -inf), then attn_exp(score - m) = 2^(fl((score - m) log2 e))
    const float2 sc2 = make_float2(scale, scale), m2 = make_float2(m, m);
    const float2 l2e = make_float2(1.44269504088896341f, 1.44269504088896341f);
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        float2 x = c0 < n_max ? mul2(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), sc2)
                              : make_float2(-INFINITY, -INFINITY);
        if (kMask) {
            if (c0 + j >= ncol) x.x = -INFINITY;
            if (c0 + j + 1 >= ncol) x.y = -INFINITY;
        }
        x = mul2(sub2(x, m2), l2e);
        float pv0, pv1;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(pv0) : "f"(x.x));
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(pv1) : "f"(x.y));
        p[off + j] = pv0;
        p[off + j + 1] = pv1;
        pack_p(pv0, pv1, w[j / 2], w[8 + j / 2]);
    }
    if (c0 < n_max) tmem_st16(base + c0, w);
}

template <bool kMask, int DH>
__device__ __forceinline__ bool softmax_lo(Smem<DH>& sm, uint32_t tmem, int half, int row, int32_t n_max,
                                           int32_t ncol, float scale, float& m_out, float (&pa)[64], bool good) {
    const int c_lo = 64 * half, c_hi = 128 + 64 * half;  // this thread's key ranges (64 keys each)
    const uint32_t base = lane_addr(tmem, kColS);
    // pass 1: the row's maximum over its keys, 64 at a time
    float mx = -INFINITY;
#pragma unroll
    for (int rg = 0; rg < 2; ++rg) {
        const int c0 = rg == 0 ? c_lo : c_hi;
        if (good && c0 < n_max) {
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
    // the partial maxima meet, and every consumer learns whether the scores' wait succeeded everywhere
    if (consumer_any(!good)) return false;
    const float m = ncol > 0 ? __fmul_rn(fmaxf(sm.xmax[0][row], sm.xmax[1][row]), scale) : 0.0f;
    m_out = m;
    // pass 2, keys below 128: four blocks of 16, the next block read while one is computed
    uint32_t ra[16], rb[16];
    load16(base, c_lo, n_max, ra);
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        const int ca = c_lo + 16 * blk;
        ptx::tmem_ld_wait();
        if (blk % 2 == 0) {
            reg_fence<16>(ra);
            if (blk + 1 < 4) load16(base, ca + 16, n_max, rb);
            p_block16<kMask>(base, ca, n_max, ncol, scale, m, ra, pa, blk * 16);
        } else {
            reg_fence<16>(rb);
            if (blk + 1 < 4) load16(base, ca + 16, n_max, ra);
            p_block16<kMask>(base, ca, n_max, ncol, scale, m, rb, pa, blk * 16);
        }
    }
    return true;
}

// Second phase: p of the thread's keys 128 + 32b + i, the group sums in the
// decode routine's tree (pair sums pa + pb, the xor-butterfly), P words of
// these keys to TMEM.  Leaves w01 (lower half: groups 0 + 1) or xsum (upper
// half: groups 2 and 3).
template <bool kMask, int DH>
__device__ __forceinline__ void softmax_hi(Smem<DH>& sm, uint32_t tmem, int half, int row, int32_t n_max,
                                           int32_t ncol, float scale, float m, const float (&pa)[64], float& w01) {
    const int c_hi = 128 + 64 * half;
    const uint32_t base = lane_addr(tmem, kColS);
    float pb[64];
    uint32_t ra[16], rb[16];
    load16(base, c_hi, n_max, ra);
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        const int cb = c_hi + 16 * blk;
        ptx::tmem_ld_wait();
        if (blk % 2 == 0) {
            reg_fence<16>(ra);
            if (blk + 1 < 4) load16(base, cb + 16, n_max, rb);
            p_block16<kMask>(base, cb, n_max, ncol, scale, m, ra, pb, blk * 16);
        } else {
            reg_fence<16>(rb);
            if (blk + 1 < 4) load16(base, cb + 16, n_max, ra);
            p_block16<kMask>(base, cb, n_max, ncol, scale, m, rb, pb, blk * 16);
        }
    }
    // group gi: pairs (pa, pb) of keys 32b + i, i = 0..31, summed pairwise then
    // by the butterfly (16 first: i with i + 16, then 8, 4, 2, 1)
    float w[2];
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {  // 0 + p = p exactly (p >= 0)
            const float2 t = add2(make_float2(pa[32 * gi + i], pa[32 * gi + i + 1]),
                                  make_float2(pb[32 * gi + i], pb[32 * gi + i + 1]));
            v[i] = t.x;
            v[i + 1] = t.y;
        }
#pragma unroll
        for (int off = 16; off >= 2; off >>= 1)
#pragma unroll
            for (int i = 0; i < off; i += 2) {
                const float2 t = add2(make_float2(v[i], v[i + 1]), make_float2(v[i + off], v[i + off + 1]));
                v[i] = t.x;
                v[i + 1] = t.y;
            }
        w[gi] = __fadd_rn(v[0], v[1]);
    }
    if (half == 0) {
        w01 = __fadd_rn(w[0], w[1]);
    } else {
        sm.xsum[0][row] = w[0];
        sm.xsum[1][row] = w[1];
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

// The producer warp (every lane calls it): TMA page boxes of keys
// [k0, k0 + n) of KV head g into a chunk buffer (one box per 16-key page and
// 64-dim region: rows of 128 bytes, 128-byte swizzle), counted on bar.  The
// lanes read the chunk's page-table entries together; lane 0 issues.
template <int DH>
__device__ __forceinline__ void issue_chunk(uint8_t (*dst)[kKeyRegion], const CUtensorMap* map, uint64_t* bar,
                                            const int32_t* page_row, int32_t k0, int32_t n, int32_t g,
                                            const AttnGeom& geo) {
    constexpr int kRegions = DH / 64;
    const int lane = threadIdx.x & 31;
    const int32_t np = (n + BI_PAGE - 1) / BI_PAGE;  // <= 16
    int32_t pg = 0;
    if (lane < np) {
        const int32_t lp = k0 / BI_PAGE + lane;
        pg = lp < geo.max_pages ? __ldg(page_row + lp) : -1;
        if (pg < 0 || pg >= geo.num_pages) {
            report(geo.status, BI_DEV_BAD_PAGE);
            pg = 0;
        }
    }
    if (lane == 0) ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(np * kRegions * BI_PAGE * 128));
    for (int i = 0; i < np; ++i) {
        const int32_t pi = __shfl_sync(0xffffffffu, pg, i);
        if (lane == 0) {
            const int32_t y = (pi * geo.Hkv + g) * BI_PAGE;
#pragma unroll
            for (int h = 0; h < kRegions; ++h) ptx::tma_load_2d(&dst[h][i * BI_PAGE * 128], map, bar, h * 64, y);
        }
    }
}

// Every consumer thread: bounded wait for the phase of bar with the given
// parity; the outcome is the same in every consumer thread (a failure
// anywhere fails them all).
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, volatile int32_t* abort) {
    return !consumer_any(!wait_bounded(bar, parity, abort));
}

// A finished run whose output is still in tensor memory (running O).
struct PendingOut {
    bool on;
    int32_t t0, tokens, g;  // first token, tokens of the run, KV head
};

// out = O * fl(1 / L) of a finished run, staged through shared memory and written
// with 16-byte stores.  Every thread takes part: each writes its half of its
// row (a row without keys: zeros), then all copy whole rows out.  bf16 rows
// fit the stage at once, fp32 rows in two passes of half the dims.
template <int G, int DH>
__device__ __forceinline__ void write_out(Smem<DH>& sm, uint32_t tmem, const AttnGeom& geo, const PendingOut& po,
                                          int half, int row, bool has, float L_lower) {
    constexpr int kHalfDims = DH / 2;
    constexpr int kCPR = DH / 8;  // 16-byte chunks per stage row (DH * 2 bytes)
    const float L = half == 0 ? L_lower : sm.xL[row];
    const float rl = __frcp_rn(L);  // out = O * fl(1 / L), as the decode merge computes it
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
                for (int x = 0; x < 32; ++x) val[x] = has ? __fmul_rn(__uint_as_float(O[x]), rl) : 0.0f;
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
        consumer_sync();
        for (int k = threadIdx.x; k < kRows * kCPR; k += kConsumers) {
            const int r = k / kCPR, c = k % kCPR;
            const int ti = r / G;
            if (ti < po.tokens) {
                const int64_t orow = static_cast<int64_t>(po.t0 + ti) * geo.H + static_cast<int64_t>(po.g) * G + r % G;
                char* dst = reinterpret_cast<char*>(geo.out) + (orow * DH) * esize + p * (DH / 2) * 4 + c * 16;
                *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&sm.stage[r * DH * 2 + ((c ^ (r % kCPR)) << 4)]);
            }
        }
        consumer_sync();
    }
}

// The producer warp: walks this CTA's tiles (NT consecutive entries of one
// KV head; tiles strided by the grid) as runs of one request each, writes a
// descriptor per run, and issues its copies as the buffers come free: the
// queries and keys of a chunk once the previous chunk's scores are done, its
// values once the previous chunk's PV product is done.  It runs up to two
// runs ahead of the consumers (the descriptor ring) and a chunk ahead in the
// copies.  Ends with a descriptor of -1 tokens, then waits (bounded) until
// every copy it issued has landed.
template <int G, int DH>
__device__ __forceinline__ void produce(Smem<DH>& sm, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                        const CUtensorMap* tmQ, const AttnGeom& geo, const EntryMap& em,
                                        int32_t n_entries) {
    constexpr int NT = kRows / G;
    constexpr int kRegions = DH / 64;
    const int lane = threadIdx.x & 31;
    const int32_t n_tiles = ((n_entries + NT - 1) / NT) * geo.Hkv;
    volatile int32_t* abort = &sm.abort;
    uint32_t runs = 0, chunks = 0, q_runs = 0;  // descriptors written, chunks and queries issued
    bool ok = true;
    // lane 0 waits (bounded), the warp follows its outcome
    auto wait = [&](uint64_t* bar, uint32_t parity) {
        bool r = true;
        if (lane == 0) r = wait_bounded(bar, parity, abort);
        return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    auto take_slot = [&]() {  // the descriptor slot for run `runs`, once its previous run was read
        const int slot = runs & 1;
        if (runs >= 2 && !wait(&sm.rd_empty[slot], ((runs >> 1) - 1) & 1u)) return -1;
        return slot;
    };
    for (int32_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int32_t g = tile % geo.Hkv;
        const int32_t e_begin = (tile / geo.Hkv) * NT;
        const int32_t e_end = min(e_begin + NT, n_entries);
        for (int32_t e0 = e_begin; e0 < e_end && ok;) {
            const int slot = take_slot();
            if (slot < 0) {
                ok = false;
                break;
            }
            RunDesc& rd = sm.rd[slot];
            // the run: token first.t + i is query row i * G + head for the heads of group g
            const Entry first = get_entry(em, e0);
            int32_t tok = 0, kmax = 0, kmin = INT_MAX;
            for (int i = lane; i < NT; i += 32) {
                const int32_t e = e0 + i;
                int32_t keys = 0;
                bool mine = false;
                if (e < e_end) {
                    Entry en;
                    if (em.kind == 2) {  // entries are tokens; the request's tokens end at cu_q[r + 1]
                        mine = e < em.a[first.r + 1];
                        en = Entry{e, first.r, first.p + i};
                    } else {
                        en = get_entry(em, e);
                        mine = en.r == first.r;
                    }
                    if (mine) {
                        const int32_t s_len = en.p + 1;
                        // the queries are read as one box of consecutive tokens from first.t
                        const bool valid =
                            en.p >= 0 && (s_len + BI_PAGE - 1) / BI_PAGE <= geo.max_pages && en.t == first.t + i;
                        if (!valid) report(geo.status, BI_DEV_BAD_POSITION);
                        keys = valid ? s_len : 0;
                    }
                }
#pragma unroll
                for (int hh = 0; hh < G; ++hh) rd.keys[i * G + hh] = keys;
                if (mine) {
                    ++tok;
                    kmax = max(kmax, keys);
                    kmin = min(kmin, keys);
                }
            }
            tok = __reduce_add_sync(0xffffffffu, tok);
            kmax = __reduce_max_sync(0xffffffffu, kmax);
            kmin = __reduce_min_sync(0xffffffffu, kmin);
            const int32_t count = (kmax + kChunk - 1) / kChunk;
            if (lane == 0) {
                rd.tokens = tok;
                rd.t0 = first.t;
                rd.g = g;
                rd.r = first.r;
                rd.s_max = kmax;
                rd.s_min = kmin;
                rd.count = count;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.rd_full[slot]);  // releases the descriptor
            ++runs;
            const int32_t* page_row = geo.page_table + static_cast<int64_t>(first.r) * geo.max_pages;
            for (int32_t j = 0; j < count && ok; ++j) {
                const int32_t k0 = j * kChunk, n = min(kChunk, kmax - k0);
                // the K (and Q) buffer is free once the previous chunk's scores are done
                if (chunks > 0 && !(ok = wait(&sm.s_done, (chunks - 1) & 1u))) break;
                if (j == 0) {
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(&sm.q_full, static_cast<uint32_t>(kRegions * kQRegion));
#pragma unroll
                        for (int h = 0; h < kRegions; ++h)
                            ptx::tma_load_3d(&sm.q[h][0], tmQ, &sm.q_full, h * 64, g * G, first.t,
                                             ptx::policy_evict_first());
                    }
                    ++q_runs;
                }
                issue_chunk<DH>(sm.k, tmK, &sm.k_full, page_row, k0, n, g, geo);
                // the V buffer is free once the previous chunk's PV product is done
                if (chunks > 0 && !(ok = wait(&sm.pv_done, (chunks - 1) & 1u))) break;
                issue_chunk<DH>(sm.v, tmV, &sm.v_full, page_row, k0, n, g, geo);
                ++chunks;
            }
            e0 += tok;
        }
    }
    if (ok) {
        const int slot = take_slot();
        if (slot >= 0) {
            if (lane == 0) {
                sm.rd[slot].tokens = -1;
                mbar_arrive(&sm.rd_full[slot]);
            }
        } else {
            ok = false;
        }
    }
    if (!ok && lane == 0) {
        report(geo.status, BI_DEV_TIMEOUT_ATTENTION);
        *abort = 1;
    }
    // every copy issued has landed before the shared memory is released
    volatile int32_t none = 0;
    if (lane == 0) {
        if (q_runs > 0) ptx::mbar_wait_bounded(&sm.q_full, (q_runs - 1) & 1u, &none);
        if (chunks > 0) {
            ptx::mbar_wait_bounded(&sm.k_full, (chunks - 1) & 1u, &none);
            ptx::mbar_wait_bounded(&sm.v_full, (chunks - 1) & 1u, &none);
        }
    }
    __syncwarp();
}

// The MMA thread (lane 0 of warp 9): per chunk S = Q K^T once the chunk's
// keys (and the run's queries) have landed and the previous chunk's PV
// product is done; PV of keys 0-127 once the consumers have written their P
// and the values have landed; PV of keys 128-255 once that P is written.
// Reads the run descriptors to know the chunk counts.  Before it returns no
// product is in flight.
template <int DH>
__device__ __forceinline__ void issue_products(Smem<DH>& sm, uint32_t tmem) {
    const uint32_t idesc_s = ptx::idesc_bf16_f32(kRows, kChunk);
    const uint32_t idesc_pv = ptx::idesc_bf16_f32(kRows, DH) | (1u << 16);  // B (V) MN-major
    volatile int32_t* abort = &sm.abort;
    uint32_t runs = 0, chunks = 0, q_runs = 0;
    bool ok = true, issued = false;
    auto pv_steps = [&](int k_begin, int k_end) {  // 16-key steps: the hi part, then the lo part
        for (int ks = k_begin; ks < k_end; ++ks) {
            const uint64_t bd = desc(smem_u32(&sm.v[0][0]) + static_cast<uint32_t>(ks * 2048), kVLbo, kVSbo);
            mma_ts(tmem + kColO, tmem + kColS + 16 * ks, bd, idesc_pv, 1u);
            mma_ts(tmem + kColO, tmem + kColS + 16 * ks + 8, bd, idesc_pv, 1u);
        }
    };
    while (ok) {
        const int slot = runs & 1;
        if (!(ok = wait_bounded(&sm.rd_full[slot], (runs >> 1) & 1u, abort))) break;
        const int32_t tokens = sm.rd[slot].tokens, count = sm.rd[slot].count, s_max = sm.rd[slot].s_max;
        mbar_arrive(&sm.rd_empty[slot]);
        ++runs;
        if (tokens < 0) break;
        for (int32_t j = 0; j < count; ++j, ++chunks) {
            const int32_t n_max = min(kChunk, s_max - j * kChunk);
            const int steps = (n_max + 15) / 16;
            if (j == 0 && !(ok = wait_bounded(&sm.q_full, (q_runs++) & 1u, abort))) break;
            // the previous chunk's PV product has read its P (in the S columns)
            if (issued && !(ok = wait_bounded(&sm.pv_done, (chunks - 1) & 1u, abort))) break;
            if (!(ok = wait_bounded(&sm.k_full, chunks & 1u, abort))) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < DH / 16; ++ks) {
                const uint32_t step = static_cast<uint32_t>((ks % 4) * 32);
                ptx::tc_mma_f16<1>(tmem + kColS, desc(smem_u32(&sm.q[ks / 4][0]) + step, 16, 1024),
                                   desc(smem_u32(&sm.k[ks / 4][0]) + step, 16, 1024), idesc_s, ks > 0);
            }
            ptx::tc_commit<1>(&sm.s_done);
            issued = true;
            if (!(ok = wait_bounded(&sm.pa_ready, chunks & 1u, abort))) break;
            if (!(ok = wait_bounded(&sm.v_full, chunks & 1u, abort))) break;
            ptx::tc_fence_after();
            pv_steps(0, min(steps, 8));
            if (!(ok = wait_bounded(&sm.pb_ready, chunks & 1u, abort))) break;
            ptx::tc_fence_after();
            pv_steps(8, steps);
            ptx::tc_commit<1>(&sm.pv_done);
        }
    }
    if (!ok) *abort = 1;
    // no product may be in flight when tensor memory is freed
    if (issued) {
        ptx::tc_commit<1>(&sm.drain);
        volatile int32_t none = 0;
        ptx::mbar_wait_bounded(&sm.drain, 0, &none);
    }
}

// Persistent CTAs, one per SM: warps 0-7 consume runs (two threads per query
// row: softmax, fold, output), warp 8 produces them (descriptors and copies),
// lane 0 of warp 9 issues the tensor-core products; warps 10 and 11 complete
// that warpgroup, whose registers go to the consumers.
template <int G, int DH>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, AttnGeom geo, EntryMap em, int32_t n_entries) {
    pdl_trigger();
    pdl_wait();
    constexpr int kHalfDims = DH / 2;  // head dims of o and O per thread
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    Smem<DH>& sm = *reinterpret_cast<Smem<DH>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
    if (tid == 0) {
        sm.abort = 0;
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmQ);
        ptx::mbar_init(&sm.q_full, 1);
        ptx::mbar_init(&sm.k_full, 1);
        ptx::mbar_init(&sm.v_full, 1);
        ptx::mbar_init(&sm.s_done, 1);
        ptx::mbar_init(&sm.pv_done, 1);
        ptx::mbar_init(&sm.drain, 1);
        ptx::mbar_init(&sm.pa_ready, kConsumers);
        ptx::mbar_init(&sm.pb_ready, kConsumers);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.rd_full[i], 1);
            ptx::mbar_init(&sm.rd_empty[i], kConsumers + 1);  // the consumers and the MMA thread
        }
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
    if (warp >= kConsumers / 32) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
        if (warp == kConsumers / 32) {
            produce<G, DH>(sm, &tmK, &tmV, &tmQ, geo, em, n_entries);
        } else if (warp == kConsumers / 32 + 1 && lane == 0) {
            issue_products<DH>(sm, tmem);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
        const int half = warp >> 2;              // which half of the row's keys and dims
        const int row = 32 * (warp & 3) + lane;  // the row, = its TMEM lane
        const uint32_t col_o = kColO + half * kHalfDims, col_run = kColRun + half * kHalfDims;
        volatile int32_t* abort = &sm.abort;
        zero_cols<kHalfDims>(lane_addr(tmem, col_o));  // o starts at zero (and is zeroed after every fold)
        uint32_t runs = 0, chunks = 0;
        bool ok = true;
        PendingOut po{false, 0, 0, 0};
        bool po_has = false;  // this thread's row of the pending run has keys
        float po_L = 0.0f;
        // P written (TMEM stores and generic shared-memory writes done) before the products read it
        auto p_ready = [&](uint64_t* bar) {
            tmem_st_wait();
            ptx::tc_fence_before();
            mbar_arrive(bar);
        };
        while (ok) {
            // ---- the next run's descriptor ----
            const int slot = runs & 1;
            if (!(ok = wait_all(&sm.rd_full[slot], (runs >> 1) & 1u, abort))) break;
            const RunDesc& rd = sm.rd[slot];
            const int32_t tokens = rd.tokens;
            if (tokens < 0) break;
            const int32_t t0 = rd.t0, g = rd.g, s_max = rd.s_max, s_min = rd.s_min, count = rd.count;
            const int32_t keys = rd.keys[row];
            const bool mine = row / G < tokens;
            mbar_arrive(&sm.rd_empty[slot]);
            ++runs;
            // the previous run's output, while this run's first scores are computed
            if (po.on) {
                write_out<G, DH>(sm, tmem, geo, po, half, row, po_has, po_L);
                po.on = false;
            }
            float M = 0.0f, L = 0.0f;
            for (int32_t j = 0; j < count && ok; ++j, ++chunks) {
                const int32_t k0 = j * kChunk;
                const int32_t n_max = min(kChunk, s_max - k0);
                const int32_t ncol = mine ? min(max(keys - k0, 0), kChunk) : 0;
                const bool masked = k0 + kChunk > s_min;  // some row of the run stops inside this chunk
                bool good = warp_wait(&sm.s_done, chunks & 1u, abort);
                ptx::tc_fence_after();
                float m, w01, pa[64];
                const bool agreed = masked ? softmax_lo<true, DH>(sm, tmem, half, row, n_max, ncol, geo.scale, m, pa, good)
                                           : softmax_lo<false, DH>(sm, tmem, half, row, n_max, ncol, geo.scale, m, pa, good);
                if (!agreed) {
                    ok = false;
                    break;
                }
                // V rows past the last key up to the 16-key step meet p = 0 in the MMAs:
                // zeros, not whatever the page holds there
                if (n_max & 15) {
                    constexpr int kRegions = DH / 64;
                    good = warp_wait(&sm.v_full, chunks & 1u, abort);
                    if (good) {
                        const int pad = ((n_max + 15) & ~15) - n_max;
                        for (int i = tid; i < pad * 8 * kRegions; i += kConsumers) {
                            const int r = n_max + i / (8 * kRegions), rem = i % (8 * kRegions);
                            *reinterpret_cast<uint4*>(&sm.v[rem / 8][sw128(r, rem % 8)]) = make_uint4(0u, 0u, 0u, 0u);
                        }
                        ptx::fence_proxy_async_smem();
                    }
                }
                p_ready(&sm.pa_ready);  // PV of keys 0-127 runs during the second phase
                if (masked)
                    softmax_hi<true, DH>(sm, tmem, half, row, n_max, ncol, geo.scale, m, pa, w01);
                else
                    softmax_hi<false, DH>(sm, tmem, half, row, n_max, ncol, geo.scale, m, pa, w01);
                p_ready(&sm.pb_ready);
                good = good && warp_wait(&sm.pv_done, chunks & 1u, abort);
                if (consumer_any(!good)) {  // also publishes the upper half's group sums
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // l in the decode routine's order: ((group 0 + group 1) + group 2) + group 3
                const float l = half == 0 ? __fadd_rn(__fadd_rn(w01, sm.xsum[0][row]), sm.xsum[1][row]) : 0.0f;
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
                tmem_st_wait();  // O before it is read again (next fold, or the output)
            }
            if (!ok) break;
            // the run's output is written while the next run's first scores are computed
            if (half == 0) sm.xL[row] = L;
            po = PendingOut{true, t0, tokens, g};
            po_has = keys > 0 && count > 0;
            po_L = L;
        }
        if (ok && po.on) {
            consumer_sync();  // xL of the last run
            write_out<G, DH>(sm, tmem, geo, po, half, row, po_has, po_L);
        }
        if (!ok && tid == 0) {
            // a copy or a product did not complete in time: stop the other roles
            report(geo.status, BI_DEV_TIMEOUT_ATTENTION);
            *abort = 1;
        }
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
        // the consumers' register increase relies on the launch giving every
        // thread kLaunchRegs: refuse to launch a build that gives fewer
        cudaFuncAttributes fa{};
        if (attr_err == cudaSuccess) attr_err = cudaFuncGetAttributes(&fa, prefill_tc_kernel<G, DH>);
        if (attr_err == cudaSuccess && fa.numRegs < kLaunchRegs) attr_err = cudaErrorInvalidConfiguration;
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tmK, tmV, tmQ;
    if (!encode_kv_map(&tmK, g.kc, g.num_pages, g.Hkv, DH) || !encode_kv_map(&tmV, g.vc, g.num_pages, g.Hkv, DH) ||
        !encode_q_map(&tmQ, g.q, q_rows, g.H, DH, G))
        return cudaErrorInvalidValue;
    const int64_t tiles = static_cast<int64_t>((n + NT - 1) / NT) * g.Hkv;
    const int64_t ctas = std::min<int64_t>(tiles, num_sms());
    return launch_pdl(prefill_tc_kernel<G, DH>, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), smem, s, tmK, tmV,
                      tmQ, g, em, n);
}

}  // namespace tc_prefill
}  // namespace bi
