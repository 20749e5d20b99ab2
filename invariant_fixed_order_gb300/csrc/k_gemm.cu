// Batch-invariant GEMM on the 5th-generation tensor cores.
//
// "Batch invariance and reproducible inference", "2 · Cross-block
// accumulation" and "3 · Kernel selection changing with shape": split-K and
// M-dependent kernel choice are what make a GEMM's per-element order follow
// the batch.  Here every output element of a weight matrix, for every M, is
// produced by the same sequence: tcgen05.mma products (bf16 in, fp32
// accumulated in TMEM, K = 16), K tiles of 64 in ascending order, inside a K
// tile the four 16-deep MMAs in ascending order, all into one accumulator.
// The instruction forms and widths below give every element the same bits
// (tested bit for bit), so which one runs is data movement:
//   * N <= 65536 (the projections of a layer): the CTA-pair form, M = 256
//     over a cluster of two CTAs on two SMs.  The pair's MMA takes 128 rows of
//     A from each CTA's shared memory and half its weight rows from each, so
//     a layer projection with only 32-48 output tiles of 128 columns keeps
//     twice the SMs busy (one MMA costs the same in either form: 32.7 ns at
//     N = 128, measured with resident operands).  With at most 64 rows (and
//     no fused RoPE) the pair takes M = 128 instead, 64 rows per CTA, so each
//     tensor core reads half the A rows per MMA;
//   * N > 65536 (a vocabulary projection): the single-CTA form, M = 128.
//     Its hundreds of tiles fill every SM many times over, and one SM then
//     consumes 4 KB of weights per MMA instead of the pair's 2 KB, which is
//     what lets the weight stream run at the copy bandwidth.
//
// What may follow M is only how that work is laid out, never the arithmetic
// of an element:
//   * tile width: 128 columns for M <= 256 and 256 for larger M, one MMA of
//     that width per 16-deep step (N = 256: the A slice is read from shared
//     memory once per step instead of once per 128 columns, which is what
//     lets a prefill GEMM keep the tensor pipe busy: 63 -> 87 % active);
//   * the TMA box of A covers the smallest power of two >= min(M, 128) rows
//     (16..128); A stages are packed at that stride, so the MMA's rows past
//     the box read neighbouring stages: those rows of the accumulator are
//     never stored, and a row's result depends only on its own A row (pinned
//     by the row-invariance tests);
//   * ring depth and K tiles per ring stage.
//
// The kernel is persistent (one CTA per SM) with warp roles: warp 0 of each
// CTA streams its K tiles of A and W by TMA into its own ring, counting the
// bytes of the whole group on the issuing CTA's barrier, and owns the TMEM
// allocation; warp 1 of the issuing CTA (the even CTA of a pair) issues the
// MMAs (one thread) and commits each consumed ring stage to every producer;
// warps 4-7 of each CTA read that CTA's 128 accumulator rows back (warp w:
// TMEM lanes 32*(w%4)..+31), run the fused epilogue and release the
// accumulator to the MMA issuer.  The accumulator is double buffered in TMEM
// so a tile's epilogue overlaps the next tile's main loop.  Weights do not
// depend on the kernel before this one in the stream, so while that kernel
// finishes the producers already pull the first tile's weight slab;
// activations are read only after the dependency wait.  Every wait is
// bounded: a wait that runs out sets an abort flag in every CTA of the group
// and a device status code, every role winds down, copies and MMAs in flight
// are drained and TMEM is freed.
//
// With a fused RMSNorm (a few contiguous rows: the forward step's norms at
// small batch) the producer brings the raw rows x into the A ring as usual,
// counted on a separate barrier; warps 2-3 of the issuing CTA then normalise
// each landed stage in place and release it to the MMA issuer.  Each row's
// rinv is taken first, by warps 2-7 of the issuing CTA, from x in global
// memory in the RMSNorm kernel's order (a warp per row, lane l over 16-byte
// chunks l, l + 32, ... with fused multiply-adds, then the xor-butterfly), and
// every element becomes bf16((x * rinv) * gamma): the A operand is bit for bit
// the RMSNorm kernel's output, so whether a step normalises in a kernel or in
// the GEMM does not change a row's bits.
//
// BI_VARIANT splits K over CTAs into an fp32 workspace when the output has
// fewer 128x128 tiles than SMs and adds the partials in split order in a
// second kernel: deterministic run to run, but its order depends on M.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace bi {

constexpr int kBM = BI_GEMM_BLOCK_M;   // 128: accumulator rows of one CTA
constexpr int kUN = BI_GEMM_UMMA_N;    // 128: N of one MMA
constexpr int kEpi = 64;               // epilogue column chunk (a SwiGLU gate|up group pair)
constexpr int kBK = BI_GEMM_BLOCK_K;   // 64
constexpr int kMaxStages = 16;
constexpr int kGemmThreads = 256;
constexpr int kGroupM = 16;            // M tiles per rasterisation band
constexpr int kBarrierBytes = 1024;
constexpr int kRingBudget = 212 * 1024;  // shared memory for the A and W rings
constexpr int kMaxSmem = 226 * 1024;  // dynamic shared memory; the kernel's few static bytes fit beside it

struct GemmArgs {
    void* C;
    const uint16_t* residual;
    int64_t M;
    int32_t N, K;
    int32_t c_f32;
    int32_t ep;
    int32_t kb_per_split;
    int32_t nkb_total;
    int32_t m_tiles, n_tiles, total_tiles;
    int64_t split_stride;  // elements between split partials (fp32), variant only
    int32_t a_box_rows;    // rows of A per TMA box (16..128)
    int32_t a_stride;      // bytes between A box slots (a_box_rows * 128)
    int32_t a_region;      // bytes of the A region (slots + pad for the last window)
    int32_t stages;        // ring stages
    int32_t kps;           // 64-deep K tiles per stage
    int32_t w_early;       // 1: W may be read before the dependency wait (no earlier kernel writes it)
    unsigned long long* am_keys;  // fused greedy argmax (fp32 output only): per-row winning key, or null
    int32_t* am_tokens;
    unsigned int* am_counter;
    int32_t rope_on;       // 1: the epilogue applies RoPE and appends K/V (rope) instead of storing C
    RopeFuse rope;
    int32_t* status;
    uint64_t wait_ns;      // bound of every wait (2 s; shorter in the wait test)
    int32_t skip_stage;    // wait test: the ring stage (in issue order) whose copies are withheld, else -1
    int32_t norm_on;       // 1: A = bf16((x * rinv) * gamma) of x's first M rows (M <= kNormMaxM), A loads raw x
    const uint4* norm_x;   // [M.., K / 8]
    const uint4* norm_gamma;
    float norm_eps;
    const int32_t* norm_rows;  // the rows the caller means (must be 0..M-1), or null
};

// Rows up to which a GEMM may take its A operand through a fused RMSNorm:
// warps 2-3 then rescale every landed A stage of every output tile they visit
// in shared memory, M x 64 elements per K tile of the stage.
constexpr int64_t kNormMaxM = 8;

__device__ __forceinline__ float silu_mul(float g, float u) {
    const float s = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
    return __fmul_rn(s, u);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}


// Epilogue of one 64-column group (one MMA's worth) of one row: 64 fp32
// accumulators in r, output columns n0 .. n0+63 of the GEMM.
__device__ __forceinline__ void epilogue_group(const GemmArgs& args, int64_t row, int32_t n0, int32_t split,
                                               const uint32_t (&r)[4][16]) {
    if (args.ep == BI_EP_SWIGLU) {
        // columns 0..31 gate, 32..63 up of the same 32 hidden units
        uint32_t hv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c0 = 2 * i, c1 = 2 * i + 1;
            const float g0 = __uint_as_float(r[c0 / 16][c0 % 16]);
            const float g1 = __uint_as_float(r[c1 / 16][c1 % 16]);
            const float u0 = __uint_as_float(r[2 + c0 / 16][c0 % 16]);
            const float u1 = __uint_as_float(r[2 + c1 / 16][c1 % 16]);
            hv[i] = pack_bf16x2(silu_mul(g0, u0), silu_mul(g1, u1));
        }
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(args.C) + row * (args.N / 2) + n0 / 2);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
    } else if (args.c_f32) {
        float* dst = reinterpret_cast<float*>(args.C) + split * args.split_stride + row * args.N + n0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                reinterpret_cast<uint4*>(dst + c * 16)[i] =
                    make_uint4(r[c][4 * i], r[c][4 * i + 1], r[c][4 * i + 2], r[c][4 * i + 3]);
    } else {
        uint16_t* dst = reinterpret_cast<uint16_t*>(args.C) + row * args.N + n0;
        const uint16_t* res = args.ep == BI_EP_RESIDUAL ? args.residual + row * args.N + n0 : nullptr;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t rw[8];
            if (res) {
                const uint4 a = reinterpret_cast<const uint4*>(res + c * 16)[0];
                const uint4 b = reinterpret_cast<const uint4*>(res + c * 16)[1];
                rw[0] = a.x; rw[1] = a.y; rw[2] = a.z; rw[3] = a.w;
                rw[4] = b.x; rw[5] = b.y; rw[6] = b.z; rw[7] = b.w;
            }
            uint32_t ov[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float v0 = __uint_as_float(r[c][2 * i]);
                float v1 = __uint_as_float(r[c][2 * i + 1]);
                if (res) {
                    v0 = __fadd_rn(v0, bf16_lo(rw[i]));
                    v1 = __fadd_rn(v1, bf16_hi(rw[i]));
                }
                ov[i] = pack_bf16x2(v0, v1);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 16);
            d4[0] = make_uint4(ov[0], ov[1], ov[2], ov[3]);
            d4[1] = make_uint4(ov[4], ov[5], ov[6], ov[7]);
        }
    }
}

// Accumulator column (within a tile's TMEM buffer) of output column o of the
// tile.  A tile is one MMA wide (N = BN): in a pair, the MMA's first BN/2
// columns are the even CTA's W rows (the tile's first half) and the rest the
// odd CTA's, so in either form the column is o itself.
template <int BN, int CG>
__device__ __forceinline__ uint32_t acc_col(int32_t o) {
    return static_cast<uint32_t>(o);
}

// RoPE + KV append of one GEMM row (token), the arithmetic of rope_append_kernel: rotate-half pairs
// (i, i + Dh/2) of q and k heads as r0 = x0 c - x1 s, r1 = x1 c + x0 s in fp32, one bf16 rounding; q to q_out,
// k and v to the token's page slot.  The row's position and page are looked up once (bad ones reported).
struct RopeRow {
    bool ok;
    int32_t pos, page, slot;
    const float* crow;
    const float* srow;
};

__device__ __forceinline__ RopeRow rope_row(const GemmArgs& args, int64_t row, bool live) {
    const RopeFuse& rp = args.rope;
    RopeRow r{false, 0, 0, 0, nullptr, nullptr};
    if (live) {
        r.pos = rp.tok_pos[row];
        const int32_t req = rp.tok_req[row];
        r.ok = r.pos >= 0 && r.pos < rp.max_pos && (r.pos / BI_PAGE) < rp.max_pages;
        if (r.ok) {
            r.page = rp.page_table[static_cast<int64_t>(req) * rp.max_pages + r.pos / BI_PAGE];
            if (r.page < 0 || r.page >= rp.num_pages) {
                report(args.status, BI_DEV_BAD_PAGE);
                r.ok = false;
            }
        } else {
            report(args.status, BI_DEV_BAD_POSITION);
        }
    }
    const int32_t half = rp.Dh / 2;
    r.slot = r.pos & (BI_PAGE - 1);
    r.crow = rp.rc + static_cast<int64_t>(r.ok ? r.pos : 0) * half;
    r.srow = rp.rs + static_cast<int64_t>(r.ok ? r.pos : 0) * half;
    return r;
}

// Destination of one head of the row (q_out, or the K/V cache slot), or null (k/v of a row without a slot).
__device__ __forceinline__ uint16_t* rope_dst(const RopeFuse& rp, const RopeRow& rr, int64_t row, int32_t head) {
    if (head < rp.H) return rp.q_out + (row * rp.H + head) * rp.Dh;
    if (!rr.ok) return nullptr;
    const bool is_k = head < rp.H + rp.Hkv;
    const int32_t g = is_k ? head - rp.H : head - rp.H - rp.Hkv;
    return (is_k ? rp.kc : rp.vc) + ((static_cast<int64_t>(rr.page) * rp.Hkv + g) * BI_PAGE + rr.slot) * rp.Dh;
}

// Elements c .. c+15 of both halves of one head: ra = x[c..], rb = x[half + c..] (fp32 bits); rotated when rot
// (q and k heads), stored to d[c..] and d[half + c..].
__device__ __forceinline__ void rope_chunk16(const RopeRow& rr, int32_t half, int32_t c, bool rot,
                                             const uint32_t (&ra)[16], const uint32_t (&rb)[16], uint16_t* dst) {
    float cs16[16], sn16[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const float4 cv = rr.ok ? reinterpret_cast<const float4*>(rr.crow + c)[v] : make_float4(1.f, 1.f, 1.f, 1.f);
        const float4 sv = rr.ok ? reinterpret_cast<const float4*>(rr.srow + c)[v] : make_float4(0.f, 0.f, 0.f, 0.f);
        cs16[4 * v] = cv.x; cs16[4 * v + 1] = cv.y; cs16[4 * v + 2] = cv.z; cs16[4 * v + 3] = cv.w;
        sn16[4 * v] = sv.x; sn16[4 * v + 1] = sv.y; sn16[4 * v + 2] = sv.z; sn16[4 * v + 3] = sv.w;
    }
    uint32_t o0[8], o1[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
        float r0[2], r1[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float x0 = __uint_as_float(ra[e + u]), x1 = __uint_as_float(rb[e + u]);
            if (rot) {
                const float cs = cs16[e + u];
                const float sn = sn16[e + u];
                r0[u] = __fsub_rn(__fmul_rn(x0, cs), __fmul_rn(x1, sn));
                r1[u] = __fadd_rn(__fmul_rn(x1, cs), __fmul_rn(x0, sn));
            } else {
                r0[u] = x0;
                r1[u] = x1;
            }
        }
        o0[e / 2] = pack_bf16x2(r0[0], r0[1]);
        o1[e / 2] = pack_bf16x2(r1[0], r1[1]);
    }
    uint4* d0 = reinterpret_cast<uint4*>(dst + c);
    uint4* d1 = reinterpret_cast<uint4*>(dst + half + c);
    d0[0] = make_uint4(o0[0], o0[1], o0[2], o0[3]);
    d0[1] = make_uint4(o0[4], o0[5], o0[6], o0[7]);
    d1[0] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    d1[1] = make_uint4(o1[4], o1[5], o1[6], o1[7]);
}

// The row's heads of one tile from its TMEM lane.  Every lane loads (the TMEM loads are warp-wide); only
// rows < M store.
template <int BN, int CG>
__device__ __forceinline__ void rope_epilogue(const GemmArgs& args, uint32_t taddr, int64_t row, int32_t n_tile) {
    const RopeFuse& rp = args.rope;
    const int32_t Dh = rp.Dh, half = Dh / 2;
    const bool live = row < args.M;
    const RopeRow rr = rope_row(args, row, live);
#pragma unroll 1
    for (int32_t hs = 0; hs < BN / Dh; ++hs) {
        const int32_t head = (n_tile * BN + hs * Dh) / Dh;
        const bool rot = head < rp.H + rp.Hkv;
        uint16_t* dst = live ? rope_dst(rp, rr, row, head) : nullptr;
        const uint32_t ta = acc_col<BN, CG>(hs * Dh), tb = acc_col<BN, CG>(hs * Dh + half);
#pragma unroll 1
        for (int32_t c = 0; c < half; c += 16) {
            uint32_t ra[16], rb[16];
            ptx::tmem_ld16(taddr + ta + c, ra);
            ptx::tmem_ld16(taddr + tb + c, rb);
            ptx::tmem_ld_wait();
            if (dst != nullptr) rope_chunk16(rr, half, c, rot, ra, rb, dst);
        }
    }
}

// Fused RMSNorm: rinv of the rows r = wi, wi + 6, ... (< M) of x, one warp per row (wi = 0..5: warps 2-7 of
// the issuing CTA), in the RMSNorm kernel's order: lane l adds the squares of 16-byte chunks l, l + 32, ... in
// ascending element order with fused multiply-adds, the lane sums meet in an xor-butterfly (16, 8, 4, 2, 1),
// then rinv = 1 / sqrt(sum / K + eps).  A lane issues all its loads of a row before it uses any.
__device__ __forceinline__ void norm_rinv_rows(const GemmArgs& args, float* rinv_out, int wi) {
    const int lane = threadIdx.x & 31;
    const int32_t d8 = args.K / 8;
    constexpr int kMaxPerLane = 16;  // K <= 4096
    for (int32_t r = wi; r < args.M; r += 6) {
        const uint4* xr = args.norm_x + static_cast<int64_t>(r) * d8;
        uint4 v[kMaxPerLane];
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i)
            if (lane + 32 * i < d8) v[i] = xr[lane + 32 * i];
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            if (lane + 32 * i < d8) {
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
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
        const float mean = __fdiv_rn(ss, static_cast<float>(args.K));
        if (lane == 0) rinv_out[r] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, args.norm_eps)));
    }
}

// HALF: the CTA-pair MMA with M = 128 (64 rows of A and of the accumulator per CTA).  Its accumulator holds, in
// CTA c, lanes 0-63 = rows 64c + lane for the tile's first 64 columns and lanes 64-127 = the same rows for the
// last 64 (measured), so warp q's lanes are rows 64c + 32 (q % 2) + lane of column half q / 2.
template <int BN, int CG, bool HALF = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, GemmArgs args) {
    static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair");
    static_assert(!HALF || (CG == 2 && BN == kUN), "the half-row pair form has 128-wide tiles");
    constexpr int kRowsCta = HALF ? kBM / 2 : kBM;  // rows of A (and of the accumulator) in one CTA
    constexpr int kTileM = CG * kRowsCta;     // rows of a tile (the MMA's M)
    constexpr int kMmaN = BN;                  // one MMA per 16-deep step covers the tile (N = 128 or 256)
    constexpr int kGroups = BN / kMmaN;        // MMAs per 16-deep step
    constexpr int kWRows = BN / CG;            // W rows (output columns) this CTA holds per K tile
    constexpr int kWBytes = kWRows * kBK * 2;  // bytes of one K tile of W in this CTA
    constexpr int kChunks = BN / kEpi;         // epilogue chunks per tile
    constexpr uint32_t kTmemCols = 2 * BN;     // two accumulator buffers
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTileM, kMmaN);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // both CTAs of a pair use identical offsets: the MMA descriptors and the
    // cluster addresses below name the same offset in either CTA
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sW = smem + args.a_region;
    uint64_t* full = reinterpret_cast<uint64_t*>(sW + args.stages * args.kps * kWBytes);
    uint64_t* empty = full + kMaxStages;
    uint64_t* a_full = empty + kMaxStages;       // fused RMSNorm: the raw A rows of a stage landed
    uint64_t* acc_full = a_full + kMaxStages;    // [2]
    uint64_t* acc_empty = acc_full + 2;          // [2]
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ float norm_rinv[kNormMaxM];  // fused RMSNorm: each row's rinv
    int32_t* abort_word = reinterpret_cast<int32_t*>(tmem_holder + 1);
    volatile int32_t* abort_flag = abort_word;

    uint32_t rank = 0;  // 0: the CTA that issues the MMAs (the even CTA of a pair)
    if constexpr (CG == 2) rank = ptx::cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int32_t unit = static_cast<int32_t>(blockIdx.x) / CG;  // this CTA's pair (or the CTA itself)
    const int32_t nunits = static_cast<int32_t>(gridDim.x) / CG;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
    const int32_t split = blockIdx.y;
    const int32_t kb0 = split * args.kb_per_split;
    const int32_t nkb = min(args.kb_per_split, args.nkb_total - kb0);
    const int S = args.stages, kps = args.kps;

    auto tile_coords = [&](int32_t lin, int32_t& m_tile, int32_t& n_tile) {
        const int32_t band = kGroupM * args.n_tiles;
        const int32_t first_m = (lin / band) * kGroupM;
        const int32_t band_m = min(kGroupM, args.m_tiles - first_m);
        m_tile = first_m + (lin % band) % band_m;
        n_tile = (lin % band) / band_m;
    };
    // a role that gives up stops every CTA of the group
    auto raise_abort = [&]() {
        *abort_flag = 1;
        if constexpr (CG == 2) ptx::st_shared_cluster_u32(ptx::mapa_shared(smem_u32(abort_word), peer), 1u);
    };

    pdl_trigger();
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmW);
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], args.norm_on ? 2 : 1);  // + the A writers' arrival
            ptx::mbar_init(&empty[s], 1);
            ptx::mbar_init(&a_full[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 4 * CG);  // one arrival per epilogue warp of the group
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp >= 4) {
        // the A region starts zeroed: rows no TMA box covers read as zero
        uint4* z = reinterpret_cast<uint4*>(sA);
        for (int i = threadIdx.x - 128; i < args.a_region / 16; i += 128) z[i] = make_uint4(0, 0, 0, 0);
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0) {
        __syncwarp();
        ptx::tmem_alloc<CG>(tmem_holder, kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    if constexpr (CG == 2)
        ptx::cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
    else
        __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    bool tmem_ok = true;
    // a pair's MMAs write the even CTA's column address in both CTAs
    if constexpr (CG == 2) tmem_ok = ptx::ld_shared_cluster_u32(ptx::mapa_shared(smem_u32(tmem_holder), peer)) == tmem;
    if (!(warp == 0 && lane == 0)) pdl_wait();  // the producer waits in its role below

    if (!tmem_ok) {
        if (warp == 0 && lane == 0) {
            pdl_wait();
            if (rank == 0) report(args.status, BI_DEV_PAIR_TMEM);
        }
    } else if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer (every CTA): per stage one box of A and one of W, each kps K tiles deep ----
            const uint64_t pol_w = ptx::policy_evict_first();  // weights stream through once
            const uint64_t pol_a = ptx::policy_evict_last();   // activations are re-read by every N tile
            // boxes always land whole (out-of-range rows and K tiles are zero-filled); the
            // issuing CTA's full barrier counts the bytes of every CTA of the group
            const uint32_t stage_tx =
                static_cast<uint32_t>(CG * kps) * (static_cast<uint32_t>(args.norm_on ? 0 : args.a_stride) + kWBytes);
            const int32_t a_row0 = static_cast<int32_t>(rank) * kRowsCta;  // this CTA's rows of the tile
            const int32_t w_row0 = static_cast<int32_t>(rank) * kWRows;  // this CTA's W rows of the tile
            auto load = [&](void* dst, const CUtensorMap* map, int s_, int32_t y, int32_t z, uint64_t pol) {
                if constexpr (CG == 2)
                    ptx::tma_load_3d_pair(dst, map, ptx::mapa_shared(smem_u32(&full[s_]), 0), 0, y, z, pol);
                else
                    ptx::tma_load_3d(dst, map, &full[s_], 0, y, z, pol);
            };
            // A of a stage: counted with W on the group's full barrier, or (fused RMSNorm) the issuing CTA's raw
            // rows on a_full for the A writers, who then complete full themselves (the other CTA's rows lie
            // past M and keep their zeros)
            auto load_a = [&](int s_, int32_t y, int32_t z) {
                if (!args.norm_on) {
                    load(sA + s_ * kps * args.a_stride, &tmA, s_, y, z, pol_a);
                } else if (rank == 0) {
                    ptx::mbar_arrive_expect_tx(&a_full[s_], static_cast<uint32_t>(kps * args.a_stride));
                    ptx::tma_load_3d(sA + s_ * kps * args.a_stride, &tmA, &a_full[s_], 0, y, z, pol_a);
                }
            };
            // Weights do not depend on the kernel before this one: when the
            // caller guarantees that nothing still in flight writes them, the
            // first tile's first stages of W are requested before the
            // dependency wait and only A waits for the previous kernel.
            uint32_t pre = 0;
            if (args.w_early && unit < args.total_tiles) {
                int32_t m_tile, n_tile;
                tile_coords(unit, m_tile, n_tile);
                const int32_t first_stages = (nkb + kps - 1) / kps;
                pre = static_cast<uint32_t>(min(S, first_stages));
                for (uint32_t q = 0; q < pre; ++q) {
                    if (rank == 0) ptx::mbar_arrive_expect_tx(&full[q], stage_tx);
                    load(sW + q * kps * kWBytes, &tmW, static_cast<int>(q), n_tile * BN + w_row0,
                         kb0 + static_cast<int32_t>(q) * kps, pol_w);
                }
            }
            pdl_wait();
            uint32_t issued = 0;  // stages issued
            int s = 0;            // stage and its phase, advanced incrementally
            uint32_t ph = 0;
            bool ok = true;
            for (int32_t tile = unit; tile < args.total_tiles && ok; tile += nunits) {
                int32_t m_tile, n_tile;
                tile_coords(tile, m_tile, n_tile);
                const int32_t a_row = m_tile * kTileM + a_row0;
                for (int32_t kb = 0; kb < nkb; kb += kps) {
                    if (issued < pre) {
                        // armed, W already requested: only A is missing
                        load_a(s, a_row, kb0 + kb);
                    } else {
                        if (!ptx::mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag, args.wait_ns)) {
                            if (!*abort_flag) report(args.status, BI_DEV_TIMEOUT_PRODUCER);
                            raise_abort();
                            ok = false;
                            break;
                        }
                        if (static_cast<int32_t>(issued) != args.skip_stage) {
                            if (rank == 0) ptx::mbar_arrive_expect_tx(&full[s], stage_tx);
                            load_a(s, a_row, kb0 + kb);
                            load(sW + s * kps * kWBytes, &tmW, s, n_tile * BN + w_row0, kb0 + kb, pol_w);
                        }
                    }
                    ++issued;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // drain: every issued copy of the group lands on the issuing CTA's
            // barriers, and must land before any CTA of the group may exit
            if (rank == 0) {
                const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0u;
                for (uint32_t q = first; q < issued; ++q) {
                    const int qs = static_cast<int>(q % S);
                    const uint32_t qph = (q / S) & 1u;
                    const uint64_t t0 = globaltimer_ns();
                    while (!ptx::mbar_try_wait(smem_u32(&full[qs]), qph) ||
                           (args.norm_on && !ptx::mbar_try_wait(smem_u32(&a_full[qs]), qph))) {
                        if (globaltimer_ns() - t0 > args.wait_ns) {
                            report(args.status, BI_DEV_TIMEOUT_DRAIN);
                            break;
                        }
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---- MMA issuer (one thread of the issuing CTA) ----
            // Descriptors are built once; a slot or a 16-deep K step only moves
            // the start-address field (16-byte units; shared memory < 256 KB so
            // the 14-bit field never carries).
            const uint64_t a_desc0 = ptx::smem_desc_sw128(smem_u32(sA));
            const uint64_t w_desc0 = ptx::smem_desc_sw128(smem_u32(sW));
            const uint32_t a_step = static_cast<uint32_t>(args.a_stride) >> 4;
            constexpr uint32_t w_step = kWBytes >> 4;
            constexpr uint32_t g_step = ((kMmaN / CG) * kBK * 2) >> 4;  // the next MMA's W rows in each CTA
            int s = 0;
            uint32_t ph = 0;
            int32_t i = 0;
            bool ok = true;
            for (int32_t tile = unit; tile < args.total_tiles && ok; tile += nunits, ++i) {
                const int b = i & 1;
                if (!ptx::mbar_wait_bounded(&acc_empty[b], ((static_cast<uint32_t>(i) >> 1) & 1u) ^ 1u, abort_flag,
                                            args.wait_ns)) {
                    if (!*abort_flag) report(args.status, BI_DEV_TIMEOUT_MMA);
                    raise_abort();
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t acc = tmem + static_cast<uint32_t>(b * BN);
                for (int32_t kb = 0; kb < nkb; kb += kps) {
                    const int cnt = min(kps, nkb - kb);
                    if (!ptx::mbar_wait_bounded(&full[s], ph, abort_flag, args.wait_ns)) {
                        if (!*abort_flag) report(args.status, BI_DEV_TIMEOUT_MMA);
                        raise_abort();
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    for (int j = 0; j < cnt; ++j) {
                        const uint32_t slot = static_cast<uint32_t>(s * kps + j);
                        const uint64_t ad = a_desc0 + slot * a_step;
                        const uint64_t wd = w_desc0 + slot * w_step;
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
#pragma unroll
                            for (int g = 0; g < kGroups; ++g)
                                ptx::tc_mma_f16<CG>(acc + g * kMmaN, ad + 2u * k, wd + g * g_step + 2u * k, kIdesc,
                                                    (kb + j > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    ptx::tc_commit<CG>(&empty[s]);  // the stage is free (in every CTA) once read
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) ptx::tc_commit<CG>(&acc_full[b]);
            }
            // no MMA may be in flight when any CTA frees TMEM or exits
            ptx::tc_commit<CG>(drain);
        }
        if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!ptx::mbar_try_wait(smem_u32(drain), 0)) {
                if (globaltimer_ns() - t0 > args.wait_ns) {
                    report(args.status, BI_DEV_TIMEOUT_DRAIN);
                    break;
                }
            }
        }
    } else if ((warp == 2 || warp == 3) && args.norm_on && rank == 0) {
        // ---- A writers (fused RMSNorm): warps 2-3 of the issuing CTA; the tile's rows < M all lie in this
        // CTA's 128 rows (the pair's other CTA keeps its zeroed A region) ----
        norm_rinv_rows(args, norm_rinv, warp - 2);
        if (args.norm_rows != nullptr && blockIdx.x == 0 && threadIdx.x == 64) {
            // the fused norm reads x's first M rows: a caller's row list that says otherwise is reported
            for (int32_t r = 0; r < static_cast<int32_t>(args.M); ++r)
                if (args.norm_rows[r] != r) report(args.status, BI_DEV_BAD_LOGIT_ROWS);
        }
        asm volatile("bar.sync 2, 192;" ::: "memory");  // every row's rinv (warps 2-7)
        const int t = threadIdx.x - 64;  // 0..63
        const int32_t rows = static_cast<int32_t>(args.M);
        int s = 0;
        uint32_t ph = 0;
        for (int32_t tile = unit; tile < args.total_tiles; tile += nunits) {
            bool ok = true;
            for (int32_t kb = 0; kb < nkb; kb += kps) {
                if (!ptx::mbar_wait_bounded(&a_full[s], ph, abort_flag, args.wait_ns)) {
                    if (!*abort_flag) report(args.status, BI_DEV_TIMEOUT_PRODUCER);
                    raise_abort();
                    ok = false;
                    break;
                }
                // in place: chunk position p of row r of K tile j holds the 8 elements of chunk p ^ (r % 8)
                // (the 128-byte swizzle of the TMA box)
                const int32_t cnt = min(kps, nkb - kb);
                const int32_t total = rows * cnt * 8;
                uint8_t* stage_a = sA + s * kps * args.a_stride;
                constexpr int kIt = static_cast<int>(kNormMaxM) * 4 * 8 / 64;
                // passes of 64 * kIt cells over the stage (one pass for up to 4 K tiles of 8 rows); in each,
                // every read first, then the arithmetic and the writes
                for (int32_t base = 0; base < total; base += 64 * kIt) {
                    uint4 v[kIt], g[kIt];
                    uint4* cell[kIt];
                    float rinv[kIt];
#pragma unroll
                    for (int u = 0; u < kIt; ++u) {
                        const int32_t i = base + t + 64 * u;
                        if (i < total) {
                            const int32_t r = i / (cnt * 8), rem = i % (cnt * 8), j = rem / 8, pos = rem % 8;
                            cell[u] = reinterpret_cast<uint4*>(stage_a + j * args.a_stride + r * 128 + pos * 16);
                            v[u] = *cell[u];
                            g[u] = __ldg(args.norm_gamma + (kb0 + kb + j) * 8 + (pos ^ (r & 7)));
                            rinv[u] = norm_rinv[r];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kIt; ++u) {
                        if (base + t + 64 * u < total) {
                            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                            const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float x0 = __fmul_rn(__fmul_rn(bf16_lo(w[e]), rinv[u]), bf16_lo(gw[e]));
                                const float x1 = __fmul_rn(__fmul_rn(bf16_hi(w[e]), rinv[u]), bf16_hi(gw[e]));
                                o[e] = pack_bf16x2(x0, x1);
                            }
                            *cell[u] = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
                ptx::fence_proxy_async_smem();  // the generic writes before the MMAs (async proxy) read them
                asm volatile("bar.sync 3, 64;" ::: "memory");
                if (t == 0) mbar_arrive(&full[s]);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
        }
    } else if (warp >= 4) {
        // ---- epilogue: warps 4..7 of each CTA, on that CTA's 128 rows ----
        if (args.norm_on && rank == 0) {  // first, rinv of some rows for the A writers
            norm_rinv_rows(args, norm_rinv, warp - 2);
            asm volatile("bar.sync 2, 192;" ::: "memory");
        }
        const int q = warp & 3;
        int32_t i = 0;
        for (int32_t tile = unit; tile < args.total_tiles; tile += nunits, ++i) {
            const int b = i & 1;
            int32_t m_tile, n_tile;
            tile_coords(tile, m_tile, n_tile);
            const int64_t row = HALF ? static_cast<int64_t>(m_tile) * kTileM + rank * kRowsCta + (q & 1) * 32 + lane
                                     : static_cast<int64_t>(m_tile) * kTileM + rank * kBM + q * 32 + lane;
            if (args.rope_on && row < args.M) {
                // the row's cos/sin table rows are read after the MMAs: fetch them into L1 meanwhile
                const int32_t pos = args.rope.tok_pos[row];
                if (pos >= 0 && pos < args.rope.max_pos) {
                    const int32_t half = args.rope.Dh / 2;
                    const char* cp = reinterpret_cast<const char*>(args.rope.rc + static_cast<int64_t>(pos) * half);
                    const char* sp = reinterpret_cast<const char*>(args.rope.rs + static_cast<int64_t>(pos) * half);
                    for (int32_t o = 0; o < half * 4; o += 128) {
                        asm volatile("prefetch.global.L1 [%0];" ::"l"(cp + o));
                        asm volatile("prefetch.global.L1 [%0];" ::"l"(sp + o));
                    }
                }
            }
            const bool ready =
                ptx::mbar_wait_bounded(&acc_full[b], (static_cast<uint32_t>(i) >> 1) & 1u, abort_flag, args.wait_ns);
            if (!ready && !*abort_flag) report(args.status, BI_DEV_TIMEOUT_EPILOGUE);
            if (!__all_sync(0xffffffffu, ready && !*abort_flag)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN);
            unsigned long long best = kArgmaxKeyNone;
            if (args.rope_on) rope_epilogue<BN, CG>(args, taddr, row, n_tile);
#pragma unroll 1
            for (int j = 0; j < (args.rope_on ? 0 : (HALF ? 1 : kChunks)); ++j) {
                uint32_t r[4][16];
#pragma unroll
                for (int c = 0; c < 4; ++c) ptx::tmem_ld16(taddr + j * kEpi + c * 16, r[c]);
                ptx::tmem_ld_wait();
                // accumulator columns 64j..64j+63 are the tile's output columns 64j.. (half form: this warp's
                // lanes hold column half q / 2 in accumulator columns 0-63)
                const int32_t n0 = HALF ? n_tile * BN + (q >> 1) * kEpi : n_tile * BN + j * kEpi;
                if (row < args.M && args.C != nullptr) epilogue_group(args, row, n0, split, r);
                if (args.am_keys != nullptr) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const unsigned long long key = argmax_key(__uint_as_float(r[c][e]), n0 + c * 16 + e);
                            best = key < best ? key : best;
                        }
                }
            }
            if (args.am_keys != nullptr && row < args.M) atomicMin(args.am_keys + row, best);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0)
                    mbar_arrive(&acc_empty[b]);
                else
                    ptx::mbar_arrive_cluster(ptx::mapa_shared(smem_u32(&acc_empty[b]), 0));
            }
        }
    }

    // teardown: MMAs drained (every CTA saw the drain commit), copies drained
    // by the issuing CTA's producer; after the (cluster) barrier no CTA
    // touches another's shared or tensor memory
    if (args.am_keys != nullptr) __threadfence();  // this CTA's argmax keys before its count below
    ptx::tc_fence_before();
    if constexpr (CG == 2)
        ptx::cluster_sync();
    else
        __syncthreads();
    if (warp == 0) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc<CG>(tmem, kTmemCols);
    }
    if (args.am_keys != nullptr) {
        // the last CTA to finish turns every row's key into its token id
        __shared__ uint32_t am_last;
        if (threadIdx.x == 0) {
            const unsigned int done = atomicAdd(args.am_counter, 1u);
            am_last = done == gridDim.x * gridDim.y - 1u ? 1u : 0u;
        }
        __syncthreads();
        if (am_last) {
            __threadfence();
            for (int64_t r = threadIdx.x; r < args.M; r += blockDim.x)
                args.am_tokens[r] = static_cast<int32_t>(__ldcg(args.am_keys + r) & 0xffffffffull);
            if (threadIdx.x == 0) *args.am_counter = 0u;
        }
    }
}

// Split-K reduction (variant mode): partials added in split order, then the epilogue.
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int32_t splits, int64_t split_stride, int64_t M,
                                     int32_t N, void* C, int32_t c_f32, const uint16_t* residual, int32_t ep) {
    pdl_trigger();
    pdl_wait();
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (ep == BI_EP_SWIGLU) {
        const int32_t nout = N / 2;
        if (idx >= M * nout) return;
        const int64_t row = idx / nout;
        const int32_t c = static_cast<int32_t>(idx % nout);
        const int32_t gcol = (c / 32) * 64 + (c % 32), ucol = gcol + 32;
        float g = ws[row * N + gcol], u = ws[row * N + ucol];
        for (int s = 1; s < splits; ++s) {
            g = __fadd_rn(g, ws[s * split_stride + row * N + gcol]);
            u = __fadd_rn(u, ws[s * split_stride + row * N + ucol]);
        }
        reinterpret_cast<uint16_t*>(C)[row * nout + c] = f32_to_bf16(silu_mul(g, u));
        return;
    }
    if (idx >= M * N) return;
    float a = ws[idx];
    for (int s = 1; s < splits; ++s) a = __fadd_rn(a, ws[s * split_stride + idx]);
    if (c_f32) {
        reinterpret_cast<float*>(C)[idx] = a;
    } else {
        if (ep == BI_EP_RESIDUAL) a = __fadd_rn(a, bf16_to_f32(residual[idx]));
        reinterpret_cast<uint16_t*>(C)[idx] = f32_to_bf16(a);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major [rows, K] bf16 matrix seen as three dimensions (64 elements of a
// K tile, row, K tile), so that one box of (64, box_rows, depth) brings
// `depth` consecutive K tiles of box_rows rows, each tile laid out as rows of
// 128 bytes with the 128-byte swizzle (the layout the MMA descriptors read).
// One large copy per operand and ring stage keeps enough bytes in flight per
// SM; small copies are limited by how fast one thread can re-arm and issue.
static bool make_kslab_map(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows,
                           uint32_t depth) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kBK), rows, K / kBK};
    cuuint64_t strides[2] = {K * 2, static_cast<cuuint64_t>(kBK) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), box_rows, depth};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_kv_map(CUtensorMap* map, const bi_bf16* cache, int64_t num_pages, int32_t Hkv, int32_t Dh) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(Dh), static_cast<cuuint64_t>(num_pages) * Hkv * BI_PAGE};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(Dh) * 2};
    cuuint32_t box[2] = {64, BI_PAGE};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bi_bf16*>(cache), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap* map, const bi_bf16* q, int64_t rows, int32_t H, int32_t Dh, int32_t G) {
    auto fn = encode_fn();
    if (!fn || G <= 0 || 128 % G != 0 || rows <= 0) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(Dh), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(Dh) * 2, static_cast<cuuint64_t>(H) * Dh * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(128 / G)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<bi_bf16*>(q), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

GemmPlan gemm_plan(int64_t M, int32_t N, int32_t K, bi_mode mode) {
    GemmPlan p{1};
    if (mode != BI_VARIANT || M <= 0) return p;
    const int64_t tiles = ((M + kBM - 1) / kBM) * (N / kUN);
    const int sms = num_sms();
    if (tiles >= sms) return p;
    const int32_t nkb = K / kBK;
    int64_t s = sms / tiles;
    if (s > nkb / 4) s = nkb / 4;
    if (s > 16) s = 16;
    if (s < 1) s = 1;
    const int32_t per = static_cast<int32_t>((nkb + s - 1) / s);
    p.splits = (nkb + per - 1) / per;
    return p;
}

size_t gemm_ws_bytes(int64_t M, int32_t N, int32_t K, bi_mode mode) {
    const GemmPlan p = gemm_plan(M, N, K, mode);
    if (p.splits <= 1) return 0;
    return static_cast<size_t>(p.splits) * static_cast<size_t>(M) * N * sizeof(float) + 256;
}

namespace {

struct Layout {
    int32_t cg, bn, a_box, a_stride, a_region, stages, kps;
    bool half;  // CTA-pair MMA with M = 128: 64 rows per CTA
    size_t smem;
};

// The MMA instruction form: weight matrices up to kPairMaxN columns have few
// enough 128-wide output tiles that a tile must be spread over two SMs to use
// the GPU, and take the pair form (256x128x16 over two SMs, 2 KB of weights
// per SM per MMA); wider ones (a vocabulary projection) fill every SM many
// times over and are bound by how fast the tensor cores consume weights,
// which the single-CTA form (128x128x16, 4 KB of weights per MMA) does faster.
constexpr int32_t kPairMaxN = 65536;
// The two forms give every element the same bits (tested: the same product
// through either form, bit for bit, at decode and prefill sizes), so the
// choice is data movement like the tile width.  (Taking the single-CTA form
// for the gate/up projection at decode sizes, whose 224 tiles fill every SM,
// was measured no faster: ~50 us either way at M = 64.)
int mma_group(int32_t N) { return N <= kPairMaxN ? 2 : 1; }

// Rows up to which the pair form takes 8 K tiles per ring stage (below).
constexpr int64_t kDeepStageMaxM = 16;

// Layout of one launch.  Only data movement depends on M here; the MMA
// sequence of every output element is the same for all layouts.
// Rows up to which a pair-form product with 128-wide tiles takes the half-row pair MMA (M = 128: 64 rows of A
// per CTA).  Each CTA's tensor core then reads 64 rows of A per MMA instead of 128, most of them padding at
// decode sizes; the per-element arithmetic is the same (tested bit for bit against the full pair form).
constexpr int64_t kHalfMaxM = 64;

Layout choose_layout(int64_t M, int32_t N, int32_t K, bool half_ok) {
    Layout L{};
    L.cg = mma_group(N);
    // 256-wide tiles (one 256-wide MMA per step: half the A re-reads from L2
    // and from shared memory) for M > 256; for fewer rows 128-wide tiles
    // spread the output over twice the tiles
    L.bn = (M > 2 * kBM && N % 256 == 0) ? 256 : kUN;
    L.half = half_ok && L.cg == 2 && L.bn == kUN && M <= kHalfMaxM;
    const int32_t rows_cta = L.half ? kBM / 2 : kBM;  // rows of A the MMA reads in one CTA
    int32_t box = 16;
    while (box < rows_cta && box < M) box *= 2;
    L.a_box = box;
    L.a_stride = box * kBK * 2;
    const int32_t w_tile = (L.bn / L.cg) * kBK * 2;  // one K tile of this CTA's W rows
    const int32_t pad = rows_cta * kBK * 2 - L.a_stride;  // the last slot's MMA window reaches this far past it
    const int32_t budget = kRingBudget - pad;
    const int32_t per_k = L.a_stride + w_tile;  // bytes of one K tile of A and W
    // deep stages (one large copy per operand) while at least two still fit
    // (few rows: 8 K tiles per stage in the pair form.  One SM's copy engine handles a few boxes per
    // microsecond whatever their size up to tens of KB, so with 16-row A boxes the larger stages bring the
    // weights in faster: measured 310 / 316 / 337 us per decode step at 1 / 4 / 8 tokens against 318 / 325 /
    // 344 with 4 K tiles, and no better with 5-7; with more rows the A boxes grow and 4 stays best)
    L.kps = std::max(1, std::min({L.bn == 256 ? 2 : (L.cg == 2 && M <= kDeepStageMaxM ? 8 : 4), K / kBK,
                                  budget / (2 * per_k)}));
    int32_t stages = budget / (L.kps * per_k);
    stages = std::min(std::max(stages, 2), kMaxStages);
    L.stages = stages;
    L.a_region = stages * L.kps * L.a_stride + pad;
    L.smem = 1024 + static_cast<size_t>(L.a_region) + static_cast<size_t>(stages) * L.kps * w_tile + kBarrierBytes;
    return L;
}

template <int BN, int CG, bool HALF = false>
cudaError_t prepare_tiles() {
    static_assert(BN % kUN == 0, "a tile is a whole number of MMAs wide");
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(gemm_tc_kernel<BN, CG, HALF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kMaxSmem);
    });
    return err;
}

// Pairs of CTAs that fit on the GPU at once (one CTA per SM).
int resident_pairs() {
    static int pairs = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int n = 0;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kGemmThreads);
        cfg.dynamicSmemBytes = kMaxSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (prepare_tiles<kUN, 2>() != cudaSuccess ||
            cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<kUN, 2>, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = num_sms() / 2;
        }
        pairs = std::max(1, std::min(n, num_sms() / 2));
    });
    return pairs;
}

// Units (pairs or CTAs) launched: one per tile up to what fits at once.
template <int BN, int CG, bool HALF = false>
cudaError_t launch_tiles(const CUtensorMap& tmA, const CUtensorMap& tmW, const GemmArgs& a, int64_t tiles,
                         int splits, size_t smem, cudaStream_t s) {
    cudaError_t e = prepare_tiles<BN, CG, HALF>();
    if (e != cudaSuccess) return e;
    if constexpr (CG == 2) {
        const int64_t pairs = std::min<int64_t>(tiles, std::max(1, resident_pairs() / splits));
        return launch_pair_pdl(gemm_tc_kernel<BN, CG, HALF>, dim3(static_cast<unsigned>(2 * pairs), splits),
                               dim3(kGemmThreads), smem, s, tmA, tmW, a);
    } else {
        const int64_t ctas = std::min<int64_t>(tiles, std::max(1, num_sms() / splits));
        return launch_pdl(gemm_tc_kernel<BN, CG>, dim3(static_cast<unsigned>(ctas), splits), dim3(kGemmThreads),
                          smem, s, tmA, tmW, a);
    }
}

}  // namespace

bool gemm_can_fuse_rope(int64_t M, int32_t N, int32_t K, bi_mode mode, int32_t Dh) {
    // tiles (128 or 256 columns, at multiples of their width) then hold whole heads
    return M > 0 && N > 0 && gemm_plan(M, N, K, mode).splits == 1 && (Dh == 64 || Dh == 128);
}

bool gemm_can_fuse_norm(int64_t M, int32_t N, int32_t K, bi_mode mode) {
    return M > 0 && M <= kNormMaxM && N > 0 && K % kBK == 0 && K <= 4096 && gemm_plan(M, N, K, mode).splits == 1;
}

bi_status run_gemm(const bi_bf16* A, const bi_bf16* W, void* C, bi_dtype c_dtype, const bi_bf16* residual,
                   bi_epilogue ep, int64_t M, int32_t N, int32_t K, bi_mode mode, void* ws, size_t ws_bytes,
                   int32_t* status, cudaStream_t s, bool weights_settled, const ArgmaxFuse* am,
                   const RopeFuse* rope, const GemmWaitTest* wait_test, const NormFuse* norm) {
    if (M == 0) return BI_OK;
    if (norm != nullptr) {
        if (!gemm_can_fuse_norm(M, N, K, mode) || wait_test != nullptr)
            return fail(BI_ERR_INVALID, "fused RMSNorm needs at most 8 rows, K <= 4096 and no split-K");
        A = norm->x;  // the A ring receives the raw rows
    }
    const GemmPlan plan = gemm_plan(M, N, K, mode);
    // (the fused RoPE rotates pairs (i, i + Dh/2) of one row, which the half-row form puts in two warps)
    const Layout L = choose_layout(M, N, K, rope == nullptr);

    if (L.smem > static_cast<size_t>(kMaxSmem)) return fail(BI_ERR_UNSUPPORTED, "bi_gemm: no ring layout fits");
    const int32_t nkb = K / kBK;
    const int32_t per = (nkb + plan.splits - 1) / plan.splits;
    CUtensorMap tmA, tmW;
    if (!make_kslab_map(&tmA, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), static_cast<uint32_t>(L.a_box),
                        static_cast<uint32_t>(L.kps)) ||
        !make_kslab_map(&tmW, W, static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                        static_cast<uint32_t>(L.bn / L.cg), static_cast<uint32_t>(L.kps)))
        return fail(BI_ERR_CUDA, "cuTensorMapEncodeTiled failed");

    GemmArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.kb_per_split = per;
    a.nkb_total = nkb;
    const int64_t tile_m = L.half ? kBM : static_cast<int64_t>(L.cg) * kBM;
    a.m_tiles = static_cast<int32_t>((M + tile_m - 1) / tile_m);
    a.n_tiles = N / L.bn;
    a.a_box_rows = L.a_box;
    a.a_stride = L.a_stride;
    a.a_region = L.a_region;
    a.stages = L.stages;
    a.kps = L.kps;
    a.w_early = weights_settled && wait_test == nullptr ? 1 : 0;
    a.status = status;
    a.wait_ns = wait_test != nullptr ? wait_test->wait_ns : kWaitLimitNs;
    a.skip_stage = wait_test != nullptr ? wait_test->skip_stage : -1;
    if (norm != nullptr) {
        a.norm_on = 1;
        a.norm_x = reinterpret_cast<const uint4*>(norm->x);
        a.norm_gamma = reinterpret_cast<const uint4*>(norm->gamma);
        a.norm_eps = norm->eps;
        a.norm_rows = norm->rows;
    }
    if (rope != nullptr) {
        if (!gemm_can_fuse_rope(M, N, K, mode, rope->Dh) || am != nullptr || ep != BI_EP_NONE ||
            N != (rope->H + 2 * rope->Hkv) * rope->Dh)
            return fail(BI_ERR_INVALID, "fused RoPE needs a pair-form QKV GEMM without split-K or other epilogue");
        a.rope_on = 1;
        a.rope = *rope;
    } else if (am != nullptr) {
        if (plan.splits != 1 || c_dtype != BI_F32 || ep != BI_EP_NONE)
            return fail(BI_ERR_INVALID, "fused argmax needs an fp32 GEMM without epilogue or split-K");
        a.am_keys = am->keys;
        a.am_tokens = am->tokens;
        a.am_counter = am->counter;
    } else if (C == nullptr) {
        return fail(BI_ERR_INVALID, "bi_gemm: null output");
    }
    if (plan.splits > 1) {
        if (ws == nullptr || ws_bytes < gemm_ws_bytes(M, N, K, mode) || (reinterpret_cast<uintptr_t>(ws) & 15u))
            return fail(BI_ERR_WORKSPACE, "bi_gemm: variant split-K workspace too small or not 16-byte aligned");
        a.C = ws;
        a.c_f32 = 1;
        a.ep = BI_EP_NONE;
        a.residual = nullptr;
        a.split_stride = M * N;
    } else {
        a.C = C;
        a.c_f32 = c_dtype == BI_F32;
        a.ep = ep;
        a.residual = reinterpret_cast<const uint16_t*>(residual);
        a.split_stride = 0;
    }
    const int64_t tiles = static_cast<int64_t>(a.m_tiles) * a.n_tiles;
    if (tiles > 0x7fffffffLL) return fail(BI_ERR_SHAPE, "bi_gemm: too many tiles");
    a.total_tiles = static_cast<int32_t>(tiles);
    cudaError_t e;
    if (L.cg == 2)
        e = L.bn == 256 ? launch_tiles<256, 2>(tmA, tmW, a, tiles, plan.splits, L.smem, s)
            : L.half    ? launch_tiles<kUN, 2, true>(tmA, tmW, a, tiles, plan.splits, L.smem, s)
                        : launch_tiles<kUN, 2>(tmA, tmW, a, tiles, plan.splits, L.smem, s);
    else
        e = L.bn == 256 ? launch_tiles<256, 1>(tmA, tmW, a, tiles, plan.splits, L.smem, s)
                        : launch_tiles<kUN, 1>(tmA, tmW, a, tiles, plan.splits, L.smem, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm_tc_kernel launch");
    if (plan.splits > 1) {
        const int64_t n_out = ep == BI_EP_SWIGLU ? M * (N / 2) : M * N;
        const int threads = 256;
        const int64_t blocks = (n_out + threads - 1) / threads;
        e = launch_pdl(splitk_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s,
                       static_cast<const float*>(ws), plan.splits, M * N, M, N, C, static_cast<int32_t>(c_dtype == BI_F32),
                       reinterpret_cast<const uint16_t*>(residual), static_cast<int32_t>(ep));
        if (e != cudaSuccess) return cuda_fail(e, "splitk_reduce_kernel launch");
    }
    return BI_OK;
}

}  // namespace bi
