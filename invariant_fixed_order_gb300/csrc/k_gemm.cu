// Batch-invariant GEMM on the 5th-generation tensor cores.
//
// "Batch invariance and reproducible inference", "2 · Cross-block
// accumulation" and "3 · Kernel selection changing with shape": split-K and
// M-dependent tile choice are what make a GEMM's per-element order follow the
// batch.  Here every M runs the same configuration: 128-row M tiles, 64-column
// N tiles, 64-deep K tiles loaded by TMA with 128-byte swizzle, and one
// tcgen05.mma shape (M=128, N=64, K=16, bf16 in, fp32 accumulate in TMEM).  An
// output element's K sum is always: K tiles in ascending order, within a tile
// the four 16-deep MMAs in ascending order, accumulated in place in TMEM.
// Nothing in that sequence depends on M, on the position of the row inside its
// tile or on the other rows.
//
// Warp roles (192 threads): warp 0 issues TMA loads into a ring of shared-
// memory stages and owns the TMEM allocation; warp 1 issues the MMAs; warps
// 2-5 read the accumulator back (warp w reads TMEM lanes 32*(w%4)..+31, i.e.
// rows of the tile) and apply the fused epilogue.  Every wait is bounded: a
// wait that runs out sets an abort flag and a device status code, every role
// then winds down, in-flight copies and MMAs are drained, TMEM is freed.
//
// BI_VARIANT splits K over CTAs into an fp32 workspace when the output has
// fewer tiles than SMs (the fast path for small M) and adds the partials in
// split order in a second kernel: deterministic run to run, but its order
// depends on M.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace bi {

constexpr int kBM = BI_GEMM_BLOCK_M;   // 128
constexpr int kBN = BI_GEMM_UMMA_N;    // 64
constexpr int kBK = BI_GEMM_BLOCK_K;   // 64
constexpr int kStages = 8;
constexpr int kGemmThreads = 192;
constexpr int kABytes = kBM * kBK * 2;                // 16 KB
constexpr int kBBytes = kBN * kBK * 2;                // 8 KB
constexpr int kStageBytes = kABytes + kBBytes;        // 24 KB
constexpr int kTmemCols = 64;                         // fp32 accumulator columns
constexpr int kGroupM = 16;                           // M tiles per rasterisation band
constexpr size_t kGemmSmem = 1024 + static_cast<size_t>(kStages) * kStageBytes + 256;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBM, kBN);

struct GemmArgs {
    void* C;
    const uint16_t* residual;
    int64_t M;
    int32_t N, K;
    int32_t c_f32;
    int32_t ep;
    int32_t kb_per_split;
    int32_t nkb_total;
    int32_t m_tiles, n_tiles;
    int64_t split_stride;  // elements between split partials (fp32), variant only
    int32_t* status;
};

__device__ __forceinline__ float silu_mul(float g, float u) {
    const float s = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
    return __fmul_rn(s, u);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, GemmArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* accum = empty + kStages;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(accum + 1);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_holder + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;

    // grouped rasterisation: bands of kGroupM M tiles sweep the N tiles together
    const int32_t lin = blockIdx.x;
    const int32_t band = kGroupM * args.n_tiles;
    const int32_t first_m = (lin / band) * kGroupM;
    const int32_t band_m = min(kGroupM, args.m_tiles - first_m);
    const int32_t m_tile = first_m + (lin % band) % band_m;
    const int32_t n_tile = (lin % band) / band_m;
    const int32_t split = blockIdx.y;
    const int32_t kb0 = split * args.kb_per_split;
    const int32_t nkb = min(args.kb_per_split, args.nkb_total - kb0);

    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmW);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(accum, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0) {
        __syncwarp();
        ptx::tmem_alloc(tmem_holder, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer ----
            const uint64_t pol_w = ptx::policy_evict_first();  // weights stream through once
            const uint64_t pol_a = ptx::policy_evict_last();   // activations are re-read by every N tile
            int32_t last_phase[kStages];
            for (int s = 0; s < kStages; ++s) last_phase[s] = -1;
            for (int32_t kb = 0; kb < nkb; ++kb) {
                const int s = kb % kStages;
                const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
                if (!ptx::mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) {
                    if (!*abort_flag) report(args.status, BI_DEV_TIMEOUT_PRODUCER);
                    *abort_flag = 1;
                    break;
                }
                uint8_t* sa = smem + s * kStageBytes;
                ptx::mbar_arrive_expect_tx(&full[s], kStageBytes);
                const int32_t kx = (kb0 + kb) * kBK;
                ptx::tma_load_2d(sa, &tmA, &full[s], kx, m_tile * kBM, pol_a);
                ptx::tma_load_2d(sa + kABytes, &tmW, &full[s], kx, n_tile * kBN, pol_w);
                last_phase[s] = static_cast<int32_t>(ph);
            }
            // drain: every issued copy must land before the CTA may exit
            for (int s = 0; s < kStages; ++s) {
                if (last_phase[s] >= 0 &&
                    !ptx::mbar_wait_bounded(&full[s], static_cast<uint32_t>(last_phase[s]), abort_flag)) {
                    // the wait above also returns early on abort: wait once more without the abort exit
                    const uint64_t t0 = globaltimer_ns();
                    while (!ptx::mbar_try_wait(smem_u32(&full[s]), static_cast<uint32_t>(last_phase[s]))) {
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            report(args.status, BI_DEV_TIMEOUT_DRAIN);
                            break;
                        }
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer ----
            for (int32_t kb = 0; kb < nkb; ++kb) {
                const int s = kb % kStages;
                const uint32_t ph = static_cast<uint32_t>(kb / kStages) & 1u;
                if (!ptx::mbar_wait_bounded(&full[s], ph, abort_flag)) {
                    if (!*abort_flag) report(args.status, BI_DEV_TIMEOUT_MMA);
                    *abort_flag = 1;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * kStageBytes);
                const uint32_t sb = sa + kABytes;
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {
                    const uint64_t ad = ptx::smem_desc_sw128(sa + k * 32);
                    const uint64_t bd = ptx::smem_desc_sw128(sb + k * 32);
                    ptx::tc_mma_f16(tmem, ad, bd, kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
                }
                ptx::tc_commit(&empty[s]);  // stage s is free once these MMAs have read it
            }
            ptx::tc_commit(accum);  // always: the epilogue and teardown wait on it
        }
    } else {
        // ---- epilogue: warps 2..5 ----
        const int q = warp & 3;
        const int64_t row = static_cast<int64_t>(m_tile) * kBM + q * 32 + lane;
        const bool ready = ptx::mbar_wait_bounded(accum, 0, abort_flag);
        if (!ready && !*abort_flag) report(args.status, BI_DEV_TIMEOUT_EPILOGUE);
        const bool go = __all_sync(0xffffffffu, ready && !*abort_flag && nkb > 0);
        if (go) {
            ptx::tc_fence_after();
            uint32_t r[4][16];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld16(taddr + c * 16, r[c]);
            ptx::tmem_ld_wait();
            if (row < args.M) {
                const int32_t col0 = n_tile * kBN;
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
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(args.C) +
                                                          row * (args.N / 2) + col0 / 2);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
                } else if (args.c_f32) {
                    float* dst = reinterpret_cast<float*>(args.C) + split * args.split_stride + row * args.N + col0;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            reinterpret_cast<uint4*>(dst + c * 16)[i] =
                                make_uint4(r[c][4 * i], r[c][4 * i + 1], r[c][4 * i + 2], r[c][4 * i + 3]);
                } else {
                    uint16_t* dst = reinterpret_cast<uint16_t*>(args.C) + row * args.N + col0;
                    const uint16_t* res = args.ep == BI_EP_RESIDUAL ? args.residual + row * args.N + col0 : nullptr;
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
        }
    }

    // teardown: all MMAs have completed once `accum` fired (or its wait gave
    // up); warp 0 frees TMEM.
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// Split-K reduction (variant mode): partials added in split order, then the epilogue.
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int32_t splits, int64_t split_stride, int64_t M,
                                     int32_t N, void* C, int32_t c_f32, const uint16_t* residual, int32_t ep) {
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

// Row-major [rows, K] bf16 matrix, box of box_rows x 64 with 128-byte swizzle.
static bool make_kmajor_map(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {K * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

GemmPlan gemm_plan(int64_t M, int32_t N, int32_t K, bi_mode mode) {
    GemmPlan p{1};
    if (mode != BI_VARIANT || M <= 0) return p;
    const int64_t tiles = ((M + kBM - 1) / kBM) * (N / kBN);
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

bi_status run_gemm(const bi_bf16* A, const bi_bf16* W, void* C, bi_dtype c_dtype, const bi_bf16* residual,
                   bi_epilogue ep, int64_t M, int32_t N, int32_t K, bi_mode mode, void* ws, size_t ws_bytes,
                   int32_t* status, cudaStream_t s) {
    if (M == 0) return BI_OK;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kGemmSmem));
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(gemm)");

    const GemmPlan plan = gemm_plan(M, N, K, mode);
    const int32_t nkb = K / kBK;
    const int32_t per = (nkb + plan.splits - 1) / plan.splits;
    CUtensorMap tmA, tmW;
    if (!make_kmajor_map(&tmA, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M), kBM) ||
        !make_kmajor_map(&tmW, W, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kBN))
        return fail(BI_ERR_CUDA, "cuTensorMapEncodeTiled failed");

    GemmArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.kb_per_split = per;
    a.nkb_total = nkb;
    a.m_tiles = static_cast<int32_t>((M + kBM - 1) / kBM);
    a.n_tiles = N / kBN;
    a.status = status;
    if (plan.splits > 1) {
        if (ws == nullptr || ws_bytes < gemm_ws_bytes(M, N, K, mode))
            return fail(BI_ERR_WORKSPACE, "bi_gemm: variant split-K workspace too small");
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
    dim3 grid(static_cast<unsigned>(tiles), plan.splits);
    gemm_tc_kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(tmA, tmW, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "gemm_tc_kernel launch");
    if (plan.splits > 1) {
        const int64_t n_out = ep == BI_EP_SWIGLU ? M * (N / 2) : M * N;
        const int threads = 256;
        const int64_t blocks = (n_out + threads - 1) / threads;
        splitk_reduce_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
            reinterpret_cast<const float*>(ws), plan.splits, M * N, M, N, C, c_dtype == BI_F32,
            reinterpret_cast<const uint16_t*>(residual), ep);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "splitk_reduce_kernel launch");
    }
    return BI_OK;
}

}  // namespace bi
