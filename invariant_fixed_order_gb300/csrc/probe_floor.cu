// Microbenchmarks behind the tensor-core GEMM's layout choices.  Not part of
// libbi: built beside it as libbi_probe.so and run by `bench.py --floor`.
//
//   bip_mma_ns   time per tcgen05.mma.kind::f16 instruction of one form
//                (single CTA, M = 64 or 128; CTA pair, M = 128 or 256), with both
//                operands resident in shared memory and the issue loop fully
//                unrolled: a chain into one accumulator, or alternating over
//                independent accumulators (each its own chain);
//   bip_ingest   how fast CTAs, one per SM, take in a stream from global
//                memory: TMA 2-D boxes of 128 rows x 128 bytes (contiguous),
//                1-D bulk copies of 16 KB, or TMA 3-D boxes shaped as the
//                GEMM's weight ring (64 rows x 4 K tiles of 64 bf16, rows of
//                one long matrix, 128-byte swizzle).
//
// Every wait is bounded (2 s against microseconds of work).  A wait that runs
// out is reported; the MMA probe then leaves its tensor memory allocated
// rather than free it under MMAs that may still run (the calling process is
// expected to end), and the copy probe waits, bounded again, for its copies
// in flight before it returns.
#include <cudaTypedefs.h>

#include <vector>

#include "internal.h"
#include "tc_ptx.cuh"

namespace bi {
namespace probe {

constexpr int kTile = 128 * 128;  // one 128-row, 64-deep bf16 K tile with the 128-byte swizzle (16 KB)
constexpr int kKT = 4;            // resident K tiles of each operand
constexpr int kMmaSmem = 2 * kKT * kTile + 2048;
constexpr uint64_t kLimitNs = 2000000000ull;

template <int CG, int NACC>
__global__ void __launch_bounds__(128, 1)
    mma_kernel(uint32_t idesc, int32_t ncols, int32_t iters, unsigned long long* ns, int32_t* err) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = sm;
    uint8_t* sB = sm + kKT * kTile;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sB + kKT * kTile);
    uint32_t* holder = reinterpret_cast<uint32_t*>(bar + 1);
    int32_t* ok_word = reinterpret_cast<int32_t*>(holder + 1);
    const int warp = threadIdx.x / 32;
    uint32_t rank = 0;
    if constexpr (CG == 2) rank = ptx::cluster_ctarank();
    // operands: bf16 1.0 everywhere (the values do not change the time)
    for (int i = threadIdx.x; i < 2 * kKT * kTile / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(sm)[i] = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
    ptx::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        *ok_word = 1;
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        __syncwarp();
        ptx::tmem_alloc<CG>(holder, 512);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    if constexpr (CG == 2)
        ptx::cluster_sync();
    else
        __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *holder;
    if (rank == 0 && threadIdx.x == 0) {
        const uint64_t a0 = ptx::smem_desc_sw128(smem_u32(sA)), b0 = ptx::smem_desc_sw128(smem_u32(sB));
        uint32_t acc[NACC];
#pragma unroll
        for (int q = 0; q < NACC; ++q) acc[q] = tmem + static_cast<uint32_t>(q * ncols);
        const uint64_t t0 = globaltimer_ns();
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int q = u % NACC, step = u / NACC;
                const int j = (step >> 2) % kKT, k = step & 3;
                ptx::tc_mma_f16<CG>(acc[q], a0 + j * (kTile >> 4) + 2 * k, b0 + j * (kTile >> 4) + 2 * k, idesc,
                                    (it > 0 || step > 0) ? 1u : 0u);
            }
        }
        ptx::tc_commit<CG>(bar);
        bool done = false;
        while (!(done = ptx::mbar_try_wait(smem_u32(bar), 0)))
            if (globaltimer_ns() - t0 > kLimitNs) break;
        ns[0] = globaltimer_ns() - t0;
        if (!done) {
            *err = 1;
            *ok_word = 0;
            if constexpr (CG == 2) ptx::st_shared_cluster_u32(ptx::mapa_shared(smem_u32(ok_word), 1), 0u);
        }
    }
    // both CTAs of a pair always meet here, then both read the same verdict
    if constexpr (CG == 2)
        ptx::cluster_sync();
    else
        __syncthreads();
    if (*reinterpret_cast<volatile int32_t*>(ok_word) == 0) return;  // MMAs may still run: TMEM stays allocated
    ptx::tc_fence_before();
    if constexpr (CG == 2)
        ptx::cluster_sync();
    else
        __syncthreads();
    if (warp == 0) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc<CG>(tmem, 512);
    }
}

constexpr int kRing = 192 * 1024;  // copy ring per CTA
constexpr int kIngestSmem = kRing + 2048;

// mode 0: TMA 2-D boxes of 128 rows x 64 bf16 from a contiguous slab; mode 1: 1-D bulk copies of 16 KB;
// mode 2: TMA 3-D boxes of (64 bf16, 64 rows, 4 K tiles) walking a 64-row slab of a [rows, kWideK] matrix.
constexpr int64_t kWideK = 65536;

__global__ void __launch_bounds__(128, 1) ingest_kernel(const __grid_constant__ CUtensorMap tm, const uint8_t* src,
                                                        int64_t per_cta, int32_t mode, unsigned long long* ns,
                                                        int32_t* err) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int box = mode == 2 ? 32768 : 16384;
    const int stages = kRing / box;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kRing);
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) ptx::mbar_init(&full[s], 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    const int64_t n = per_cta / box;
    const uint8_t* base = src + static_cast<int64_t>(blockIdx.x) * per_cta;
    const int32_t row0 = static_cast<int32_t>(static_cast<int64_t>(blockIdx.x) * (per_cta / 128));
    auto issue = [&](int64_t i) {
        const int s = static_cast<int>(i % stages);
        ptx::mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(box));
        if (mode == 0) {
            ptx::tma_load_2d(sm + s * box, &tm, &full[s], 0, row0 + static_cast<int32_t>(i * 128));
        } else if (mode == 1) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(sm + s * box)),
                "l"(base + i * box), "r"(box), "r"(smem_u32(&full[s]))
                : "memory");
        } else {
            ptx::tma_load_3d(sm + s * box, &tm, &full[s], 0, static_cast<int32_t>(blockIdx.x) * 64,
                             static_cast<int32_t>(i * 4), ptx::policy_evict_first());
        }
    };
    const uint64_t t0 = globaltimer_ns();
    for (int64_t i = 0; i < stages && i < n; ++i) issue(i);
    bool ok = true;
    int64_t landed = 0;
    for (int64_t i = 0; i < n && ok; ++i) {
        const int s = static_cast<int>(i % stages);
        const uint32_t ph = static_cast<uint32_t>((i / stages) & 1);
        while (!ptx::mbar_try_wait(smem_u32(&full[s]), ph))
            if (globaltimer_ns() - t0 > kLimitNs) {
                ok = false;
                break;
            }
        if (!ok) break;
        landed = i + 1;
        if (i + stages < n) issue(i + stages);
    }
    ns[blockIdx.x] = globaltimer_ns() - t0;
    if (!ok) {
        *err = 1;
        // the copies still in flight land on this CTA's barriers: wait for them (bounded) before leaving
        const int64_t issued = landed + stages < n ? landed + stages : n;
        for (int64_t i = landed; i < issued; ++i) {
            const int s = static_cast<int>(i % stages);
            const uint32_t ph = static_cast<uint32_t>((i / stages) & 1);
            const uint64_t tw = globaltimer_ns();
            while (!ptx::mbar_try_wait(smem_u32(&full[s]), ph))
                if (globaltimer_ns() - tw > kLimitNs) break;
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
}

template <int CG, int NACC>
int run_mma(uint32_t idesc, int32_t ncols, double* ns_per_mma) {
    unsigned long long* d_ns = nullptr;
    int32_t* d_err = nullptr;
    if (cudaMalloc(&d_ns, 8) != cudaSuccess || cudaMalloc(&d_err, 4) != cudaSuccess) return 1;
    int rc = 0;
    const int32_t iters = 512;  // 8192 MMAs
    unsigned long long best = ~0ull;
    if (cudaMemset(d_err, 0, 4) != cudaSuccess ||
        cudaFuncSetAttribute(mma_kernel<CG, NACC>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem) !=
            cudaSuccess)
        rc = 1;
    for (int rep = 0; rep < 5 && rc == 0; ++rep) {
        cudaError_t e = CG == 2 ? launch_pair_pdl(mma_kernel<CG, NACC>, dim3(2), dim3(128), kMmaSmem, nullptr, idesc,
                                                  ncols, iters, d_ns, d_err)
                                : launch_pdl(mma_kernel<CG, NACC>, dim3(1), dim3(128), kMmaSmem, nullptr, idesc, ncols,
                                             iters, d_ns, d_err);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        unsigned long long h = 0;
        int32_t herr = 0;
        if (e == cudaSuccess) e = cudaMemcpy(&h, d_ns, 8, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(&herr, d_err, 4, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) rc = 1;
        else if (herr) rc = 2;
        else if (h < best) best = h;
    }
    cudaFree(d_ns);
    cudaFree(d_err);
    if (rc == 0) *ns_per_mma = static_cast<double>(best) / (16.0 * iters);
    return rc;
}

}  // namespace probe
}  // namespace bi

using namespace bi;
using namespace bi::probe;

// ns per MMA instruction.  cg = 1: M = 64 or 128, N a multiple of 16 (8 for M = 64) up to 128; cg = 2: M = 256
// with N a multiple of 16 up to 256, or M = 128 with N a multiple of 32 up to 256.  nacc = 1, 2 or 4 accumulators of N columns (nacc * N <= 512).  Returns 0, or
// -1 (bad arguments), 1 (CUDA error), 2 (a wait ran out).
extern "C" int bip_mma_ns(int cg, int M, int N, int nacc, double* ns_per_mma) {
    if (ns_per_mma == nullptr) return -1;
    const bool shape_ok = cg == 1 ? ((M == 128 && N % 16 == 0 && N >= 16 && N <= 128) ||
                                     (M == 64 && N % 8 == 0 && N >= 8 && N <= 128))
                                  : (cg == 2 && ((M == 256 && N % 16 == 0 && N >= 16 && N <= 256) ||
                                                 (M == 128 && N % 32 == 0 && N >= 32 && N <= 256)));
    if (!shape_ok || (nacc != 1 && nacc != 2 && nacc != 4) || nacc * N > 512) return -1;
    const uint32_t idesc = ptx::idesc_bf16_f32(static_cast<uint32_t>(M), static_cast<uint32_t>(N));
    if (cg == 1) {
        if (nacc == 1) return run_mma<1, 1>(idesc, N, ns_per_mma);
        if (nacc == 2) return run_mma<1, 2>(idesc, N, ns_per_mma);
        return run_mma<1, 4>(idesc, N, ns_per_mma);
    }
    if (nacc == 1) return run_mma<2, 1>(idesc, N, ns_per_mma);
    if (nacc == 2) return run_mma<2, 2>(idesc, N, ns_per_mma);
    return run_mma<2, 4>(idesc, N, ns_per_mma);
}

// Stream 8 MB into each of `ctas` CTAs (1..152, one per SM) by `mode` (see ingest_kernel) after writing a
// 256 MB buffer (so the stream starts in HBM).  Returns 0, -1, 1 or 2 as bip_mma_ns; gbps_cta is the mean of
// the CTAs' own rates, gbps_total the bytes of all CTAs over the slowest CTA's time.
extern "C" int bip_ingest(int mode, int ctas, double* gbps_cta, double* gbps_total) {
    if (mode < 0 || mode > 2 || ctas < 1 || ctas > 152 || gbps_cta == nullptr || gbps_total == nullptr) return -1;
    const int64_t per_cta = 8ll << 20;
    const int64_t total = per_cta * ctas;
    auto enc = encoder();
    if (enc == nullptr) return 1;
    uint8_t *src = nullptr, *flush = nullptr;
    unsigned long long* d_ns = nullptr;
    int32_t* d_err = nullptr;
    int rc = 0;
    if (cudaMalloc(&src, total) != cudaSuccess || cudaMalloc(&flush, 256ll << 20) != cudaSuccess ||
        cudaMalloc(&d_ns, 8 * ctas) != cudaSuccess || cudaMalloc(&d_err, 4) != cudaSuccess)
        rc = 1;
    CUtensorMap tm{};
    if (rc == 0 && (cudaMemset(src, 1, total) != cudaSuccess || cudaMemset(d_err, 0, 4) != cudaSuccess))
        rc = 1;
    if (rc == 0) {
        CUresult r;
        cuuint32_t es[3] = {1, 1, 1};
        if (mode == 2) {
            // [rows = total / (kWideK * 2), kWideK] seen as (64, rows, kWideK / 64); box (64, 64, 4)
            cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(total / (kWideK * 2)), kWideK / 64};
            cuuint64_t strides[2] = {kWideK * 2, 128};
            cuuint32_t box[3] = {64, 64, 4};
            r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, src, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(total / 128)};
            cuuint64_t strides[1] = {128};
            cuuint32_t box[2] = {64, 128};
            r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, src, dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) rc = 1;
    }
    if (rc == 0 && (cudaFuncSetAttribute(ingest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kIngestSmem) !=
                        cudaSuccess ||
                    cudaMemset(flush, 0, 256ll << 20) != cudaSuccess))
        rc = 1;
    if (rc == 0) {
        cudaError_t e = launch_pdl(ingest_kernel, dim3(ctas), dim3(128), kIngestSmem, nullptr, tm,
                                   static_cast<const uint8_t*>(src), per_cta, mode, d_ns, d_err);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        std::vector<unsigned long long> h(ctas);
        int32_t herr = 0;
        if (e == cudaSuccess) e = cudaMemcpy(h.data(), d_ns, 8 * ctas, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(&herr, d_err, 4, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) {
            rc = 1;
        } else if (herr) {
            rc = 2;
        } else {
            double sum = 0.0, mx = 0.0;
            for (int i = 0; i < ctas; ++i) {
                sum += per_cta / static_cast<double>(h[i]);
                mx = static_cast<double>(h[i]) > mx ? static_cast<double>(h[i]) : mx;
            }
            *gbps_cta = sum / ctas;
            *gbps_total = static_cast<double>(total) / mx;
        }
    }
    cudaFree(src);
    cudaFree(flush);
    cudaFree(d_ns);
    cudaFree(d_err);
    return rc;
}
