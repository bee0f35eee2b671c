// smla_peak_gather.cu -- a microbenchmark of random-row gathers into shared
// memory on sm_103a, built into libsmla_peak.so beside the tensor-core one.
//
// Every CTA (one per SM) streams `chunks` chunks of 128 rows of a pool of
// 576-byte rows, at the row numbers the caller gives, into a ring of three
// 72 KB stages laid out as the decode kernel lays out its KV tiles (four
// 128-byte latent blocks with the 128-byte swizzle, then the 64-byte rope
// block with the 64-byte swizzle). Nothing consumes the rows: a stage is
// refilled as soon as its previous chunk has landed, so the launch time
// measures the gather alone. Three ways of gathering, as the decode can:
//   0: cp.async, 16 bytes per thread, from `issuers` warps;
//   1: TMA tile::gather4 (four rows per instruction: four 128-byte latent
//      boxes and one 64-byte rope box), one thread in each of `issuers`
//      warps issuing;
//   2: as 1, in clusters of two CTAs that share each chunk: each CTA gathers
//      half of its rows with multicast into both, and a stage is refilled
//      once both CTAs have seen its chunk land (each arrives on the other's
//      stage barrier), the protocol of the decode's paired head groups.
// Every wait is bounded by the global timer; a wait that gives up sets the
// caller's error word and the kernel returns.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "smla_ptx.cuh"

namespace smla_gather {

using namespace smla;

constexpr int kRows = 128;
constexpr int kRowBytes = 576;
constexpr int kStageBytes = 4 * kRows * 128 + kRows * 64;  // 73,728
constexpr int kStages = 3;
constexpr int kThreads = 512;
constexpr int kBarOffset = kStages * kStageBytes;
constexpr int kSmem = kBarOffset + 256 + 1024;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct Args {
    CUtensorMap latent;  // {576 bytes, rows}, boxes of 128 bytes x 1 row, 128-byte swizzle
    CUtensorMap rope;    // boxes of 64 bytes x 1 row, 64-byte swizzle
    const uint8_t* pool;
    const int32_t* idx;  // [units][chunks][128]; a unit is a CTA (methods 0, 1) or a pair (2)
    int32_t chunks;
    int32_t* error;
};

template <int METHOD, int ISSUERS>
__global__ void __launch_bounds__(kThreads, 1) gather_kernel(const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOffset);  // [kStages] the stage's chunk landed
    uint64_t* free_ = full + kStages;                                  // [kStages] pairs: landed in both CTAs
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2 * kStages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr bool kPair = METHOD == 2;
    const uint32_t half = kPair ? static_cast<uint32_t>(blockIdx.x & 1) : 0u;
    const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], METHOD == 0 ? ISSUERS * 32 : 1);
            mbar_init(&free_[s], 2);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if constexpr (kPair)
        cluster_sync_all();
    else
        __syncthreads();

    const int32_t* idx = a.idx + static_cast<int64_t>(unit) * a.chunks * kRows;
    const bool issuer = warp < ISSUERS;
    bool ok = true;
    // paired: once chunk x has landed here, tell both CTAs (thread 0, two
    // chunks behind the issue, so that it rarely waits)
    auto confirm = [&](int x) {
        ok &= mbar_wait_bounded(&full[x % kStages], static_cast<uint32_t>((x / kStages) & 1), abort_flag,
                                kWaitLimitNs);
        mbar_arrive_cluster(map_to_rank(smem_u32(&free_[x % kStages]), 0));
        mbar_arrive_cluster(map_to_rank(smem_u32(&free_[x % kStages]), 1));
    };
    if (issuer) {
        for (int c = 0; c < a.chunks && ok; ++c) {
            const int b = c % kStages;
            if (kPair && tid == 0 && c >= kStages - 1) confirm(c - (kStages - 1));
            const uint32_t parity_prev = static_cast<uint32_t>(((c - kStages) / kStages) & 1);
            if (c >= kStages) {
                if constexpr (kPair)
                    ok &= mbar_wait_cluster_bounded(&free_[b], parity_prev, abort_flag, kWaitLimitNs);
                else
                    ok &= mbar_wait_bounded(&full[b], parity_prev, abort_flag, kWaitLimitNs);
            }
            const uint32_t stage = sbase + b * kStageBytes;
            const int32_t* ci = idx + c * kRows;
            if constexpr (METHOD == 0) {
                for (int k = warp; k < kRows; k += ISSUERS) {
                    const uint8_t* src = a.pool + static_cast<int64_t>(ci[k]) * kRowBytes + lane * 16;
                    cp_async_16(stage + (lane >> 3) * kRows * 128 + (k >> 3) * 1024 + (k & 7) * 128 +
                                    (((lane & 7) ^ (k & 7)) << 4),
                                src, 16u);
                }
                for (int j = warp; j < kRows / 8; j += ISSUERS) {
                    const int k = j * 8 + (lane >> 2), u = lane & 3;
                    cp_async_16(stage + 4 * kRows * 128 + (k >> 3) * 512 + (k & 7) * 64 + ((u ^ ((k >> 1) & 3)) << 4),
                                a.pool + static_cast<int64_t>(ci[k]) * kRowBytes + 512 + u * 16, 16u);
                }
                cp_async_arrive_noinc(&full[b]);
            } else if (lane == 0) {
                if (warp == 0) mbar_arrive_expect_tx(&full[b], kStageBytes);
                const int first = kPair ? static_cast<int>(half) * (kRows / 2) : 0;
                const int last = kPair ? first + kRows / 2 : kRows;
                for (int k = first + 4 * warp; k < last; k += 4 * ISSUERS) {
                    const int32_t r0 = ci[k], r1 = ci[k + 1], r2 = ci[k + 2], r3 = ci[k + 3];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t dst = stage + j * kRows * 128 + (k >> 3) * 1024 + (k & 7) * 128;
                        if constexpr (kPair)
                            tma_gather4_multicast(dst, &a.latent, j * 128, r0, r1, r2, r3, &full[b], 3);
                        else
                            tma_gather4(dst, &a.latent, j * 128, r0, r1, r2, r3, &full[b]);
                    }
                    const uint32_t dst = stage + 4 * kRows * 128 + (k >> 3) * 512 + (k & 7) * 64;
                    if constexpr (kPair)
                        tma_gather4_multicast(dst, &a.rope, 512, r0, r1, r2, r3, &full[b], 3);
                    else
                        tma_gather4(dst, &a.rope, 512, r0, r1, r2, r3, &full[b]);
                }
            }
            if (!ok) *abort_flag = 1;
        }
        if (kPair && tid == 0)
            for (int x = a.chunks > kStages - 1 ? a.chunks - (kStages - 1) : 0; x < a.chunks && ok; ++x) confirm(x);
        // every chunk has landed (paired: in both CTAs, whose arrivals on
        // this CTA's barriers have then all been made)
        for (int c = a.chunks > kStages ? a.chunks - kStages : 0; c < a.chunks; ++c) {
            const uint32_t parity = static_cast<uint32_t>((c / kStages) & 1);
            if constexpr (kPair)
                ok &= mbar_wait_cluster_bounded(&free_[c % kStages], parity, abort_flag, kWaitLimitNs);
            else
                ok &= mbar_wait_bounded(&full[c % kStages], parity, abort_flag, kWaitLimitNs);
        }
        if constexpr (METHOD == 0) cp_async_wait_all();
    }
    if (!ok) {
        *abort_flag = 1;
        atomicExch(a.error, 1);
    }
    if constexpr (kPair)
        cluster_sync_all();  // neither CTA leaves while the other may still signal it
    else
        __syncthreads();
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool encode(CUtensorMap* map, const void* pool, int64_t rows, int box, CUtensorMapSwizzle swizzle) {
    auto enc = encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRowBytes), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
    const cuuint32_t boxes[2] = {static_cast<cuuint32_t>(box), 1};
    const cuuint32_t steps[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, boxes, steps,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int METHOD, int ISSUERS>
int run(const Args& a, int ctas, float* ms) {
    auto kernel = gather_kernel<METHOD, ISSUERS>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) return -3;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = METHOD == 2 ? 2 : 1;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return -3;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return -3;
    }
    int rc = 0;
    cudaEventRecord(e0);
    if (cudaLaunchKernelEx(&cfg, kernel, a) != cudaSuccess) rc = -3;
    cudaEventRecord(e1);
    if (cudaDeviceSynchronize() != cudaSuccess) rc = -3;
    if (rc == 0) cudaEventElapsedTime(ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return rc;
}

}  // namespace smla_gather

// One launch of the gather benchmark: `ctas` CTAs (even for method 2) each
// stream `chunks` chunks of 128 rows of `pool` (`rows` rows of 576 bytes,
// device memory, 16-byte aligned) at the row numbers in `idx` (device int32
// [units][chunks][128], every entry in [0, rows); a unit is a CTA, or a CTA
// pair for method 2). `error` is a device int32 the kernel sets to 1 when a
// bounded wait gives up. Writes the launch's CUDA-event time to `ms`.
// Returns 0, -1 for a method / issuer count this benchmark does not build,
// -2 for bad arguments, -3 for a CUDA error.
extern "C" int smla_peak_gather(int method, int issuers, const void* pool, long long rows, const int* idx, int ctas,
                                int chunks, int* error, float* ms) {
    using namespace smla_gather;
    if (pool == nullptr || idx == nullptr || error == nullptr || ms == nullptr || rows <= 0 || rows > 0x7FFFFFFF ||
        ctas <= 0 || chunks <= 0 || (method == 2 && ctas % 2 != 0) || (reinterpret_cast<uintptr_t>(pool) & 15u))
        return -2;
    Args a;
    std::memset(&a, 0, sizeof(a));
    a.pool = static_cast<const uint8_t*>(pool);
    a.idx = idx;
    a.chunks = chunks;
    a.error = error;
    if (method != 0 && (!encode(&a.latent, pool, rows, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
                        !encode(&a.rope, pool, rows, 64, CU_TENSOR_MAP_SWIZZLE_64B)))
        return -3;
#define SMLA_GATHER_CASE(M, I) \
    if (method == M && issuers == I) return run<M, I>(a, ctas, ms);
    SMLA_GATHER_CASE(0, 7)
    SMLA_GATHER_CASE(0, 16)
    SMLA_GATHER_CASE(1, 1)
    SMLA_GATHER_CASE(1, 4)
    SMLA_GATHER_CASE(1, 7)
    SMLA_GATHER_CASE(1, 16)
    SMLA_GATHER_CASE(2, 7)
    SMLA_GATHER_CASE(2, 16)
#undef SMLA_GATHER_CASE
    return -1;
}
