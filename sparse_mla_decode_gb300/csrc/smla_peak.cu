// smla_peak.cu -- a microbenchmark of the FP8 tensor cores of sm_103a
// (tcgen05.mma kind::f8f6f4, E4M3 x E4M3 -> FP32 in TMEM), built as its own
// library (libsmla_peak.so) beside libsmla.so.
//
// It measures what the decode kernel's products cost, shape by shape:
//   * one CTA (or one CTA pair for cta_group::2) issuing a long run of
//     K = 32 MMAs into one accumulator: cycles per MMA, the issue-to-drain
//     rate of one SM's tensor core fed from shared memory;
//   * every SM doing the same: achieved TFLOP/s of the whole GPU, the dense
//     FP8 peak that the decode's tensor fraction is quoted against.
// Operand tiles are laid out as the decode reads them: K-major tiles with the
// 128-byte swizzle (rows of 128 bytes, 8-row atoms of 1 KB), and MN-major
// tiles (the latent block read as V^T, 128B swizzle; P^T of 64 heads, 64B
// swizzle). The operands are fixed bytes: the rate does not depend on them.
//
// Every wait is bounded by the global timer; a wait that gives up sets an
// error flag that the host reads back, and the kernel still frees its TMEM.

#include <cuda_runtime.h>

#include <cstdint>

namespace smla_peak {

constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    const uint64_t start = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && global_timer_ns() - start > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t columns) {
    if constexpr (CG == 2)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                     "r"(columns)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                     "r"(columns)
                     : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t columns) {
    if constexpr (CG == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(columns) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(columns) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    if constexpr (CG == 2)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrives once on the mbarrier at shared::cluster address `bar` (this CTA's
// or its peer's) when every tcgen05 operation this thread issued completed.
template <int CG>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    if constexpr (CG == 2)
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(swizzle) << 61;
    return d;
}

constexpr uint32_t kSwizzle128B = 2;
constexpr uint32_t kSwizzle64B = 4;
constexpr uint32_t kSwizzle32B = 6;

__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n, int a_mn, int b_mn) {
    return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Shared memory: the A tile (128 rows x 128 bytes = 16 KB: 128 rows of one K
// atom K-major, or 128 K-rows of 128 M-bytes MN-major) at 0, the B tile
// (K-major: up to 256 rows x 128 bytes; MN-major: 128 K-rows x NB bytes) at
// 16 KB, the barrier and the TMEM address after 48 KB.
constexpr int kA = 0;
constexpr int kB = 16384;
constexpr int kBar = 16384 + 32768;
// 128 KB requested, so that one CTA runs per SM when every SM takes part.
constexpr int kSmem = 128 * 1024;

// Each CTA of the launch: the elected thread of the issuing CTA runs `iters`
// groups of four K = 32 MMAs into CH TMEM accumulators of N columns (MMA ks
// of a group into accumulator ks % CH, so that CH independent chains
// interleave) and commits; `cycles` (when non-null) gets the clock64 span of
// CTA 0's run.
template <int CG, int N, int AMN, int BMN, int CH, int COMMIT = 0>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int iters, long long* cycles, int* error) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* done = reinterpret_cast<uint64_t*>(smem + kBar);
    uint64_t* every = done + 4;  // COMMIT: a commit after each group of four lands here; nothing waits on it
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBar + 16);
    const int tid = threadIdx.x;
    const uint32_t rank = CG == 2 ? cluster_rank() : 0u;

    // operands: E4M3 bytes without NaN codes
    for (int i = tid; i < (kBar - kA) / 4; i += blockDim.x) {
        const uint32_t x = static_cast<uint32_t>(i) * 2654435761u + rank * 97u;
        reinterpret_cast<uint32_t*>(smem)[i] = (x ^ (x >> 13)) & 0x76767676u;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (tid == 0) {
        mbar_init(done, 1);
        mbar_init(every, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    static_assert(CH == 1 || CH == 2 || CH == 4, "one, two or four chains");
    constexpr int kCols = N * CH < 32 ? 32 : N * CH;
    if (tid < 32) tmem_alloc<CG>(tmem_slot, kCols);
    tc_fence_before_sync();
    if constexpr (CG == 2)
        cluster_sync_all();
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (tid == 0 && rank == 0) {
        constexpr int M = CG == 2 ? 256 : 128;
        constexpr uint32_t idesc = idesc_e4m3(M, N, AMN, BMN);
        constexpr int NB = N / CG;  // B rows (K-major) or bytes per K-row (MN-major) in this CTA
        // K-major A: 128 rows of one 128-byte atom, a K step moves 32 bytes.
        // MN-major A: 128 M-bytes per K-row, 8-row atoms of 1 KB, a K step
        // moves 32 rows (4 KB).
        const uint64_t a_desc = smem_desc(sbase + kA, 1024, 1024, kSwizzle128B);
        const uint32_t a_step = AMN ? (32 * 128) >> 4 : 32 >> 4;
        uint64_t b_desc;
        uint32_t b_step;
        if constexpr (BMN) {
            // MN-major B of NB bytes per K-row, 8-row atoms of 8 NB bytes, the
            // swizzle of the row width (none for 16 bytes), as the decode's P^T
            static_assert(NB == 16 || NB == 32 || NB == 64 || NB == 128, "MN-major B of 16..128 bytes per K-row");
            constexpr uint32_t kSw = NB == 128 ? kSwizzle128B : NB == 64 ? kSwizzle64B : NB == 32 ? kSwizzle32B : 0u;
            b_desc = smem_desc(sbase + kB, 8 * NB, 8 * NB, kSw);
            b_step = (32 * NB) >> 4;
        } else {
            b_desc = smem_desc(sbase + kB, 1024, 1024, kSwizzle128B);
            b_step = 32 >> 4;
        }
        const long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f8<CG>(tmem + (ks % CH) * N, a_desc + ks * a_step, b_desc + ks * b_step, idesc,
                           (it != 0 || ks >= CH) ? 1u : 0u);
            if constexpr (COMMIT != 0) mma_commit<CG>(smem_u32(every));
        }
        mma_commit<CG>(smem_u32(done));
        if constexpr (CG == 2) mma_commit<CG>(map_to_rank(smem_u32(done), 1));
        ok = mbar_wait_bounded(done, 0);
        const long long t1 = clock64();
        if (cycles != nullptr && blockIdx.x == 0) *cycles = t1 - t0;
    } else if (tid == 0) {
        ok = mbar_wait_bounded(done, 0);  // the pair's MMAs wrote this CTA's TMEM
    }
    if (!ok) atomicExch(error, 1);
    tc_fence_before_sync();
    if constexpr (CG == 2)
        cluster_sync_all();
    else
        __syncthreads();
    tc_fence_after_sync();
    if (tid < 32) tmem_dealloc<CG>(tmem, kCols);
}

// N = 64 K-major FP8 MMAs from thread 0 (groups of four into one
// accumulator at column 0) while the other three warps keep another unit
// busy, as the decode's softmax and producers do beside its MMA warp:
//   MODE 1: tcgen05.ld / tcgen05.st of 16 columns at a time on columns
//           64..127 of their TMEM lanes (the softmax's logit reads and O^T
//           rescales);
//   MODE 2: no other warp; each group of four FP8 MMAs follows one BF16
//           kind::f16 MMA (K = 16) into the same accumulator (the rope);
//   MODE 3: 16-byte st.shared by every lane into the shared memory past the
//           operand tiles (the producers' landing rows);
//   MODE 4: warps 4 and 8 (on thread 0's SM sub-partition, as the decode's
//           softmax warps 0 and 4 share one with its MMA warp) run chains of
//           FMAs;
//   MODE 5: no other warp, and `cycles` gets the span of thread 0's issue of
//           the first group of four MMAs and its commit alone (the issue
//           cost, before any back-pressure of the pipe).
// The busy warps run until thread 0's MMAs have drained (a flag in shared
// memory), at most `iters` * 64 rounds. `cycles` gets thread 0's clock64
// span from its first issue to the drain.
template <int MODE>
__global__ void __launch_bounds__(384, 1) mma_contend_kernel(int iters, long long* cycles, int* error) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* done = reinterpret_cast<uint64_t*>(smem + kBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBar + 16);
    volatile int* stop = reinterpret_cast<volatile int*>(smem + kBar + 32);
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < (kBar - kA) / 4; i += blockDim.x) {
        const uint32_t x = static_cast<uint32_t>(i) * 2654435761u;
        reinterpret_cast<uint32_t*>(smem)[i] = (x ^ (x >> 13)) & 0x36363636u;  // E4M3 and BF16 without NaN or Inf
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (tid == 0) {
        mbar_init(done, 1);
        mbar_init(done + 1, 1);
        *stop = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < 32) tmem_alloc<1>(tmem_slot, 128);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    if (tid == 0) {
        constexpr uint32_t idesc = idesc_e4m3(128, 64, 0, 0);
        // kind::f16, BF16 A and B, FP32 D, K-major
        constexpr uint32_t idesc16 = (1u << 4) | (1u << 7) | (1u << 10) | (64u >> 3 << 17) | (128u >> 4 << 24);
        const uint64_t a_desc = smem_desc(sbase + kA, 1024, 1024, kSwizzle128B);
        const uint64_t b_desc = smem_desc(sbase + kB, 1024, 1024, kSwizzle128B);
        const long long t0 = clock64();
        long long t_first = 0;
        for (int it = 0; it < iters; ++it) {
            if constexpr (MODE == 2) {
                asm volatile(
                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                    "l"(a_desc), "l"(b_desc), "r"(idesc16), "r"(it != 0 ? 1u : 0u)
                    : "memory");
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f8<1>(tmem, a_desc + ks * 2, b_desc + ks * 2, idesc, (it != 0 || ks != 0 || MODE == 2) ? 1u : 0u);
            if (MODE == 5 && it == 0) {
                mma_commit<1>(smem_u32(done + 1));
                t_first = clock64();
            }
        }
        mma_commit<1>(smem_u32(done));
        ok = mbar_wait_bounded(done, 0);
        const long long t1 = clock64();
        *stop = 1;
        if (cycles != nullptr && blockIdx.x == 0) *cycles = MODE == 5 ? t_first - t0 : t1 - t0;
    } else if (warp >= 1 && warp < 4 && MODE == 1) {
        const uint32_t col = tmem + (static_cast<uint32_t>(warp * 32) << 16) + 64;
        for (int r = 0; r < iters * 64; ++r) {
            // the warp leaves together: the .sync.aligned TMEM accesses need every lane
            if (__shfl_sync(0xFFFFFFFFu, *stop, 0) != 0) break;
            uint32_t v[16];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
                "tcgen05.wait::ld.sync.aligned;"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                : "r"(col + 16 * (r & 3))
                : "memory");
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] ^= 1u;
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
                "tcgen05.wait::st.sync.aligned;" ::"r"(col + 16 * (r & 3)),
                "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
                "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                : "memory");
            __syncwarp();
        }
    } else if ((warp == 4 || warp == 8) && MODE == 4) {
        float x = static_cast<float>(tid), y = 1.0f;
        for (int r = 0; r < iters * 64; ++r) {
            if (__shfl_sync(0xFFFFFFFFu, *stop, 0) != 0) break;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                x = fmaf(x, 0.999f, y);
                y = fmaf(y, 1.001f, x);
            }
        }
        if (x == 12345.0f) *stop = 2;  // keeps the chain live
    } else if (warp >= 1 && warp < 4 && MODE == 3) {
        const uint32_t base = sbase + 64 * 1024 + static_cast<uint32_t>(tid - 32) * 16;  // 96 lanes x 16 bytes
        for (int r = 0; r < iters * 64; ++r) {
            if (__shfl_sync(0xFFFFFFFFu, *stop, 0) != 0) break;
            const uint32_t a = base + static_cast<uint32_t>((r & 31) * 96 * 16);  // within 64 KB .. 112 KB
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(static_cast<uint32_t>(r)) : "memory");
        }
    }
    if (!ok) atomicExch(error, 1);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (tid < 32) tmem_dealloc<1>(tmem, 128);
}

template <int MODE>
int run_contend(int iters, long long* cycles_out) {
    auto kernel = mma_contend_kernel<MODE>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) return -3;
    long long* d_cycles = nullptr;
    int* d_error = nullptr;
    if (cudaMalloc(&d_cycles, sizeof(long long)) != cudaSuccess) return -3;
    if (cudaMalloc(&d_error, sizeof(int)) != cudaSuccess) {
        cudaFree(d_cycles);
        return -3;
    }
    cudaMemset(d_error, 0, sizeof(int));
    int rc = 0;
    for (int pass = 0; pass < 2 && rc == 0; ++pass) {
        kernel<<<1, MODE == 4 ? 384 : 128, kSmem>>>(iters, d_cycles, d_error);
        if (cudaDeviceSynchronize() != cudaSuccess) rc = -3;
    }
    int err = 0;
    if (rc == 0) {
        cudaMemcpy(cycles_out, d_cycles, sizeof(long long), cudaMemcpyDeviceToHost);
        cudaMemcpy(&err, d_error, sizeof(int), cudaMemcpyDeviceToHost);
        if (err != 0) rc = -4;
    }
    cudaFree(d_cycles);
    cudaFree(d_error);
    return rc;
}

template <int CG, int N, int AMN, int BMN, int CH, int COMMIT = 0>
int run(int iters, int ctas, long long* cycles_out, float* ms_out) {
    auto kernel = mma_rate_kernel<CG, N, AMN, BMN, CH, COMMIT>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) return -3;
    long long* d_cycles = nullptr;
    int* d_error = nullptr;
    if (cudaMalloc(&d_cycles, sizeof(long long)) != cudaSuccess) return -3;
    if (cudaMalloc(&d_error, sizeof(int)) != cudaSuccess) {
        cudaFree(d_cycles);
        return -3;
    }
    cudaMemset(d_error, 0, sizeof(int));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = CG;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    int rc = 0;
    // one warm-up launch, then the timed one
    for (int pass = 0; pass < 2 && rc == 0; ++pass) {
        if (pass == 1) cudaEventRecord(e0);
        if (cudaLaunchKernelEx(&cfg, kernel, iters, d_cycles, d_error) != cudaSuccess) rc = -3;
        if (pass == 1) cudaEventRecord(e1);
        if (cudaDeviceSynchronize() != cudaSuccess) rc = -3;
    }
    int err = 0;
    if (rc == 0) {
        cudaEventElapsedTime(ms_out, e0, e1);
        cudaMemcpy(cycles_out, d_cycles, sizeof(long long), cudaMemcpyDeviceToHost);
        cudaMemcpy(&err, d_error, sizeof(int), cudaMemcpyDeviceToHost);
        if (err != 0) rc = -4;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(d_cycles);
    cudaFree(d_error);
    return rc;
}

}  // namespace smla_peak

// Runs the shape (cta_group 1 or 2, N, A / B MN-major) on `ctas` CTAs (a
// multiple of cta_group), each issuing 4 * iters MMAs of K = 32. Writes CTA
// 0's clock64 span of its run and the launch's elapsed time. Returns 0, -1
// for a shape this benchmark does not build, -3 for a CUDA error, -4 when a
// bounded wait gave up.
extern "C" int smla_peak_mma(int cta_group, int n, int a_mn, int b_mn, int iters, int ctas, long long* cycles,
                             float* ms) {
    using namespace smla_peak;
    if (cycles == nullptr || ms == nullptr || iters <= 0 || ctas <= 0 || ctas % cta_group != 0) return -1;
#define SMLA_PEAK_CASE(CG, N, AMN, BMN) \
    if (cta_group == CG && n == N && a_mn == AMN && b_mn == BMN) return run<CG, N, AMN, BMN, 1>(iters, ctas, cycles, ms);
    SMLA_PEAK_CASE(1, 16, 0, 0)
    SMLA_PEAK_CASE(1, 16, 1, 1)
    SMLA_PEAK_CASE(1, 32, 0, 0)
    SMLA_PEAK_CASE(1, 32, 1, 1)
    SMLA_PEAK_CASE(1, 64, 0, 0)
    SMLA_PEAK_CASE(1, 128, 0, 0)
    SMLA_PEAK_CASE(1, 256, 0, 0)
    SMLA_PEAK_CASE(1, 64, 1, 1)
    SMLA_PEAK_CASE(1, 128, 1, 1)
    SMLA_PEAK_CASE(1, 64, 1, 0)
    SMLA_PEAK_CASE(2, 128, 0, 0)
    SMLA_PEAK_CASE(2, 256, 0, 0)
    SMLA_PEAK_CASE(2, 128, 1, 1)
    SMLA_PEAK_CASE(2, 256, 1, 1)
    SMLA_PEAK_CASE(2, 128, 1, 0)
#undef SMLA_PEAK_CASE
    return -1;
}

// The same with `chains` (1, 2 or 4) accumulators of N columns that the
// MMAs of each group of four take in turn: whether independent accumulators
// overlap where one chain does not. Returns as smla_peak_mma.
extern "C" int smla_peak_mma_chains(int cta_group, int n, int a_mn, int b_mn, int chains, int iters, int ctas,
                                    long long* cycles, float* ms) {
    using namespace smla_peak;
    if (cycles == nullptr || ms == nullptr || iters <= 0 || ctas <= 0 || ctas % cta_group != 0) return -1;
    if (chains == 1) return smla_peak_mma(cta_group, n, a_mn, b_mn, iters, ctas, cycles, ms);
#define SMLA_PEAK_CHAINS(N, AMN, BMN, CH)                                        \
    if (cta_group == 1 && n == N && a_mn == AMN && b_mn == BMN && chains == CH) \
        return run<1, N, AMN, BMN, CH>(iters, ctas, cycles, ms);
    SMLA_PEAK_CHAINS(16, 0, 0, 2)
    SMLA_PEAK_CHAINS(16, 0, 0, 4)
    SMLA_PEAK_CHAINS(32, 0, 0, 2)
    SMLA_PEAK_CHAINS(32, 0, 0, 4)
    SMLA_PEAK_CHAINS(64, 0, 0, 2)
    SMLA_PEAK_CHAINS(64, 0, 0, 4)
    SMLA_PEAK_CHAINS(64, 1, 1, 2)
    SMLA_PEAK_CHAINS(64, 1, 1, 4)
    SMLA_PEAK_CHAINS(128, 0, 0, 2)
#undef SMLA_PEAK_CHAINS
    return -1;
}

// One accumulator with a tcgen05.commit (to an mbarrier nothing waits on)
// after every group of four MMAs, as a pipeline that hands each accumulator
// to its consumer issues them: whether commits slow the tensor pipe. N = 64,
// operands K-major (a_mn = b_mn = 0) or MN-major (1, 1). Returns as
// smla_peak_mma.
extern "C" int smla_peak_mma_commit4(int n, int a_mn, int b_mn, int iters, int ctas, long long* cycles, float* ms) {
    using namespace smla_peak;
    if (cycles == nullptr || ms == nullptr || iters <= 0 || ctas <= 0 || n != 64 || a_mn != b_mn) return -1;
    return a_mn ? run<1, 64, 1, 1, 1, 1>(iters, ctas, cycles, ms) : run<1, 64, 0, 0, 1, 1>(iters, ctas, cycles, ms);
}

// One CTA: N = 64 K-major FP8 MMAs (4 * iters of them, plus iters BF16 ones in
// mode 2) beside the other warps' work of `mode` (1: TMEM loads and stores,
// 2: BF16 MMAs interleaved, 3: shared-memory stores, 4: FMA chains on the
// issuing warp's sub-partition, 5: nothing, timing the first four issues).
// Writes the clock64 span of the MMAs (mode 5: of the first four issues and
// their commit). Returns as smla_peak_mma.
extern "C" int smla_peak_mma_contend(int mode, int iters, long long* cycles) {
    using namespace smla_peak;
    if (cycles == nullptr || iters <= 0) return -1;
    if (mode == 1) return run_contend<1>(iters, cycles);
    if (mode == 2) return run_contend<2>(iters, cycles);
    if (mode == 3) return run_contend<3>(iters, cycles);
    if (mode == 4) return run_contend<4>(iters, cycles);
    if (mode == 5) return run_contend<5>(iters, cycles);
    return -1;
}
