// smla_ds_mla.cu -- sparse MLA decode over fp8_ds_mla cache rows of 656
// bytes (Kimi K3.1 dsa_indexer_mxfp4 page, mxfp4_fused_prologue: the
// mla_cache of [num_blocks, block_size, 656] bytes that the insert fills with
// [kv_c_normed | k_pe] and views as FP8, float32 and BF16).
//
// Row layout (the plainest reading of 656 = 512 + 16 + 128; the page prints
// no row): bytes 0..511 the E4M3 codes of the 512 latents, bytes 512..527
// four little-endian FP32 scales s_0..s_3 (scale b covers latents 128 b ..
// 128 b + 127), bytes 528..655 the 64 rope values as little-endian BF16.
// Latent j is dec(code_j) * s_(j / 128).
//
// What is computed is the 576-byte decode's definition (DeepSeek-V4.1
// sparse_mla_cute page, "What this module computes") with K the 576 values of
// a row and V its 512 latents; the row scales take the place of k_scale.
//
// The scales vary per key and per 128-latent block, so neither product can
// take them as one factor:
//   * QK: one E4M3 accumulator per latent block (S^T_b = codes_b . Q_b^T) and
//     a BF16 product for the rope (kind::f16); the softmax forms each key's
//     logits as sum_b s_b S^T_b + S^T_rope in FP32.
//   * PV: latent block b takes P'_b = P * s_b / sigma_b as its B operand, in
//     E4M3, where sigma_b is the running maximum of |s_b| over the keys seen
//     so far (so |P'_b| <= |P| <= 448). O^T block b lives in the frame of
//     sigma_b: when sigma_b rises, the block is rescaled by sigma_old /
//     sigma_new together with the running-max factor, and the epilogue
//     multiplies it by sigma_b.
// One CTA handles 32 heads of one token over all its keys (no key split):
// chunks of 128 keys in two stages of 82 KB, the softmax in one warpgroup
// (thread t owns key t of each chunk and latent row t of each O^T block),
// one MMA-issuing warp, seven cp.async producer warps. TMEM: two S buffers of
// five 32-column accumulators and four O^T blocks, 448 of 512 columns.
// Every wait is bounded; a timeout sets an error bit and the kernel returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "smla.h"
#include "smla_ptx.cuh"

namespace smla {
void note_cuda_error(int code);
int32_t* device_error_word();
bool dependent_launch();
bool encode_bytes_map(CUtensorMap* map, const void* base, uint32_t rank, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, int swizzle, int promotion);

namespace dsmla {

constexpr int kN = 32;            // heads per CTA
constexpr int kC = 128;           // keys per chunk = the MMA's M
constexpr int kRowBytes = 656;
constexpr int kScaleAt = 512;     // byte offset of the scales in a row
constexpr int kRopeAt = 528;      // byte offset of the rope in a row
constexpr int kThreads = 384;
constexpr int kMmaWarp = 4;
constexpr int kProducerWarp = 5;  // first of seven
constexpr int kProducerThreads = 224;
constexpr int kFirstThreads = 128 + kProducerThreads;  // chunk 0: the softmax warps and the producers
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2P = 8.80735492205760410744f;  // log2(448): P of the running max
constexpr float kLog2e = 1.44269504088896340736f;

// Shared memory (offsets from a 1024-byte aligned base). A stage: the four
// 128-byte latent blocks of 128 keys (128B swizzle), the 128-byte BF16 rope
// rows (128B swizzle) and the keys' four scales (16 bytes each, plain).
constexpr int kLat = 0;
constexpr int kRope = 4 * kC * 128;
constexpr int kScale = kRope + kC * 128;
constexpr int kStage = kScale + kC * 16;
constexpr int kQ = 2 * kStage;                // Q latent: four blocks of 32 heads x 128 bytes
constexpr int kQRope = kQ + 4 * kN * 128;     // Q rope: 32 heads x 128 bytes (BF16)
constexpr int kPBlock = kC * kN;              // P'_b^T: 128 keys x 32 heads of E4M3
constexpr int kP = kQRope + kN * 128;         // [2 buffers][4 blocks]
constexpr int kIdx = kP + 2 * 4 * kPBlock;    // int32 [2][128]: each key's row, -1 masked
constexpr int kRed = kIdx + 2 * kC * 4;       // float [4 warps][32 heads]
constexpr int kSig = kRed + 4 * kN * 4;       // float [4 warps][4 blocks], sigma[4], beta[4]
constexpr int kHead = kSig + 128;             // float [4][32]: m_run, bias, alpha, l
constexpr int kBar = kHead + 4 * kN * 4;      // 16 mbarriers
constexpr int kMisc = kBar + 16 * 8;          // TMEM base, abort flag
constexpr int kBytes = kMisc + 64;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 227 * 1024, "one CTA's shared memory");
static_assert(kStage % 1024 == 0 && kQ % 1024 == 0 && kQRope % 1024 == 0 && kP % 1024 == 0, "aligned tiles");

// TMEM columns: S buffer b at b * 160 (latent blocks at +0, 32, 64, 96, the
// rope at +128), O^T block j at 320 + 32 j.
constexpr int kSCols = 5 * kN;
constexpr int kOCol = 2 * kSCols;
constexpr int kTmemCols = 512;

struct Params {
    CUtensorMap q_latent;  // {512 bytes, H, T}: boxes of 128 bytes x 32 heads, 128B swizzle
    CUtensorMap q_rope;    // {128 bytes, H, T}: boxes of 128 bytes x 32 heads, 128B swizzle
    const uint8_t* pool0;
    const uint8_t* pool1;
    int64_t rows0, rows1;
    const int32_t* indices;
    int64_t idx_stride;
    const int32_t* lens;
    const float* sinks;
    __nv_bfloat16* out;
    int64_t out_stride_token, out_stride_head;
    float* lse;
    int64_t lse_stride_token;
    int32_t width, pool_split, num_pools;
    float scale_log2, out_scale;
    int32_t* error;
};

// kind::f16 instruction descriptor: BF16 A and B (format 1), FP32 D, K-major.
constexpr uint32_t idesc_bf16_kmajor(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// P'^T of one block: 128 keys x 32 heads, MN-major (each key's 32 heads
// contiguous), 32-byte swizzle: 16-byte unit u of key k at k * 32 + ((u ^
// ((k >> 2) & 1)) << 4).
__device__ __forceinline__ uint32_t p_unit(int key, int unit) {
    return static_cast<uint32_t>(key * kN + ((unit ^ ((key >> 2) & 1)) << 4));
}

// The row `id` of key column `col` (pool by the split column).
__device__ __forceinline__ const uint8_t* row_of(const Params& p, int col, int32_t id) {
    const bool second = p.num_pools == 2 && col >= p.pool_split;
    return (second ? p.pool1 : p.pool0) + static_cast<int64_t>(id) * kRowBytes;
}

// Copies the rows of one chunk (`ids` of its 128 keys, -1 masked: zero
// filled) into a stage, as warp `w` of `warps`.
__device__ __forceinline__ void gather_chunk(const Params& p, uint32_t stage, const int32_t* ids, int col0, int w,
                                             int warps, int lane) {
    for (int k = w; k < kC; k += warps) {  // latent codes: 32 lanes x 16 bytes
        const int32_t id = ids[k];
        const uint8_t* src = row_of(p, col0 + k, id >= 0 ? id : 0) + lane * 16;
        const uint32_t dst = stage + kLat + (lane >> 3) * kC * 128 + (k >> 3) * 1024 + (k & 7) * 128 +
                             (((lane & 7) ^ (k & 7)) << 4);
        cp_async_16(dst, src, id >= 0 ? 16u : 0u);
    }
    for (int j = w; j < kC / 4; j += warps) {  // rope: four keys of 8 x 16 bytes per instruction
        const int k = 4 * j + (lane >> 3), u = lane & 7;
        const int32_t id = ids[k];
        const uint8_t* src = row_of(p, col0 + k, id >= 0 ? id : 0) + kRopeAt + u * 16;
        const uint32_t dst = stage + kRope + (k >> 3) * 1024 + (k & 7) * 128 + ((u ^ (k & 7)) << 4);
        cp_async_16(dst, src, id >= 0 ? 16u : 0u);
    }
    for (int j = w; j < kC / 32; j += warps) {  // scales: one key per lane
        const int k = 32 * j + lane;
        const int32_t id = ids[k];
        const uint8_t* src = row_of(p, col0 + k, id >= 0 ? id : 0) + kScaleAt;
        cp_async_16(stage + kScale + k * 16, src, id >= 0 ? 16u : 0u);
    }
}

// Resolves key column `col` (< count) of the token to a row, or -1 (a hole,
// or an index past its pool: masked and flagged).
__device__ __forceinline__ int32_t resolve(const Params& p, int col, int32_t raw) {
    if (raw < 0) return -1;
    const bool second = p.num_pools == 2 && col >= p.pool_split;
    if (raw < (second ? p.rows1 : p.rows0)) return raw;
    atomicOr(p.error, SMLA_DEV_INDEX_RANGE);
    return -1;
}

// Writes the BF16 tile [heads][512] in shared memory to out[token][head0 + h],
// 16 bytes per thread and step where the output rows allow it, else 4.
__device__ __forceinline__ void store_tile(const Params& p, const __nv_bfloat16* tile, int token, int head0, int heads,
                                           int tid, int threads) {
    __nv_bfloat16* out = p.out + static_cast<int64_t>(token) * p.out_stride_token +
                         static_cast<int64_t>(head0) * p.out_stride_head;
    const bool wide_rows = ((reinterpret_cast<uintptr_t>(p.out) | static_cast<uintptr_t>(p.out_stride_token * 2) |
                             static_cast<uintptr_t>(p.out_stride_head * 2)) & 15u) == 0;
    if (wide_rows) {
        for (int i = tid; i < heads * 512 / 8; i += threads) {
            const int h = i / 64, e = (i % 64) * 8;
            *reinterpret_cast<uint4*>(out + static_cast<int64_t>(h) * p.out_stride_head + e) =
                *reinterpret_cast<const uint4*>(tile + h * 512 + e);
        }
    } else {
        for (int i = tid; i < heads * 512 / 2; i += threads) {
            const int h = i / 256, e = (i % 256) * 2;
            *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(h) * p.out_stride_head + e) =
                *reinterpret_cast<const uint32_t*>(tile + h * 512 + e);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) ds_mla_decode_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBar);
    uint64_t* kv_full = bars + 0;   // [2] a stage's rows landed (224 cp.async arrivals + 1)
    uint64_t* pv_done = bars + 2;   // [2] PV of the stage's chunk finished
    uint64_t* s_full = bars + 4;    // [2] QK of a chunk finished
    uint64_t* p_full = bars + 6;    // P' written, O^T rescaled (128 softmax arrivals)
    uint64_t* drain = bars + 7;     // every MMA finished
    uint64_t* q_full = bars + 8;    // the Q tiles landed
    uint64_t* kv_first = bars + 9;  // chunk 0 landed (352 cp.async arrivals + 1)
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + kIdx);
    float* red = reinterpret_cast<float*>(smem + kRed);
    float* sig_red = reinterpret_cast<float*>(smem + kSig);  // [4 warps][4 blocks]
    float* sig_run = sig_red + 16;                            // [4]
    float* sig_beta = sig_run + 4;                            // [4]
    float* m_run_s = reinterpret_cast<float*>(smem + kHead);
    float* bias_s = m_run_s + kN;
    float* alpha_s = m_run_s + 2 * kN;
    float* l_s = m_run_s + 3 * kN;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head0 = static_cast<int>(blockIdx.x) * kN;
    const int token = blockIdx.y;

    // ---- set-up (reads no input, so it overlaps the previous kernel) -------
    if (tid == 0) {
        mbar_init(&kv_full[0], kProducerThreads + 1);
        mbar_init(&kv_full[1], kProducerThreads + 1);
        mbar_init(&pv_done[0], 1);
        mbar_init(&pv_done[1], 1);
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(p_full, 128);
        mbar_init(drain, 1);
        mbar_init(q_full, 1);
        mbar_init(kv_first, kFirstThreads + 1);
        misc[1] = 0;
        mbar_init_fence();
    }
    if (tid < kN) {
        m_run_s[tid] = -INFINITY;
        bias_s[tid] = -INFINITY;
        alpha_s[tid] = 1.0f;
        l_s[tid] = 0.0f;
    }
    if (tid < 4) {
        sig_run[tid] = 0.0f;
        sig_beta[tid] = 1.0f;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(misc, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensor_map(&p.q_latent);
        prefetch_tensor_map(&p.q_rope);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    grid_dependency_wait();  // inputs are read only after this point
    if (warp == kProducerWarp && lane == 0) {
        mbar_arrive_expect_tx(q_full, kN * 512 + kN * 128);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
            tma_load_3d(sbase + kQ + kb * kN * 128, &p.q_latent, kb * 128, head0, token, q_full);
        tma_load_3d(sbase + kQRope, &p.q_rope, 0, head0, token, q_full);
    }
    const int32_t* idx_row = p.indices + static_cast<int64_t>(token) * p.idx_stride;
    int32_t raw_first = -1;
    if (tid < kC && tid < p.width) raw_first = idx_row[tid];
    const int count = min(max(p.lens[token], 0), p.width);
    const float sink_of_head = (tid < kN && p.sinks != nullptr) ? p.sinks[head0 + tid] * kLog2e : -INFINITY;
    const int nch = (count + kC - 1) / kC;
    grid_launch_dependents();

    bool ok = true;
    auto kv_bar = [&](int c) -> uint64_t* { return c == 0 ? kv_first : &kv_full[c & 1]; };
    auto kv_parity = [&](int c) -> uint32_t {
        return c == 0 ? 0u : static_cast<uint32_t>(((c >> 1) - ((c & 1) ? 0 : 1)) & 1);
    };
    auto pv_wait = [&](int c) {
        ok &= mbar_wait_bounded(&pv_done[c & 1], static_cast<uint32_t>((c >> 1) & 1), abort_flag, kWaitLimitNs);
    };

    if (warp != kMmaWarp && nch > 0) {
        // ===================== chunk 0 by the softmax and producer warps
        if (tid < kC) idx_s[tid] = tid < count ? resolve(p, tid, raw_first) : -1;
        named_barrier(5, kFirstThreads);
        if (tid == 0) mbar_arrive(kv_first);  // every idx_s entry (release)
        gather_chunk(p, sbase, idx_s, 0, warp < kMmaWarp ? warp : warp - 1, kFirstThreads / 32, lane);
        cp_async_arrive_noinc(kv_first);
    }

    if (warp >= kProducerWarp) {
        // ================================================== producers
        const int g = tid - kProducerWarp * 32;
        for (int c = 1; c < nch; ++c) {
            const int b = c & 1;
            const int col = c * kC + g;
            const int32_t raw = (g < kC && col < count) ? idx_row[col] : -1;
            if (c >= 2) pv_wait(c - 2);
            if (g < kC) idx_s[b * kC + g] = col < count ? resolve(p, col, raw) : -1;
            named_barrier(3, kProducerThreads);
            if (g == 0) mbar_arrive(&kv_full[b]);
            gather_chunk(p, sbase + b * kStage, idx_s + b * kC, c * kC, g >> 5, kProducerThreads / 32, lane);
            cp_async_arrive_noinc(&kv_full[b]);
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        // ================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_e4m3(kC, kN, 0, 0);
            constexpr uint32_t kIdescRope = idesc_bf16_kmajor(kC, kN);
            constexpr uint32_t kIdescPV = idesc_e4m3(kC, kN, 1, 1);
            const uint64_t d_kv = smem_desc(sbase + kLat, 1024, 1024, kSwizzle128B);
            const uint64_t d_kv_rope = smem_desc(sbase + kRope, 1024, 1024, kSwizzle128B);
            const uint64_t d_q = smem_desc(sbase + kQ, 1024, 1024, kSwizzle128B);
            const uint64_t d_q_rope = smem_desc(sbase + kQRope, 1024, 1024, kSwizzle128B);
            const uint64_t d_p = smem_desc(sbase + kP, 8 * kN, 8 * kN, kSwizzle32B);
            int next_qk = 0, next_pv = 0;
            bool q_ready = false;
            uint64_t idle_since = 0;
            while (next_pv < nch) {
                bool progressed = false;
                if (!q_ready) q_ready = mbar_test_wait(q_full, 0);
                if (q_ready && next_qk < nch && next_qk <= next_pv + 1 &&
                    mbar_test_wait(kv_bar(next_qk), kv_parity(next_qk))) {
                    const int c = next_qk;
                    fence_proxy_async_smem();  // the producers' cp.async data, for the tensor cores
                    tc_fence_after_sync();
                    const uint32_t stage16 = static_cast<uint32_t>((c & 1) * kStage) >> 4;
                    const uint32_t d_s = tmem + (c & 1) * kSCols;
#pragma unroll
                    for (int a = 0; a < 4; ++a) {  // latent block a: its own accumulator
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_f8(d_s + a * kN, d_kv + stage16 + ((a * kC * 128 + ks * 32) >> 4),
                                   d_q + ((a * kN * 128 + ks * 32) >> 4), kIdescQK, ks != 0 ? 1u : 0u);
                    }
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)  // the rope: BF16, 16 values (32 bytes) a step
                        mma_bf16(d_s + 4 * kN, d_kv_rope + stage16 + ((ks * 32) >> 4), d_q_rope + ((ks * 32) >> 4),
                                 kIdescRope, ks != 0 ? 1u : 0u);
                    mma_commit(&s_full[c & 1]);
                    ++next_qk;
                    progressed = true;
                }
                if (next_pv < next_qk && mbar_test_wait(p_full, next_pv & 1)) {
                    const int c = next_pv;
                    tc_fence_after_sync();
                    const uint32_t stage16 = static_cast<uint32_t>((c & 1) * kStage) >> 4;
                    const uint32_t p16 = static_cast<uint32_t>((c & 1) * 4 * kPBlock) >> 4;
#pragma unroll
                    for (int kk = 0; kk < kC / 32; ++kk) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_f8(tmem + kOCol + j * kN, d_kv + stage16 + ((j * kC * 128 + kk * 32 * 128) >> 4),
                                   d_p + p16 + ((j * kPBlock + kk * 32 * kN) >> 4), kIdescPV,
                                   (c > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&pv_done[c & 1]);
                    ++next_pv;
                    progressed = true;
                }
                if (progressed) {
                    idle_since = 0;
                } else {
                    const uint64_t now = global_timer_ns();
                    if (idle_since == 0) idle_since = now;
                    if (*abort_flag || now - idle_since > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!q_ready) ok &= mbar_wait_bounded(q_full, 0, abort_flag, kWaitLimitNs);  // no copy outlives the CTA
            mma_commit(drain);
        }
        __syncwarp();
    } else {
        // ===================================================== softmax
        // Thread t owns key t of each chunk (TMEM lane t of S^T) and latent
        // row t of each O^T block.
        const int t = tid;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const float scale_log2 = p.scale_log2;
        float lsum[kN];
#pragma unroll
        for (int h = 0; h < kN; ++h) lsum[h] = 0.0f;

        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            ok &= mbar_wait_bounded(kv_bar(c), kv_parity(c), abort_flag, kWaitLimitNs);
            ok &= mbar_wait_bounded(&s_full[b], (c >> 1) & 1, abort_flag, kWaitLimitNs);
            tc_fence_after_sync();
            const bool active = idx_s[b * kC + t] >= 0;
            const float4 sc = *reinterpret_cast<const float4*>(smem + b * kStage + kScale + t * 16);
            // logits of this key: sum_b s_b S_b + S_rope (FP32)
            float s[kN];
            {
                const uint32_t col = tmem + lane_base + b * kSCols;
                tmem_load16x2(col + 4 * kN, col + 4 * kN + 16, s);
                const float sb[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    float v[kN];
                    tmem_load16x2(col + a * kN, col + a * kN + 16, v);
#pragma unroll
                    for (int h = 0; h < kN; ++h) s[h] = fmaf(sb[a], v[h], s[h]);
                }
            }
            // chunk maxima per head (transposing butterfly: lane l ends with
            // head l) and per block the largest |scale| of the active keys
            {
                float m[kN / 2];
                {
                    const bool up = (lane & 16) != 0;
#pragma unroll
                    for (int i = 0; i < kN / 2; ++i) {
                        const float lo = active ? s[i] : -INFINITY, hi = active ? s[i + kN / 2] : -INFINITY;
                        m[i] = fmaxf(up ? hi : lo, __shfl_xor_sync(0xFFFFFFFFu, up ? lo : hi, 16));
                    }
                }
#pragma unroll
                for (int o = 8, n = kN / 2; n > 1; o >>= 1, n >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < n / 2; ++i) {
                        const float send = up ? m[i] : m[i + n / 2];
                        const float keep = up ? m[i + n / 2] : m[i];
                        m[i] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
                    }
                }
                red[warp * kN + lane] = m[0];
                float g4[4] = {active ? fabsf(sc.x) : 0.0f, active ? fabsf(sc.y) : 0.0f, active ? fabsf(sc.z) : 0.0f,
                               active ? fabsf(sc.w) : 0.0f};
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int a = 0; a < 4; ++a) g4[a] = fmaxf(g4[a], __shfl_xor_sync(0xFFFFFFFFu, g4[a], o));
                if (lane < 4) sig_red[warp * 4 + lane] = g4[lane];
            }
            named_barrier(1, 128);
            if (t < kN) {
                const float cm = fmaxf(fmaxf(red[t], red[kN + t]), fmaxf(red[2 * kN + t], red[3 * kN + t]));
                const float mo = m_run_s[t];
                const float mn = fmaxf(mo, cm * scale_log2);
                alpha_s[t] = (mo == -INFINITY) ? 1.0f : fast_exp2(mo - mn);
                bias_s[t] = mn - kLog2P;
                m_run_s[t] = mn;
            } else if (t >= 64 && t < 68) {
                const int a = t - 64;
                const float so = sig_run[a];
                const float sn = fmaxf(so, fmaxf(fmaxf(sig_red[a], sig_red[4 + a]), fmaxf(sig_red[8 + a], sig_red[12 + a])));
                sig_beta[a] = (so > 0.0f && sn > so) ? so / sn : 1.0f;
                sig_run[a] = sn;
            }
            named_barrier(1, 128);

            // P = 2^(s * scale_log2 - m + log2 448) (FP32 sums of the
            // unrounded P) and P'_a = P * s_a / sigma_a as E4M3 into the four
            // P'^T blocks of buffer b (PV of chunk c - 2 has read them)
            if (c >= 2) pv_wait(c - 2);
            {
                float ratio[4];
                {
                    const float sb[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        const float sg = sig_run[a];
                        ratio[a] = sg > 0.0f ? sb[a] / sg : 0.0f;
                    }
                }
                uint8_t* pbuf = smem + kP + b * 4 * kPBlock;
#pragma unroll
                for (int g = 0; g < kN / 16; ++g) {
                    uint32_t words[4][4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int j = 16 * g + 4 * q4;
                        const float4 bi = reinterpret_cast<const float4*>(bias_s)[j / 4];
                        const float4 al = reinterpret_cast<const float4*>(alpha_s)[j / 4];
                        float pr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        if (active) {
                            pr[0] = fast_exp2(fmaf(s[j + 0], scale_log2, -bi.x));
                            pr[1] = fast_exp2(fmaf(s[j + 1], scale_log2, -bi.y));
                            pr[2] = fast_exp2(fmaf(s[j + 2], scale_log2, -bi.z));
                            pr[3] = fast_exp2(fmaf(s[j + 3], scale_log2, -bi.w));
                        }
                        lsum[j + 0] = fmaf(lsum[j + 0], al.x, pr[0]);
                        lsum[j + 1] = fmaf(lsum[j + 1], al.y, pr[1]);
                        lsum[j + 2] = fmaf(lsum[j + 2], al.z, pr[2]);
                        lsum[j + 3] = fmaf(lsum[j + 3], al.w, pr[3]);
#pragma unroll
                        for (int a = 0; a < 4; ++a)
                            words[a][q4] = e4m3x2(pr[0] * ratio[a], pr[1] * ratio[a]) |
                                           (e4m3x2(pr[2] * ratio[a], pr[3] * ratio[a]) << 16);
                    }
#pragma unroll
                    for (int a = 0; a < 4; ++a)
                        *reinterpret_cast<uint4*>(pbuf + a * kPBlock + p_unit(t, g)) =
                            make_uint4(words[a][0], words[a][1], words[a][2], words[a][3]);
                }
            }

            // O^T block a *= alpha(head) * beta(a) where either moved (PV of
            // chunk c - 1 is done)
            if (c >= 1) {
                pv_wait(c - 1);
                tc_fence_after_sync();
                bool any_alpha = false;
#pragma unroll
                for (int j4 = 0; j4 < kN / 4; ++j4) {
                    const float4 v4 = reinterpret_cast<const float4*>(alpha_s)[j4];
                    any_alpha |= (v4.x != 1.0f) | (v4.y != 1.0f) | (v4.z != 1.0f) | (v4.w != 1.0f);
                }
#pragma unroll 1
                for (int a = 0; a < 4; ++a) {
                    const float beta = sig_beta[a];
                    if (!any_alpha && beta == 1.0f) continue;
                    const uint32_t col = tmem + lane_base + kOCol + a * kN;
                    float v[kN];
                    tmem_load16x2(col, col + 16, v);
#pragma unroll
                    for (int j4 = 0; j4 < kN / 4; ++j4) {
                        const float4 al = reinterpret_cast<const float4*>(alpha_s)[j4];
                        v[4 * j4 + 0] *= al.x * beta;
                        v[4 * j4 + 1] *= al.y * beta;
                        v[4 * j4 + 2] *= al.z * beta;
                        v[4 * j4 + 3] *= al.w * beta;
                    }
                    tmem_store16x2(col, col + 16, v);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(p_full);
        }
        if (nch > 0) pv_wait(nch - 1);
        tc_fence_after_sync();

        // per-head totals of the per-thread partial sums
#pragma unroll
        for (int j = 0; j < kN; ++j) {
            float v = lsum[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == j) red[warp * kN + j] = v;
        }
        named_barrier(1, 128);
        if (t < kN) l_s[t] = (red[t] + red[kN + t]) + (red[2 * kN + t] + red[3 * kN + t]);
    }
    if (!ok) {
        *abort_flag = 1;
        atomicOr(p.error, SMLA_DEV_TIMEOUT);
    }
    cp_async_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // ================================================ epilogue
    // bias_s becomes each head's output factor; O^T rows -> BF16 [32][512]
    // in the free KV stage, then 16-byte stores to out.
    if (tid < kN) {
        const int h = head0 + tid;
        const float m = m_run_s[tid];
        float scale = 0.0f, lse2 = -INFINITY;
        if (m != -INFINITY) {
            float top = m, extra = 0.0f;
            if (p.sinks != nullptr) {
                top = fmaxf(m, sink_of_head);
                extra = 448.0f * fast_exp2(sink_of_head - top);
            }
            const float w = fast_exp2(m - top);
            const float total = l_s[tid] * w + extra;
            scale = p.out_scale * w / total;
            lse2 = top - kLog2P + log2f(total);
        }
        bias_s[tid] = scale;
        if (p.lse != nullptr) p.lse[static_cast<int64_t>(token) * p.lse_stride_token + h] = lse2;
    }
    __syncthreads();
    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem + kLat);
    if (warp < 4) {
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
        for (int a = 0; a < 4; ++a) {
            float v[kN];
            const uint32_t col = tmem + lane_base + kOCol + a * kN;
            tmem_load16x2(col, col + 16, v);
            const float sg = sig_run[a];
            const int lat = a * 128 + tid;
            // a head without active keys has factor 0 and gets +0.0 (its
            // O^T block may never have been written)
#pragma unroll
            for (int h = 0; h < kN; ++h) {
                const float f = sg * bias_s[h];
                tile[h * 512 + lat] = __float2bfloat16_rn(f == 0.0f ? 0.0f : v[h] * f);
            }
        }
    }
    __syncthreads();
    store_tile(p, tile, token, head0, kN, tid, kThreads);

    // ---- teardown: every MMA and TMEM access has finished -----------------
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        if (!mbar_wait_bounded(drain, 0, abort_flag, kWaitLimitNs)) {
            if (lane == 0) atomicOr(p.error, SMLA_DEV_TIMEOUT);
        }
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// 64 heads per CTA. The same arithmetic, step for step and in the same order,
// as the 32-head kernel above; what changes is where the products live:
//   * TMEM: the four O^T blocks of 64 heads take 256 columns, so the five
//     accumulators of a chunk's QK (the rope first, then latent blocks 0..3)
//     take turns in a ring of four 64-column slots. The softmax reads each
//     slot into registers as soon as its product lands and frees it at once,
//     so the next chunk's products start while it works on this one.
//   * shared memory: two stages of 82 KB and a 40 KB Q leave room for two
//     P'_b^T buffers of 8 KB, which take P'_0 and P'_1; P'_2 and P'_3 take
//     the chunk's 16 KB of rope rows, which nothing reads once its QK is done
//     and nothing writes before its PV is done (the stage is refilled only
//     then).
// Two softmax warpgroups (32 heads each), six producer warps and two issuing
// warps: one for the QK products, one for PV, so that neither waits behind
// the other's bursts (a burst of four MMAs and its commit takes a few hundred
// cycles to issue).
namespace wide {

constexpr int kN = 64;
constexpr int kThreads = 512;
constexpr int kMmaWarp = 8;         // issues the QK products (and holds the TMEM allocation)
constexpr int kProducerWarp = 9;    // first of six
constexpr int kPvWarp = 15;         // issues the PV products
constexpr int kGatherThreads = 192;  // warps 9..14
constexpr int kFirstThreads = 256 + kGatherThreads;  // chunk 0: the softmax and producer warps
constexpr int kQ = 2 * kStage;
constexpr int kQRope = kQ + 4 * kN * 128;
constexpr int kPBlock = kC * kN;              // P'_b^T: 128 keys x 64 heads of E4M3
constexpr int kP = kQRope + kN * 128;         // P'_0, P'_1 (P'_2, P'_3 in the stage's rope rows)
static_assert(2 * kPBlock == kC * 128 && kRope % 1024 == 0, "two P' blocks fill the rope rows of a stage");
constexpr int kIdx = kP + 2 * kPBlock;        // int32 [2][128]
constexpr int kRed = kIdx + 2 * kC * 4;       // float [4 warps][64 heads]
constexpr int kSig = kRed + 4 * kN * 4;       // per warpgroup: float [4 warps][4 blocks], sigma[4], beta[4]
constexpr int kSigBytes = 128;
constexpr int kHead = kSig + 2 * kSigBytes;   // float [4][64]: m_run, bias, alpha, l
constexpr int kBar = kHead + 4 * kN * 4;      // 32 mbarriers
constexpr int kMisc = kBar + 32 * 8;
constexpr int kBytes = kMisc + 64;
constexpr int kAlloc = kBytes + 1024;
static_assert(kAlloc <= 227 * 1024, "one CTA's shared memory");
static_assert(kQ % 1024 == 0 && kQRope % 1024 == 0 && kP % 1024 == 0, "aligned tiles");
static_assert(kN * 512 * 2 <= kStage, "the epilogue's BF16 tile fits in a stage");

// TMEM columns: O^T block j at 64 j, S slot i at 256 + 64 i.
constexpr int kSlot0 = 4 * kN;
constexpr int kTmemCols = 512;
constexpr int kAccPerChunk = 5;  // the rope, then latent blocks 0..3

// P'^T of one block: 128 keys x 64 heads, MN-major, 64-byte swizzle.
__device__ __forceinline__ uint32_t p_unit64(int key, int unit) {
    return static_cast<uint32_t>(key * kN + ((unit ^ ((key >> 1) & 3)) << 4));
}

__global__ void __launch_bounds__(kThreads, 1) ds_mla_decode_kernel64(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBar);
    uint64_t* kv_full = bars + 0;      // [2] a stage's rows landed (192 cp.async arrivals + 1)
    uint64_t* stage_free = bars + 2;   // [2] PV of the stage's chunk finished
    uint64_t* slot_full = bars + 4;    // [4] a QK product landed in the slot
    uint64_t* slot_free = bars + 8;    // [4] the softmax read the slot (one arrival per softmax warp)
    uint64_t* p_full = bars + 12;      // [4] P'_b written, O^T block b rescaled (256 arrivals)
    uint64_t* drain = bars + 16;       // every MMA of both issuing threads finished
    uint64_t* q_full = bars + 17;      // the Q tiles landed
    uint64_t* kv_first = bars + 18;    // chunk 0 landed (448 cp.async arrivals + 1)
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + kIdx);
    float* red = reinterpret_cast<float*>(smem + kRed);
    float* m_run_s = reinterpret_cast<float*>(smem + kHead);
    float* bias_s = m_run_s + kN;
    float* alpha_s = m_run_s + 2 * kN;
    float* l_s = m_run_s + 3 * kN;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int head0 = static_cast<int>(blockIdx.x) * kN;
    const int token = blockIdx.y;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kv_full[i], kGatherThreads + 1);
            mbar_init(&stage_free[i], 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&slot_full[i], 1);
            mbar_init(&slot_free[i], 8);
            mbar_init(&p_full[i], 256);
        }
        mbar_init(drain, 2);  // one commit from each issuing thread
        mbar_init(q_full, 1);
        mbar_init(kv_first, kFirstThreads + 1);
        misc[1] = 0;
        mbar_init_fence();
    }
    if (tid < kN) {
        m_run_s[tid] = -INFINITY;
        bias_s[tid] = -INFINITY;
        alpha_s[tid] = 1.0f;
        l_s[tid] = 0.0f;
    }
    if (tid < 8) {  // each warpgroup's sigma[4] and beta[4]
        float* sg = reinterpret_cast<float*>(smem + kSig + (tid >> 2) * kSigBytes) + 16;
        sg[tid & 3] = 0.0f;
        sg[4 + (tid & 3)] = 1.0f;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(misc, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensor_map(&p.q_latent);
        prefetch_tensor_map(&p.q_rope);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    grid_dependency_wait();  // inputs are read only after this point
    if (warp == kProducerWarp && lane == 0) {
        mbar_arrive_expect_tx(q_full, kN * 512 + kN * 128);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
            tma_load_3d(sbase + kQ + kb * kN * 128, &p.q_latent, kb * 128, head0, token, q_full);
        tma_load_3d(sbase + kQRope, &p.q_rope, 0, head0, token, q_full);
    }
    const int32_t* idx_row = p.indices + static_cast<int64_t>(token) * p.idx_stride;
    int32_t raw_first = -1;
    if (tid < kC && tid < p.width) raw_first = idx_row[tid];
    const int count = min(max(p.lens[token], 0), p.width);
    const float sink_of_head = (tid < kN && p.sinks != nullptr) ? p.sinks[head0 + tid] * kLog2e : -INFINITY;
    const int nch = (count + kC - 1) / kC;
    grid_launch_dependents();

    bool ok = true;
    auto kv_bar = [&](int c) -> uint64_t* { return c == 0 ? kv_first : &kv_full[c & 1]; };
    auto kv_parity = [&](int c) -> uint32_t {
        return c == 0 ? 0u : static_cast<uint32_t>(((c >> 1) - ((c & 1) ? 0 : 1)) & 1);
    };

    if (warp != kMmaWarp && warp != kPvWarp && nch > 0) {
        // ===================== chunk 0 by the softmax and producer warps
        if (tid < kC) idx_s[tid] = tid < count ? resolve(p, tid, raw_first) : -1;
        named_barrier(5, kFirstThreads);
        if (tid == 0) mbar_arrive(kv_first);  // every idx_s entry (release)
        gather_chunk(p, sbase, idx_s, 0, warp < kMmaWarp ? warp : warp - 1, kFirstThreads / 32, lane);
        cp_async_arrive_noinc(kv_first);
    }

    if (warp >= kProducerWarp && warp < kPvWarp) {
        // ================================================== producers
        const int g = tid - kProducerWarp * 32;
        for (int c = 1; c < nch; ++c) {
            const int b = c & 1;
            const int col = c * kC + g;
            const int32_t raw = (g < kC && col < count) ? idx_row[col] : -1;
            if (c >= 2)
                ok &= mbar_wait_bounded(&stage_free[b], static_cast<uint32_t>(((c - 2) >> 1) & 1), abort_flag,
                                        kWaitLimitNs);
            if (g < kC) idx_s[b * kC + g] = col < count ? resolve(p, col, raw) : -1;
            named_barrier(3, kGatherThreads);
            if (g == 0) mbar_arrive(&kv_full[b]);
            gather_chunk(p, sbase + b * kStage, idx_s + b * kC, c * kC, g >> 5, kGatherThreads / 32, lane);
            cp_async_arrive_noinc(&kv_full[b]);
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        // ===================================== QK issuer: the five products
        // of each chunk into the slot ring, in order
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_e4m3(kC, kN, 0, 0);
            constexpr uint32_t kIdescRope = idesc_bf16_kmajor(kC, kN);
            const uint64_t d_kv = smem_desc(sbase + kLat, 1024, 1024, kSwizzle128B);
            const uint64_t d_kv_rope = smem_desc(sbase + kRope, 1024, 1024, kSwizzle128B);
            const uint64_t d_q = smem_desc(sbase + kQ, 1024, 1024, kSwizzle128B);
            const uint64_t d_q_rope = smem_desc(sbase + kQRope, 1024, 1024, kSwizzle128B);
            ok &= mbar_wait_bounded(q_full, 0, abort_flag, kWaitLimitNs);  // also: no copy outlives the CTA
            for (int acc = 0; ok && acc < kAccPerChunk * nch; ++acc) {
                const int c = acc / kAccPerChunk, a = acc % kAccPerChunk;
                const int slot = acc & 3, use = acc >> 2;
                if (a == 0) {
                    ok &= mbar_wait_bounded(kv_bar(c), kv_parity(c), abort_flag, kWaitLimitNs);
                    fence_proxy_async_smem();  // the producers' cp.async data, for the tensor cores
                }
                if (use >= 1)
                    ok &= mbar_wait_bounded(&slot_free[slot], static_cast<uint32_t>((use - 1) & 1), abort_flag,
                                            kWaitLimitNs);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t stage16 = static_cast<uint32_t>((c & 1) * kStage) >> 4;
                const uint32_t d_s = tmem + kSlot0 + slot * kN;
                if (a == 0) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)  // the rope: BF16, 16 values (32 bytes) a step
                        mma_bf16(d_s, d_kv_rope + stage16 + ((ks * 32) >> 4), d_q_rope + ((ks * 32) >> 4),
                                 kIdescRope, ks != 0 ? 1u : 0u);
                } else {
                    const int lb = a - 1;  // latent block
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f8(d_s, d_kv + stage16 + ((lb * kC * 128 + ks * 32) >> 4),
                               d_q + ((lb * kN * 128 + ks * 32) >> 4), kIdescQK, ks != 0 ? 1u : 0u);
                }
                mma_commit(&slot_full[slot]);
            }
            mma_commit(drain);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ===================================== PV issuer: block by block as
        // the softmax hands each P' block over
        if (lane == 0) {
            constexpr uint32_t kIdescPV = idesc_e4m3(kC, kN, 1, 1);
            const uint64_t d_kv = smem_desc(sbase + kLat, 1024, 1024, kSwizzle128B);
            const uint64_t d_p = smem_desc(sbase + kP, 8 * kN, 8 * kN, kSwizzle64B);
            const uint64_t d_p_rope = smem_desc(sbase + kRope, 8 * kN, 8 * kN, kSwizzle64B);
            for (int c = 0; ok && c < nch; ++c) {
                const uint32_t stage16 = static_cast<uint32_t>((c & 1) * kStage) >> 4;
                for (int j = 0; j < 4; ++j) {
                    ok &= mbar_wait_bounded(&p_full[j], static_cast<uint32_t>(c & 1), abort_flag, kWaitLimitNs);
                    if (!ok) break;
                    tc_fence_after_sync();
                    // P'_0, P'_1 in their own buffers, P'_2, P'_3 in the chunk's rope rows
                    const uint64_t d_pj = j < 2 ? d_p + ((j * kPBlock) >> 4)
                                                : d_p_rope + stage16 + (((j - 2) * kPBlock) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kC / 32; ++kk)
                        mma_f8(tmem + j * kN, d_kv + stage16 + ((j * kC * 128 + kk * 32 * 128) >> 4),
                               d_pj + ((kk * 32 * kN) >> 4), kIdescPV, (c > 0 || kk > 0) ? 1u : 0u);
                    if (j == 3) mma_commit(&stage_free[c & 1]);
                }
            }
            mma_commit(drain);
        }
        __syncwarp();
    } else {
        // ===================================================== softmax
        // Warpgroup wg owns heads 32 wg .. 32 wg + 31; thread t owns key t of
        // each chunk (TMEM lane t) and latent row t of each O^T block.
        const int wg = warp >> 2, t = tid & 127, hb = 32 * wg;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float scale_log2 = p.scale_log2;
        float* sig_red = reinterpret_cast<float*>(smem + kSig + wg * kSigBytes);  // [4 warps][4 blocks]
        float* sig_run = sig_red + 16;
        float* sig_beta = sig_red + 20;
        float lsum[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) lsum[h] = 0.0f;

        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            ok &= mbar_wait_bounded(kv_bar(c), kv_parity(c), abort_flag, kWaitLimitNs);
            const bool active = idx_s[b * kC + t] >= 0;
            const float4 sc = *reinterpret_cast<const float4*>(smem + b * kStage + kScale + t * 16);
            const float sb[4] = {sc.x, sc.y, sc.z, sc.w};
            // logits of this key: S_rope + sum_b s_b S_b (FP32), slot by slot
            float s[32];
#pragma unroll 1
            for (int a = 0; a < kAccPerChunk; ++a) {
                const int acc = kAccPerChunk * c + a, slot = acc & 3;
                ok &= mbar_wait_bounded(&slot_full[slot], static_cast<uint32_t>((acc >> 2) & 1), abort_flag,
                                        kWaitLimitNs);
                tc_fence_after_sync();
                const uint32_t col = tmem + lane_base + kSlot0 + slot * kN + hb;
                if (a == 0) {
                    tmem_load16x2(col, col + 16, s);
                } else {
                    const float f = a == 1 ? sb[0] : a == 2 ? sb[1] : a == 3 ? sb[2] : sb[3];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float v[16];
                        tmem_load16x1(col + 16 * half, v);
#pragma unroll
                        for (int h = 0; h < 16; ++h) s[16 * half + h] = fmaf(f, v[h], s[16 * half + h]);
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&slot_free[slot]);
            }
            // chunk maxima per head (transposing butterfly: lane l ends with
            // head hb + l) and per block the largest |scale| of the active keys
            {
                float m[16];
                {
                    const bool up = (lane & 16) != 0;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float lo = active ? s[i] : -INFINITY, hi = active ? s[i + 16] : -INFINITY;
                        m[i] = fmaxf(up ? hi : lo, __shfl_xor_sync(0xFFFFFFFFu, up ? lo : hi, 16));
                    }
                }
#pragma unroll
                for (int o = 8, n = 16; n > 1; o >>= 1, n >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < n / 2; ++i) {
                        const float send = up ? m[i] : m[i + n / 2];
                        const float keep = up ? m[i + n / 2] : m[i];
                        m[i] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
                    }
                }
                red[(warp & 3) * kN + hb + lane] = m[0];
                float g4[4] = {active ? fabsf(sc.x) : 0.0f, active ? fabsf(sc.y) : 0.0f, active ? fabsf(sc.z) : 0.0f,
                               active ? fabsf(sc.w) : 0.0f};
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int a = 0; a < 4; ++a) g4[a] = fmaxf(g4[a], __shfl_xor_sync(0xFFFFFFFFu, g4[a], o));
                if (lane < 4) sig_red[(warp & 3) * 4 + lane] = g4[lane];
            }
            named_barrier(1 + wg, 128);
            if (t < 32) {
                const int h = hb + t;
                const float cm = fmaxf(fmaxf(red[h], red[kN + h]), fmaxf(red[2 * kN + h], red[3 * kN + h]));
                const float mo = m_run_s[h];
                const float mn = fmaxf(mo, cm * scale_log2);
                alpha_s[h] = (mo == -INFINITY) ? 1.0f : fast_exp2(mo - mn);
                bias_s[h] = mn - kLog2P;
                m_run_s[h] = mn;
            } else if (t >= 64 && t < 68) {
                const int a = t - 64;
                const float so = sig_run[a];
                const float sn = fmaxf(so, fmaxf(fmaxf(sig_red[a], sig_red[4 + a]), fmaxf(sig_red[8 + a], sig_red[12 + a])));
                sig_beta[a] = (so > 0.0f && sn > so) ? so / sn : 1.0f;
                sig_run[a] = sn;
            }
            named_barrier(1 + wg, 128);

            // P = 2^(s * scale_log2 - m + log2 448) in place of s (FP32 sums of
            // the unrounded P)
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
                const float4 bi = reinterpret_cast<const float4*>(bias_s + hb)[j4];
                const float4 al = reinterpret_cast<const float4*>(alpha_s + hb)[j4];
                const int j = 4 * j4;
                float pr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (active) {
                    pr[0] = fast_exp2(fmaf(s[j + 0], scale_log2, -bi.x));
                    pr[1] = fast_exp2(fmaf(s[j + 1], scale_log2, -bi.y));
                    pr[2] = fast_exp2(fmaf(s[j + 2], scale_log2, -bi.z));
                    pr[3] = fast_exp2(fmaf(s[j + 3], scale_log2, -bi.w));
                }
                lsum[j + 0] = fmaf(lsum[j + 0], al.x, pr[0]);
                lsum[j + 1] = fmaf(lsum[j + 1], al.y, pr[1]);
                lsum[j + 2] = fmaf(lsum[j + 2], al.z, pr[2]);
                lsum[j + 3] = fmaf(lsum[j + 3], al.w, pr[3]);
                s[j + 0] = pr[0];
                s[j + 1] = pr[1];
                s[j + 2] = pr[2];
                s[j + 3] = pr[3];
            }
            bool any_alpha = false;
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
                const float4 v4 = reinterpret_cast<const float4*>(alpha_s + hb)[j4];
                any_alpha |= (v4.x != 1.0f) | (v4.y != 1.0f) | (v4.z != 1.0f) | (v4.w != 1.0f);
            }

            // PV of chunk c - 1 has finished: its P'_0 and P'_1 buffers are free
            // and its O^T blocks final for this step
            if (c >= 1)
                ok &= mbar_wait_bounded(&stage_free[(c - 1) & 1], static_cast<uint32_t>(((c - 1) >> 1) & 1),
                                        abort_flag, kWaitLimitNs);
            // block by block: P'_a = P * s_a / sigma_a as E4M3 (P'_0 and P'_1
            // into their buffers, P'_2 and P'_3 into this chunk's rope rows,
            // which its QK has finished reading), then O^T block a *= alpha(head)
            // * beta(a) where either moved; PV of the block may start at once
#pragma unroll 1
            for (int a = 0; a < 4; ++a) {
                const float sg = sig_run[a];
                const float ratio = sg > 0.0f ? (a == 0 ? sb[0] : a == 1 ? sb[1] : a == 2 ? sb[2] : sb[3]) / sg : 0.0f;
                uint8_t* pbuf = a < 2 ? smem + kP + a * kPBlock : smem + b * kStage + kRope + (a - 2) * kPBlock;
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    uint32_t words[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int j = 16 * g + 4 * q4;
                        words[q4] = e4m3x2(s[j + 0] * ratio, s[j + 1] * ratio) |
                                    (e4m3x2(s[j + 2] * ratio, s[j + 3] * ratio) << 16);
                    }
                    *reinterpret_cast<uint4*>(pbuf + p_unit64(t, 2 * wg + g)) =
                        make_uint4(words[0], words[1], words[2], words[3]);
                }
                const float beta = sig_beta[a];
                if (c >= 1 && (any_alpha || beta != 1.0f)) {
                    tc_fence_after_sync();
                    const uint32_t col = tmem + lane_base + a * kN + hb;
                    float v[32];
                    tmem_load16x2(col, col + 16, v);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 al = reinterpret_cast<const float4*>(alpha_s + hb)[j4];
                        v[4 * j4 + 0] *= al.x * beta;
                        v[4 * j4 + 1] *= al.y * beta;
                        v[4 * j4 + 2] *= al.z * beta;
                        v[4 * j4 + 3] *= al.w * beta;
                    }
                    tmem_store16x2(col, col + 16, v);
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&p_full[a]);
            }
        }
        // every PV finished
        if (nch > 0)
            ok &= mbar_wait_bounded(&stage_free[(nch - 1) & 1], static_cast<uint32_t>(((nch - 1) >> 1) & 1),
                                    abort_flag, kWaitLimitNs);
        tc_fence_after_sync();

        // per-head totals of the per-thread partial sums
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            float v = lsum[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == j) red[(warp & 3) * kN + hb + j] = v;
        }
        named_barrier(1 + wg, 128);
        if (t < 32) {
            const int h = hb + t;
            l_s[h] = (red[h] + red[kN + h]) + (red[2 * kN + h] + red[3 * kN + h]);
        }
    }
    if (!ok) {
        *abort_flag = 1;
        atomicOr(p.error, SMLA_DEV_TIMEOUT);
    }
    cp_async_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // ================================================ epilogue
    // bias_s becomes each head's output factor; O^T rows -> BF16 [64][512]
    // in the free KV stage, then 16-byte stores to out.
    if (tid < kN) {
        const int h = head0 + tid;
        const float m = m_run_s[tid];
        float scale = 0.0f, lse2 = -INFINITY;
        if (m != -INFINITY) {
            float top = m, extra = 0.0f;
            if (p.sinks != nullptr) {
                top = fmaxf(m, sink_of_head);
                extra = 448.0f * fast_exp2(sink_of_head - top);
            }
            const float w = fast_exp2(m - top);
            const float total = l_s[tid] * w + extra;
            scale = p.out_scale * w / total;
            lse2 = top - kLog2P + log2f(total);
        }
        bias_s[tid] = scale;
        if (p.lse != nullptr) p.lse[static_cast<int64_t>(token) * p.lse_stride_token + h] = lse2;
    }
    __syncthreads();
    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem + kLat);
    if (warp < 8) {
        const int wg = warp >> 2, hb = 32 * wg;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float* sig_run = reinterpret_cast<const float*>(smem + kSig) + 16;  // warpgroup 0's copy
#pragma unroll 1
        for (int a = 0; a < 4; ++a) {
            float v[32];
            const uint32_t col = tmem + lane_base + a * kN + hb;
            tmem_load16x2(col, col + 16, v);
            const float sg = sig_run[a];
            const int lat = a * 128 + (tid & 127);
            // a head without active keys has factor 0 and gets +0.0 (its
            // O^T block may never have been written)
#pragma unroll
            for (int h = 0; h < 32; ++h) {
                const float f = sg * bias_s[hb + h];
                tile[(hb + h) * 512 + lat] = __float2bfloat16_rn(f == 0.0f ? 0.0f : v[h] * f);
            }
        }
    }
    __syncthreads();
    store_tile(p, tile, token, head0, kN, tid, kThreads);

    // ---- teardown: every MMA and TMEM access has finished -----------------
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        if (!mbar_wait_bounded(drain, 0, abort_flag, kWaitLimitNs)) {
            if (lane == 0) atomicOr(p.error, SMLA_DEV_TIMEOUT);
        }
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace wide

bool g_configured[64] = {};
bool g_configured_wide[64] = {};

// Heads per CTA for the shape: 64 where H allows it and the 64-head grid
// takes fewer waves of the device's SMs than the 32-head grid (its CTAs land
// each row in half as many SMs), else 32; `forced` 32 or 64 overrides.
int head_tile_for(int tokens, int heads, int forced, int num_sms) {
    if (forced == 32 || forced == 64) return forced;
    if (heads % 64 != 0 || num_sms <= 0) return 32;
    const int64_t ctas32 = static_cast<int64_t>(tokens) * (heads / 32), ctas64 = ctas32 / 2;
    const int64_t waves32 = (ctas32 + num_sms - 1) / num_sms, waves64 = (ctas64 + num_sms - 1) / num_sms;
    return waves64 < waves32 ? 64 : 32;
}

int device_sms(int dev) {
    static std::atomic<int> cached[64];
    if (dev < 0 || dev >= 64) return 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0 && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
        cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace dsmla
}  // namespace smla

extern "C" int smla_decode_ds_mla(const smla_ds_mla_shape* shape, const void* q_latent, const void* q_rope,
                                  const smla_pool* kv_pools, const int32_t* indices, const int32_t* lens,
                                  const float* sinks, float bmm1_scale, float bmm2_scale, void* out, float* lse,
                                  void* stream) {
    using namespace smla::dsmla;
    if (shape == nullptr) return SMLA_EINVAL;
    const smla_ds_mla_shape& s = *shape;
    if (s.tokens < 0 || s.width < 0 || s.heads <= 0 || s.heads % kN != 0) return SMLA_EINVAL;
    if (s.head_tile != 0 && s.head_tile != 32 && s.head_tile != 64) return SMLA_EINVAL;
    if (s.head_tile == 64 && s.heads % 64 != 0) return SMLA_EINVAL;
    if (s.heads > 1024 || s.tokens > 65535) return SMLA_EUNSUPPORTED;
    if (s.num_pools != 1 && s.num_pools != 2) return SMLA_EUNSUPPORTED;
    if (s.num_pools == 2 && (s.pool_split < 0 || s.pool_split > s.width)) return SMLA_EINVAL;
    if (s.q_stride_token < 0 || s.q_stride_head < 0 || s.q_stride_token % 16 || s.q_stride_head % 16 ||
        (s.heads > 1 && s.q_stride_head < 512))
        return SMLA_EINVAL;
    if (s.rope_stride_token < 0 || s.rope_stride_head < 0 || s.rope_stride_token % 8 || s.rope_stride_head % 8 ||
        (s.heads > 1 && s.rope_stride_head < 64))
        return SMLA_EINVAL;
    if (s.idx_stride_token < s.width || s.out_stride_token < 0 || s.lse_stride_token < 0) return SMLA_EINVAL;
    if ((s.heads > 1 && s.out_stride_head < 512) || s.out_stride_head < 0 || s.out_stride_token % 2 ||
        s.out_stride_head % 2)
        return SMLA_EINVAL;
    if (s.tokens == 0) return SMLA_OK;
    if (q_latent == nullptr || q_rope == nullptr || kv_pools == nullptr || lens == nullptr || out == nullptr)
        return SMLA_EINVAL;
    if (indices == nullptr && s.width > 0) return SMLA_EINVAL;
    if ((reinterpret_cast<uintptr_t>(q_latent) & 15u) || (reinterpret_cast<uintptr_t>(q_rope) & 15u) ||
        (reinterpret_cast<uintptr_t>(out) & 3u))
        return SMLA_EINVAL;
    for (int i = 0; i < s.num_pools; ++i) {
        const smla_pool& pl = kv_pools[i];
        if (pl.data == nullptr || pl.rows < 0 || pl.row_bytes != kRowBytes) return SMLA_EINVAL;
        if (reinterpret_cast<uintptr_t>(pl.data) & 15u) return SMLA_EINVAL;
        if (pl.rows > 0x7FFFFFFFll) return SMLA_EUNSUPPORTED;
    }
    if (!std::isfinite(bmm1_scale) || !std::isfinite(bmm2_scale) || !(bmm1_scale > 0.0f)) return SMLA_EINVAL;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        smla::note_cuda_error(static_cast<int>(e));
        return SMLA_ECUDA;
    }
    const int tile = head_tile_for(s.tokens, s.heads, s.head_tile, device_sms(dev));

    Params p;
    std::memset(&p, 0, sizeof(p));
    {
        // Q latent as {512 bytes, H, T} and Q rope as {128 bytes, H, T}: boxes
        // of one 128-byte row x the CTA's heads (a one-token call's token
        // stride is never used; it is given a legal value)
        const int64_t qt = s.tokens == 1 && s.q_stride_token < s.q_stride_head * s.heads
                               ? s.q_stride_head * s.heads : s.q_stride_token;
        const int64_t rt = s.tokens == 1 && s.rope_stride_token < s.rope_stride_head * s.heads
                               ? s.rope_stride_head * s.heads : s.rope_stride_token;
        const cuuint64_t qdims[3] = {512, static_cast<cuuint64_t>(s.heads), static_cast<cuuint64_t>(s.tokens)};
        const cuuint64_t qstrides[2] = {static_cast<cuuint64_t>(s.heads > 1 ? s.q_stride_head : 512),
                                        static_cast<cuuint64_t>(qt > 0 ? qt : 512)};
        const cuuint64_t rdims[3] = {128, static_cast<cuuint64_t>(s.heads), static_cast<cuuint64_t>(s.tokens)};
        const cuuint64_t rstrides[2] = {static_cast<cuuint64_t>(s.heads > 1 ? s.rope_stride_head * 2 : 128),
                                        static_cast<cuuint64_t>(rt > 0 ? rt * 2 : 128)};
        const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(tile), 1};
        if (!smla::encode_bytes_map(&p.q_latent, q_latent, 3, qdims, qstrides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B) ||
            !smla::encode_bytes_map(&p.q_rope, q_rope, 3, rdims, rstrides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
            return SMLA_EUNSUPPORTED;
    }
    const smla_pool& second = s.num_pools == 2 ? kv_pools[1] : kv_pools[0];
    p.pool0 = static_cast<const uint8_t*>(kv_pools[0].data);
    p.rows0 = kv_pools[0].rows;
    p.pool1 = static_cast<const uint8_t*>(second.data);
    p.rows1 = second.rows;
    p.indices = indices;
    p.idx_stride = s.idx_stride_token;
    p.lens = lens;
    p.sinks = sinks;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.out_stride_token = s.out_stride_token;
    p.out_stride_head = s.out_stride_head;
    p.lse = lse;
    p.lse_stride_token = s.lse_stride_token;
    p.width = s.width;
    p.pool_split = s.num_pools == 2 ? s.pool_split : 0;
    p.num_pools = s.num_pools;
    p.scale_log2 = static_cast<float>(static_cast<double>(bmm1_scale) * 1.4426950408889634);
    p.out_scale = bmm2_scale;
    p.error = smla::device_error_word();

    if (p.error == nullptr) e = cudaErrorInvalidSymbol;
    const bool wide64 = tile == 64;
    bool* configured = wide64 ? g_configured_wide : g_configured;
    if (e == cudaSuccess && dev < 64 && !configured[dev]) {
        e = wide64 ? cudaFuncSetAttribute(wide::ds_mla_decode_kernel64, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          wide::kAlloc)
                   : cudaFuncSetAttribute(ds_mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
        if (e == cudaSuccess) configured[dev] = true;
    }
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(s.heads / tile), static_cast<unsigned>(s.tokens), 1);
        cfg.blockDim = dim3(wide64 ? wide::kThreads : kThreads, 1, 1);
        cfg.dynamicSmemBytes = wide64 ? wide::kAlloc : kAlloc;
        cfg.stream = static_cast<cudaStream_t>(stream);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = smla::dependent_launch() ? 1 : 0;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = wide64 ? cudaLaunchKernelEx(&cfg, wide::ds_mla_decode_kernel64, p)
                   : cudaLaunchKernelEx(&cfg, ds_mla_decode_kernel, p);
    }
    if (e != cudaSuccess) {
        smla::note_cuda_error(static_cast<int>(e));
        return SMLA_ECUDA;
    }
    return SMLA_OK;
}

extern "C" int smla_ds_mla_head_tile(const smla_ds_mla_shape* shape, int num_sms) {
    using namespace smla::dsmla;
    if (shape == nullptr || shape->tokens < 0 || shape->heads <= 0 || shape->heads % kN != 0) return SMLA_EINVAL;
    if (shape->head_tile != 0 && shape->head_tile != 32 && shape->head_tile != 64) return SMLA_EINVAL;
    if (shape->head_tile == 64 && shape->heads % 64 != 0) return SMLA_EINVAL;
    if (num_sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ECUDA;
        num_sms = device_sms(dev);
        if (num_sms <= 0) return SMLA_ECUDA;
    }
    return head_tile_for(shape->tokens, shape->heads, shape->head_tile, num_sms);
}
