// smla_decode.cu -- sparse MLA decode attention for sm_103a, and the C ABI
// declared in include/smla.h.
//
// The operation is the one stated on the DeepSeek-V4.1 "sparse_mla_cute" page
// (module docstring, "What this module computes"): per token and head, softmax
// attention over the token's active gathered KV rows, with optional per-head
// sinks. The datapath follows the Kimi K3.1 "attn_sparse" page (module
// docstring, per-chunk steps and "Precision"; SparseDcpDecode.merge): FP32
// logits, base-2 online softmax per chunk, P rounded to E4M3 at 448 of the
// running maximum, FP32 sums of the unrounded P, FP32 accumulation, an FP32
// merge of the key splits across a thread-block cluster, one BF16 rounding.
//
// GB300 design (one CTA per SM, 512 threads, 16 warps = 4 per SM sub-partition):
//   warps 0-7  softmax: for a 64-head tile two warpgroups of 32 heads each, for
//              16 or 32 heads one warpgroup; one thread per key of a chunk
//              (the TMEM lane of S^T), per-head maxima by a shuffle butterfly
//              + shared memory, P as E4M3 into shared memory, rescale of O^T
//              in TMEM, epilogue/merge; unpaired, they also gather the first
//              chunk;
//   warp 8     allocates TMEM and issues QK from one thread, each chunk's as
//              soon as its rows landed and its S^T buffer is free;
//   warp 15    issues PV from one thread, each chunk's as soon as its P is
//              ready (two issuing threads: a burst of MMAs takes hundreds of
//              cycles to issue, and neither product waits behind the other's);
//   warps 9-14 producers. Unpaired: 16-byte cp.async copies of the chunk's KV
//              rows, one row per warp instruction, straight into the swizzled
//              K-major tiles the MMAs read (masked columns are zero-filled);
//              each thread's arrival on the stage barrier fires when its
//              copies land. Paired (two head tiles of a token in one
//              cluster): tile::gather4 of half of each chunk's rows, one lane
//              per warp, multicast into the stage of both CTAs. The Q tile
//              comes by TMA tile loads.
// Chunks hold 128 keys in two stages, or 96 keys in three where the planner
// finds the deeper ring pays (unpaired CTAs streaming many chunks).
// Both products put the long side on the MMA's M = 128 and the heads on N, as
// the DeepSeek page sketches:
//   S^T[key, head]   = KV[key, :] . Q[head, :]      (A = KV K-major, B = Q K-major)
//   O^T[lat, head]  += V^T[lat, key] . P^T[key, head] (A = the same KV tile read
//                      MN-major, B = P^T K-major), four 128-latent blocks.
// TMEM holds two S^T buffers (one accumulator over the whole row: a single
// chain runs at the same smem-bound rate as two) and O^T.
// Key splits of one (token, head tile) form a cluster and merge over DSMEM.
// Every wait is bounded; a timeout sets an error bit and the kernel still
// returns (and frees its TMEM).
// Head groups of 128 heads may also run on the CTA-pair kernel of
// smla_pair.cu, whose products run at the tensor core's full FP8 rate.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "smla.h"
#include "smla_pair.cuh"
#include "smla_ptx.cuh"

namespace smla {

constexpr int kRows = 128;  // the MMA's M: rows of S^T, latents of an O^T block
constexpr int kLatent = 512;
constexpr int kThreads = 512;
constexpr int kSoftmaxRange = 256;  // warps 0-7: one or two softmax warpgroups
constexpr int kMmaWarp = 8;       // issues QK (and holds the TMEM allocation)
constexpr int kProducerWarp = 9;  // first of six
constexpr int kProducerThreads = 192;
constexpr int kPvWarp = 15;       // issues PV
// Unpaired chunk 0 is gathered by every warp but the two issuing warps: the
// softmax range and the producers.
constexpr int kFirstGatherThreads = kSoftmaxRange + kProducerThreads;
constexpr int kMaxSplits = 16;
constexpr float kLog2P = 8.80735492205760410744f;  // log2(448): P of the running max
constexpr float kLog2e = 1.44269504088896340736f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait, then give up

__device__ int32_t g_device_error;

struct Params {
    // Tensor maps (64-byte aligned kernel parameters) of the Q tile of one
    // token and head group: 128-byte latent boxes (128B swizzle) and the
    // 64-byte rope box (64B swizzle).
    CUtensorMap q_latent;
    CUtensorMap q_rope;
    // Row gathers of pool 0 for paired CTAs (tile::gather4, one row high):
    // 128-byte latent boxes (128B swizzle) and the 64-byte rope box.
    CUtensorMap kv_latent;
    CUtensorMap kv_rope;
    const uint8_t* q;
    int64_t q_stride_token, q_stride_head;
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
    int32_t width, pool_split, num_pools, splits;
    int32_t pair;  // head groups sharing each gathered chunk (1 or 2; 2 needs one pool)
    float scale_log2, out_scale;
};

// The split merge's inbox holds splits x ceil(16 / splits) latent slices of
// 32; the most over 1..kMaxSplits splits (30, at 15).
constexpr int max_inbox_slices() {
    int most = 0;
    for (int s = 1; s <= kMaxSplits; ++s) most = most > s * ((16 + s - 1) / s) ? most : s * ((16 + s - 1) / s);
    return most;
}

// Shared-memory map of one CTA for N heads and D-byte rows (offsets from a
// 1024-byte aligned base; every MMA operand tile starts on 1024 bytes).
template <int N, int D, int C>
struct Layout {
    // A tile of R rows: four 128-byte latent K blocks (128B swizzle, 8-row
    // atoms of 1 KB) then, for 576-byte rows, the 64-byte rope block (64B
    // swizzle, 8-row atoms of 512 bytes).
    // C keys per chunk: 128 in two stages, or 96 in three (the MMAs still
    // read 128 rows; the 32 past a 96-key block are the next block's or the
    // next area's bytes, and their S^T rows are masked, their P^T rows never
    // read).
    static constexpr bool kRope = D == 576;
    static constexpr int kStages = C == 128 ? 2 : 3;
    static constexpr int kStage = 4 * C * 128 + (kRope ? C * 64 : 0);
    static constexpr int kKv = 0;                                 // kStages stages of KV rows
    static constexpr int kQ = kStages * kStage;                   // the Q tile
    static constexpr int kQBytes = 4 * N * 128 + (kRope ? N * 64 : 0);
    static constexpr int kP = kQ + kQBytes;                       // 2 buffers of P^T (C x N bytes)
    static constexpr int kIdx = kP + 2 * C * N;            // int32 [kStages][C] row of each key, -1 masked
    static constexpr int kRed = kIdx + kStages * C * 4;    // float [4][N] per-warp partials
    static constexpr int kHead = kRed + 4 * N * 4;      // float [4][N]: m_run, bias, alpha, l
    static constexpr int kBar = kHead + 4 * N * 4;      // 16 mbarriers
    static constexpr int kMisc = kBar + 16 * 8;         // tmem base, abort flag
    // 16-head tiles: the split merge's inbox, stats and weights in their own
    // area (the KV tiles stay untouched), so that a CTA may receive its
    // partners' partials without first waiting for the cluster to leave the
    // main loop. Larger tiles reuse the KV tiles and wait.
    static constexpr bool kOwnInbox = N == 16;
    static constexpr int kInboxBytes = max_inbox_slices() * N * 32 * 4 + kMaxSplits * 2 * N * 4 + kMaxSplits * N * 4;
    static constexpr int kInbox = (kMisc + 64 + 1023) / 1024 * 1024;
    static constexpr int kBytes = kOwnInbox ? kInbox + kInboxBytes : kMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(C == 128 || C == 96, "chunks of 128 or 96 keys");
    static_assert(kAlloc <= 227 * 1024, "one CTA's shared memory");
    static_assert(kStage % 1024 == 0 && kQ % 1024 == 0 && kP % 512 == 0, "operand tiles stay aligned");
    // TMEM columns: S^T of buffers 0/1 at [0, 2N), O^T blocks at [2N, 6N)
    // (the allocation is a power of two).
    static constexpr int kTmemCols = 8 * N;
};

// P^T for PV: B operand of N heads x 128 keys, MN-major (each key's N heads
// are contiguous). Rows of N bytes, 8-row atoms of 8N bytes, swizzled with the
// atom width: 64 heads -> 64B swizzle, 32 -> 32B swizzle, 16 -> none.
template <int N>
__device__ __forceinline__ uint32_t p_unit(int key, int unit) {
    int u = unit;
    if constexpr (N == 64) u ^= (key >> 1) & 3;
    if constexpr (N == 32) u ^= (key >> 2) & 1;
    return static_cast<uint32_t>(key * N + (u << 4));
}

template <int N>
__host__ __device__ constexpr uint32_t p_swizzle() {
    return N == 64 ? kSwizzle64B : (N == 32 ? kSwizzle32B : kSwizzleNone);
}

// Writes the BF16 tile [N heads][512] from shared memory to out[token][head0
// + h][:], 16 bytes per thread per step when the output rows allow it.
template <int N>
__device__ __forceinline__ void store_rows(const Params& p, const __nv_bfloat16* tile, int token, int head0,
                                           int tid) {
    __nv_bfloat16* out = p.out + static_cast<int64_t>(token) * p.out_stride_token +
                         static_cast<int64_t>(head0) * p.out_stride_head;
    const bool wide = ((reinterpret_cast<uintptr_t>(p.out) | static_cast<uintptr_t>(p.out_stride_token * 2) |
                        static_cast<uintptr_t>(p.out_stride_head * 2)) & 15u) == 0;
    if (wide) {
        for (int i = tid; i < N * kLatent / 8; i += kSoftmaxRange) {
            const int h = i / (kLatent / 8), e = (i % (kLatent / 8)) * 8;
            *reinterpret_cast<uint4*>(out + static_cast<int64_t>(h) * p.out_stride_head + e) =
                *reinterpret_cast<const uint4*>(tile + h * kLatent + e);
        }
    } else {
        for (int i = tid; i < N * kLatent / 2; i += kSoftmaxRange) {
            const int h = i / (kLatent / 2), e = (i % (kLatent / 2)) * 2;
            *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(h) * p.out_stride_head + e) =
                *reinterpret_cast<const uint32_t*>(tile + h * kLatent + e);
        }
    }
}

// Logits of the H heads (H = 16 or 32) of this thread's key, from the S^T
// accumulator at TMEM address `col` (one round trip).
template <int H>
__device__ __forceinline__ void load_logits(uint32_t col, float (&s)[H]) {
    if constexpr (H == 16)
        tmem_load16x1(col, s);
    else
        tmem_load16x2(col, col + 16, s);
}

template <int N, int D, int C>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_decode_kernel(const __grid_constant__ Params p) {
    using L = Layout<N, D, C>;
    constexpr int NS = L::kStages;
    constexpr int NG = N == 64 ? 2 : 1;  // softmax warpgroups
    constexpr int HW = N / NG;           // heads per softmax warpgroup (16 or 32)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* kv_full = bars + 0;   // [NS] a stage's rows landed (192 cp.async arrivals + 1)
    // pv_done[st]: PV of the chunk in stage st finished (its KV stage is free,
    // O^T holds it). One barrier per stage, so that no waiter is ever more
    // than one phase behind the barrier it waits on.
    uint64_t* pv_done = bars + 3;   // [NS] commit
    uint64_t* s_full = bars + 6;    // [2] QK of a chunk done (commit)
    uint64_t* p_full = bars + 8;    // P^T written, O^T rescaled (softmax arrivals)
    uint64_t* drain = bars + 9;     // every MMA of both issuing threads done (commits)
    uint64_t* q_full = bars + 10;   // the Q tile landed (TMA transaction bytes)
    uint64_t* kv_first = bars + 11; // chunk 0 landed (448 cp.async arrivals + 1, the producers' at once
                                    // when they do not help); later chunks use kv_full
    // stage_free[st] (paired): PV of the chunk in stage st finished in both
    // CTAs of the pair (one multicast commit from each), so either may refill
    // the stage in both.
    uint64_t* stage_free = bars + 12;  // [NS]
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + L::kIdx);
    float* red = reinterpret_cast<float*>(smem + L::kRed);
    float* m_run_s = reinterpret_cast<float*>(smem + L::kHead);
    float* bias_s = m_run_s + N;
    float* alpha_s = m_run_s + 2 * N;
    float* l_s = m_run_s + 3 * N;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int splits = p.splits;
    const bool paired = p.pair == 2;
    // The cluster holds the splits of `pair` consecutive head groups of one
    // token: rank = half * splits + split.
    const int rank = static_cast<int>(blockIdx.x) % (splits * p.pair);
    const int split = rank % splits;
    const int half = rank / splits;
    const int head0 = (static_cast<int>(blockIdx.x) / splits) * N;
    // the CTA of the same split in the other head group of the pair, and both
    const uint16_t pair_mask = static_cast<uint16_t>((1u << split) | (1u << (splits + split)));
    const int token = blockIdx.y;

    // ---- set-up (reads no input, so it overlaps the previous kernel) -------
    if (tid == 0) {
        // paired: the producer's expect-tx arrival; else every producer
        // thread's cp.async arrival and one index-release arrival
        for (int st = 0; st < NS; ++st) {
            mbar_init(&kv_full[st], paired ? 1 : kProducerThreads + 1);
            mbar_init(&stage_free[st], 2);
            mbar_init(&pv_done[st], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(p_full, NG * 128);
        mbar_init(drain, 2);  // one commit from each issuing thread
        mbar_init(kv_first, kFirstGatherThreads + 1);
        misc[1] = 0;
        mbar_init_fence();
    }
    if (tid < N) {
        m_run_s[tid] = -INFINITY;
        bias_s[tid] = -INFINITY;
        alpha_s[tid] = 1.0f;
        l_s[tid] = 0.0f;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(misc, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensor_map(&p.q_latent);
        if constexpr (L::kRope) prefetch_tensor_map(&p.q_rope);
        if (paired) {
            prefetch_tensor_map(&p.kv_latent);
            if constexpr (L::kRope) prefetch_tensor_map(&p.kv_rope);
        }
    }
    tc_fence_before_sync();
    if (paired)
        cluster_sync_all();  // the partner's barriers are initialised before anything reaches them
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    grid_dependency_wait();  // inputs are read only after this point
    if (warp == kProducerWarp && lane == 0) {
        // The Q tile of this CTA's heads, before anything else is known.
        mbar_arrive_expect_tx(q_full, N * D);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
            tma_load_3d(sbase + L::kQ + kb * N * 128, &p.q_latent, kb * 128, head0, token, q_full);
        if constexpr (L::kRope) tma_load_3d(sbase + L::kQ + 4 * N * 128, &p.q_rope, 512, head0, token, q_full);
    }
    // The first chunk's raw indices, loaded while the count loads: the
    // chunk this split starts with when the count fills the width (always
    // for split 0). Thread k of the chunk's resolvers (the softmax range
    // unpaired, the producers paired) takes column k; the count masks them
    // later, and a split whose first chunk turns out elsewhere reloads.
    const int chunks_w = (p.width + C - 1) / C;
    const int col_guess = split * ((chunks_w + splits - 1) / splits) * C;
    const int resolver = paired ? tid - kProducerWarp * 32 : tid;
    int32_t raw_guess = -1;
    if (resolver >= 0 && resolver < C && col_guess + resolver < p.width)
        raw_guess = p.indices[static_cast<int64_t>(token) * p.idx_stride + col_guess + resolver];
    const int count = min(max(p.lens[token], 0), p.width);
    // this thread's head's sink (threads < N), read now so that the epilogue
    // does not wait for it
    const float sink_of_head = (tid < N && p.sinks != nullptr) ? p.sinks[head0 + tid] * kLog2e : -INFINITY;
    // This split's chunks of the token: ceil(chunks / splits) consecutive
    // chunks each, dealt over the token's own count (later splits may be empty).
    const int chunks_total = (count + C - 1) / C;
    const int per_split = (chunks_total + splits - 1) / splits;
    const int c_first = split * per_split;
    const int nch = max(0, min(per_split, chunks_total - c_first));
    grid_launch_dependents();
    // Chunk c lives in stage c % NS. Its stage barrier and the parity of its
    // phase: unpaired, chunk 0 has its own barrier and stage 0's barrier
    // serves chunks NS, 2 NS, ... from its first phase; paired CTAs use the
    // stage barriers from chunk 0 on. A phase of pv_done / stage_free
    // completes per chunk of its stage, chunk c's being phase c / NS.
    bool ok = true;
    auto kv_bar = [&](int c) -> uint64_t* { return (c == 0 && !paired) ? kv_first : &kv_full[c % NS]; };
    auto kv_parity = [&](int c) -> uint32_t {
        if (paired) return static_cast<uint32_t>((c / NS) & 1);
        return c == 0 ? 0u : static_cast<uint32_t>(((c / NS) - (c % NS == 0 ? 1 : 0)) & 1);
    };
    auto pv_wait = [&](int c) {  // PV of chunk c has finished
        ok &= mbar_wait_bounded(&pv_done[c % NS], static_cast<uint32_t>((c / NS) & 1), abort_flag, kWaitLimitNs);
    };

    // Unpaired chunk 0 is gathered by the softmax-range warps (idle until the
    // first QK), and by the producers too when it is the CTA's only chunk (it
    // is on every CTA's critical path, and more issuing warps stream it
    // faster); with more chunks the producers start on chunk 1 at once.
    const bool producers_help = nch == 1;
    const bool producer = warp >= kProducerWarp && warp < kPvWarp;
    if (producer && nch > 1 && !paired) cp_async_arrive_noinc(kv_first);  // nothing in flight yet
    if (warp != kMmaWarp && warp != kPvWarp && nch > 0 && !paired && (warp < kMmaWarp || producers_help)) {
        // ============================================= chunk 0
        const int gw = warp < kMmaWarp ? warp : warp - 1;  // 0 .. 13
        const int gather_warps = producers_help ? kFirstGatherThreads / 32 : kSoftmaxRange / 32;
        const int32_t* idx_row = p.indices + static_cast<int64_t>(token) * p.idx_stride;
        const int col0 = c_first * C;
        if (tid < C) {
            const int col = col0 + tid;
            int32_t id = -1;
            if (col < count) {
                const int32_t raw = col0 == col_guess ? raw_guess : idx_row[col];
                const bool second = p.num_pools == 2 && col >= p.pool_split;
                if (raw >= 0) {
                    if (raw < (second ? p.rows1 : p.rows0))
                        id = raw;
                    else
                        atomicOr(&g_device_error, SMLA_DEV_INDEX_RANGE);
                }
            }
            idx_s[tid] = id;
        }
        named_barrier(5, producers_help ? kFirstGatherThreads : kSoftmaxRange);
        if (tid == 0) mbar_arrive(kv_first);  // every idx_s entry (release)
        const uint32_t stage = sbase + L::kKv;
        const uint32_t lane_part = stage + (lane >> 3) * C * 128;
        for (int k = gw; k < C; k += gather_warps) {
            const int32_t id = idx_s[k];
            const bool second = p.num_pools == 2 && col0 + k >= p.pool_split;
            const uint8_t* src = (second ? p.pool1 : p.pool0) + static_cast<int64_t>(id >= 0 ? id : 0) * D + lane * 16;
            const uint32_t dst = lane_part + (k >> 3) * 1024 + (k & 7) * 128 + (((lane & 7) ^ (k & 7)) << 4);
            cp_async_16(dst, src, id >= 0 ? 16u : 0u);
        }
        if constexpr (L::kRope) {
            for (int j = gw; j < C / 8; j += gather_warps) {
                const int k = j * 8 + (lane >> 2), u = lane & 3;
                const int32_t id = idx_s[k];
                const bool second = p.num_pools == 2 && col0 + k >= p.pool_split;
                const uint8_t* src =
                    (second ? p.pool1 : p.pool0) + static_cast<int64_t>(id >= 0 ? id : 0) * D + 512 + u * 16;
                const uint32_t dst = stage + 4 * C * 128 + (k >> 3) * 512 + (k & 7) * 64 + ((u ^ ((k >> 1) & 3)) << 4);
                cp_async_16(dst, src, id >= 0 ? 16u : 0u);
            }
        }
        cp_async_arrive_noinc(kv_first);
    }
    if (producer && paired) {
        // =========================================== paired producers
        // Both CTAs of the pair hold the same token and split, so the same
        // chunks. Each resolves all 128 indices (the softmax masks by them)
        // and gathers its half of the rows with tile::gather4, multicast into
        // the stage of both CTAs; a stage is refilled once PV has released it
        // in both. Masked keys get a row past the pool's end (zero fill).
        const int g = tid - kProducerWarp * 32;
        const int32_t* idx_row = p.indices + static_cast<int64_t>(token) * p.idx_stride;
        const int32_t past_end = static_cast<int32_t>(p.rows0);
        for (int c = 0; c < nch; ++c) {
            const int b = c % NS;
            const int col0 = (c_first + c) * C;
            const int32_t raw = (g < C && col0 + g < count)
                                    ? ((c == 0 && col0 == col_guess) ? raw_guess : idx_row[col0 + g])
                                    : -1;
            if (c >= NS)
                ok &= mbar_wait_bounded(&stage_free[b], ((c - NS) / NS) & 1, abort_flag, kWaitLimitNs);
            if (g < C) {
                int32_t id = -1;
                if (raw >= 0) {
                    if (raw < p.rows0)
                        id = raw;
                    else
                        atomicOr(&g_device_error, SMLA_DEV_INDEX_RANGE);
                }
                idx_s[b * C + g] = id;
            }
            named_barrier(3, kProducerThreads);
            if (g == 0) mbar_arrive_expect_tx(&kv_full[b], L::kStage);  // both halves; also releases idx_s
            if (lane == 0) {
                // one lane per producer warp: the TMA instructions of one
                // thread issue one after another, several threads overlap
                const uint32_t stage = sbase + L::kKv + b * L::kStage;
                for (int k = half * (C / 2) + 4 * (g >> 5); k < (half + 1) * (C / 2);
                     k += 4 * (kProducerThreads / 32)) {
                    int32_t r[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int32_t id = idx_s[b * C + k + i];
                        r[i] = id >= 0 ? id : past_end;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tma_gather4_multicast(stage + j * C * 128 + (k >> 3) * 1024 + (k & 7) * 128, &p.kv_latent,
                                              j * 128, r[0], r[1], r[2], r[3], &kv_full[b], pair_mask);
                    if constexpr (L::kRope)
                        tma_gather4_multicast(stage + 4 * C * 128 + (k >> 3) * 512 + (k & 7) * 64, &p.kv_rope,
                                              512, r[0], r[1], r[2], r[3], &kv_full[b], pair_mask);
                }
            }
        }
        // The partner's commits for the last chunks have reached this CTA's
        // stage barriers before either CTA moves on to its exit.
        if (g == 0)
            for (int c = max(0, nch - NS); c < nch; ++c)
                ok &= mbar_wait_bounded(&stage_free[c % NS], (c / NS) & 1, abort_flag, kWaitLimitNs);
    } else if (producer) {
        // ================================================== producers
        // Thread g < 128 resolves key g's row; warp w then copies keys w,
        // w + 6, ..., one 512-byte latent row per instruction (lane l: bytes
        // 16 l .. 16 l + 15), and the 64-byte ropes of eight keys per
        // instruction. Masked keys are zero-filled. Thread 0 also arrives
        // after the index barrier, so that the stage barrier releases idx_s.
        const int g = tid - kProducerWarp * 32;
        const int pw = g >> 5;
        const int32_t* idx_row = p.indices + static_cast<int64_t>(token) * p.idx_stride;
        for (int c = 1; c < nch; ++c) {  // chunk 0 is gathered by the softmax-range warps
            const int b = c % NS;
            const int col0 = (c_first + c) * C;
            // This chunk's index is loaded before the wait for its stage, so
            // that its latency overlaps the wait.
            const int32_t raw = (g < C && col0 + g < count) ? idx_row[col0 + g] : -1;
            if (c >= NS) pv_wait(c - NS);
            if (g < C) {
                const int col = col0 + g;
                int32_t id = -1;
                if (col < count) {
                    const bool second = p.num_pools == 2 && col >= p.pool_split;
                    if (raw >= 0) {
                        if (raw < (second ? p.rows1 : p.rows0))
                            id = raw;
                        else
                            atomicOr(&g_device_error, SMLA_DEV_INDEX_RANGE);
                    }
                }
                idx_s[b * C + g] = id;
            }
            named_barrier(3, kProducerThreads);
            if (g == 0) mbar_arrive(&kv_full[b]);
            const uint32_t stage = sbase + L::kKv + b * L::kStage;
            const uint32_t lane_part = stage + (lane >> 3) * C * 128;
            for (int k = pw; k < C; k += kProducerThreads / 32) {
                const int32_t id = idx_s[b * C + k];
                const bool second = p.num_pools == 2 && col0 + k >= p.pool_split;
                const uint8_t* src = (second ? p.pool1 : p.pool0) + static_cast<int64_t>(id >= 0 ? id : 0) * D + lane * 16;
                const uint32_t dst = lane_part + (k >> 3) * 1024 + (k & 7) * 128 + (((lane & 7) ^ (k & 7)) << 4);
                cp_async_16(dst, src, id >= 0 ? 16u : 0u);
            }
            if constexpr (L::kRope) {
                for (int j = pw; j < C / 8; j += kProducerThreads / 32) {
                    const int k = j * 8 + (lane >> 2), u = lane & 3;
                    const int32_t id = idx_s[b * C + k];
                    const bool second = p.num_pools == 2 && col0 + k >= p.pool_split;
                    const uint8_t* src =
                        (second ? p.pool1 : p.pool0) + static_cast<int64_t>(id >= 0 ? id : 0) * D + 512 + u * 16;
                    const uint32_t dst = stage + 4 * C * 128 + (k >> 3) * 512 + (k & 7) * 64 + ((u ^ ((k >> 1) & 3)) << 4);
                    cp_async_16(dst, src, id >= 0 ? 16u : 0u);
                }
            }
            cp_async_arrive_noinc(&kv_full[b]);
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        // ================================================== QK issuer
        // QK(c) once chunk c landed and S buffer c % 2 is free (the softmax
        // of chunk c - 2 has handed over its P).
        if (lane == 0) {
            constexpr uint32_t kIdescQK = idesc_e4m3(kRows, N, 0, 0);
            // Descriptors of every operand tile; moving a descriptor by b
            // bytes adds b >> 4 to its start field (no carry: shared
            // addresses stay below 256 KB).
            const uint64_t d_q = smem_desc(sbase + L::kQ, 1024, 1024, kSwizzle128B);
            const uint64_t d_q_rope = smem_desc(sbase + L::kQ + 4 * N * 128, 512, 512, kSwizzle64B);
            const uint64_t d_kv = smem_desc(sbase + L::kKv, 1024, 1024, kSwizzle128B);
            const uint64_t d_kv_rope = smem_desc(sbase + L::kKv + 4 * C * 128, 512, 512, kSwizzle64B);
            ok &= mbar_wait_bounded(q_full, 0, abort_flag, kWaitLimitNs);  // also: no copy outlives the CTA
            for (int c = 0; ok && c < nch; ++c) {
                if (c >= 2) ok &= mbar_wait_bounded(p_full, static_cast<uint32_t>(c & 1), abort_flag, kWaitLimitNs);
                ok &= mbar_wait_bounded(kv_bar(c), kv_parity(c), abort_flag, kWaitLimitNs);
                if (!ok) break;
                fence_proxy_async_smem();  // the producers' cp.async data, for the tensor cores
                tc_fence_after_sync();
                const uint32_t stage16 = static_cast<uint32_t>((c % NS) * L::kStage) >> 4;
                // one accumulator: the 16 latent K steps, then the rope's two
                const uint32_t d_s = tmem + (c & 1) * N;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int kb = i >> 2, ks = i & 3;
                    const uint32_t a = stage16 + ((kb * C * 128 + ks * 32) >> 4);
                    const uint32_t bq = (kb * N * 128 + ks * 32) >> 4;
                    mma_f8(d_s, d_kv + a, d_q + bq, kIdescQK, i != 0 ? 1u : 0u);
                }
                if constexpr (L::kRope) {
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_f8(d_s, d_kv_rope + stage16 + ((ks * 32) >> 4), d_q_rope + ((ks * 32) >> 4),
                               kIdescQK, 1u);
                }
                mma_commit(&s_full[c & 1]);
            }
            mma_commit(drain);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ================================================== PV issuer
        // PV(c) as soon as P(c) is ready (and O^T rescaled); a separate thread
        // from QK's, so that neither waits behind the other's burst of MMAs.
        if (lane == 0) {
            constexpr uint32_t kIdescPV = idesc_e4m3(kRows, N, 1, 1);
            const uint64_t d_kv = smem_desc(sbase + L::kKv, 1024, 1024, kSwizzle128B);
            const uint64_t d_p = smem_desc(sbase + L::kP, 8 * N, 8 * N, p_swizzle<N>());
            for (int c = 0; ok && c < nch; ++c) {
                // p_full completes once per chunk; chunk c's is phase c
                ok &= mbar_wait_bounded(p_full, static_cast<uint32_t>(c & 1), abort_flag, kWaitLimitNs);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t stage16 = static_cast<uint32_t>((c % NS) * L::kStage) >> 4;
                const uint32_t p16 = static_cast<uint32_t>((c & 1) * C * N) >> 4;
#pragma unroll
                for (int kk = 0; kk < C / 32; ++kk) {  // the four latent blocks are independent chains
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t a_off = stage16 + ((j * C * 128 + kk * 32 * 128) >> 4);
                        const uint32_t b_off = p16 + ((kk * 32 * N) >> 4);
                        mma_f8(tmem + 2 * N + j * N, d_kv + a_off, d_p + b_off, kIdescPV, (c > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&pv_done[c % NS]);
                if (paired) mma_commit_multicast(&stage_free[c % NS], pair_mask);
            }
            mma_commit(drain);
        }
        __syncwarp();
    } else if (warp < 4 * NG) {
        // ===================================================== softmax
        // Warpgroup wg owns heads hb .. hb + HW - 1. Thread t owns key t of
        // each chunk (TMEM lane t of S^T) and, for O^T, latent rows t of each
        // 128-latent block.
        const int wg = warp >> 2, t = tid & 127, hb = wg * HW;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float scale_log2 = p.scale_log2;
        float lsum[HW];
#pragma unroll
        for (int h = 0; h < HW; ++h) lsum[h] = 0.0f;

        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            ok &= mbar_wait_bounded(kv_bar(c), kv_parity(c), abort_flag, kWaitLimitNs);
            ok &= mbar_wait_bounded(&s_full[b], (c >> 1) & 1, abort_flag, kWaitLimitNs);
            tc_fence_after_sync();
            const bool active = t < C && idx_s[(c % NS) * C + t] >= 0;
            // this key's logits of the warpgroup's heads, kept for the P pass
            float s[HW];
            load_logits<HW>(tmem + lane_base + b * N + hb, s);

            // chunk maxima per head, in logit units (bmm1_scale > 0 keeps the
            // order; masked keys are -inf)
            {
                // a transposing butterfly: each step hands half of a lane's
                // heads to its partner; with 32 heads lane l ends with head l,
                // with 16 lanes 2 h and 2 h + 1 share head h. The first step
                // reads the logits and leaves them in place.
                float m[HW / 2];
                {
                    const bool up = (lane & 16) != 0;
#pragma unroll
                    for (int i = 0; i < HW / 2; ++i) {
                        const float lo = active ? s[i] : -INFINITY, hi = active ? s[i + HW / 2] : -INFINITY;
                        m[i] = fmaxf(up ? hi : lo, __shfl_xor_sync(0xFFFFFFFFu, up ? lo : hi, 16));
                    }
                }
#pragma unroll
                for (int o = 8, n = HW / 2; n > 1; o >>= 1, n >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < n / 2; ++i) {
                        const float send = up ? m[i] : m[i + n / 2];
                        const float keep = up ? m[i + n / 2] : m[i];
                        m[i] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
                    }
                }
                if constexpr (HW == 16) {
                    m[0] = fmaxf(m[0], __shfl_xor_sync(0xFFFFFFFFu, m[0], 1));
                    if ((lane & 1) == 0) red[(warp & 3) * N + hb + (lane >> 1)] = m[0];
                } else {
                    red[(warp & 3) * N + hb + lane] = m[0];
                }
            }
            named_barrier(1 + wg, 128);
            if (t < HW) {
                const int h = hb + t;
                const float cm = fmaxf(fmaxf(red[h], red[N + h]), fmaxf(red[2 * N + h], red[3 * N + h]));
                const float mo = m_run_s[h];
                const float mn = fmaxf(mo, cm * scale_log2);
                alpha_s[h] = (mo == -INFINITY) ? 1.0f : fast_exp2(mo - mn);
                bias_s[h] = mn - kLog2P;
                m_run_s[h] = mn;
            }
            named_barrier(1 + wg, 128);

            // P = 2^(s * scale_log2 - m + log2 448) as E4M3 into P^T[b] (PV of
            // chunk c-2 has finished reading it); FP32 sums of the unrounded P
            if (c >= 2) pv_wait(c - 2);  // its P^T buffer is free
            {
                uint8_t* pbuf = smem + L::kP + b * C * N;
#pragma unroll
                for (int g = 0; g < HW / 16; ++g) {
                    uint32_t words[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int j = 16 * g + 4 * q4;
                        const float4 bi = reinterpret_cast<const float4*>(bias_s + hb)[j / 4];
                        const float4 al = reinterpret_cast<const float4*>(alpha_s + hb)[j / 4];
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
                        words[q4] = e4m3x2(pr[0], pr[1]) | (e4m3x2(pr[2], pr[3]) << 16);
                    }
                    if (t < C)
                        *reinterpret_cast<uint4*>(pbuf + p_unit<N>(t, hb / 16 + g)) =
                            make_uint4(words[0], words[1], words[2], words[3]);
                }
            }

            // O^T *= alpha where a head's running maximum rose (PV of chunk c-1 is done)
            if (c >= 1) {
                pv_wait(c - 1);
                tc_fence_after_sync();
#pragma unroll
                for (int g = 0; g < HW / 16; ++g) {
                    float a[16];
                    bool rescale = false;
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const float4 v4 = reinterpret_cast<const float4*>(alpha_s + hb + 16 * g)[j4];
                        a[4 * j4 + 0] = v4.x;
                        a[4 * j4 + 1] = v4.y;
                        a[4 * j4 + 2] = v4.z;
                        a[4 * j4 + 3] = v4.w;
                        rescale |= (v4.x != 1.0f) | (v4.y != 1.0f) | (v4.z != 1.0f) | (v4.w != 1.0f);
                    }
                    if (rescale) {
                        const uint32_t col = tmem + lane_base + 2 * N + hb + 16 * g;
                        float v[64];
                        tmem_load16x4(col, col + N, col + 2 * N, col + 3 * N, v);
#pragma unroll
                        for (int i = 0; i < 64; ++i) v[i] *= a[i & 15];
                        tmem_store16x4(col, col + N, col + 2 * N, col + 3 * N, v);
                    }
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
        for (int j = 0; j < HW; ++j) {
            float v = lsum[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == j) red[(warp & 3) * N + hb + j] = v;
        }
        named_barrier(1 + wg, 128);
        if (t < HW) {
            const int h = hb + t;
            l_s[h] = (red[h] + red[N + h]) + (red[2 * N + h] + red[3 * N + h]);
        }
    }
    if (!ok) {
        *abort_flag = 1;
        atomicOr(&g_device_error, SMLA_DEV_TIMEOUT);
    }
    cp_async_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // ================================================ epilogue / merge
    // Warps 0-7 (softmax range); warpgroup wg < NG holds heads hb .. hb + HW - 1.
    const bool split_empty = (m_run_s[0] == -INFINITY);  // no active key in this split
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int wg = warp >> 2, hb = wg * HW;
    const bool has_heads = warp < 4 * NG;
    if (splits == 1) {
        if (tid < N) {
            const int h = head0 + tid;
            const float m = m_run_s[tid];
            float scale = 0.0f, lse2 = -INFINITY;
            if (m != -INFINITY) {
                float top = m, extra = 0.0f;
                if (p.sinks != nullptr) {
                    const float s2 = sink_of_head;
                    top = fmaxf(m, s2);
                    extra = 448.0f * fast_exp2(s2 - top);
                }
                const float w = fast_exp2(m - top);
                const float total = l_s[tid] * w + extra;
                scale = p.out_scale * w / total;
                lse2 = top - kLog2P + log2f(total);
            }
            bias_s[tid] = scale;
            if (p.lse != nullptr) p.lse[static_cast<int64_t>(token) * p.lse_stride_token + h] = lse2;
        }
        named_barrier(4, kThreads);
        __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem + L::kKv);
        if (has_heads) {
            // O^T rows (one latent index per thread, this warpgroup's heads)
            // -> BF16 [N][512] in shared memory (the KV tiles are free now)
#pragma unroll 1
            for (int blk = 0; blk < 4; blk += 64 / HW) {  // 64 values per TMEM round trip
                float v[64];
                const uint32_t col = tmem + lane_base + 2 * N + hb;
                if constexpr (HW == 32)
                    tmem_load16x4(col + blk * N, col + blk * N + 16, col + (blk + 1) * N, col + (blk + 1) * N + 16, v);
                else
                    tmem_load16x4(col, col + N, col + 2 * N, col + 3 * N, v);
                // Heads j, j + 1 of latents d, d + 1 (lanes l, l ^ 1) as two
                // BF16 words: the even lane stores head j, the odd lane head
                // j + 1, each after one exchange with its neighbour.
                const bool odd = lane & 1;
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    const int bb = HW == 32 ? blk + i / 32 : i / 16;  // latent block of value i
                    const int j = HW == 32 ? i % 32 : i % 16;        // head (even) within the warpgroup
                    const float x0 = split_empty ? 0.0f : v[i] * bias_s[hb + j];
                    const float x1 = split_empty ? 0.0f : v[i + 1] * bias_s[hb + j + 1];
                    const float other = __shfl_xor_sync(0xFFFFFFFFu, odd ? x0 : x1, 1);
                    const __nv_bfloat162 two = odd ? __floats2bfloat162_rn(other, x1) : __floats2bfloat162_rn(x0, other);
                    const int lat = bb * 128 + (warp & 3) * 32 + (lane & ~1);
                    *reinterpret_cast<__nv_bfloat162*>(tile + (hb + j + (odd ? 1 : 0)) * kLatent + lat) = two;
                }
            }
        }
        named_barrier(4, kThreads);
        if (tid < kSoftmaxRange) store_rows<N>(p, tile, token, head0, tid);
    } else {
        // Partials of every split of this (token, head tile) meet at the CTA
        // owning their latent slice: slice s (latent 32 s .. 32 s + 31, s < 16)
        // belongs to rank s % splits. The areas reuse the KV and Q tiles.
        const int slots = (16 + splits - 1) / splits;
        constexpr int kInboxAt = L::kOwnInbox ? L::kInbox : 0;
        const uint32_t inbox = sbase + kInboxAt;                        // float [S][slots][N][32]
        const uint32_t stats = inbox + splits * slots * N * 32 * 4;     // float [S][2][N]
        float* stats_f = reinterpret_cast<float*>(smem + kInboxAt + splits * slots * N * 32 * 4);
        float* weight_f = stats_f + splits * 2 * N;                     // float [S][N]
        const float* inbox_f = reinterpret_cast<const float*>(smem + kInboxAt);
        if (!L::kOwnInbox) cluster_sync_relaxed();  // every CTA of the cluster is past its main loop
        if (tid < N) {
            for (int r = 0; r < splits; ++r) {
                st_cluster_f32(map_to_rank(stats + ((split * 2 + 0) * N + tid) * 4, half * splits + r), m_run_s[tid]);
                st_cluster_f32(map_to_rank(stats + ((split * 2 + 1) * N + tid) * 4, half * splits + r), l_s[tid]);
            }
        }
        if (has_heads && !split_empty) {
            auto send_block = [&](int blk, const float* v) {
                const int slice = blk * 4 + (warp & 3);
                const int owner = slice % splits, slot = slice / splits;
                const uint32_t dst =
                    map_to_rank(inbox + (((split * slots + slot) * N + hb) * 32 + lane) * 4, half * splits + owner);
#pragma unroll
                for (int j = 0; j < HW; ++j) st_cluster_f32(dst + j * 32 * 4, v[j]);
            };
            const uint32_t col = tmem + lane_base + 2 * N + hb;
            if constexpr (HW == 16) {
                float v[64];  // the four blocks of this warp's 16 heads, one TMEM round trip
                tmem_load16x4(col, col + N, col + 2 * N, col + 3 * N, v);
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) send_block(blk, v + 16 * blk);
            } else {
#pragma unroll 1
                for (int blk = 0; blk < 4; blk += 2) {  // two blocks of 32 heads a round trip
                    float v[64];
                    tmem_load16x4(col + blk * N, col + blk * N + 16, col + (blk + 1) * N, col + (blk + 1) * N + 16, v);
                    send_block(blk, v);
                    send_block(blk + 1, v + 32);
                }
            }
        }
        cluster_sync_all();  // every partial has landed
        if (tid < N) {
            // the splits' loops unrolled to the maximum split count, so that
            // their loads and exponentials issue together
            const int h = head0 + tid;
            const float sink2 = sink_of_head;
            float m[kMaxSplits], l[kMaxSplits];
#pragma unroll
            for (int s = 0; s < kMaxSplits; ++s) {
                m[s] = s < splits ? stats_f[(s * 2) * N + tid] : -INFINITY;
                l[s] = s < splits ? stats_f[(s * 2 + 1) * N + tid] : 0.0f;
            }
            float top = -INFINITY;
#pragma unroll
            for (int s = 0; s < kMaxSplits; ++s) top = fmaxf(top, m[s]);
            float lse2 = -INFINITY;
            if (top == -INFINITY) {
                for (int s = 0; s < splits; ++s) weight_f[s * N + tid] = 0.0f;
            } else {
                float extra = 0.0f;
                if (p.sinks != nullptr) {
                    top = fmaxf(top, sink2);
                    extra = 448.0f * fast_exp2(sink2 - top);
                }
                float w[kMaxSplits];
                float total = 0.0f;
#pragma unroll
                for (int s = 0; s < kMaxSplits; ++s) {
                    w[s] = (m[s] == -INFINITY) ? 0.0f : fast_exp2(m[s] - top);
                    total += w[s] * l[s];
                }
                total += extra;
                const float inverse = p.out_scale / total;
#pragma unroll
                for (int s = 0; s < kMaxSplits; ++s)
                    if (s < splits) weight_f[s * N + tid] = w[s] * inverse;
                lse2 = top - kLog2P + log2f(total);
            }
            if (split == 0 && p.lse != nullptr) p.lse[static_cast<int64_t>(token) * p.lse_stride_token + h] = lse2;
        }
        named_barrier(4, kThreads);
        {
            // Every thread: eight latent values of one (owned slice, head),
            // merged from the splits' partials and stored as 16 bytes.
            const int owned = (16 - split + splits - 1) / splits;
            __nv_bfloat16* out = p.out + static_cast<int64_t>(token) * p.out_stride_token +
                                 static_cast<int64_t>(head0) * p.out_stride_head;
            const bool wide = ((reinterpret_cast<uintptr_t>(p.out) | static_cast<uintptr_t>(p.out_stride_token * 2) |
                                static_cast<uintptr_t>(p.out_stride_head * 2)) & 15u) == 0;
            for (int it = tid; it < owned * N * 4; it += kThreads) {
                const int q8 = it & 3, h = (it >> 2) % N, k = (it >> 2) / N;
                const int slice = split + k * splits;
                float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
                for (int s = 0; s < splits; ++s) {
                    const float w = weight_f[s * N + h];
                    if (w == 0.0f) continue;
                    const float4* src = reinterpret_cast<const float4*>(inbox_f + ((s * slots + k) * N + h) * 32 + q8 * 8);
                    const float4 a = src[0], b = src[1];
                    acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
                    acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
                }
                __nv_bfloat16* dst = out + static_cast<int64_t>(h) * p.out_stride_head + slice * 32 + q8 * 8;
                uint32_t packed[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 two = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
                    packed[e] = *reinterpret_cast<const uint32_t*>(&two);
                }
                if (wide) {
                    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) reinterpret_cast<uint32_t*>(dst)[e] = packed[e];
                }
            }
        }
    }

    // ---- teardown: every MMA and TMEM access has finished -----------------
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        if (!mbar_wait_bounded(drain, 0, abort_flag, kWaitLimitNs)) {
            if (lane == 0) atomicOr(&g_device_error, SMLA_DEV_TIMEOUT);
        }
        __syncwarp();
        tmem_dealloc(tmem, L::kTmemCols);
    }
    if (paired) cluster_sync_all();  // neither CTA of a pair leaves while the other may still signal it
}

// ============================================================== host side

thread_local int t_last_cuda_error = 0;

void note_cuda_error(int code) { t_last_cuda_error = code; }

int head_tile_for(int heads) {
    if (heads % 64 == 0) return 64;
    if (heads % 32 == 0) return 32;
    return 16;
}

template <int N, int D, int C>
int smem_bytes() {
    return Layout<N, D, C>::kAlloc;
}

int tmem_for(int n) { return 8 * n; }

// Whether the merge area of `splits` splits fits the KV + Q tiles it reuses
// (chunks of c keys).
bool merge_fits(int n, int d, int c, int splits) {
    const int stage = 4 * c * 128 + (d == 576 ? c * 64 : 0);
    const int limit = (c == 128 ? 2 : 3) * stage + 4 * n * 128 + (d == 576 ? n * 64 : 0);  // KV stages + Q tile
    const int slots = (16 + splits - 1) / splits;
    return splits * slots * n * 32 * 4 + splits * 3 * n * 4 <= limit;
}

// Programmatic dependent launch (the kernel's set-up overlaps the previous
// kernel in the stream) unless the environment variable SMLA_PDL is "0", for
// measuring what it gains.
bool dependent_launch() {
    static const bool on = [] {
        const char* env = std::getenv("SMLA_PDL");
        return !(env != nullptr && env[0] == '0');
    }();
    return on;
}

// Opts the kernel into its shared-memory size and non-portable clusters, once
// per device.
template <int N, int D, int C>
cudaError_t configure() {
    auto kernel = sparse_mla_decode_kernel<N, D, C>;
    constexpr int kSmem = Layout<N, D, C>::kAlloc;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

// CTAs in clusters of `splits` that the current device holds at once (the
// occupancy API's cluster count x splits; GPC boundaries make it smaller than
// the SM count for wide clusters). 0 when the query fails.
template <int N, int D, int C>
int resident_ctas_query(int splits) {
    if (configure<N, D, C>() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(splits), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Layout<N, D, C>::kAlloc;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(splits);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, sparse_mla_decode_kernel<N, D, C>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters * splits;
}

// The kernel's variants, by head tile n, row bytes d and chunk keys c.
struct Variant {
    int (*smem)();
    int (*resident)(int splits);
    cudaError_t (*launch)(const Params& p, dim3 grid, int cluster, cudaStream_t stream);
};

template <int N, int D, int C>
cudaError_t launch(const Params& p, dim3 grid, int cluster, cudaStream_t stream);

template <int N, int D, int C>
Variant variant() {
    return {smem_bytes<N, D, C>, resident_ctas_query<N, D, C>, launch<N, D, C>};
}

const Variant& variant_for(int n, int d, int c) {
    static const Variant table[3][2][2] = {
        {{variant<64, 576, 128>(), variant<64, 576, 96>()}, {variant<64, 512, 128>(), variant<64, 512, 96>()}},
        {{variant<32, 576, 128>(), variant<32, 576, 96>()}, {variant<32, 512, 128>(), variant<32, 512, 96>()}},
        // 16-head tiles keep 128-key chunks: their own merge inbox leaves no room for a third stage
        {{variant<16, 576, 128>(), variant<16, 576, 128>()}, {variant<16, 512, 128>(), variant<16, 512, 128>()}},
    };
    return table[n == 64 ? 0 : n == 32 ? 1 : 2][d == 576 ? 0 : 1][c == 128 ? 0 : 1];
}

int smem_for(int n, int d, int c) { return variant_for(n, d, c).smem(); }

// `dev` is the current device (the query runs on it).
int resident_ctas_on_device(int dev, int n, int d, int c, int splits) {
    static std::mutex mu;
    static int cache[64][3][2][2][kMaxSplits + 1] = {};
    if (dev < 0 || dev >= 64 || splits < 1 || splits > kMaxSplits) return 0;
    const int ni = n == 64 ? 0 : n == 32 ? 1 : 2;
    const int di = d == 576 ? 0 : 1;
    const int ci = c == 128 ? 0 : 1;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev][ni][di][ci][splits] != 0) return cache[dev][ni][di][ci][splits];
    }
    const int r = variant_for(n, d, c).resident(splits);
    if (r > 0) {
        std::lock_guard<std::mutex> lock(mu);
        cache[dev][ni][di][ci][splits] = r;
    }
    return r;
}

template <int N, int D, int C>
cudaError_t launch(const Params& p, dim3 grid, int cluster, cudaStream_t stream) {
    auto kernel = sparse_mla_decode_kernel<N, D, C>;
    constexpr int kSmem = Layout<N, D, C>::kAlloc;
    cudaError_t e = configure<N, D, C>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = dependent_launch() ? 1 : 0;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Every argument of one tiled tensor-map encode of bytes; the cache below
// compares them whole (the struct is zeroed before it is filled).
struct MapKey {
    const void* base;
    uint32_t rank;
    int32_t swizzle, promotion;
    cuuint64_t dims[3];
    cuuint64_t strides[2];
    cuuint32_t box[3];
};

// cuTensorMapEncodeTiled through a small cache of recent encodes: a decode's
// Q and pool maps repeat from call to call (fixed buffers, or a few rotating
// ones), and an encode costs microseconds of host time. Sixteen entries,
// replaced round robin; a map is a plain 128-byte value, so a hit copies it.
bool encode_cached(CUtensorMap* map, const MapKey& k) {
    constexpr int kEntries = 16;
    static std::mutex mu;
    static MapKey keys[kEntries];
    static CUtensorMap maps[kEntries];
    static bool used[kEntries] = {};
    static int next = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < kEntries; ++i)
            if (used[i] && std::memcmp(&keys[i], &k, sizeof(MapKey)) == 0) {
                *map = maps[i];
                return true;
            }
    }
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint32_t steps[3] = {1, 1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, k.rank, const_cast<void*>(k.base), k.dims, k.strides, k.box, steps,
            CU_TENSOR_MAP_INTERLEAVE_NONE, static_cast<CUtensorMapSwizzle>(k.swizzle),
            static_cast<CUtensorMapL2promotion>(k.promotion), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    keys[next] = k;
    maps[next] = *map;
    used[next] = true;
    next = (next + 1) % kEntries;
    return true;
}

// A tiled map of bytes of rank 2 or 3 (dims[0] innermost, strides of the
// outer dimensions in bytes), through the cache; for the library's other
// translation units.
bool encode_bytes_map(CUtensorMap* map, const void* base, uint32_t rank, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, int swizzle, int promotion) {
    if (rank < 2 || rank > 3) return false;
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.base = base;
    k.rank = rank;
    k.swizzle = swizzle;
    k.promotion = promotion;
    for (uint32_t i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank) k.strides[i] = strides[i];
    }
    return encode_cached(map, k);
}

// Q as [T][H][D] bytes with the caller's strides, read in boxes of `box`
// bytes x n heads of one token.
bool encode_q_map(CUtensorMap* map, const void* q, const smla_shape* s, int n, int box, CUtensorMapSwizzle swizzle) {
    const int64_t head_stride = s->q_stride_head;
    int64_t token_stride = s->q_stride_token;
    if (s->tokens == 1 && token_stride < head_stride * s->heads) token_stride = head_stride * s->heads;  // unused
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.base = q;
    k.rank = 3;
    k.swizzle = swizzle;
    k.promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    k.dims[0] = static_cast<cuuint64_t>(s->head_dim);
    k.dims[1] = static_cast<cuuint64_t>(s->heads);
    k.dims[2] = static_cast<cuuint64_t>(s->tokens);
    k.strides[0] = static_cast<cuuint64_t>(head_stride);
    k.strides[1] = static_cast<cuuint64_t>(token_stride);
    k.box[0] = static_cast<cuuint32_t>(box);
    k.box[1] = static_cast<cuuint32_t>(n);
    k.box[2] = 1;
    return encode_cached(map, k);
}

// Pool rows of `d` bytes, read by tile::gather4 in boxes of `box` bytes x 1 row.
bool encode_kv_map(CUtensorMap* map, const void* pool, int64_t rows, int d, int box, CUtensorMapSwizzle swizzle) {
    if (rows <= 0) return false;
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.base = pool;
    k.rank = 2;
    k.swizzle = swizzle;
    k.promotion = CU_TENSOR_MAP_L2_PROMOTION_NONE;
    k.dims[0] = static_cast<cuuint64_t>(d);
    k.dims[1] = static_cast<cuuint64_t>(rows);
    k.strides[0] = static_cast<cuuint64_t>(d);
    k.box[0] = static_cast<cuuint32_t>(box);
    k.box[1] = 1;
    return encode_cached(map, k);
}

int device_sms() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && cache[dev] > 0) return cache[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev < 64) cache[dev] = sms;
    return sms;
}

// The device address of this device's error word, for kernels of other
// translation units (which take it as a parameter).
int32_t* device_error_word() {
    static std::mutex mu;
    static int32_t* cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] != nullptr) return cache[dev];
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int32_t*>(ptr);
    return cache[dev];
}

// CTA pairs of the 128-head kernel the current device holds at once, cached.
int pair_resident_on_device(int d) {
    static std::mutex mu;
    static int cache[64][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 0;
    const int di = d == 576 ? 0 : 1;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev][di] != 0) return cache[dev][di];
    }
    const int r = pair_resident_clusters(d);
    if (r > 0) {
        std::lock_guard<std::mutex> lock(mu);
        cache[dev][di] = r;
    }
    return r;
}

int validate(const smla_shape* s) {
    if (s == nullptr) return SMLA_EINVAL;
    if (s->tokens < 0 || s->width < 0 || s->heads <= 0) return SMLA_EINVAL;
    if (s->heads % 16 != 0) return SMLA_EINVAL;
    if (s->heads > 1024 || s->tokens > 65535) return SMLA_EUNSUPPORTED;
    if (s->head_dim != 576 && s->head_dim != 512) return SMLA_EUNSUPPORTED;
    if (s->num_pools != 1 && s->num_pools != 2) return SMLA_EUNSUPPORTED;
    if (s->num_pools == 2 && (s->pool_split < 0 || s->pool_split > s->width)) return SMLA_EINVAL;
    if (s->q_stride_token < 0 || s->q_stride_head < 0 || s->idx_stride_token < 0 || s->out_stride_head < 0)
        return SMLA_EINVAL;
    if (s->q_stride_token % 16 != 0 || s->q_stride_head % 16 != 0) return SMLA_EINVAL;
    if (s->q_stride_head < s->head_dim && s->heads > 1) return SMLA_EINVAL;
    if (s->idx_stride_token < s->width) return SMLA_EINVAL;
    if (s->out_stride_head < kLatent && s->heads > 1) return SMLA_EINVAL;
    if (s->out_stride_token < 0 || s->lse_stride_token < 0) return SMLA_EINVAL;
    return SMLA_OK;
}

}  // namespace smla

using namespace smla;

extern "C" int smla_plan_for(const smla_shape* shape, int num_sms, smla_plan* plan) {
    if (plan == nullptr) return SMLA_EINVAL;
    const int rc = validate(shape);
    if (rc != SMLA_OK) return rc;
    const bool query_device = num_sms <= 0;
    int dev = -1;
    if (query_device) {
        num_sms = device_sms();
        if (num_sms <= 0 || cudaGetDevice(&dev) != cudaSuccess) return SMLA_ECUDA;
    }
    // Keys per chunk: tiles and splits are chosen for chunks of 128 keys in
    // two stages; SMLA_CHUNK=96 or 128 forces the chunk (96 keys in three
    // stages needs a 32- or 64-head tile).
    const int forced_chunk = [] {
        const char* env = std::getenv("SMLA_CHUNK");
        const int v = env != nullptr ? std::atoi(env) : 0;
        return v == 96 || v == 128 ? v : 0;
    }();
    auto chunk_for = [&](int tile) { return forced_chunk == 96 && tile >= 32 ? 96 : 128; };
    const int max_tile = head_tile_for(shape->heads);
    int forced_tile = 0, forced_splits = 0;
    if (const char* env = std::getenv("SMLA_HEAD_TILE")) {
        const int f = std::atoi(env);
        if ((f == 16 || f == 32 || f == 64) && shape->heads % f == 0) forced_tile = f;
    }
    if (const char* env = std::getenv("SMLA_SPLITS")) forced_splits = std::max(0, std::atoi(env));

    // Head groups of 128 heads may run on the CTA-pair kernel (smla_pair.cu)
    // when SMLA_KERNEL=pair asks for it and no tile or split count of the
    // tile kernel is forced. On GB300 the tile kernel with paired gathers
    // measured faster at the 128-head shapes of the sweep (the pair kernel's
    // three cross-SM handoffs per chunk cost about a microsecond each), so it
    // stays the default.
    const bool use_pair = shape->heads % kPairHeads == 0 && forced_tile == 0 && forced_splits == 0 && [] {
        const char* env = std::getenv("SMLA_KERNEL");
        return env != nullptr && std::strcmp(env, "pair") == 0;
    }();
    const int pair_chunks = (shape->width + kPairChunk - 1) / kPairChunk;
    const long pair_units = static_cast<long>(shape->tokens) * (shape->heads / kPairHeads);
    // Pairing (two head groups share each gathered chunk) pays once a CTA
    // streams at least four chunks, where the gather bounds the pipeline
    // (up to 12% at 128-256 tokens x 128 heads on GB300); at one or two
    // chunks per CTA its multicast latency costs up to 8%.
    int pair_mode = -1;  // -1: by chunks per CTA; 0: never; 1: whenever the shape allows
    if (const char* env = std::getenv("SMLA_PAIR")) pair_mode = std::atoi(env) != 0 ? 1 : 0;
    auto can_pair = [&](int tile) {
        return pair_mode != 0 && shape->num_pools == 1 && (shape->heads / tile) % 2 == 0;
    };
    auto resident = [&](int tile, int s) {
        const int r = query_device ? resident_ctas_on_device(dev, tile, shape->head_dim, chunk_for(tile), s) : 0;
        return r > 0 ? r : (num_sms / s) * s;
    };

    // Head tile and split count. One CTA runs per SM and pays a fixed cost
    // (Q, TMEM, epilogue; larger for wider head tiles) besides its chunks, and
    // a chunk costs more the more CTAs share the HBM. Among the (tile, splits)
    // whose clusters are all resident at once, the one of least estimated
    // time wins:
    //   a(tile) + 0.71 log2(splits) + per * (b(tile) + 0.62 ctas / num_sms) us,
    // per = chunks per CTA; a = 5.1 / 6.3 / 8.0 and b = 2.24 / 2.28 / 2.82 for
    // 16 / 32 / 64 heads (a least-squares fit of the tokens x heads x top-k
    // sweep on GB300). A launch that needs a second wave at any tile takes the
    // widest tile and no split: splitting then only adds fixed costs and
    // merges, and wider tiles read each gathered row for more heads.
    int n = forced_tile > 0 ? forced_tile : max_tile;
    int best = 1;
    double best_cost = 1e300;
    auto chunks_for = [&](int tile) { return (shape->width + chunk_for(tile) - 1) / chunk_for(tile); };
    if (forced_splits == 0) {
        for (int tile = 64; tile >= 16; tile /= 2) {
            if (shape->heads % tile != 0 || (forced_tile > 0 && tile != forced_tile)) continue;
            const int chunks = chunks_for(tile);
            const int max_splits = chunks < 8 ? (chunks < 1 ? 1 : chunks) : 8;
            const long units = static_cast<long>(shape->tokens) * (shape->heads / tile);
            const int pair = 1;  // pairing is decided for the chosen tile and splits
            const double a = tile == 64 ? 8.05 : tile == 32 ? 6.34 : 5.13;
            const double b = tile == 64 ? 2.82 : tile == 32 ? 2.28 : 2.24;
            for (int s = 1; s <= max_splits; ++s) {
                if (s > 1 && !merge_fits(tile, shape->head_dim, chunk_for(tile), s)) continue;
                const int per = chunks > 0 ? (chunks + s - 1) / s : 0;
                if (per > 0 && (chunks + per - 1) / per != s) continue;  // same chunks per CTA as fewer splits
                if (pair * s > kMaxSplits) continue;
                const long ctas = units * s;
                if (ctas > resident(tile, pair * s)) continue;
                const double cost = a + 0.71 * std::log2(static_cast<double>(s)) +
                                    per * (b + 0.62 * static_cast<double>(ctas) / num_sms);
                if (cost < best_cost - 1e-9) {
                    best_cost = cost;
                    n = tile;
                    best = s;
                }
            }
        }
    } else {
        int s = forced_splits;
        const int chunks = chunks_for(n);
        const int cap = chunks < kMaxSplits ? (chunks < 1 ? 1 : chunks) : kMaxSplits;
        if (s > cap) s = cap;
        while (s > 1 && !merge_fits(n, shape->head_dim, chunk_for(n), s)) --s;
        if (can_pair(n) && pair_mode == 1 && 2 * s > kMaxSplits) s = kMaxSplits / 2;
        const int per = chunks > 0 ? (chunks + s - 1) / s : 0;
        best = per > 0 ? (chunks + per - 1) / per : 1;
    }
    if (use_pair) {
        int pair_resident = query_device ? pair_resident_on_device(shape->head_dim) : 0;
        if (pair_resident <= 0) pair_resident = num_sms / 2;
        plan->head_tile = kPairHeads;
        plan->head_groups = shape->heads / kPairHeads;
        plan->chunk = kPairChunk;
        plan->chunks = pair_chunks;
        plan->splits = 1;
        plan->chunks_per_split = pair_chunks;
        plan->ctas = static_cast<int32_t>(2 * pair_units);
        plan->threads = kPairThreads;
        plan->smem_bytes = pair_smem_bytes(shape->head_dim);
        plan->tmem_columns = kPairTmemColumns;
        plan->num_sms = num_sms;
        plan->resident_ctas = 2 * pair_resident;
        plan->pair = 2;
        return SMLA_OK;
    }
    const int groups = shape->heads / n;
    const long units = static_cast<long>(shape->tokens) * groups;
    int chunk = chunk_for(n);
    int chunks = chunks_for(n);
    const int per_cta = chunks > 0 ? (chunks + best - 1) / best : 0;
    int pair = 1;
    if (can_pair(n) && (pair_mode == 1 || per_cta >= 4) && 2 * best <= kMaxSplits &&
        (units * best <= resident(n, best) ? units * best <= resident(n, 2 * best) : true))
        pair = 2;
    // An unpaired CTA of a 32- or 64-head tile that streams eight or more
    // chunks of 128 keys (its cp.async gathers bound the two-stage pipeline)
    // takes chunks of 96 keys in three stages instead: 4-7% faster at 128 x
    // 64 x 2048 and 256 x 64 x 1024 on GB300. A paired 64-head CTA does so
    // from sixteen chunks of 128 on (about 1% at 64 x 128 x 2048); shorter
    // paired streams measured within 4% either way, slower more often than not.
    const bool deep_ring = pair == 1 ? (n >= 32 && per_cta >= 8) : (n == 64 && per_cta >= 16);
    if (forced_chunk == 0 && deep_ring && (best == 1 || merge_fits(n, shape->head_dim, 96, best))) {
        chunk = 96;
        chunks = (shape->width + chunk - 1) / chunk;
    }
    const int best_resident = [&] {
        const int r = query_device ? resident_ctas_on_device(dev, n, shape->head_dim, chunk, pair * best) : 0;
        return r > 0 ? r : (num_sms / (pair * best)) * (pair * best);
    }();
    plan->head_tile = n;
    plan->head_groups = groups;
    plan->chunk = chunk;
    plan->chunks = chunks;
    plan->splits = best;
    plan->chunks_per_split = chunks > 0 ? (chunks + best - 1) / best : 0;
    plan->ctas = static_cast<int32_t>(units * best);
    plan->threads = kThreads;
    plan->smem_bytes = smem_for(n, shape->head_dim, chunk);
    plan->tmem_columns = tmem_for(n);
    plan->num_sms = num_sms;
    plan->resident_ctas = best_resident;
    plan->pair = pair;
    return SMLA_OK;
}

extern "C" int smla_decode(const smla_shape* shape, const void* q, const smla_pool* kv_pools,
                           const int32_t* indices, const int32_t* lens, const float* sinks,
                           float bmm1_scale, float bmm2_scale, float k_scale, void* out, float* lse,
                           void* stream) {
    int rc = validate(shape);
    if (rc != SMLA_OK) return rc;
    if (shape->tokens == 0) return SMLA_OK;
    if (q == nullptr || kv_pools == nullptr || lens == nullptr || out == nullptr) return SMLA_EINVAL;
    if (indices == nullptr && shape->width > 0) return SMLA_EINVAL;
    if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0 || (reinterpret_cast<uintptr_t>(out) & 3u) != 0)
        return SMLA_EINVAL;
    if (shape->out_stride_token % 2 != 0 || shape->out_stride_head % 2 != 0) return SMLA_EINVAL;
    for (int i = 0; i < shape->num_pools; ++i) {
        const smla_pool& pl = kv_pools[i];
        if (pl.data == nullptr || pl.rows < 0 || pl.row_bytes != shape->head_dim) return SMLA_EINVAL;
        if ((reinterpret_cast<uintptr_t>(pl.data) & 15u) != 0) return SMLA_EINVAL;
        if (pl.rows > 0x7FFFFFFFll) return SMLA_EUNSUPPORTED;
    }
    if (!std::isfinite(bmm1_scale) || !std::isfinite(bmm2_scale) || !std::isfinite(k_scale)) return SMLA_EINVAL;
    if (!(bmm1_scale > 0.0f)) return SMLA_EINVAL;  // a softmax scale; its sign orders the maxima

    smla_plan plan;
    rc = smla_plan_for(shape, 0, &plan);
    if (rc != SMLA_OK) return rc;

    const smla_pool& second = shape->num_pools == 2 ? kv_pools[1] : kv_pools[0];
    const float scale_log2 = static_cast<float>(static_cast<double>(bmm1_scale) * 1.4426950408889634);
    const float out_scale = static_cast<float>(static_cast<double>(bmm2_scale) * static_cast<double>(k_scale));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;

    if (plan.head_tile == kPairHeads) {
        // the CTA-pair kernel: each CTA loads Q of 64 of the pair's 128 heads
        PairParams pp;
        std::memset(&pp, 0, sizeof(pp));
        const bool rope = shape->head_dim == 576;
        if (!encode_q_map(&pp.q_latent, q, shape, kPairHeads / 2, 128, CU_TENSOR_MAP_SWIZZLE_128B))
            return SMLA_EUNSUPPORTED;
        if (rope && !encode_q_map(&pp.q_rope, q, shape, kPairHeads / 2, 64, CU_TENSOR_MAP_SWIZZLE_64B))
            return SMLA_EUNSUPPORTED;
        pp.error = device_error_word();
        if (pp.error == nullptr) {
            t_last_cuda_error = static_cast<int>(cudaGetLastError());
            return SMLA_ECUDA;
        }
        pp.pool0 = static_cast<const uint8_t*>(kv_pools[0].data);
        pp.rows0 = kv_pools[0].rows;
        pp.pool1 = static_cast<const uint8_t*>(second.data);
        pp.rows1 = second.rows;
        pp.indices = indices;
        pp.idx_stride = shape->idx_stride_token;
        pp.lens = lens;
        pp.sinks = sinks;
        pp.out = static_cast<__nv_bfloat16*>(out);
        pp.out_stride_token = shape->out_stride_token;
        pp.out_stride_head = shape->out_stride_head;
        pp.lse = lse;
        pp.lse_stride_token = shape->lse_stride_token;
        pp.width = shape->width;
        pp.pool_split = shape->num_pools == 2 ? shape->pool_split : 0;
        pp.num_pools = shape->num_pools;
        pp.scale_log2 = scale_log2;
        pp.out_scale = out_scale;
        pp.peer_tma = encode_kv_map(&pp.kv0, kv_pools[0].data, kv_pools[0].rows, shape->head_dim, 128,
                                    CU_TENSOR_MAP_SWIZZLE_128B) &&
                      (shape->num_pools == 1 ||
                       encode_kv_map(&pp.kv1, second.data, second.rows, shape->head_dim, 128,
                                     CU_TENSOR_MAP_SWIZZLE_128B));
        e = launch_pair(pp, shape->head_dim, plan.head_groups, shape->tokens, dependent_launch(), st);
        if (e != cudaSuccess) {
            t_last_cuda_error = static_cast<int>(e);
            return SMLA_ECUDA;
        }
        return SMLA_OK;
    }

    Params p;
    std::memset(&p, 0, sizeof(p));
    {
        const int n = plan.head_tile;
        const bool rope = shape->head_dim == 576;
        if (!encode_q_map(&p.q_latent, q, shape, n, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return SMLA_EUNSUPPORTED;
        if (rope && !encode_q_map(&p.q_rope, q, shape, n, 64, CU_TENSOR_MAP_SWIZZLE_64B)) return SMLA_EUNSUPPORTED;
    }
    p.q = static_cast<const uint8_t*>(q);
    p.q_stride_token = shape->q_stride_token;
    p.q_stride_head = shape->q_stride_head;
    p.pool0 = static_cast<const uint8_t*>(kv_pools[0].data);
    p.rows0 = kv_pools[0].rows;
    p.pool1 = static_cast<const uint8_t*>(second.data);
    p.rows1 = second.rows;
    p.indices = indices;
    p.idx_stride = shape->idx_stride_token;
    p.lens = lens;
    p.sinks = sinks;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.out_stride_token = shape->out_stride_token;
    p.out_stride_head = shape->out_stride_head;
    p.lse = lse;
    p.lse_stride_token = shape->lse_stride_token;
    p.width = shape->width;
    p.pool_split = shape->num_pools == 2 ? shape->pool_split : 0;
    p.num_pools = shape->num_pools;
    p.splits = plan.splits;
    p.pair = plan.pair;
    if (plan.pair == 2) {
        const bool rope = shape->head_dim == 576;
        if (!encode_kv_map(&p.kv_latent, kv_pools[0].data, kv_pools[0].rows, shape->head_dim, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B) ||
            (rope && !encode_kv_map(&p.kv_rope, kv_pools[0].data, kv_pools[0].rows, shape->head_dim, 64,
                                    CU_TENSOR_MAP_SWIZZLE_64B)))
            p.pair = 1;  // an empty pool (nothing to gather): unpaired
    }
    p.scale_log2 = scale_log2;
    p.out_scale = out_scale;

    const dim3 grid(static_cast<unsigned>(plan.head_groups * plan.splits), static_cast<unsigned>(shape->tokens), 1);
    const int cluster = plan.splits * p.pair;
    e = variant_for(plan.head_tile, shape->head_dim, plan.chunk).launch(p, grid, cluster, st);
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return SMLA_ECUDA;
    }
    return SMLA_OK;
}

namespace smla {

// Where the stream-ordered read of the error word leaves the bits it took, for
// the copy back to the host.
__device__ int32_t g_error_taken;

// Takes the error word's bits and clears it in one atomic step, in stream
// order after the kernels queued before it.
__global__ void take_error_kernel() { g_error_taken = atomicExch(&g_device_error, 0); }

// One warp: thread 0 sets up an mbarrier that expects one arrival and, with
// `arrive` set, arrives on it; every lane then waits with the library's
// bounded wait and `limit_ns`. A wait that gives up records SMLA_DEV_TIMEOUT.
__global__ void bounded_wait_selftest_kernel(int arrive, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncwarp();
    if (threadIdx.x == 0 && arrive) mbar_arrive(&bar);
    const bool ok = mbar_wait_bounded(&bar, 0, &abort_flag, limit_ns);
    if (!ok && threadIdx.x == 0) atomicOr(&g_device_error, SMLA_DEV_TIMEOUT);
}

}  // namespace smla

extern "C" int smla_read_device_error(void* stream, int32_t* bits) {
    if (bits == nullptr) return SMLA_EINVAL;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &capture);
    if (e == cudaSuccess && capture != cudaStreamCaptureStatusNone) return SMLA_EINVAL;
    // one staging word per device: the launch, the copy and the wait of one
    // read finish before another thread's read starts
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int32_t v = 0;
    if (e == cudaSuccess) {
        smla::take_error_kernel<<<1, 1, 0, st>>>();
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&v, smla::g_error_taken, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return SMLA_ECUDA;
    }
    *bits = v;
    return SMLA_OK;
}

extern "C" int smla_selftest_bounded_wait(int arrive, int64_t limit_ns, void* stream) {
    if (limit_ns < 1000 || limit_ns > 1000000000) return SMLA_EINVAL;
    smla::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        arrive != 0, static_cast<uint64_t>(limit_ns));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return SMLA_ECUDA;
    }
    return SMLA_OK;
}

extern "C" int smla_device_error(int32_t* bits) {
    if (bits == nullptr) return SMLA_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    int32_t v = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    const int32_t zero = 0;
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return SMLA_ECUDA;
    }
    *bits = v;
    return SMLA_OK;
}

extern "C" const char* smla_error_string(int code) {
    switch (code) {
        case SMLA_OK: return "ok";
        case SMLA_EINVAL: return "invalid argument (null pointer, shape, stride or alignment)";
        case SMLA_EUNSUPPORTED: return "unsupported shape";
        case SMLA_ECUDA: return "CUDA runtime error";
        case SMLA_EDEVICE: return "device-side error";
        default: return "unknown error";
    }
}

extern "C" int smla_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int smla_version(void) { return 200; }
