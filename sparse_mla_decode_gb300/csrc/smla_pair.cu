// smla_pair.cu -- sparse MLA decode for head groups of 128 heads on sm_103a,
// one pair of CTAs (one cluster of two, on two SMs) per (token, head group).
//
// The operation and the datapath are those of smla_decode.cu: the DeepSeek-V4.1
// "sparse_mla_cute" page ("What this module computes") for what is computed,
// the Kimi K3.1 "attn_sparse" page (module docstring, per-chunk steps and
// "Precision") for how: FP32 logits, a base-2 online softmax per chunk, P
// rounded to E4M3 at 448 of the running maximum, FP32 sums of the unrounded P,
// FP32 accumulation, one BF16 rounding. A chunk here is 256 columns.
//
// Why a pair. With 128 heads on the MMA's N side, both products run at the
// tensor core's full FP8 rate (N = 64 is bound by the shared-memory operand
// reads to about 60% of it), but one SM's TMEM cannot hold O^T for 128 heads x
// 512 latents (512 columns) beside S^T. A cta_group::2 MMA spreads M = 256
// rows over the two SMs of a pair, each supplying half of A and half of B:
//   QK:  S^T[key, head]  = KV[key, :] . Q[head, :]   M = 256 keys (128 per
//        CTA: CTA r gathers the chunk's keys 128 r .. 128 r + 127), N = 128
//        heads (CTA r holds Q of heads 64 r .. 64 r + 63), K = 576 or 512;
//   PV:  O^T[lat, head] += V^T[lat, key] . P^T[key, head]   M = 256 latents
//        (CTA 0 owns latents 0..255, CTA 1 256..511), N = 128 heads (CTA r
//        holds P^T of heads 64 r ..), K = the chunk's 256 keys.
// TMEM per SM: two S^T buffers (2 x 128 columns) and the CTA's half of O^T
// (2 x 128 columns), 512 in all.
//
// PV needs, in each CTA, its latent half of every key of the chunk, while QK
// gave each CTA whole rows of half the keys. After QK, the two latent blocks
// that a CTA's own PV never reads are dead, and each CTA gathers into them the
// peer's keys' blocks it does need: CTA 0 reads blocks 0 and 1 of CTA 1's keys
// into its blocks 2 and 3, CTA 1 blocks 2 and 3 of CTA 0's keys into its
// blocks 0 and 1 (a second read of rows the peer just fetched, mostly from
// L2). The PV's A descriptors then name the same offsets in both CTAs.
//
// The softmax runs over all 256 keys of a chunk: each CTA reduces its 128
// keys per head, the two CTAs exchange those maxima over distributed shared
// memory and both form the same running maximum. P^T of a CTA's keys goes to
// the CTA that holds those heads (its own or its peer's shared memory).
//
// Warps (512 threads, one CTA per SM):
//   0-7   softmax: two warpgroups of 64 heads; thread t is key t of the CTA's
//         128 (TMEM lane t of S^T) and latent row t of each O^T block;
//   8     allocates TMEM (both CTAs together); in CTA 0 one thread issues the
//         pair's MMAs, in CTA 1 one thread relays that its copies landed;
//   9-13  producers of the CTA's own rows: the chunk's indices (loaded a
//         chunk ahead), 16-byte cp.async copies into 128B-swizzled K-major
//         tiles (a latent row per warp instruction, masked keys zero-filled),
//         and an L2 prefetch of the next chunk's rows;
//   14-15 producers of the peer keys' latent half, once QK is done: TMA
//         tile::gather4 (four rows of 128 bytes per instruction, on the SM's
//         TMA unit beside the warps' cp.async; rows past a pool read as zeros).
//         A warp's TMA instructions issue one after another, about 55 ns
//         each, so two warps share them.
// Every wait is bounded; a timeout sets an error bit, tells the peer, and
// the kernel still passes every barrier and frees its TMEM.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "smla.h"
#include "smla_pair.cuh"
#include "smla_ptx.cuh"

namespace smla {
namespace pair {

constexpr int kKeys = 128;   // keys of one CTA per chunk (its 128 MMA rows)
constexpr int kHalf = 64;    // heads whose Q and P^T one CTA holds
constexpr int kMmaWarp = 8;
constexpr int kProducerWarp = 9;  // first of the own-row producers
constexpr int kProducerWarps = 5;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kPeerWarp = kProducerWarp + kProducerWarps;  // 14
constexpr int kPeerWarps = 2;
constexpr int kPeerGroups = kKeys / 4 / kPeerWarps;  // groups of four peer keys per peer warp
static_assert(kPeerWarp + kPeerWarps == kPairThreads / 32, "warps");
constexpr float kLog2P = 8.80735492205760410744f;  // log2(448): P of the running max
constexpr float kLog2e = 1.44269504088896340736f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait, then give up

// Shared memory of one CTA (offsets from a 1024-byte aligned base).
template <int D>
struct Layout {
    static constexpr bool kRope = D == 576;
    static constexpr int kBlock = kKeys * 128;  // one 128-latent block of 128 keys
    static constexpr int kStage = 4 * kBlock + (kRope ? kKeys * 64 : 0);
    static constexpr int kKv = 0;  // 2 stages
    static constexpr int kQ = 2 * kStage;
    static constexpr int kQBytes = 4 * kHalf * 128 + (kRope ? kHalf * 64 : 0);
    static constexpr int kPBytes = kPairChunk * kHalf;  // P^T [256 keys][64 heads]
    static constexpr int kP = kQ + kQBytes;             // 2 buffers
    // P^T of this CTA's keys for the peer's heads, staged for one bulk copy
    // into the peer (8 KB): the rope block of the chunk's stage, which only QK
    // reads; rows of 512 bytes have no rope block and get two of their own.
    static constexpr int kPStageBytes = kKeys * kHalf;
    static constexpr int kPStage = kP + 2 * kPBytes;
    static constexpr int kIdx = kPStage + (kRope ? 0 : 2 * kPStageBytes);  // int32 [2][128] own keys' rows, -1 masked
    static constexpr int kRed = kIdx + 2 * kKeys * 4;  // float [2 warpgroups][4 warps][64]
    static constexpr int kHead = kRed + 2 * 4 * kHalf * 4;  // float [4][128]: m_run, bias, alpha, l
    static constexpr int kPeer = kHead + 4 * kPairHeads * 4;  // float [2][128] peer maxima, [128] peer sums
    static constexpr int kBar = kPeer + 3 * kPairHeads * 4;
    static constexpr int kNumBars = 24;
    static constexpr int kMisc = kBar + kNumBars * 8;  // TMEM base, abort flag
    static constexpr int kBytes = kMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 227 * 1024, "shared memory");
    static_assert(2 * kStage >= kPairHeads * 256 * 2, "the output tile reuses the stages");
    // where chunk c's staged P^T goes: stage b's rope block, or its own area
    static constexpr int p_stage(int b) { return kRope ? kKv + b * kStage + 4 * kBlock : kPStage + b * kPStageBytes; }
};

// Barriers (indices into the CTA's array).
enum : int {
    kOwnFull = 0,    // [2] this CTA's rows of a stage landed (producer cp.async arrivals + index release)
    kPeerFull = 2,   // [2] the peer keys' latent half landed (TMA bytes + the peer warp's cp.async arrivals)
    kSFull = 4,      // [2] QK of the stage's chunk done (commit of the pair's MMAs)
    kPvDone = 6,     // [2] PV of the stage's chunk done (commit)
    kQFull = 8,      // this CTA's Q half landed (TMA bytes)
    kPmaxFull = 9,   // [2 buffers][2 warpgroups] the peer's chunk maxima arrived (st.async bytes + local arm)
    kLFull = 13,     // the peer's per-head sums arrived
    kDrain = 14,     // CTA 0: every MMA done
    kRelayOwn = 15,  // CTA 0: [2] CTA 1's rows of a stage landed
    kRelayPeer = 17, // CTA 0: [2] CTA 1's peer half of a stage landed
    kRelayQ = 19,    // CTA 0: CTA 1's Q half landed
    kPLocal = 20,    // P^T written here and O^T rescaled (the CTA's eight softmax warps), per chunk
    kPRemote = 21,   // [2] the peer's part of this CTA's P^T landed (bulk-copy bytes + local arm)
    kRelayP = 23,    // CTA 0: CTA 1's P^T complete and O^T rescaled, per chunk
};
static_assert(kRelayP < Layout<576>::kNumBars, "barriers");

__device__ __forceinline__ const uint8_t* row_of(const PairParams& p, int col, int32_t id, int d) {
    const bool second = p.num_pools == 2 && col >= p.pool_split;
    return (second ? p.pool1 : p.pool0) + static_cast<int64_t>(id >= 0 ? id : 0) * d;
}

// Column `col`'s row, or -1 when it is a hole, past the count (raw = -1) or
// at or beyond its pool (then also flagged).
__device__ __forceinline__ int32_t resolve(const PairParams& p, int col, int32_t raw) {
    if (raw < 0) return -1;
    const bool second = p.num_pools == 2 && col >= p.pool_split;
    if (raw < (second ? p.rows1 : p.rows0)) return raw;
    atomicOr(p.error, SMLA_DEV_INDEX_RANGE);
    return -1;
}

template <int D>
__global__ void __launch_bounds__(kPairThreads, 1) sparse_mla_decode_pair_kernel(const __grid_constant__ PairParams p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    int32_t* idx_s = reinterpret_cast<int32_t*>(smem + L::kIdx);
    float* red = reinterpret_cast<float*>(smem + L::kRed);
    float* m_run_s = reinterpret_cast<float*>(smem + L::kHead);
    float* bias_s = m_run_s + kPairHeads;
    float* alpha_s = m_run_s + 2 * kPairHeads;
    float* l_s = m_run_s + 3 * kPairHeads;
    float* pmax_s = reinterpret_cast<float*>(smem + L::kPeer);  // [2][128]
    float* lpeer_s = pmax_s + 2 * kPairHeads;                   // [128]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = blockIdx.x & 1u;  // the cluster is (2, 1, 1)
    const uint32_t peer = rank ^ 1u;
    const int head0 = static_cast<int>(blockIdx.x >> 1) * kPairHeads;
    const int token = blockIdx.y;
    auto peer_addr = [&](const void* local) { return map_to_rank(smem_u32(local), peer); };
    auto leader_addr = [&](const void* local) { return map_to_rank(smem_u32(local), 0); };
    // On a timeout: stop this CTA's waits and its peer's.
    auto give_up = [&]() {
        *abort_flag = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_addr(misc + 1)), "r"(1) : "memory");
    };

    // ---- set-up (reads no input, so it overlaps the previous kernel) -------
    if (tid == 0) {
        mbar_init(&bars[kOwnFull + 0], kProducerThreads + 1);
        mbar_init(&bars[kOwnFull + 1], kProducerThreads + 1);
        // the peer warps' cp.async arrivals + one expect-tx arrival each
        mbar_init(&bars[kPeerFull + 0], kPeerWarps * 33);
        mbar_init(&bars[kPeerFull + 1], kPeerWarps * 33);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[kSFull + i], 1);
            mbar_init(&bars[kPvDone + i], 1);
            mbar_init(&bars[kRelayOwn + i], 1);
            mbar_init(&bars[kRelayPeer + i], 1);
        }
        mbar_init(&bars[kQFull], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&bars[kPmaxFull + i], 1);  // the local arm; the bytes come by st.async
        mbar_init(&bars[kLFull], 4);                                      // the peer's four head warps
        mbar_init(&bars[kDrain], 1);
        mbar_init(&bars[kRelayQ], 1);
        mbar_init(&bars[kPLocal], 8);  // the CTA's eight softmax warps
        mbar_init(&bars[kPRemote + 0], 1);
        mbar_init(&bars[kPRemote + 1], 1);
        mbar_init(&bars[kRelayP], 1);
        misc[1] = 0;
        mbar_init_fence();
    }
    if (tid < kPairHeads) {
        m_run_s[tid] = -INFINITY;
        bias_s[tid] = -INFINITY;
        alpha_s[tid] = 1.0f;
        l_s[tid] = 0.0f;
    }
    if (warp == kMmaWarp) {
        tmem_alloc_pair(misc, kPairTmemColumns);
        tmem_relinquish_pair();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensor_map(&p.q_latent);
        if constexpr (L::kRope) prefetch_tensor_map(&p.q_rope);
    }
    if (warp == kPeerWarp && lane == 0 && p.peer_tma) {
        prefetch_tensor_map(&p.kv0);
        if (p.num_pools == 2) prefetch_tensor_map(&p.kv1);
    }
    tc_fence_before_sync();
    cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    grid_dependency_wait();  // inputs are read only after this point
    if (warp == kProducerWarp && lane == 0) {
        mbar_arrive_expect_tx(&bars[kQFull], kHalf * D);
        const int qh = head0 + kHalf * static_cast<int>(rank);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
            tma_load_3d(sbase + L::kQ + kb * kHalf * 128, &p.q_latent, kb * 128, qh, token, &bars[kQFull]);
        if constexpr (L::kRope) tma_load_3d(sbase + L::kQ + 4 * kHalf * 128, &p.q_rope, 512, qh, token, &bars[kQFull]);
    }
    const int count = min(max(p.lens[token], 0), p.width);
    const int nch = (count + kPairChunk - 1) / kPairChunk;
    grid_launch_dependents();

    bool ok = true;
    if (warp >= kProducerWarp && warp < kPeerWarp) {
        // ========================================= own-row producers
        // Thread g < 128 loads and resolves column g of the CTA's half of a
        // chunk (the load a chunk ahead); warp w copies the CTA's keys w,
        // w + 6, ... (one 512-byte latent row per instruction, lane l: bytes
        // 16 l .. 16 l + 15) and the 64-byte ropes of eight keys per
        // instruction, then asks L2 for the next chunk's rows.
        const int g = tid - kProducerWarp * 32;
        const int pw = g >> 5;
        const int32_t* idx_row = p.indices + static_cast<int64_t>(token) * p.idx_stride;
        const int own0 = kKeys * static_cast<int>(rank);
        int32_t raw = -1;
        if (g < kKeys && own0 + g < count) raw = idx_row[own0 + g];
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            const int col0 = c * kPairChunk;
            const int next_col = col0 + kPairChunk + own0 + g;
            int32_t raw_next = -1;
            if (g < kKeys && next_col < count) raw_next = idx_row[next_col];
            if (c >= 2) ok &= mbar_wait_bounded(&bars[kPvDone + b], ((c - 2) >> 1) & 1, abort_flag, kWaitLimitNs);
            if (g < kKeys) idx_s[b * kKeys + g] = resolve(p, col0 + own0 + g, raw);
            named_barrier(3, kProducerThreads);
            if (g == 0) mbar_arrive(&bars[kOwnFull + b]);  // also releases idx_s to the softmax
            const uint32_t stage = sbase + L::kKv + b * L::kStage;
            for (int k = pw; k < kKeys; k += kProducerWarps) {
                const int32_t id = idx_s[b * kKeys + k];
                const uint8_t* src = row_of(p, col0 + own0 + k, id, D) + lane * 16;
                const uint32_t dst =
                    stage + (lane >> 3) * L::kBlock + (k >> 3) * 1024 + (k & 7) * 128 + (((lane & 7) ^ (k & 7)) << 4);
                cp_async_16(dst, src, id >= 0 ? 16u : 0u);
            }
            if constexpr (L::kRope) {
                for (int j = pw; j < kKeys / 8; j += kProducerWarps) {
                    const int k = j * 8 + (lane >> 2), u = lane & 3;
                    const int32_t id = idx_s[b * kKeys + k];
                    const uint8_t* src = row_of(p, col0 + own0 + k, id, D) + 512 + u * 16;
                    const uint32_t dst =
                        stage + 4 * L::kBlock + (k >> 3) * 512 + (k & 7) * 64 + ((u ^ ((k >> 1) & 3)) << 4);
                    cp_async_16(dst, src, id >= 0 ? 16u : 0u);
                }
            }
            cp_async_arrive_noinc(&bars[kOwnFull + b]);
            // the next chunk's rows start their way from HBM into L2 now
            if (g < kKeys && raw_next >= 0) {
                const bool second = p.num_pools == 2 && next_col >= p.pool_split;
                if (raw_next < (second ? p.rows1 : p.rows0)) prefetch_l2(row_of(p, next_col, raw_next, D), D);
            }
            raw = raw_next;
        }
        cp_async_wait_all();
    } else if (warp >= kPeerWarp) {
        // ========================================== peer-half producers
        // Lane l < 16 of peer warp v takes keys 4 q .. 4 q + 3 of the peer's
        // half of a chunk, q = 16 v + l. Once
        // QK of the chunk has read this CTA's dead blocks, the lane's four
        // rows' 256 latent bytes this CTA multiplies in PV (CTA 0: bytes
        // 0..255 into its blocks 2, 3; CTA 1: 256..511 into its blocks 0, 1)
        // come by two tile::gather4 copies; a masked key names a row past its
        // pool (zero fill). Four keys that straddle the pools' boundary, or a
        // pool without a tensor map, are copied by cp.async instead.
        const int32_t* idx_row = p.indices + static_cast<int64_t>(token) * p.idx_stride;
        const int other0 = kKeys * static_cast<int>(peer);
        const int src_x = rank == 0 ? 0 : 256;
        const int dst_blk = rank == 0 ? 2 : 0;
        const bool has_group = lane < kPeerGroups;
        const int q = (warp - kPeerWarp) * kPeerGroups + lane;  // this lane's group (when it has one)
        int32_t raw[4], raw_next[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int col = other0 + 4 * q + i;
            raw[i] = (has_group && col < count) ? idx_row[col] : -1;
        }
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            const int col0 = c * kPairChunk + other0 + 4 * q;  // this lane's first column
            int32_t id[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // out-of-pool indices are flagged by the CTA that owns the column
                const bool second = p.num_pools == 2 && col0 + i >= p.pool_split;
                id[i] = (raw[i] >= 0 && raw[i] < (second ? p.rows1 : p.rows0)) ? raw[i] : -1;
                const int col = col0 + kPairChunk + i;
                raw_next[i] = (has_group && col < count) ? idx_row[col] : -1;
            }
            const bool first_second = p.num_pools == 2 && col0 >= p.pool_split;
            const bool last_second = p.num_pools == 2 && col0 + 3 >= p.pool_split;
            const bool by_tma = has_group && p.peer_tma && first_second == last_second;
            const uint32_t tma_lanes = __ballot_sync(0xFFFFFFFFu, by_tma);
            ok &= mbar_wait_bounded(&bars[kSFull + b], (c >> 1) & 1, abort_flag, kWaitLimitNs);
            const uint32_t stage = sbase + L::kKv + b * L::kStage;
            const int k = 4 * q;  // first of the lane's four keys in the tile
            if (lane == 0) mbar_arrive_expect_tx(&bars[kPeerFull + b], __popc(tma_lanes) * 4 * 256);
            __syncwarp();
            if (by_tma) {
                const void* map = first_second ? static_cast<const void*>(&p.kv1) : static_cast<const void*>(&p.kv0);
                const int32_t past_end = static_cast<int32_t>(first_second ? p.rows1 : p.rows0);
                int32_t r[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) r[i] = id[i] >= 0 ? id[i] : past_end;
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tma_gather4(stage + (dst_blk + h) * L::kBlock + (k >> 3) * 1024 + (k & 7) * 128, map,
                                src_x + 128 * h, r[0], r[1], r[2], r[3], &bars[kPeerFull + b]);
            } else if (has_group) {
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    const uint8_t* row = row_of(p, col0 + i, id[i], D) + src_x;
                    const int kk = k + i;
#pragma unroll
                    for (int v = 0; v < 16; ++v) {
                        const int u = v & 7;
                        const uint32_t dst = stage + (dst_blk + (v >> 3)) * L::kBlock + (kk >> 3) * 1024 +
                                             (kk & 7) * 128 + ((u ^ (kk & 7)) << 4);
                        cp_async_16(dst, row + v * 16, id[i] >= 0 ? 16u : 0u);
                    }
                }
            }
            cp_async_arrive_noinc(&bars[kPeerFull + b]);
#pragma unroll
            for (int i = 0; i < 4; ++i) raw[i] = raw_next[i];
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        if (lane == 0 && rank == 0) {
            // ================================================ MMA issuer
            // QK(c) once chunk c's rows landed in both CTAs and S buffer c % 2
            // is free (PV(c - 2) issued, so the softmax of c - 2 is done); PV(c)
            // once P(c) is written (and O^T rescaled) in both CTAs and the peer
            // halves landed. Whichever is due goes first.
            constexpr uint32_t kIdescQK = idesc_e4m3(256, kPairHeads, 0, 0);
            constexpr uint32_t kIdescPV = idesc_e4m3(256, kPairHeads, 1, 1);
            // Descriptors; moving one by b bytes adds b >> 4 to its start
            // field (no carry: shared addresses stay below 256 KB).
            const uint64_t d_q = smem_desc(sbase + L::kQ, 1024, 1024, kSwizzle128B);
            const uint64_t d_q_rope = smem_desc(sbase + L::kQ + 4 * kHalf * 128, 512, 512, kSwizzle64B);
            const uint64_t d_kv = smem_desc(sbase + L::kKv, 1024, 1024, kSwizzle128B);
            const uint64_t d_kv_rope = smem_desc(sbase + L::kKv + 4 * L::kBlock, 512, 512, kSwizzle64B);
            const uint64_t d_p = smem_desc(sbase + L::kP, 512, 512, kSwizzle64B);
            const uint32_t s_full_peer = peer_addr(&bars[kSFull]);
            const uint32_t pv_done_peer = peer_addr(&bars[kPvDone]);
            int next_qk = 0, next_pv = 0, armed = 0;  // armed: chunks whose P^T bytes this thread expects
            bool q_ready = false;
            uint64_t idle_since = 0;
            while (next_pv < nch) {
                bool progressed = false;
                if (!q_ready) q_ready = mbar_test_wait(&bars[kQFull], 0) && mbar_test_wait_cluster(&bars[kRelayQ], 0);
                if (q_ready && next_qk < nch && next_qk <= next_pv + 1) {
                    const int c = next_qk, b = c & 1;
                    const uint32_t par = (c >> 1) & 1;
                    if (mbar_test_wait(&bars[kOwnFull + b], par) && mbar_test_wait_cluster(&bars[kRelayOwn + b], par)) {
                        fence_proxy_async_all();  // the producers' cp.async data, for the tensor cores
                        tc_fence_after_sync();
                        const uint32_t stage16 = static_cast<uint32_t>(b * L::kStage) >> 4;
                        const uint32_t d_s = tmem + b * kPairHeads;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int kb = i >> 2, ks = i & 3;
                            mma_f8_pair(d_s, d_kv + stage16 + ((kb * L::kBlock + ks * 32) >> 4),
                                        d_q + ((kb * kHalf * 128 + ks * 32) >> 4), kIdescQK, i != 0 ? 1u : 0u);
                        }
                        if constexpr (L::kRope) {
#pragma unroll
                            for (int ks = 0; ks < 2; ++ks)
                                mma_f8_pair(d_s, d_kv_rope + stage16 + ((ks * 32) >> 4), d_q_rope + ((ks * 32) >> 4),
                                            kIdescQK, 1u);
                        }
                        mma_commit_pair(smem_u32(&bars[kSFull + b]));
                        mma_commit_pair(s_full_peer + 8 * b);
                        ++next_qk;
                        progressed = true;
                    }
                }
                if (next_pv < next_qk) {
                    const int c = next_pv, b = c & 1;
                    const uint32_t par = (c >> 1) & 1;
                    if (armed == c) {  // the peer's bulk copy of this chunk's P^T part
                        mbar_arrive_expect_tx(&bars[kPRemote + b], L::kPStageBytes);
                        ++armed;
                    }
                    // this CTA's barriers first (CTA-scope tests are cheap), the
                    // ones the peer completes after
                    if (mbar_test_wait(&bars[kPLocal], c & 1) && mbar_test_wait(&bars[kPeerFull + b], par) &&
                        mbar_test_wait_cluster(&bars[kPRemote + b], par) && mbar_test_wait_cluster(&bars[kRelayP], c & 1) &&
                        mbar_test_wait_cluster(&bars[kRelayPeer + b], par)) {
                        fence_proxy_async_all();
                        tc_fence_after_sync();
                        const uint32_t stage16 = static_cast<uint32_t>(b * L::kStage) >> 4;
                        const uint32_t p16 = static_cast<uint32_t>(b * L::kPBytes) >> 4;
#pragma unroll
                        for (int grp = 0; grp < 2; ++grp) {
#pragma unroll
                            for (int ks = 0; ks < 8; ++ks) {
                                // keys 0..127 (CTA 0's) sit in block grp, keys
                                // 128..255 (CTA 1's) in block 2 + grp, in both CTAs
                                const int blk = ks < 4 ? grp : 2 + grp;
                                const uint32_t a_off = stage16 + ((blk * L::kBlock + (ks & 3) * 32 * 128) >> 4);
                                const uint32_t b_off = p16 + ((ks * 32 * kHalf) >> 4);
                                mma_f8_pair(tmem + 2 * kPairHeads + grp * kPairHeads, d_kv + a_off, d_p + b_off,
                                            kIdescPV, (c > 0 || ks > 0) ? 1u : 0u);
                            }
                        }
                        mma_commit_pair(smem_u32(&bars[kPvDone + b]));
                        mma_commit_pair(pv_done_peer + 8 * b);
                        ++next_pv;
                        progressed = true;
                    }
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
            if (!q_ready) ok &= mbar_wait_bounded(&bars[kQFull], 0, abort_flag, kWaitLimitNs);  // no copy outlives the CTA
            mma_commit_pair(smem_u32(&bars[kDrain]));
        } else if (lane == 0) {
            // ======================================= relay (CTA 1)
            // The leader's MMAs read this CTA's shared memory: tell it when
            // the Q half, a stage's own rows and a stage's peer half landed.
            ok &= mbar_wait_bounded(&bars[kQFull], 0, abort_flag, kWaitLimitNs);
            fence_proxy_async_all();
            mbar_arrive_cluster(leader_addr(&bars[kRelayQ]));
            int next_own = 0, next_peer = 0, next_p = 0, armed = 0;
            uint64_t idle_since = 0;
            while (next_peer < nch || next_p < nch) {
                bool progressed = false;
                if (next_p < next_own) {
                    const int b = next_p & 1;
                    if (armed == next_p) {
                        mbar_arrive_expect_tx(&bars[kPRemote + b], L::kPStageBytes);
                        ++armed;
                    }
                    if (mbar_test_wait(&bars[kPLocal], next_p & 1) &&
                        mbar_test_wait_cluster(&bars[kPRemote + b], (next_p >> 1) & 1)) {
                        tc_fence_after_sync();
                        fence_proxy_async_all();
                        tc_fence_before_sync();
                        mbar_arrive_cluster(leader_addr(&bars[kRelayP]));
                        ++next_p;
                        progressed = true;
                    }
                }
                if (next_own < nch && mbar_test_wait(&bars[kOwnFull + (next_own & 1)], (next_own >> 1) & 1)) {
                    fence_proxy_async_all();
                    mbar_arrive_cluster(leader_addr(&bars[kRelayOwn + (next_own & 1)]));
                    ++next_own;
                    progressed = true;
                }
                if (next_peer < next_own && mbar_test_wait(&bars[kPeerFull + (next_peer & 1)], (next_peer >> 1) & 1)) {
                    fence_proxy_async_all();
                    mbar_arrive_cluster(leader_addr(&bars[kRelayPeer + (next_peer & 1)]));
                    ++next_peer;
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
        }
        __syncwarp();
    } else {
        // ===================================================== softmax
        // Warpgroup wg owns heads 64 wg .. 64 wg + 63 of the pair. Thread t owns
        // key t of the CTA's 128 (TMEM lane t of S^T) and latent row t of
        // each of the CTA's two O^T blocks.
        const int wg = warp >> 2, quarter = warp & 3, t = tid & 127, hw = kHalf * wg;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const float scale_log2 = p.scale_log2;
        // P^T of these heads lives in CTA wg: written straight into its own
        // buffer, or staged here and sent to the peer by one bulk copy
        const bool p_local = static_cast<uint32_t>(wg) == rank;
        const uint32_t p_row = kKeys * rank + t;  // this key's row of the chunk's P^T
        float lsum[kHalf];
#pragma unroll
        for (int h = 0; h < kHalf; ++h) lsum[h] = 0.0f;

        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            const uint32_t par = (c >> 1) & 1;
            ok &= mbar_wait_bounded(&bars[kOwnFull + b], par, abort_flag, kWaitLimitNs);
            ok &= mbar_wait_bounded(&bars[kSFull + b], par, abort_flag, kWaitLimitNs);
            tc_fence_after_sync();
            const bool active = idx_s[b * kKeys + t] >= 0;
            const uint32_t s_col = tmem + lane_base + b * kPairHeads + hw;

            // chunk maxima per head over this CTA's keys (raw logits;
            // bmm1_scale > 0 keeps the order, masked keys are -inf), 32 heads
            // at a time: a transposing butterfly, each step hands half of a
            // lane's heads to its partner, so that lane l ends with head l
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tmem_load32x1(s_col + 32 * half, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = active ? v[j] : -INFINITY;
#pragma unroll
                for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < n / 2; ++i) {
                        const float send = up ? v[i] : v[i + n / 2];
                        const float keep = up ? v[i + n / 2] : v[i];
                        v[i] = fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
                    }
                }
                red[(wg * 4 + quarter) * kHalf + 32 * half + lane] = v[0];
            }
            named_barrier(1 + wg, 128);
            if (t < kHalf) {
                // head hw + t: the CTA's maximum to the peer (st.async, the
                // bytes counted on the peer's barrier), the peer's back, and
                // the same running maximum in both CTAs
                const float* r = red + wg * 4 * kHalf + t;
                const float cm = fmaxf(fmaxf(r[0], r[kHalf]), fmaxf(r[2 * kHalf], r[3 * kHalf]));
                uint64_t* pmax_bar = &bars[kPmaxFull + 2 * b + wg];
                st_async_f32(peer_addr(&pmax_s[b * kPairHeads + hw + t]), cm, peer_addr(pmax_bar));
                if (t == 0) mbar_arrive_expect_tx(pmax_bar, kHalf * 4);
                ok &= mbar_wait_cluster_bounded(pmax_bar, par, abort_flag, kWaitLimitNs);
                const float both = fmaxf(cm, pmax_s[b * kPairHeads + hw + t]);
                const int h = hw + t;
                const float mo = m_run_s[h];
                const float mn = fmaxf(mo, both * scale_log2);
                alpha_s[h] = (mo == -INFINITY) ? 1.0f : fast_exp2(mo - mn);
                bias_s[h] = mn - kLog2P;
                m_run_s[h] = mn;
            }
            named_barrier(1 + wg, 128);

            // P = 2^(s * scale_log2 - m + log2 448) as E4M3 (PV of chunk c - 2
            // has finished reading P^T[b] in both CTAs); FP32 sums of the
            // unrounded P. Rows of 64 heads (64 bytes), 16-byte units swizzled
            // (64B) as the PV's B operand reads them.
            if (c >= 2) ok &= mbar_wait_bounded(&bars[kPvDone + b], ((c - 2) >> 1) & 1, abort_flag, kWaitLimitNs);
            {
                uint8_t* prow = p_local ? smem + L::kP + b * L::kPBytes + p_row * 64
                                        : smem + L::p_stage(b) + t * 64;
#pragma unroll
                for (int gq = 0; gq < 4; ++gq) {
                    float sv[16];
                    tmem_load16x1(s_col + 16 * gq, sv);
                    uint32_t words[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int j = 16 * gq + 4 * q4;
                        const float4 bi = reinterpret_cast<const float4*>(bias_s + hw)[j / 4];
                        const float4 al = reinterpret_cast<const float4*>(alpha_s + hw)[j / 4];
                        float pr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        if (active) {
                            pr[0] = fast_exp2(fmaf(sv[4 * q4 + 0], scale_log2, -bi.x));
                            pr[1] = fast_exp2(fmaf(sv[4 * q4 + 1], scale_log2, -bi.y));
                            pr[2] = fast_exp2(fmaf(sv[4 * q4 + 2], scale_log2, -bi.z));
                            pr[3] = fast_exp2(fmaf(sv[4 * q4 + 3], scale_log2, -bi.w));
                        }
                        lsum[j + 0] = fmaf(lsum[j + 0], al.x, pr[0]);
                        lsum[j + 1] = fmaf(lsum[j + 1], al.y, pr[1]);
                        lsum[j + 2] = fmaf(lsum[j + 2], al.z, pr[2]);
                        lsum[j + 3] = fmaf(lsum[j + 3], al.w, pr[3]);
                        words[q4] = e4m3x2(pr[0], pr[1]) | (e4m3x2(pr[2], pr[3]) << 16);
                    }
                    // the swizzle of row p_row; the staged rows (p_row - 128 r)
                    // share it, 128 r being a multiple of 8
                    *reinterpret_cast<uint4*>(prow + ((gq ^ ((p_row >> 1) & 3)) << 4)) =
                        make_uint4(words[0], words[1], words[2], words[3]);
                }
                fence_proxy_async_cta();  // for the tensor cores, or the bulk copy
                if (!p_local) {
                    named_barrier(1 + wg, 128);
                    if (t == 0)
                        bulk_copy_to_cluster(map_to_rank(sbase + L::kP + b * L::kPBytes + kKeys * rank * 64, peer),
                                             sbase + L::p_stage(b), L::kPStageBytes, peer_addr(&bars[kPRemote + b]));
                }
            }

            // O^T *= alpha for the heads whose running maximum rose (PV of chunk
            // c - 1 is done)
            if (c >= 1) {
                ok &= mbar_wait_bounded(&bars[kPvDone + ((c - 1) & 1)], ((c - 1) >> 1) & 1, abort_flag, kWaitLimitNs);
                tc_fence_after_sync();
#pragma unroll
                for (int gq = 0; gq < 4; ++gq) {
                    float a[16];
                    bool rescale = false;
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const float4 v4 = reinterpret_cast<const float4*>(alpha_s + hw + 16 * gq)[j4];
                        a[4 * j4 + 0] = v4.x;
                        a[4 * j4 + 1] = v4.y;
                        a[4 * j4 + 2] = v4.z;
                        a[4 * j4 + 3] = v4.w;
                        rescale |= (v4.x != 1.0f) | (v4.y != 1.0f) | (v4.z != 1.0f) | (v4.w != 1.0f);
                    }
                    if (rescale) {
                        const uint32_t col = tmem + lane_base + 2 * kPairHeads + hw + 16 * gq;
                        float v[32];
                        tmem_load16x2(col, col + kPairHeads, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= a[i & 15];
                        tmem_store16x2(col, col + kPairHeads, v);
                    }
                }
                tmem_wait_st();
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kPLocal]);
        }
        if (nch > 0)
            ok &= mbar_wait_bounded(&bars[kPvDone + ((nch - 1) & 1)], ((nch - 1) >> 1) & 1, abort_flag, kWaitLimitNs);
        tc_fence_after_sync();

        // per-head totals over this CTA's keys, then over the pair
#pragma unroll
        for (int j = 0; j < kHalf; ++j) {
            float v = lsum[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
            if (lane == (j & 31)) red[(wg * 4 + quarter) * kHalf + j] = v;
        }
        named_barrier(1 + wg, 128);
        if (t < kHalf) {
            const float* r = red + wg * 4 * kHalf + t;
            const float mine = (r[0] + r[kHalf]) + (r[2 * kHalf] + r[3 * kHalf]);
            l_s[hw + t] = mine;
            st_cluster_f32(peer_addr(&lpeer_s[hw + t]), mine);
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(peer_addr(&bars[kLFull]));
        }
    }
    if (!ok) {
        give_up();
        atomicOr(p.error, SMLA_DEV_TIMEOUT);
    }
    cp_async_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    // ================================================ epilogue
    // Per head: the pair's sum (both CTAs add the same two numbers), the
    // sink, the output scale and the base-2 LSE (written by CTA 0).
    if (tid < kPairHeads) {
        bool got = mbar_wait_cluster_bounded(&bars[kLFull], 0, abort_flag, kWaitLimitNs);
        if (!got) {
            give_up();
            atomicOr(p.error, SMLA_DEV_TIMEOUT);
        }
        const int h = head0 + tid;
        const float m = m_run_s[tid];
        const float l = rank == 0 ? l_s[tid] + lpeer_s[tid] : lpeer_s[tid] + l_s[tid];
        float scale = 0.0f, lse2 = -INFINITY;
        if (m != -INFINITY) {
            float top = m, extra = 0.0f;
            if (p.sinks != nullptr) {
                const float s2 = p.sinks[h] * kLog2e;
                top = fmaxf(m, s2);
                extra = 448.0f * fast_exp2(s2 - top);
            }
            const float w = fast_exp2(m - top);
            const float total = l * w + extra;
            scale = p.out_scale * w / total;
            lse2 = top - kLog2P + log2f(total);
        }
        bias_s[tid] = scale;
        if (rank == 0 && p.lse != nullptr) p.lse[static_cast<int64_t>(token) * p.lse_stride_token + h] = lse2;
    }
    __syncthreads();
    // O^T (lane = latent, column = head) -> BF16 [128 heads][256 latents] in
    // shared memory (the stages are free), then 16-byte stores of the CTA's
    // latent half of every row.
    const bool empty = m_run_s[0] == -INFINITY;  // no active key: +0.0 everywhere
    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(smem + L::kKv);
    if (warp < 8) {
        const int wg = warp >> 2, quarter = warp & 3, hw = kHalf * wg;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
#pragma unroll 1
        for (int grp = 0; grp < 2; ++grp) {
#pragma unroll 1
            for (int j0 = 0; j0 < kHalf; j0 += 32) {
                float v[32];
                tmem_load32x1(tmem + lane_base + 2 * kPairHeads + grp * kPairHeads + hw + j0, v);
                const int lat = grp * 128 + quarter * 32 + lane;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int h = hw + j0 + i;
                    tile[h * 256 + lat] = __float2bfloat16_rn(empty ? 0.0f : v[i] * bias_s[h]);
                }
            }
        }
    }
    __syncthreads();
    {
        __nv_bfloat16* out = p.out + static_cast<int64_t>(token) * p.out_stride_token +
                             static_cast<int64_t>(head0) * p.out_stride_head + 256 * rank;
        const bool wide = ((reinterpret_cast<uintptr_t>(p.out) | static_cast<uintptr_t>(p.out_stride_token * 2) |
                            static_cast<uintptr_t>(p.out_stride_head * 2)) & 15u) == 0;
        if (wide) {
            for (int i = tid; i < kPairHeads * 256 / 8; i += kPairThreads) {
                const int h = i >> 5, e = (i & 31) * 8;
                *reinterpret_cast<uint4*>(out + static_cast<int64_t>(h) * p.out_stride_head + e) =
                    *reinterpret_cast<const uint4*>(tile + h * 256 + e);
            }
        } else {
            for (int i = tid; i < kPairHeads * 256 / 2; i += kPairThreads) {
                const int h = i >> 7, e = (i & 127) * 2;
                *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(h) * p.out_stride_head + e) =
                    *reinterpret_cast<const uint32_t*>(tile + h * 256 + e);
            }
        }
    }

    // ---- teardown: every MMA, TMEM access and remote write has finished ----
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp && rank == 0) {
        tc_fence_after_sync();
        if (!mbar_wait_bounded(&bars[kDrain], 0, abort_flag, kWaitLimitNs)) {
            if (lane == 0) atomicOr(p.error, SMLA_DEV_TIMEOUT);
        }
        __syncwarp();
    }
    tc_fence_before_sync();
    cluster_sync_all();
    tc_fence_after_sync();
    if (warp == kMmaWarp) tmem_dealloc_pair(tmem, kPairTmemColumns);
}

template <int D>
cudaError_t configure() {
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(sparse_mla_decode_pair_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Layout<D>::kAlloc);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

template <int D>
cudaError_t launch(const PairParams& p, int groups, int tokens, bool dependent, cudaStream_t stream) {
    cudaError_t e = configure<D>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * groups), static_cast<unsigned>(tokens), 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = Layout<D>::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 2;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = dependent ? 1 : 0;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sparse_mla_decode_pair_kernel<D>, p);
}

template <int D>
int resident_clusters() {
    if (configure<D>() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = Layout<D>::kAlloc;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, sparse_mla_decode_pair_kernel<D>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters;
}

}  // namespace pair

int pair_smem_bytes(int head_dim) {
    return head_dim == 576 ? pair::Layout<576>::kAlloc : pair::Layout<512>::kAlloc;
}

cudaError_t launch_pair(const PairParams& p, int head_dim, int groups, int tokens, bool dependent,
                        cudaStream_t stream) {
    return head_dim == 576 ? pair::launch<576>(p, groups, tokens, dependent, stream)
                           : pair::launch<512>(p, groups, tokens, dependent, stream);
}

int pair_resident_clusters(int head_dim) {
    return head_dim == 576 ? pair::resident_clusters<576>() : pair::resident_clusters<512>();
}

}  // namespace smla
