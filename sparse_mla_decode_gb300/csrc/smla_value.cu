// Value projection and sigmoid gate after the merge of partial sets.
//
// What it computes follows the Kimi K3.1 `mla/dcp` page, DcpValue (class
// docstring and merge, after the merged rows): for token t, head h and value
// v < 128,
//   out[t, h*128 + v] = BF16(BF16(sum_j latent[t, h, j] * W_UV[h, j, v]) * sigmoid(gate[t, h*128 + v]))
// over the 512 latents, BF16 operands and FP32 accumulation; rows of a token
// whose count is <= 0 are zero.
//
// One CTA per (head, 64-token tile) computes the transposed product
// D[v][t] = sum_j W_UV[h][j][v] * latent[t][h][j] on the tensor cores: M = 128
// values (always full), N = 64 tokens (rows past the token count read as
// zeros), K = 16 latents per instruction, D in TMEM (lane = value, column =
// token). A (W_UV[h], values contiguous) is MN-major, B (the latent tile) is
// K-major, both with the 128-byte swizzle. Everything a CTA reads is in
// shared memory at once (W_UV[h] 128 KB, latents 64 KB, gates 16 KB): TMA
// brings it in eight latent blocks, each completing its own barrier, so the
// products of block kb start as soon as its bytes land. Four warps (one value
// each per lane) round, gate and write the values into the gate tile in
// place, and one TMA store writes the tile out (rows past the token count are
// clipped).
//
// The fused entry point (smla_merge_value) takes the partial sets instead of
// merged rows, as the page's owner does. A producer warp streams the sources'
// 64-token boxes of partial rows by TMA, sixteen consumer warps merge them
// block by block into a swizzled B ring with the merge kernel's own weights
// and operation order (so the rows carry the same bits as smla_merge's), and
// an MMA warp runs each block's products as soon as it is merged; the epilogue
// is the same.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "smla.h"
#include "smla_merge_row.cuh"
#include "smla_ptx.cuh"

namespace smla {
void note_cuda_error(int code);
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
int32_t* device_error_word();
}  // namespace smla

namespace vgate {

using namespace smla;

constexpr int kTile = 64;   // tokens per CTA (N)
constexpr int kJ = 512;     // latents (K)
constexpr int kV = 128;     // values per head (M)
constexpr int kBlocks = kJ / 64;              // 64-latent blocks, one swizzle atom wide
constexpr int kWBlockBytes = 64 * kV * 2;     // 64 latent rows x 128 values: two 8 KB MN atoms
constexpr int kLBlockBytes = kTile * 128;     // 64 tokens x 64 latents
constexpr int kGateBytes = kTile * kV * 2;    // 64 tokens x 128 values, unswizzled
constexpr int kW = 0;
constexpr int kL = kW + kBlocks * kWBlockBytes;
constexpr int kG = kL + kBlocks * kLBlockBytes;
constexpr int kBar = kG + kGateBytes;
constexpr int kMisc = kBar + 8 * (kBlocks + 2);
constexpr int kAlloc = kMisc + 16 + 1024;
constexpr int kWarps = 8;  // thread 0 issues the copies and the products; all eight run the epilogue
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct Params {
    CUtensorMap latent;  // {512 latents, H heads, T tokens} BF16, 128-byte swizzle, boxes of 64 x 1 x 64
                         // (fused: the partial sets, {512 latents, H, T, S sources}, boxes of 64 x 1 x 64 x 1)
    CUtensorMap w_uv;    // {64 values, 512 latents, 2 value halves, H heads} BF16, 128-byte swizzle, boxes of 64 x 64 x 2 x 1
    CUtensorMap gate;    // {H * 128, T} BF16, boxes of 128 x 64
    CUtensorMap out;     // {H * 128, T} BF16, boxes of 128 x 64
    const int32_t* lens; // [T] or null
    MergeInputs merge;   // fused: the partial sets (for the weights; the rows come by TMA)
    int32_t tokens, heads;
    int32_t* error;      // the library's device error word
};

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 1 / x by the approximate reciprocal (one MUFU operation, at most 1 ulp of
// FP32 from the exact value; subnormal results kept, 1 / inf = 0): no
// branches, so the compiler can overlap the 32 gates of a thread.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// kind::f16 instruction descriptor: BF16 A and B (format 1), FP32 D.
constexpr uint32_t idesc_bf16(int m, int n, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tma_store_2d(const void* map, int32_t x, int32_t y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, int32_t c0, int32_t c1, int32_t c2,
                                            int32_t c3, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts_u16(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(static_cast<uint16_t>(v)) : "memory");
}

// The epilogue of a CTA's tile: kEpiWarps warps (4 or 16) read D back from
// TMEM, warp w reading lanes 32 (w % 4) .. + 31, so that thread (w, lane) owns
// value v = 32 (w % 4) + lane of the kEpiWarps-dependent run of tokens from
// tb; they round, gate and write the values into the gate tile in place.
// Bit t of `live` says whether token tb + t has keys. Returns false if a
// bounded wait gave up.
// sigmoid(g) = 1 / (1 + e^-g), in FP32 to a few ulp (the value is then
// rounded to BF16, 2^-8 relative)
__device__ __forceinline__ float sigmoid_of_bf16(uint32_t bits) {
    return rcp_approx(1.0f + __expf(-__uint_as_float(bits << 16)));
}

// The gates of the epilogue thread (warp, lane) of a kEpiWarps-warp epilogue,
// as sigmoids.
template <int kEpiWarps>
__device__ __forceinline__ void epilogue_sigmoids(uint32_t tile, int warp, int lane,
                                                  float (&sig)[kTile * 4 / kEpiWarps]) {
    constexpr int kTokensPerWarp = kTile * 4 / kEpiWarps;
    const int v = 32 * (warp & 3) + lane, tb = kTokensPerWarp * (warp >> 2);
    const uint32_t slot = tile + static_cast<uint32_t>(tb * kV + v) * 2;
#pragma unroll
    for (int t = 0; t < kTokensPerWarp; ++t) sig[t] = sigmoid_of_bf16(lds_u16(slot + t * kV * 2));
}

template <int kEpiWarps, bool kHaveSigmoids = false>
__device__ __forceinline__ bool gate_epilogue(const Params& p, uint32_t tile, uint32_t tmem, uint64_t* mma_done,
                                              uint64_t* gate_full, volatile int* abort_flag, int t0, int warp,
                                              int lane, const float* sig = nullptr) {
    constexpr int kTokensPerWarp = kTile * 4 / kEpiWarps;
    const int v = 32 * (warp & 3) + lane;
    const int tb = kTokensPerWarp * (warp >> 2);
    const int t_lane = t0 + tb + (lane % kTokensPerWarp);
    const uint32_t live =
        __ballot_sync(~0u, t_lane < p.tokens && (p.lens == nullptr || p.lens[t_lane] > 0));
    bool ok = mbar_wait_bounded(mma_done, 0, abort_flag, kWaitLimitNs);
    if (!kHaveSigmoids) ok &= mbar_wait_bounded(gate_full, 0, abort_flag, kWaitLimitNs);
    __syncwarp();
    tc_fence_after_sync();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    float acc[kTokensPerWarp];
    const uint32_t col = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + tb;
    if constexpr (kTokensPerWarp == 32) {
        tmem_load16x2(col, col + 16, acc);
    } else {
        tmem_load16x1(col, acc);
    }
    const uint32_t slot = tile + static_cast<uint32_t>(tb * kV + v) * 2;  // gate / value of token tb
    uint32_t bits[kTokensPerWarp];
    if (!kHaveSigmoids) {
#pragma unroll
        for (int t = 0; t < kTokensPerWarp; ++t) bits[t] = lds_u16(slot + t * kV * 2);
    }
#pragma unroll
    for (int t = 0; t < kTokensPerWarp; ++t) {
        const float rounded = __bfloat162float(__float2bfloat16_rn(acc[t]));
        const float y = rounded * (kHaveSigmoids ? sig[t] : sigmoid_of_bf16(bits[t]));
        bits[t] = (live >> t) & 1u ? __bfloat16_as_ushort(__float2bfloat16_rn(y)) : 0u;
    }
#pragma unroll
    for (int t = 0; t < kTokensPerWarp; ++t) sts_u16(slot + t * kV * 2, bits[t]);
    fence_proxy_async_smem();  // the values, written by threads, are read by the TMA store
    return ok;
}

__global__ void __launch_bounds__(32 * kWarps, 1) value_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBar);
    uint64_t* block_full = bars;               // [kBlocks]: latent block kb and its W_UV rows landed
    uint64_t* gate_full = bars + kBlocks;      // the gate tile landed
    uint64_t* mma_done = bars + kBlocks + 1;   // every product finished (commit)
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, t0 = blockIdx.y * kTile;

    // thread 0 starts the copies as soon as its barriers exist; warp 1
    // allocates TMEM meanwhile
    if (tid == 0) {
        for (int i = 0; i < kBlocks + 2; ++i) mbar_init(bars + i, 1);
        misc[1] = 0;
        mbar_init_fence();
        prefetch_tensor_map(&p.latent);
        prefetch_tensor_map(&p.w_uv);
        prefetch_tensor_map(&p.gate);
        prefetch_tensor_map(&p.out);
    }
    if (warp == 1) {
        tmem_alloc(misc, kTile);  // D: 128 lanes (values) x 64 columns (tokens)
        tmem_relinquish();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
        for (int kb = 0; kb < kBlocks; ++kb) {
            mbar_arrive_expect_tx(block_full + kb, kLBlockBytes + kWBlockBytes);
            tma_load_3d(sbase + kL + kb * kLBlockBytes, &p.latent, kb * 64, h, t0, block_full + kb);
            tma_load_4d(sbase + kW + kb * kWBlockBytes, &p.w_uv, 0, kb * 64, 0, h, block_full + kb);
        }
        mbar_arrive_expect_tx(gate_full, kGateBytes);
        tma_load_2d(sbase + kG, &p.gate, h * kV, t0, gate_full);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    bool ok = true;
    if (tid == 0) {
        // A = W_UV^T: MN-major, 64-value atoms 8 KB apart (LBO), 8-latent
        // groups 1 KB apart (SBO); B = latents: K-major, 8-token groups 1 KB
        // apart. A step of 16 latents moves A by 16 rows of 128 bytes and B by
        // 32 bytes inside its swizzle atom.
        constexpr uint32_t kIdesc = idesc_bf16(kV, kTile, 1, 0);
        const uint64_t d_a = smem_desc(sbase + kW, kWBlockBytes / 2, 1024, kSwizzle128B);
        const uint64_t d_b = smem_desc(sbase + kL, 1024, 1024, kSwizzle128B);
        for (int kb = 0; kb < kBlocks; ++kb) {
            ok &= mbar_wait_bounded(block_full + kb, 0, abort_flag, kWaitLimitNs);
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const uint32_t a_off = static_cast<uint32_t>(kb * kWBlockBytes + s4 * 16 * 128) >> 4;
                const uint32_t b_off = static_cast<uint32_t>(kb * kLBlockBytes + s4 * 32) >> 4;
                mma_bf16(tmem, d_a + a_off, d_b + b_off, kIdesc, (kb | s4) != 0 ? 1u : 0u);
            }
        }
        mma_commit(mma_done);
    }
    __syncwarp();
    ok &= gate_epilogue<kWarps>(p, sbase + kG, tmem, mma_done, gate_full, abort_flag, t0, warp, lane);
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        if (ok) {
            tma_store_2d(&p.out, h * kV, t0, sbase + kG);
            tma_store_wait_read();
        }
    }
    if (!ok && lane == 0) atomicOr(p.error, SMLA_DEV_TIMEOUT);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTile);
    }
}

// ------------------------------------------------ fused merge + projection
//
// One CTA per (head, 64-token tile), 18 warps:
//  - warps 0-15 (the consumers) first compute every row's merge weights into
//    shared memory, then merge latent block by latent block: for block kb
//    they take the S sources' 64-token boxes from a ring in chunks of four
//    sources, thread c accumulating 8 latents (unit c % 8) of token c / 8 in
//    FP32 with the merge's own operations in source order, and write the
//    BF16 block into a 2-block B ring; at the end they run the epilogue;
//  - warp 16 (the producer) streams the gate tile and then, block after
//    block, the S boxes of partial rows into a ring of four 4-box chunks
//    (128 KB in flight, what the HBM latency asks for at this SM's share of
//    bandwidth), each chunk as soon as the consumers release it;
//  - warp 17 (the MMA warp) owns TMEM, keeps W_UV's rows three blocks ahead
//    in a 3-slot ring, and issues block kb's four products as soon as the
//    block's B rows and W_UV rows are in; their completion frees both slots.
namespace fz {
constexpr int kConsumerWarps = 16;
constexpr int kProducerWarp = 16, kMmaWarp = 17, kWarpsAll = 18;
constexpr int kChunk = 4;                              // sources' boxes behind one barrier
constexpr int kStages = 4, kWSlots = 3, kBSlots = 2;   // 4 chunks: 128 KB of partial rows in flight
constexpr int kMaxSources = 64;
constexpr int kW = 0;                                    // W_UV ring: 3 x 16 KB
constexpr int kB = kW + kWSlots * kWBlockBytes;          // B ring: 2 x 8 KB
constexpr int kP = kB + kBSlots * kLBlockBytes;          // partial-row ring: 4 chunks x 4 boxes x 8 KB
constexpr int kG = kP + kStages * kChunk * kLBlockBytes; // gate / value tile: 16 KB
constexpr int kWts = kG + kGateBytes;                    // weights: 64 tokens x S floats
constexpr int kBar = kWts + kTile * kMaxSources * 4;
constexpr int kNumBars = 2 * kStages + 2 * kWSlots + 2 * kBSlots + 2;
constexpr int kMisc = kBar + 8 * kNumBars;
constexpr int kAlloc = kMisc + 16 + 1024;
}  // namespace fz

__global__ void __launch_bounds__(32 * fz::kWarpsAll, 1) merge_value_kernel(const __grid_constant__ Params p) {
    using namespace fz;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + fz::kBar);
    uint64_t* full = bars;                          // [kStages] a chunk of partial rows landed (TMA bytes)
    uint64_t* empty = full + kStages;               // [kStages] the consumers are done with it (16 warps)
    uint64_t* w_full = empty + kStages;             // [kWSlots] W_UV rows landed (TMA bytes)
    uint64_t* w_empty = w_full + kWSlots;           // [kWSlots] their products finished (commit)
    uint64_t* b_ready = w_empty + kWSlots;          // [kBSlots] a B block written (16 warps)
    uint64_t* b_empty = b_ready + kBSlots;          // [kBSlots] its products finished (commit)
    uint64_t* gate_full = b_empty + kBSlots;        // the gate tile landed
    uint64_t* mma_done = gate_full + 1;             // every product finished (commit)
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + fz::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    float* wts = reinterpret_cast<float*>(smem + kWts);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, t0 = blockIdx.y * kTile;
    const int S = p.merge.sources;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, kConsumerWarps);
        }
        for (int i = 0; i < kWSlots; ++i) {
            mbar_init(w_full + i, 1);
            mbar_init(w_empty + i, 1);
        }
        for (int i = 0; i < kBSlots; ++i) {
            mbar_init(b_ready + i, kConsumerWarps);
            mbar_init(b_empty + i, 1);
        }
        mbar_init(gate_full, 1);
        mbar_init(mma_done, 1);
        misc[1] = 0;
        mbar_init_fence();
    }
    if (warp == kProducerWarp && lane == 0) {
        if (S > 0) prefetch_tensor_map(&p.latent);
        prefetch_tensor_map(&p.w_uv);
        prefetch_tensor_map(&p.gate);
        prefetch_tensor_map(&p.out);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(misc, kTile);
        tmem_relinquish();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = misc[0];

    bool ok = true;
    if (warp == kProducerWarp) {
        // the consumers' count and LSE loads go out before the stream of rows
        asm volatile("bar.sync 2, %0;" ::"r"(32 * (kConsumerWarps + 1)) : "memory");
        if (lane == 0) {
            mbar_arrive_expect_tx(gate_full, kGateBytes);
            tma_load_2d(sbase + fz::kG, &p.gate, h * kV, t0, gate_full);
            int n = 0;  // chunks of partial rows issued
            for (int kb = 0; kb < kBlocks && ok; ++kb) {
                for (int s0 = 0; s0 < S && ok; s0 += kChunk, ++n) {
                    const int stage = n % kStages, boxes = min(kChunk, S - s0);
                    if (n >= kStages)
                        ok &= mbar_wait_bounded(empty + stage, (n / kStages - 1) & 1, abort_flag, kWaitLimitNs);
                    mbar_arrive_expect_tx(full + stage, boxes * kLBlockBytes);
                    for (int k = 0; k < boxes; ++k)
                        tma_load_4d(sbase + kP + (stage * kChunk + k) * kLBlockBytes, &p.latent, kb * 64, h, t0,
                                    s0 + k, full + stage);
                }
            }
            if (!ok) *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            for (int kb = 0; kb < kWSlots; ++kb) {  // W_UV's first blocks
                mbar_arrive_expect_tx(w_full + kb, kWBlockBytes);
                tma_load_4d(sbase + fz::kW + kb * kWBlockBytes, &p.w_uv, 0, kb * 64, 0, h, w_full + kb);
            }
            constexpr uint32_t kIdesc = idesc_bf16(kV, kTile, 1, 0);
            const uint64_t d_b = smem_desc(sbase + kB, 1024, 1024, kSwizzle128B);
            for (int kb = 0; kb < kBlocks && ok; ++kb) {
                const int slot = kb % kWSlots, bslot = kb % kBSlots;
                ok &= mbar_wait_bounded(b_ready + bslot, (kb / kBSlots) & 1, abort_flag, kWaitLimitNs);
                ok &= mbar_wait_bounded(w_full + slot, (kb / kWSlots) & 1, abort_flag, kWaitLimitNs);
                if (!ok) break;
                tc_fence_after_sync();
                const uint64_t d_a = smem_desc(sbase + fz::kW + slot * kWBlockBytes, kWBlockBytes / 2, 1024,
                                               kSwizzle128B);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const uint32_t a_off = static_cast<uint32_t>(s4 * 16 * 128) >> 4;
                    const uint32_t b_off = static_cast<uint32_t>(bslot * kLBlockBytes + s4 * 32) >> 4;
                    mma_bf16(tmem, d_a + a_off, d_b + b_off, kIdesc, (kb | s4) != 0 ? 1u : 0u);
                }
                mma_commit(w_empty + slot);
                mma_commit(b_empty + bslot);
                if (kb + kWSlots < kBlocks) {  // refill the slot once these products have read it
                    ok &= mbar_wait_bounded(w_empty + slot, (kb / kWSlots) & 1, abort_flag, kWaitLimitNs);
                    mbar_arrive_expect_tx(w_full + slot, kWBlockBytes);
                    tma_load_4d(sbase + fz::kW + slot * kWBlockBytes, &p.w_uv, 0, (kb + kWSlots) * 64, 0, h,
                                w_full + slot);
                }
            }
            mma_commit(mma_done);
            if (!ok) *abort_flag = 1;
        }
        __syncwarp();
    } else {
        // the weights of the warp's rows warp, warp + 16, ... (one round of LSE loads)
        constexpr int kRows = kTile / kConsumerWarps;
        float l[kRows][2];
        int count[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {  // the counts and the LSEs in one round of loads
            const int tg = t0 + warp + kConsumerWarps * i;
            const bool in = tg < p.tokens;
            count[i] = in ? (p.lens == nullptr ? 1 : p.lens[tg]) : 0;
            load_row_lses(p.merge, in ? tg : 0, h, lane, l[i]);
        }
        asm volatile("bar.arrive 2, %0;" ::"r"(32 * (kConsumerWarps + 1)) : "memory");
#pragma unroll
        for (int i = 0; i < kRows; ++i)
            if (count[i] <= 0) empty_row_lses(l[i]);
#pragma unroll
        for (int i = 0; i < kRows; ++i) merge_weights(l[i], S, lane, wts + (warp + kConsumerWarps * i) * S);
        named_barrier(1, 32 * kConsumerWarps);

        // the epilogue's sigmoids while the first rows are in flight (the
        // gate tile is the producer's first copy)
        float sig[kTile * 4 / kConsumerWarps];
        ok &= mbar_wait_bounded(gate_full, 0, abort_flag, kWaitLimitNs);
        epilogue_sigmoids<kConsumerWarps>(sbase + fz::kG, warp, lane, sig);

        // then block by block, sources in order
        const int t = tid >> 3, u = tid & 7;
        const float* w_t = wts + t * S;
        int n = 0;
        for (int kb = 0; kb < kBlocks && ok; ++kb) {
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
            for (int s0 = 0; s0 < S; s0 += kChunk, ++n) {
                const int stage = n % kStages, boxes = min(kChunk, S - s0);
                ok &= mbar_wait_bounded(full + stage, (n / kStages) & 1, abort_flag, kWaitLimitNs);
                if (!ok) break;
                float w[kChunk];
                uint4 x[kChunk];
#pragma unroll
                for (int k = 0; k < kChunk; ++k)
                    if (k < boxes) {
                        w[k] = w_t[s0 + k];
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(x[k].x), "=r"(x[k].y), "=r"(x[k].z), "=r"(x[k].w)
                                     : "r"(sbase + kP + (stage * kChunk + k) * kLBlockBytes + t * 128 + u * 16));
                    }
#pragma unroll
                for (int k = 0; k < kChunk; ++k)
                    if (k < boxes && w[k] != 0.0f) add_weighted(acc, w[k], x[k]);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + stage);
            }
            if (!ok) break;
            const int bslot = kb % kBSlots;
            if (kb >= kBSlots) {  // the products of block kb - 2 have read this slot
                ok &= mbar_wait_bounded(b_empty + bslot, (kb / kBSlots - 1) & 1, abort_flag, kWaitLimitNs);
                if (!ok) break;
            }
            const uint4 bf = pack_bf16(acc);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             sbase + kB + bslot * kLBlockBytes + t * 128 + ((u ^ (t & 7)) << 4)),
                         "r"(bf.x), "r"(bf.y), "r"(bf.z), "r"(bf.w)
                         : "memory");
            fence_proxy_async_smem();  // the rows, written by threads, are read by the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(b_ready + bslot);
        }
        if (!ok) *abort_flag = 1;
        ok &= gate_epilogue<kConsumerWarps, true>(p, sbase + fz::kG, tmem, mma_done, gate_full, abort_flag, t0, warp,
                                                  lane, sig);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && ok && *abort_flag == 0) {
        tma_store_2d(&p.out, h * kV, t0, sbase + fz::kG);
        tma_store_wait_read();
    }
    if (!ok && lane == 0) atomicOr(p.error, SMLA_DEV_TIMEOUT);
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTile);
    }
}

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
    auto enc = smla::tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint32_t steps[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, steps,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace vgate

namespace vgate {

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// The tensor maps of W_UV, the gates and the output.
int encode_common(Params& p, const void* w_uv, const void* gate, int64_t gate_stride, void* out,
                  int64_t out_stride, int tokens, int heads) {
    const cuuint64_t T = static_cast<cuuint64_t>(tokens), H = static_cast<cuuint64_t>(heads);
    {
        // W_UV[h][j][v] as {64 values, 512 latents, 2 value halves, H}: one
        // box per 64-latent block lands as [value half][64 latents][64 values],
        // the two MN atoms of A
        const cuuint64_t dims[4] = {64, kJ, 2, H};
        const cuuint64_t strides[3] = {kV * 2, 64 * 2, static_cast<cuuint64_t>(kJ) * kV * 2};
        const cuuint32_t box[4] = {64, 64, 2, 1};
        if (!encode(&p.w_uv, w_uv, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return SMLA_EUNSUPPORTED;
    }
    const cuuint64_t dims[2] = {H * kV, T};
    const cuuint32_t box[2] = {kV, kTile};
    const cuuint64_t gs[1] = {static_cast<cuuint64_t>(gate_stride) * 2};
    const cuuint64_t os[1] = {static_cast<cuuint64_t>(out_stride) * 2};
    if (!encode(&p.gate, gate, 2, dims, gs, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return SMLA_EUNSUPPORTED;
    if (!encode(&p.out, out, 2, dims, os, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return SMLA_EUNSUPPORTED;
    p.tokens = tokens;
    p.heads = heads;
    return SMLA_OK;
}

// gate / out / W_UV checks shared by both entry points
bool bad_projection_args(int heads, const void* w_uv, const void* gate, int64_t gate_stride, const void* out,
                         int64_t out_stride) {
    return w_uv == nullptr || gate == nullptr || out == nullptr || !aligned16(w_uv) || !aligned16(gate) ||
           !aligned16(out) || gate_stride < static_cast<int64_t>(heads) * kV || gate_stride % 8 ||
           out_stride < static_cast<int64_t>(heads) * kV || out_stride % 8;
}

template <typename Kernel>
int launch(Kernel kernel, int threads, int smem_bytes, bool* configured, const Params& p, void* stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && p.error == nullptr) e = cudaErrorInvalidSymbol;  // the error word has no address here
    if (e == cudaSuccess && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e == cudaSuccess) configured[dev] = true;
    }
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(p.heads), static_cast<unsigned>((p.tokens + kTile - 1) / kTile), 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes;
        cfg.stream = static_cast<cudaStream_t>(stream);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, p);
    }
    if (e != cudaSuccess) {
        smla::note_cuda_error(static_cast<int>(e));
        return SMLA_ECUDA;
    }
    return SMLA_OK;
}

bool g_configured_value[64] = {}, g_configured_fused[64] = {};

}  // namespace vgate

extern "C" int smla_value_gate(const smla_value_shape* shape, const void* latent, const void* w_uv,
                               const void* gate, const int32_t* lens, void* out, void* stream) {
    using namespace vgate;
    if (shape == nullptr) return SMLA_EINVAL;
    const smla_value_shape& s = *shape;
    if (s.tokens < 0 || s.heads < 0) return SMLA_EINVAL;
    if (s.tokens == 0 || s.heads == 0) return SMLA_OK;
    if (s.tokens > 65535 * kTile || s.heads > 65535) return SMLA_EUNSUPPORTED;
    if (latent == nullptr || !aligned16(latent) ||
        bad_projection_args(s.heads, w_uv, gate, s.gate_stride_token, out, s.out_stride_token))
        return SMLA_EINVAL;
    // latent rows may sit in any order (token- or head-major) as long as each
    // row start is 16-byte aligned
    if (s.latent_stride_head <= 0 || s.latent_stride_token <= 0 || s.latent_stride_head >= (int64_t(1) << 36) ||
        s.latent_stride_token >= (int64_t(1) << 36) || s.latent_stride_head % 8 || s.latent_stride_token % 8)
        return SMLA_EINVAL;

    Params p;
    std::memset(&p, 0, sizeof(p));
    {
        const cuuint64_t dims[3] = {kJ, static_cast<cuuint64_t>(s.heads), static_cast<cuuint64_t>(s.tokens)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(s.latent_stride_head) * 2,
                                       static_cast<cuuint64_t>(s.latent_stride_token) * 2};
        const cuuint32_t box[3] = {64, 1, kTile};
        if (!encode(&p.latent, latent, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return SMLA_EUNSUPPORTED;
    }
    const int rc = encode_common(p, w_uv, gate, s.gate_stride_token, out, s.out_stride_token, s.tokens, s.heads);
    if (rc != SMLA_OK) return rc;
    p.lens = lens;
    p.error = smla::device_error_word();
    return launch(value_kernel, 32 * kWarps, kAlloc, g_configured_value, p, stream);
}

extern "C" int smla_merge_value(const smla_merge_value_shape* shape, const void* parts, const float* lses,
                                const int32_t* lens, const void* w_uv, const void* gate, void* out, void* stream) {
    using namespace vgate;
    if (shape == nullptr) return SMLA_EINVAL;
    const smla_merge_value_shape& s = *shape;
    if (s.sources < 0 || s.tokens < 0 || s.heads < 0) return SMLA_EINVAL;
    if (s.tokens == 0 || s.heads == 0) return SMLA_OK;
    if (s.tokens > 65535 * kTile || s.heads > 65535 || s.sources > fz::kMaxSources) return SMLA_EUNSUPPORTED;
    if (bad_projection_args(s.heads, w_uv, gate, s.gate_stride_token, out, s.out_stride_token)) return SMLA_EINVAL;
    if (s.sources > 0 && (parts == nullptr || lses == nullptr || !aligned16(parts))) return SMLA_EINVAL;
    if (s.part_stride_source < 0 || s.part_stride_token < 0 || s.part_stride_head < 0 || s.lse_stride_source < 0 ||
        s.lse_stride_token < 0 || s.part_stride_source % 8 || s.part_stride_token % 8 || s.part_stride_head % 8 ||
        (s.heads > 1 && s.sources > 0 && s.part_stride_head < kJ))
        return SMLA_EINVAL;

    Params p;
    std::memset(&p, 0, sizeof(p));
    const int rc = encode_common(p, w_uv, gate, s.gate_stride_token, out, s.out_stride_token, s.tokens, s.heads);
    if (rc != SMLA_OK) return rc;
    p.lens = lens;
    p.error = smla::device_error_word();
    p.merge = {static_cast<const __nv_bfloat16*>(parts), s.part_stride_source, s.part_stride_token,
               s.part_stride_head, lses, s.lse_stride_source, s.lse_stride_token, s.sources};
    if (s.sources > 0) {
        // the partial rows as {512 latents, H, T, S}: a box is 64 latents of
        // the tile's 64 tokens of one head and source, unswizzled
        const cuuint64_t dims[4] = {kJ, static_cast<cuuint64_t>(s.heads), static_cast<cuuint64_t>(s.tokens),
                                    static_cast<cuuint64_t>(s.sources)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.part_stride_head) * 2,
                                       static_cast<cuuint64_t>(s.part_stride_token) * 2,
                                       static_cast<cuuint64_t>(s.part_stride_source) * 2};
        const cuuint32_t box[4] = {64, 1, kTile, 1};
        if (!encode(&p.latent, parts, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return SMLA_EUNSUPPORTED;
    }
    return launch(merge_value_kernel, 32 * fz::kWarpsAll, fz::kAlloc, g_configured_fused, p, stream);
}
