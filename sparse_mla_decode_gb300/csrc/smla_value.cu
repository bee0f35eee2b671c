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

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "smla.h"
#include "smla_ptx.cuh"

namespace smla {
void note_cuda_error(int code);
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
}  // namespace smla

namespace vgate {

using namespace smla;

constexpr int kTile = 64;   // tokens per CTA (N)
constexpr int kJ = 512;     // latents (K)
constexpr int kV = 128;     // values per head (M)
constexpr int kBlocks = kJ / 64;              // 64-latent blocks, one swizzle atom wide
constexpr int kThreads = 256;  // 8 warps: thread 0 issues TMA and MMA; all eight run the epilogue
constexpr int kWBlockBytes = 64 * kV * 2;     // 64 latent rows x 128 values: two 8 KB MN atoms
constexpr int kLBlockBytes = kTile * 128;     // 64 tokens x 64 latents
constexpr int kGateBytes = kTile * kV * 2;    // 64 tokens x 128 values, unswizzled
constexpr int kW = 0;
constexpr int kL = kW + kBlocks * kWBlockBytes;
constexpr int kG = kL + kBlocks * kLBlockBytes;
constexpr int kBar = kG + kGateBytes;
constexpr int kMisc = kBar + 8 * (kBlocks + 2);
constexpr int kAlloc = kMisc + 16 + 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct Params {
    CUtensorMap latent;  // {512 latents, H heads, T tokens} BF16, 128-byte swizzle, boxes of 64 x 1 x 64
    CUtensorMap w_uv;    // {64 values, 512 latents, 2 value halves, H heads} BF16, 128-byte swizzle, boxes of 64 x 64 x 2 x 1
    CUtensorMap gate;    // {H * 128, T} BF16, boxes of 128 x 64
    CUtensorMap out;     // {H * 128, T} BF16, boxes of 128 x 64
    const int32_t* lens; // [T] or null
    int32_t tokens, heads;
};

__device__ int32_t g_value_error;

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

__global__ void __launch_bounds__(kThreads, 1) value_gate_kernel(const __grid_constant__ Params p) {
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

    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31, so thread (w,
    // lane) owns value v = 32 (w % 4) + lane of the 32 tokens tb .. tb + 31,
    // tb = 32 (w / 4); bit t of `live` says whether token tb + t has keys
    const int v = 32 * (warp & 3) + lane;
    const int tb = 32 * (warp >> 2);
    const int t_lane = t0 + tb + lane;
    const uint32_t live =
        __ballot_sync(~0u, t_lane < p.tokens && (p.lens == nullptr || p.lens[t_lane] > 0));
    ok &= mbar_wait_bounded(mma_done, 0, abort_flag, kWaitLimitNs);
    ok &= mbar_wait_bounded(gate_full, 0, abort_flag, kWaitLimitNs);
    __syncwarp();
    tc_fence_after_sync();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    float acc[32];
    const uint32_t col = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + tb;
    tmem_load16x2(col, col + 16, acc);
    const uint32_t slot = sbase + kG + static_cast<uint32_t>(tb * kV + v) * 2;  // gate / value of token tb
    uint32_t bits[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) bits[t] = lds_u16(slot + t * kV * 2);
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        const float gate = __uint_as_float(bits[t] << 16);
        const float rounded = __bfloat162float(__float2bfloat16_rn(acc[t]));
        // sigmoid(g) = 1 / (1 + e^-g), in FP32 to a few ulp (the value is then
        // rounded to BF16, 2^-8 relative)
        const float y = rounded * rcp_approx(1.0f + __expf(-gate));
        bits[t] = (live >> t) & 1u ? __bfloat16_as_ushort(__float2bfloat16_rn(y)) : 0u;
    }
#pragma unroll
    for (int t = 0; t < 32; ++t) sts_u16(slot + t * kV * 2, bits[t]);
    fence_proxy_async_smem();  // the values, written by threads, are read by the TMA store
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        if (ok) {
            tma_store_2d(&p.out, h * kV, t0, sbase + kG);
            tma_store_wait_read();
        }
    }
    if (!ok && lane == 0) atomicOr(&g_value_error, SMLA_DEV_TIMEOUT);
    if (warp == 1) {
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

extern "C" int smla_value_gate(const smla_value_shape* shape, const void* latent, const void* w_uv,
                               const void* gate, const int32_t* lens, void* out, void* stream) {
    using namespace vgate;
    if (shape == nullptr) return SMLA_EINVAL;
    const smla_value_shape& s = *shape;
    if (s.tokens < 0 || s.heads < 0) return SMLA_EINVAL;
    if (s.tokens == 0 || s.heads == 0) return SMLA_OK;
    if (s.tokens > 65535 * kTile || s.heads > 65535) return SMLA_EUNSUPPORTED;
    if (latent == nullptr || w_uv == nullptr || gate == nullptr || out == nullptr) return SMLA_EINVAL;
    auto aligned16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    if (!aligned16(latent) || !aligned16(w_uv) || !aligned16(gate) || !aligned16(out)) return SMLA_EINVAL;
    // latent rows may sit in any order (token- or head-major) as long as each
    // row start is 16-byte aligned; output rows may not overlap
    if (s.latent_stride_head <= 0 || s.latent_stride_token <= 0 || s.latent_stride_head >= (int64_t(1) << 36) ||
        s.latent_stride_token >= (int64_t(1) << 36) || s.latent_stride_head % 8 || s.latent_stride_token % 8 ||
        s.gate_stride_token < s.heads * kV ||
        s.gate_stride_token % 8 || s.out_stride_token < s.heads * kV || s.out_stride_token % 8)
        return SMLA_EINVAL;

    Params p;
    std::memset(&p, 0, sizeof(p));
    const cuuint64_t T = static_cast<cuuint64_t>(s.tokens), H = static_cast<cuuint64_t>(s.heads);
    {
        const cuuint64_t dims[3] = {kJ, H, T};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(s.latent_stride_head) * 2,
                                       static_cast<cuuint64_t>(s.latent_stride_token) * 2};
        const cuuint32_t box[3] = {64, 1, kTile};
        if (!encode(&p.latent, latent, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return SMLA_EUNSUPPORTED;
    }
    {
        // W_UV[h][j][v] as {64 values, 512 latents, 2 value halves, H}: one
        // box per 64-latent block lands as [value half][64 latents][64 values],
        // the two MN atoms of A
        const cuuint64_t dims[4] = {64, kJ, 2, H};
        const cuuint64_t strides[3] = {kV * 2, 64 * 2, static_cast<cuuint64_t>(kJ) * kV * 2};
        const cuuint32_t box[4] = {64, 64, 2, 1};
        if (!encode(&p.w_uv, w_uv, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return SMLA_EUNSUPPORTED;
    }
    {
        const cuuint64_t dims[2] = {H * kV, T};
        const cuuint32_t box[2] = {kV, kTile};
        const cuuint64_t gs[1] = {static_cast<cuuint64_t>(s.gate_stride_token) * 2};
        const cuuint64_t os[1] = {static_cast<cuuint64_t>(s.out_stride_token) * 2};
        if (!encode(&p.gate, gate, 2, dims, gs, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return SMLA_EUNSUPPORTED;
        if (!encode(&p.out, out, 2, dims, os, box, CU_TENSOR_MAP_SWIZZLE_NONE)) return SMLA_EUNSUPPORTED;
    }
    p.lens = lens;
    p.tokens = s.tokens;
    p.heads = s.heads;

    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(value_gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
        if (e == cudaSuccess) configured[dev] = true;
    }
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(s.heads), static_cast<unsigned>((s.tokens + kTile - 1) / kTile), 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kAlloc;
        cfg.stream = static_cast<cudaStream_t>(stream);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, value_gate_kernel, p);
    }
    if (e != cudaSuccess) {
        smla::note_cuda_error(static_cast<int>(e));
        return SMLA_ECUDA;
    }
    return SMLA_OK;
}

extern "C" int smla_value_gate_error(int32_t* bits) {
    if (bits == nullptr) return SMLA_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    int32_t v = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, vgate::g_value_error, sizeof(v));
    const int32_t zero = 0;
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(vgate::g_value_error, &zero, sizeof(zero));
    if (e != cudaSuccess) {
        smla::note_cuda_error(static_cast<int>(e));
        return SMLA_ECUDA;
    }
    *bits = v;
    return SMLA_OK;
}
