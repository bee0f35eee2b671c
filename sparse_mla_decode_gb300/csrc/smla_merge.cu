// LSE merge of partial (out, lse) sets on one GPU.
//
// What it computes follows the Kimi K3.1 `mla/dcp` page, DcpValue (class
// docstring and merge): each source s of a (token, head) weighs
// exp2(lse_s - max) / sum over the sources, in FP32; a source whose LSE is not
// finite (NaN, -inf, +inf), or every source of a token of count <= 0, weighs
// nothing; the sources' BF16 rows are summed with these weights in FP32 and
// rounded to BF16 once. A (token, head) with no weight left gets +0.0 and LSE
// -inf. The merged LSE (base 2) is max + log2(sum of weights).
//
// The pass streams every source row once and writes the merged row once, so
// it is bound by HBM bandwidth: one warp per (token, head) row, each lane 16
// consecutive latents (two 16-byte loads per source, four sources in flight),
// one resident wave of CTAs over a grid-stride loop of rows.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "smla.h"
#include "smla_merge_row.cuh"

namespace smla {
void note_cuda_error(int code);  // the thread's last CUDA error, for smla_last_cuda_error
}

namespace lse_merge {

constexpr int kLatent = 512;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kGroup = 4;  // sources whose row loads are in flight together
constexpr int kMaxPipelinedSources = 64;  // up to here a warp loads its next row's LSEs ahead

struct Params {
    smla::MergeInputs merge;  // the partial sets and their base-2 LSEs
    const int32_t* lens;      // [tokens] or null
    __nv_bfloat16* out;
    int64_t out_stride_token, out_stride_head;  // elements
    float* lse_out;                             // or null
    int64_t lse_out_stride_token;
    int32_t tokens, heads;
};

__global__ void __launch_bounds__(kThreads) lse_merge_kernel(const __grid_constant__ Params p) {
    __shared__ float wts[kWarps][kMaxPipelinedSources];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t rows = static_cast<int64_t>(p.tokens) * p.heads;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    const int64_t step = static_cast<int64_t>(gridDim.x) * kWarps;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the partial sets are read only after this point

    if (p.merge.sources <= kMaxPipelinedSources) {
        // The next row's counts and LSEs load while this row's partial rows
        // are in flight, so that a row costs one round trip to memory. The
        // weights come from the same operations as merge_row's.
        float* w_row = wts[warp];
        float l_next[2];
        int count_next = 0;
        auto load_row = [&](int64_t row, float (&l)[2], int& count) {
            const int t = static_cast<int>(row / p.heads), h = static_cast<int>(row % p.heads);
            count = p.lens == nullptr ? 1 : p.lens[t];
            smla::load_row_lses(p.merge, t, h, lane, l);
        };
        if (first < rows) load_row(first, l_next, count_next);
        for (int64_t row = first; row < rows; row += step) {
            const int t = static_cast<int>(row / p.heads), h = static_cast<int>(row % p.heads);
            float l[2] = {l_next[0], l_next[1]};
            if (count_next <= 0) smla::empty_row_lses(l);
            if (row + step < rows) load_row(row + step, l_next, count_next);
            smla::merge_weights(l, p.merge.sources, lane, w_row);
            __syncwarp();
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
            const __nv_bfloat16* base = p.merge.parts + static_cast<int64_t>(t) * p.merge.part_stride_token +
                                        static_cast<int64_t>(h) * p.merge.part_stride_head + 16 * lane;
            int s = 0;
            for (; s + kGroup <= p.merge.sources; s += kGroup) {
                float w[kGroup];
                uint4 v[2 * kGroup];
#pragma unroll
                for (int k = 0; k < kGroup; ++k) {
                    w[k] = w_row[s + k];
                    if (w[k] != 0.0f) {  // the same for every lane: an empty source's row is never read
                        const __nv_bfloat16* src = base + (s + k) * p.merge.part_stride_source;
                        v[2 * k] = smla::load_nc(src);
                        v[2 * k + 1] = smla::load_nc(src + 8);
                    }
                }
#pragma unroll
                for (int k = 0; k < kGroup; ++k)
                    if (w[k] != 0.0f) {
                        smla::add_weighted(acc, w[k], v[2 * k]);
                        smla::add_weighted(acc + 8, w[k], v[2 * k + 1]);
                    }
            }
            for (; s < p.merge.sources; ++s) {
                const float w = w_row[s];
                if (w != 0.0f) {
                    const __nv_bfloat16* src = base + s * p.merge.part_stride_source;
                    smla::add_weighted(acc, w, smla::load_nc(src));
                    smla::add_weighted(acc + 8, w, smla::load_nc(src + 8));
                }
            }
            __nv_bfloat16* dst = p.out + static_cast<int64_t>(t) * p.out_stride_token +
                                 static_cast<int64_t>(h) * p.out_stride_head + 16 * lane;
            reinterpret_cast<uint4*>(dst)[0] = smla::pack_bf16(acc);
            reinterpret_cast<uint4*>(dst)[1] = smla::pack_bf16(acc + 8);
            if (p.lse_out != nullptr) {
                // the row's largest finite LSE and the weights' sum, again by
                // merge_row's operations (cheap next to the row's bytes)
                float top = -INFINITY;
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (isfinite(l[k])) top = fmaxf(top, l[k]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) top = fmaxf(top, __shfl_xor_sync(0xFFFFFFFFu, top, o));
                float total = 0.0f;
                if (top != -INFINITY)
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        if (isfinite(l[k])) total += smla::exp2_approx(l[k] - top);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
                if (lane == 0)
                    p.lse_out[static_cast<int64_t>(t) * p.lse_out_stride_token + h] =
                        total > 0.0f ? top + log2f(total) : -INFINITY;
            }
            __syncwarp();  // w_row is rewritten for the next row
        }
    } else {
        for (int64_t row = first; row < rows; row += step) {
            const int t = static_cast<int>(row / p.heads), h = static_cast<int>(row % p.heads);
            const bool live = p.lens == nullptr || p.lens[t] > 0;
            float top, acc[16];
            const float total = smla::merge_row<kGroup>(p.merge, t, h, lane, live, top, acc);
            __nv_bfloat16* dst = p.out + static_cast<int64_t>(t) * p.out_stride_token +
                                 static_cast<int64_t>(h) * p.out_stride_head + 16 * lane;
            reinterpret_cast<uint4*>(dst)[0] = smla::pack_bf16(acc);
            reinterpret_cast<uint4*>(dst)[1] = smla::pack_bf16(acc + 8);
            if (p.lse_out != nullptr && lane == 0)
                p.lse_out[static_cast<int64_t>(t) * p.lse_out_stride_token + h] =
                    total > 0.0f ? top + log2f(total) : -INFINITY;
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

// CTAs of the merge kernel one SM holds at once (occupancy query at its
// launch shape), cached per device; -1 when the query fails.
int resident_merge_ctas() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && cache[dev] > 0) return cache[dev];
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, lse_merge_kernel, kThreads, 0) != cudaSuccess)
        return -1;
    if (dev < 64) cache[dev] = blocks;
    return blocks;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace lse_merge

using namespace lse_merge;

extern "C" int smla_merge(const smla_merge_shape* shape, const void* parts, const float* lses,
                          const int32_t* lens, void* out, float* lse_out, void* stream) {
    if (shape == nullptr) return SMLA_EINVAL;
    const smla_merge_shape& s = *shape;
    if (s.sources < 0 || s.tokens < 0 || s.heads < 0) return SMLA_EINVAL;
    if (s.tokens == 0 || s.heads == 0) return SMLA_OK;
    if (out == nullptr || (s.sources > 0 && (parts == nullptr || lses == nullptr))) return SMLA_EINVAL;
    // 16-byte loads and stores of each row
    if (!aligned16(out) || (s.sources > 0 && !aligned16(parts))) return SMLA_EINVAL;
    if (s.part_stride_source % 8 || s.part_stride_token % 8 || s.part_stride_head % 8 || s.out_stride_token % 8 ||
        s.out_stride_head % 8)
        return SMLA_EINVAL;
    if (s.part_stride_source < 0 || s.part_stride_token < 0 || s.part_stride_head < 0 || s.lse_stride_source < 0 ||
        s.lse_stride_token < 0 || s.out_stride_token < 0 || s.out_stride_head < 0 || s.lse_out_stride_token < 0)
        return SMLA_EINVAL;
    if (s.heads > 1 && (s.out_stride_head < kLatent || (s.sources > 0 && s.part_stride_head < kLatent)))
        return SMLA_EINVAL;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.merge = {static_cast<const __nv_bfloat16*>(parts), s.part_stride_source, s.part_stride_token,
               s.part_stride_head, lses, s.lse_stride_source, s.lse_stride_token, s.sources};
    p.lens = lens;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.out_stride_token = s.out_stride_token;
    p.out_stride_head = s.out_stride_head;
    p.lse_out = lse_out;
    p.lse_out_stride_token = s.lse_out_stride_token;
    p.tokens = s.tokens;
    p.heads = s.heads;

    const int sms = device_sms();
    const int per_sm = resident_merge_ctas();
    if (sms <= 0 || per_sm <= 0) return SMLA_ECUDA;
    // One resident wave (the CTAs an SM holds at the kernel's registers, from
    // the occupancy query) with a grid-stride loop, so that each warp has rows
    // after the current one and can load their LSEs ahead.
    const int64_t rows = static_cast<int64_t>(s.tokens) * s.heads;
    const int64_t want = (rows + kWarps - 1) / kWarps;
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(want < cap ? want : cap), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, lse_merge_kernel, p);
    if (e != cudaSuccess) {
        smla::note_cuda_error(static_cast<int>(e));
        return SMLA_ECUDA;
    }
    return SMLA_OK;
}
