// smla_merge_row.cuh -- the LSE merge of one (token, head) row over S partial
// sets, a warp per row and 16 latents per lane. Shared by the merge kernel and
// the fused merge + projection kernel, so that both produce the same bits.
//
// After the Kimi K3.1 `mla/dcp` page (DcpValue, merge): the weights are
// exp2(lse_s - M) / sum_s exp2(lse_s - M) over the sources whose LSE is
// finite, M their largest LSE; the row is the FP32 weighted sum, rounded to
// BF16 once by the caller.
#pragma once

#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <cstring>

namespace smla {

struct MergeInputs {
    const __nv_bfloat16* parts;
    int64_t part_stride_source, part_stride_token, part_stride_head;  // elements
    const float* lses;
    int64_t lse_stride_source, lse_stride_token;  // elements (heads contiguous)
    int32_t sources;
};

__device__ __forceinline__ uint4 load_nc(const void* ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// acc[0..7] += w * the eight BF16 values of v
__device__ __forceinline__ void add_weighted(float* acc, float w, const uint4& v) {
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 two;
        memcpy(&two, &words[e], 4);
        const float2 f = __bfloat1622float2(two);
        acc[2 * e] = fmaf(w, f.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(w, f.y, acc[2 * e + 1]);
    }
}

__device__ __forceinline__ uint4 pack_bf16(const float* x) {
    uint32_t words[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 two = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        memcpy(&words[e], &two, 4);
    }
    return make_uint4(words[0], words[1], words[2], words[3]);
}

// The weight of a source of LSE l in a row of largest finite LSE `top` and
// normalisation 1 / sum `inverse`.
__device__ __forceinline__ float merge_weight(float l, float top, float inverse) {
    return isfinite(l) ? exp2_approx(l - top) * inverse : 0.0f;
}

// The whole warp merges row (t, h): lane's latents 16 lane .. + 15 land in
// acc (zeros when nothing is merged). Returns the sum of the weights before
// normalisation (0 when the row is empty: not live, or no finite LSE) and the
// largest finite LSE in `top`. The weights' sum runs over lanes striding the
// sources and a butterfly, the weighted sum over the sources in order, kGroup
// sources' loads in flight at a time (the order of the arithmetic does not
// depend on kGroup).
template <int kGroup>
__device__ __forceinline__ float merge_row(const MergeInputs& m, int t, int h, int lane, bool live, float& top,
                                           float (&acc)[16]) {
    const float* lse_th = m.lses + static_cast<int64_t>(t) * m.lse_stride_token + h;
    top = -INFINITY;
    if (live)
        for (int s = lane; s < m.sources; s += 32) {
            const float l = lse_th[s * m.lse_stride_source];
            if (isfinite(l)) top = fmaxf(top, l);
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) top = fmaxf(top, __shfl_xor_sync(0xFFFFFFFFu, top, o));
    float total = 0.0f;
    if (top != -INFINITY)
        for (int s = lane; s < m.sources; s += 32) {
            const float l = lse_th[s * m.lse_stride_source];
            if (isfinite(l)) total += exp2_approx(l - top);
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, o);

#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
    if (total > 0.0f) {
        const float inverse = 1.0f / total;
        const __nv_bfloat16* base = m.parts + static_cast<int64_t>(t) * m.part_stride_token +
                                    static_cast<int64_t>(h) * m.part_stride_head + 16 * lane;
        int s = 0;
        for (; s + kGroup <= m.sources; s += kGroup) {
            float w[kGroup];
            uint4 v[2 * kGroup];
#pragma unroll
            for (int k = 0; k < kGroup; ++k) {
                const float l = lse_th[(s + k) * m.lse_stride_source];
                w[k] = merge_weight(l, top, inverse);
                if (w[k] != 0.0f) {  // the same for every lane: an empty source's row is never read
                    const __nv_bfloat16* src = base + (s + k) * m.part_stride_source;
                    v[2 * k] = load_nc(src);
                    v[2 * k + 1] = load_nc(src + 8);
                }
            }
#pragma unroll
            for (int k = 0; k < kGroup; ++k)
                if (w[k] != 0.0f) {
                    add_weighted(acc, w[k], v[2 * k]);
                    add_weighted(acc + 8, w[k], v[2 * k + 1]);
                }
        }
        for (; s < m.sources; ++s) {
            const float l = lse_th[s * m.lse_stride_source];
            const float w = merge_weight(l, top, inverse);
            if (w != 0.0f) {
                const __nv_bfloat16* src = base + s * m.part_stride_source;
                add_weighted(acc, w, load_nc(src));
                add_weighted(acc + 8, w, load_nc(src + 8));
            }
        }
    }
    return total;
}

}  // namespace smla

namespace smla {

// The LSEs of row (t, h) for sources lane and lane + 32 (-inf past S), for
// merge_weights; a row that is not live gets -inf for every source (apply
// with empty_row_lses once the count is known, so that the loads need not
// wait for it).
__device__ __forceinline__ void load_row_lses(const MergeInputs& m, int t, int h, int lane, float (&l)[2]) {
    const float* lse_th = m.lses + static_cast<int64_t>(t) * m.lse_stride_token + h;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int s = lane + 32 * k;
        l[k] = s < m.sources ? lse_th[s * m.lse_stride_source] : -INFINITY;
    }
}

__device__ __forceinline__ void empty_row_lses(float (&l)[2]) {
    l[0] = -INFINITY;
    l[1] = -INFINITY;
}

// The weights of a row over its S <= 64 sources, from the LSEs lane holds
// (load_row_lses), into w[0 .. S): the whole warp, the same operations in the
// same order as merge_row, so the same bits. Zeros when the row is empty.
__device__ __forceinline__ void merge_weights(const float (&l)[2], int sources, int lane, float* w) {
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
            if (isfinite(l[k])) total += exp2_approx(l[k] - top);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, o);
    const float inverse = total > 0.0f ? 1.0f / total : 0.0f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int s = lane + 32 * k;
        if (s < sources) w[s] = total > 0.0f ? merge_weight(l[k], top, inverse) : 0.0f;
    }
}

}  // namespace smla
