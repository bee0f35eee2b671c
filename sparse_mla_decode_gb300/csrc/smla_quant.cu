// MXFP4 quantisation of the indexer query, the step before sparse MLA decode
// (its top-k rows become the decode's index lists).
//
// What it computes follows the Kimi K3.1 `dsa_indexer_mxfp4` page
// (mxfp4_q_quant, _mxfp4_q_quant_kernel, _mxfp4_quant): each head's 128 query
// values, taken as FP32, form 4 blocks of 32; a block's UE8M0 scale is 2^e
// with e = ceil(log2(max(amax, 6 * 2^-126) / 6)) clamped to [-127, 127] and
// stored as e + 127 (block b in byte b of the head's int32); the values
// divided by 2^e are rounded to FP4 E2M1 (nearest, ties to even, saturating
// at 6) and packed two per byte, the even element in the low nibble; the head
// weights are multiplied by weight_scale; heads [H, P) of the padded outputs
// are zero. The ceiling of log2 is taken exactly on the FP32 quotient.
//
// One warp per 16 (BF16) or 8 (FP32) (token, padded head) rows over 4 steps:
// a head is 8 lanes of 16 BF16 values (or 16 lanes of 8 FP32 values), a
// 32-value block 2 (or 4) lanes, maxima and scale bytes by shuffles; all
// steps' loads (and head weights) are issued first and kept as raw words, so
// that enough bytes are in flight to stream from HBM; a head's 64 packed
// bytes leave as coalesced 8- (or 4-) byte stores.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "smla.h"

namespace smla {
void note_cuda_error(int code);
}

namespace mxfp4 {

constexpr int kHeadDim = 128;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

struct Params {
    const void* q;
    int64_t q_stride_token, q_stride_head;  // elements
    const float* w;
    int64_t w_stride_token;
    uint8_t* packed;
    int64_t packed_stride_token;  // bytes
    int32_t* scale;
    int64_t scale_stride_token;  // int32 elements
    float* w_out;
    int64_t w_out_stride_token;
    float weight_scale;
    int32_t tokens, heads, padded, q_is_f32;
};

// Eight FP32 values -> four bytes of E2M1 codes (value 2j in the low nibble of
// byte j, value 2j + 1 in its high nibble).
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// 16 bytes read once: not kept in L1, fetched from DRAM in 256-byte lines (a
// head's row is 256 or 512 contiguous bytes).
__device__ __forceinline__ uint4 load_stream(const uint4* ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

// The values one lane holds: 16 BF16 or 8 FP32 values, 32 raw bytes either
// way, kept as words until they are used.
template <bool kF32>
struct LaneValues {
    static constexpr int kCount = kF32 ? 8 : 16;
    uint4 w[2];
    __device__ __forceinline__ void load(const void* base, int64_t at) {
        const uint4* src = kF32 ? reinterpret_cast<const uint4*>(static_cast<const float*>(base) + at)
                                : reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + at);
        w[0] = load_stream(src);
        w[1] = load_stream(src + 1);
    }
    __device__ __forceinline__ void zero() { w[0] = w[1] = make_uint4(0u, 0u, 0u, 0u); }
    // max |value| as FP32 bits (finite values: the bit patterns of |x| order
    // like the values)
    __device__ __forceinline__ uint32_t abs_max_bits() const {
        const uint32_t u[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
        if constexpr (kF32) {
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = max(m, u[i] & 0x7FFFFFFFu);
            return m;
        } else {  // per-halfword maxima of the BF16 patterns, then the larger half
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = __vmaxu2(m, u[i] & 0x7FFF7FFFu);
            return max(m << 16, m & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ void values(float* x) const {
        const uint32_t u[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
        if constexpr (kF32) {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(u[i]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {  // BF16 -> FP32: the upper half of the word
                x[2 * e] = __uint_as_float(u[e] << 16);
                x[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
            }
        }
    }
};

// Rows (token, padded head) per CTA: kWarps warps x kSteps steps x the heads
// a warp holds per step.
template <bool kF32>
constexpr int rows_per_cta() {
    return kWarps * 4 * (32 / (128 / LaneValues<kF32>::kCount));
}

template <bool kF32>
__global__ void __launch_bounds__(kThreads) mxfp4_q_quant_kernel(const __grid_constant__ Params p) {
    using V = LaneValues<kF32>;
    constexpr int kVals = V::kCount;                     // values per lane
    constexpr int kLanesPerHead = kHeadDim / kVals;      // 8 (BF16) or 16 (FP32)
    constexpr int kHeadsPerStep = 32 / kLanesPerHead;    // 4 or 2
    constexpr int kLanesPerBlock = 32 / kVals;           // a 32-value block: 2 or 4 lanes
    constexpr int kSteps = 4;
    constexpr int kRowsPerWarp = kHeadsPerStep * kSteps;
    const int lane = threadIdx.x & 31;
    const int slot = lane / kLanesPerHead, sub = lane % kLanesPerHead;
    // rows = tokens * padded < 2^31 (checked on the host): 32-bit indices
    const uint32_t rows = static_cast<uint32_t>(p.tokens) * static_cast<uint32_t>(p.padded);
    const uint32_t first = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRowsPerWarp;
    const uint32_t padded = static_cast<uint32_t>(p.padded);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // every step's loads first (kSteps x 32 bytes per lane in flight)
    V x[kSteps];
    float wt[kSteps];  // the head weight of each step (first lane of the head)
    int tok[kSteps], head[kSteps];
    {  // (token, head) of step 0 by one division; later steps add kHeadsPerStep heads
        const uint32_t row = first + slot;
        tok[0] = static_cast<int>(row / padded);
        head[0] = static_cast<int>(row - static_cast<uint32_t>(tok[0]) * padded);
#pragma unroll
        for (int k = 1; k < kSteps; ++k) {
            int t_ = tok[k - 1], h_ = head[k - 1] + kHeadsPerStep;
            while (h_ >= p.padded) h_ -= p.padded, ++t_;
            tok[k] = t_;
            head[k] = h_;
        }
    }
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
        const uint32_t row = first + kHeadsPerStep * k + slot;
        const bool live = row < rows && head[k] < p.heads;
        const int t = live ? tok[k] : 0, h = live ? head[k] : 0;
        wt[k] = (live && sub == 0) ? p.w[static_cast<int64_t>(t) * p.w_stride_token + h] : 0.0f;
        if (live)
            x[k].load(p.q, static_cast<int64_t>(t) * p.q_stride_token + static_cast<int64_t>(h) * p.q_stride_head +
                               kVals * sub);
        else
            x[k].zero();
    }
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
        // every lane takes part in the shuffles; rows past the end store nothing
        const bool in = first + kHeadsPerStep * k + slot < rows;
        const int t = in ? tok[k] : 0, h = in ? head[k] : 0;
        const bool live = h < p.heads;
        // block maxima of |x|
        uint32_t amax = x[k].abs_max_bits();
#pragma unroll
        for (int o = 1; o < kLanesPerBlock; o <<= 1) amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        // e = ceil(log2(RN(a / 6))) for a = max(amax, 6 * 2^-126) = m * 2^E,
        // m in [1, 2): RN(a / 6) is a power of two only for m = 1.5 (then
        // 2^(E - 2)); otherwise its exponent is E - 2 for m > 1.5 and E - 3
        // below, and the ceiling adds one. So e = E - 1 for m > 1.5, else
        // E - 2 (no division; E <= 127 and E >= -124 keep e in [-126, 126]).
        const uint32_t a = max(amax, 0x01C00000u);  // 6 * 2^-126 = 1.5 * 2^-124
        const int E = static_cast<int>(a >> 23) - 127;
        const int e = (a & 0x7FFFFFu) > 0x400000u ? E - 1 : E - 2;
        // x / 2^e as x * 2^-e: the factor is a normal power of two, so the
        // product is the correctly rounded quotient
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
        float v[kVals];
        x[k].values(v);
#pragma unroll
        for (int i = 0; i < kVals; ++i) v[i] = __fmul_rn(v[i], inv);
        uint8_t* packed = p.packed + static_cast<int64_t>(t) * p.packed_stride_token + h * (kHeadDim / 2);
        if constexpr (kVals == 16) {
            const uint2 codes = make_uint2(e2m1x8(v), e2m1x8(v + 8));
            if (in) reinterpret_cast<uint2*>(packed)[sub] = live ? codes : make_uint2(0u, 0u);
        } else {
            const uint32_t codes = e2m1x8(v);
            if (in) reinterpret_cast<uint32_t*>(packed)[sub] = live ? codes : 0u;
        }
        // the head's four scale bytes: block b's byte in byte b, OR-reduced
        // over the head's lanes (every lane of a block holds its e)
        uint32_t word = static_cast<uint32_t>(e + 127) << (8 * (sub / kLanesPerBlock));
#pragma unroll
        for (int o = kLanesPerBlock; o < kLanesPerHead; o <<= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, o);
        if (in && sub == 0) {
            p.scale[static_cast<int64_t>(t) * p.scale_stride_token + h] = live ? static_cast<int32_t>(word) : 0;
            p.w_out[static_cast<int64_t>(t) * p.w_out_stride_token + h] = live ? __fmul_rn(wt[k], p.weight_scale) : 0.0f;
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

bool aligned(const void* ptr, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(ptr) & (bytes - 1)) == 0; }

}  // namespace mxfp4

extern "C" int smla_mxfp4_q_quant(const smla_mxfp4_shape* shape, const void* q, const float* weights,
                                  float weight_scale, void* q_packed, int32_t* q_scale, float* w_out,
                                  void* stream) {
    using namespace mxfp4;
    if (shape == nullptr) return SMLA_EINVAL;
    const smla_mxfp4_shape& s = *shape;
    if (s.tokens < 0 || s.heads < 0 || s.padded_heads < s.heads) return SMLA_EINVAL;
    if (s.head_dim != kHeadDim) return SMLA_EUNSUPPORTED;
    if (s.q_dtype != SMLA_DTYPE_BF16 && s.q_dtype != SMLA_DTYPE_F32) return SMLA_EUNSUPPORTED;
    if (s.tokens == 0 || s.padded_heads == 0) return SMLA_OK;
    if (q_packed == nullptr || q_scale == nullptr || w_out == nullptr) return SMLA_EINVAL;
    if (s.heads > 0 && (q == nullptr || weights == nullptr)) return SMLA_EINVAL;
    // two 16-byte loads per lane (16 BF16 or 8 FP32 values); 8-byte packed stores
    if ((s.heads > 0 && !aligned(q, 16)) || !aligned(q_packed, 8)) return SMLA_EINVAL;
    if (s.q_stride_token % 8 || s.q_stride_head % 8 || s.packed_stride_token % 8) return SMLA_EINVAL;
    if (s.q_stride_token < 0 || s.q_stride_head < 0 || s.w_stride_token < 0 || s.packed_stride_token < 0 ||
        s.scale_stride_token < 0 || s.w_out_stride_token < 0)
        return SMLA_EINVAL;
    if (s.heads > 1 && s.q_stride_head < kHeadDim) return SMLA_EINVAL;

    Params p;
    std::memset(&p, 0, sizeof(p));
    p.q = q;
    p.q_stride_token = s.q_stride_token;
    p.q_stride_head = s.q_stride_head;
    p.w = weights;
    p.w_stride_token = s.w_stride_token;
    p.packed = static_cast<uint8_t*>(q_packed);
    p.packed_stride_token = s.packed_stride_token;
    p.scale = q_scale;
    p.scale_stride_token = s.scale_stride_token;
    p.w_out = w_out;
    p.w_out_stride_token = s.w_out_stride_token;
    p.weight_scale = weight_scale;
    p.tokens = s.tokens;
    p.heads = s.heads;
    p.padded = s.padded_heads;
    p.q_is_f32 = s.q_dtype == SMLA_DTYPE_F32;

    const int64_t rows = static_cast<int64_t>(s.tokens) * s.padded_heads;
    if (rows + 2 * rows_per_cta<false>() >= (int64_t{1} << 31)) return SMLA_EUNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    const int64_t per_cta = p.q_is_f32 ? rows_per_cta<true>() : rows_per_cta<false>();
    cfg.gridDim = dim3(static_cast<unsigned>((rows + per_cta - 1) / per_cta), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = p.q_is_f32 ? cudaLaunchKernelEx(&cfg, mxfp4_q_quant_kernel<true>, p)
                                     : cudaLaunchKernelEx(&cfg, mxfp4_q_quant_kernel<false>, p);
    if (e != cudaSuccess) {
        smla::note_cuda_error(static_cast<int>(e));
        return SMLA_ECUDA;
    }
    return SMLA_OK;
}
