// smla_pair.cuh -- the 128-head CTA-pair decode kernel's launch interface,
// shared by its own translation unit (smla_pair.cu) and the C ABI's host code
// (smla_decode.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace smla {

struct PairParams {
    // Tensor maps (64-byte aligned kernel parameters) of one CTA's half of the
    // Q tile: 64 heads of one token, 128-byte latent boxes (128B swizzle) and
    // the 64-byte rope box (64B swizzle).
    CUtensorMap q_latent;
    CUtensorMap q_rope;
    // Row gathers of each pool (tile::gather4, boxes of 128 bytes x 1 row,
    // 128B swizzle), used when peer_tma is set.
    CUtensorMap kv0;
    CUtensorMap kv1;
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
    int32_t peer_tma;  // both pools have row-gather maps
    int32_t* error;    // the library's device error word
};

// Keys of one chunk of the pair (128 per CTA), heads per pair.
constexpr int kPairChunk = 256;
constexpr int kPairHeads = 128;
constexpr int kPairThreads = 512;
constexpr int kPairTmemColumns = 512;

// Dynamic shared memory of one CTA for rows of `head_dim` bytes (576 or 512).
int pair_smem_bytes(int head_dim);

// Opts the kernel into its shared memory (once per device) and launches
// `groups` head groups of 128 heads x `tokens` tokens as clusters of two CTAs,
// with programmatic stream serialization when `dependent` is set.
cudaError_t launch_pair(const PairParams& p, int head_dim, int groups, int tokens, bool dependent,
                        cudaStream_t stream);

// CTA pairs of the kernel that the current device holds at once (occupancy
// query), 0 when the query fails.
int pair_resident_clusters(int head_dim);

}  // namespace smla
