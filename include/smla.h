/*
 * smla.h -- C ABI of the sparse MLA decode library (libsmla.so, sm_103a).
 *
 * The operation (DeepSeek-V4.1 page "sparse_mla_cute", module docstring, "The
 * problem" and "What this module computes"; Kimi K3.1 page "attn_sparse",
 * module docstring and its "Precision" paragraph):
 *
 *   for each token t and head h, over the token's active columns c
 *   (c < clamp(lens[t], 0, width) and indices[t, c] >= 0):
 *     s_c  = bmm1_scale * q[t, h, :] . kv_c[:]          (all head_dim bytes)
 *     out[t, h, j] = bmm2_scale * k_scale * sum_c p_c kv_c[j] / den,  j < 512
 *     p_c  = exp(s_c - m),  den = sum_c p_c + exp(sink_h - m),  m = max(s, sink)
 *     lse[t, h] = log2(den) + m * log2(e)               (base 2)
 *   where kv_c is row indices[t, c] of pool 0 when c < pool_split and of pool 1
 *   otherwise (a single pool serves every column when num_pools == 1).
 *   A token without active columns gets out = +0.0 and lse = -inf.
 *
 * Datapath: E4M3 q and KV, FP32 logits, a base-2 online softmax over chunks of
 * the plan's `chunk` columns (128, or 96 where the planner takes three stages),
 * P rounded to E4M3 (RN, satfinite) at 448 of the running maximum
 * of the split, FP32 sums of the unrounded P, FP32 accumulation, an FP32 merge
 * of the key splits over distributed shared memory, one BF16 rounding.
 *
 * All functions are thread-safe. Device buffers are owned by the caller; the
 * library allocates no device memory.
 */
#ifndef SMLA_H
#define SMLA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define SMLA_OK 0
#define SMLA_EINVAL (-1)       /* null pointer, bad shape, stride or alignment */
#define SMLA_EUNSUPPORTED (-2) /* a shape outside what the kernels handle */
#define SMLA_ECUDA (-3)        /* a CUDA runtime call failed (see smla_last_cuda_error) */
#define SMLA_EDEVICE (-4)      /* the device reported an error (smla_device_error) */

/* Device error bits, set by the kernels in the library's device error word.
 *
 * The error word: one 32-bit word per device, shared by every kernel of this
 * library on that device (decode, merge-and-project, project-and-gate) and by
 * every stream and host thread that launches them. Kernels OR bits into it;
 * nothing clears it but a read (smla_read_device_error, smla_device_error),
 * which takes every bit present at that moment and leaves zero. So bits cannot
 * be attributed to one stream when other streams run the library's kernels at
 * the same time: a stream-ordered read sees every bit that work queued before
 * it on its stream set, plus whatever concurrent work on other streams had set
 * when the read ran, and two reads never report the same bit twice. */
#define SMLA_DEV_INDEX_RANGE 1 /* an index >= pool rows (that column was masked) */
#define SMLA_DEV_TIMEOUT 2     /* a bounded wait gave up; outputs are invalid */

/* One KV pool: `rows` rows of `row_bytes` E4M3 bytes, rows contiguous, in
 * device memory; data 16-byte aligned. row_bytes must equal shape.head_dim. */
typedef struct smla_pool {
    const void* data;
    int64_t rows;
    int32_t row_bytes;
    int32_t reserved; /* 0 */
} smla_pool;

/* Sizes and strides of one call.
 *   tokens T >= 0, heads H (a positive multiple of 16, <= 1024), width W >= 0,
 *   head_dim D in {512, 576} (576 = 512 latent + 64 rope; V is the first 512),
 *   num_pools in {1, 2}, pool_split in [0, W] (used when num_pools == 2).
 *   q element (t, h, d) at q + t*q_stride_token + h*q_stride_head + d (bytes;
 *   both strides multiples of 16, q 16-byte aligned).
 *   indices element (t, c) at indices[t*idx_stride_token + c] (int32 elements,
 *   idx_stride_token >= W).
 *   out element (t, h, j) at out[t*out_stride_token + h*out_stride_head + j]
 *   (bf16 elements; strides even, out 4-byte aligned).
 *   lse element (t, h) at lse[t*lse_stride_token + h] (float elements). */
typedef struct smla_shape {
    int32_t tokens, heads, width, head_dim;
    int32_t num_pools, pool_split;
    int64_t q_stride_token, q_stride_head;
    int64_t idx_stride_token;
    int64_t out_stride_token, out_stride_head;
    int64_t lse_stride_token;
} smla_shape;

/* The launch the library picks for a shape (returned for tests, sweeps and
 * the emulating oracle, which replays `splits` and `chunk`). */
typedef struct smla_plan {
    int32_t head_tile;        /* heads per CTA (16, 32 or 64) */
    int32_t head_groups;      /* heads / head_tile */
    int32_t chunk;            /* columns per chunk: 128 in two stages, or 96 in
                                 three for a 32/64-head tile that streams 8 or
                                 more chunks of 128 unpaired, 16 or more paired
                                 (64-head tiles) */
    int32_t chunks;           /* ceil(width / chunk) */
    int32_t splits;           /* CTAs per (token, head group) = cluster size */
    int32_t chunks_per_split; /* ceil(chunks / splits); a token of c active-count
                                 chunks gives each split ceil(c / splits) */
    int32_t ctas;             /* tokens * head_groups * splits */
    int32_t threads;          /* threads per CTA */
    int32_t smem_bytes;       /* dynamic shared memory per CTA */
    int32_t tmem_columns;     /* tensor-memory columns allocated per CTA */
    int32_t num_sms;          /* SM count the plan was made for */
    int32_t resident_ctas;    /* CTAs in clusters of pair * splits the GPU holds
                                 at once (occupancy query; with an explicit
                                 num_sms: c * floor(num_sms / c), c the cluster) */
    int32_t pair;             /* head groups sharing each gathered chunk: 2 when
                                 one pool, an even number of head groups and at
                                 least 4 chunks per CTA (the pair's CTAs each
                                 gather half of a chunk's rows into both), else 1 */
} smla_plan;

/* Fills *plan for `shape` on a GPU of `num_sms` SMs (num_sms <= 0: the current
 * device, whose SM count and cluster occupancy are queried; needs a CUDA
 * device). Pure host logic otherwise.
 * The head tile (16, 32 or 64 heads per CTA, dividing `heads`) and the split
 * count are chosen together: among the choices whose tokens * head_groups *
 * splits CTAs are all resident at once, the least estimated time (a fixed cost
 * per CTA that grows with the tile, plus the chunks per CTA at a rate that
 * grows with the CTAs sharing the HBM); when no choice fits one wave, the
 * widest tile without splits.
 * Environment overrides (for measurement): SMLA_HEAD_TILE=16|32|64 forces the
 * tile when it divides `heads`; SMLA_PAIR=0 / 1 turns pairing off / on wherever
 * the shape allows it; SMLA_SPLITS=n (n > 0) forces the split count,
 * clamped to [1, min(chunks, 16 / pair)], with the widest tile unless one is
 * forced; SMLA_CHUNK=96|128 forces the chunk (96 only on 32/64-head tiles).
 * Returns SMLA_OK, SMLA_EINVAL, SMLA_EUNSUPPORTED or SMLA_ECUDA. */
int smla_plan_for(const smla_shape* shape, int num_sms, smla_plan* plan);

/* Sparse MLA decode (the operation above), asynchronous on `stream`.
 *   shape     host pointer, see smla_shape.
 *   q         device, E4M3 [T, H, D] bytes.
 *   kv_pools  host array of shape->num_pools descriptors (data in device memory).
 *   indices   device, int32 [T, >= W], -1 marks a hole (may be NULL when W == 0).
 *   lens      device, int32 [T], active count per token, clamped to [0, W].
 *   sinks     device, float [H] per-head sink in score units, or NULL.
 *   bmm1_scale  multiplies the q.kv dot products (fold q and k scales in here).
 *   bmm2_scale, k_scale  multiply the output.
 *   out       device, BF16 [T, H, 512].
 *   lse       device, float [T, H] base-2 log-sum-exp, or NULL.
 *   stream    a cudaStream_t (NULL: the legacy default stream).
 * Launched with programmatic dependent launch: the kernel reads its inputs only
 * after the previous kernel in the stream has completed (SMLA_PDL=0 in the
 * environment launches without it, for measurement).
 * Captureable in a CUDA graph (no allocation, no synchronisation).
 * Errors: SMLA_EINVAL / SMLA_EUNSUPPORTED before anything is launched,
 * SMLA_ECUDA when the launch fails. Device-side conditions (an index beyond its
 * pool, a wait that timed out) are recorded in the device error word. */
int smla_decode(const smla_shape* shape, const void* q, const smla_pool* kv_pools,
                const int32_t* indices, const int32_t* lens, const float* sinks,
                float bmm1_scale, float bmm2_scale, float k_scale, void* out, float* lse,
                void* stream);

/* ---------------------------------------------------------------- LSE merge
 * The merge of partial (out, lse) sets of one decode step, e.g. the key
 * shards of a context-parallel decode, after the Kimi K3.1 `mla/dcp` page
 * (DcpValue, class docstring and merge): for each (token t, head h), source
 * s weighs w_s = exp2(lse_s - M) / sum_s' exp2(lse_s' - M) with M the largest
 * finite lse_s (FP32); a source whose LSE is not finite (NaN, +-inf) weighs
 * nothing, and so does every source of a token whose count is <= 0;
 * out[t, h, :] = BF16_RN(sum_s w_s * parts[s, t, h, :]) with the sum in FP32;
 * lse_out[t, h] = M + log2(sum_s exp2(lse_s - M)), base 2. A (token, head)
 * with no weight left gets +0.0 and LSE -inf. */
typedef struct smla_merge_shape {
    int32_t sources;  /* S partial sets (0: every row is empty) */
    int32_t tokens;   /* T */
    int32_t heads;    /* H */
    int32_t reserved; /* 0 */
    /* BF16 elements between consecutive sources / tokens / heads of `parts`
     * (multiples of 8; the 512 latents of a row are contiguous) */
    int64_t part_stride_source, part_stride_token, part_stride_head;
    /* float elements between consecutive sources / tokens of `lses` (heads
     * contiguous) */
    int64_t lse_stride_source, lse_stride_token;
    /* BF16 elements between consecutive tokens / heads of `out` (multiples of 8) */
    int64_t out_stride_token, out_stride_head;
    /* float elements between consecutive tokens of `lse_out` (heads contiguous) */
    int64_t lse_out_stride_token;
} smla_merge_shape;

/* Merges S partial sets into out (and lse_out).
 *   parts    device, BF16 [S, T, H, 512] at the shape's strides, 16-byte aligned.
 *   lses     device, float [S, T, H] base-2 LSEs at the shape's strides.
 *   lens     device, int32 [T] counts (<= 0: the token is empty), or NULL.
 *   out      device, BF16 [T, H, 512] at the shape's strides, 16-byte aligned;
 *            must not overlap the inputs.
 *   lse_out  device, float [T, H], or NULL.
 *   stream   a cudaStream_t (NULL: the legacy default stream).
 * Every buffer belongs to the caller; nothing is allocated. Launched with
 * programmatic dependent launch (inputs are read after the previous kernel in
 * the stream completed); captureable in a CUDA graph.
 * Errors: SMLA_EINVAL (null buffers, negative sizes or strides, unaligned rows)
 * before anything is launched; SMLA_ECUDA when the launch fails. */
int smla_merge(const smla_merge_shape* shape, const void* parts, const float* lses,
               const int32_t* lens, void* out, float* lse_out, void* stream);

/* -------------------------------------------- MXFP4 indexer query quantisation
 * The step before the decode: the indexer's query in the MXFP4 format of its
 * key cache, after the Kimi K3.1 `dsa_indexer_mxfp4` page (mxfp4_q_quant and
 * _mxfp4_quant). For token t and head h < H, the 128 values q[t, h, :] (taken
 * as FP32) form 4 blocks of 32; block b's scale is 2^e, e = ceil(log2(max(amax,
 * 6 * 2^-126) / 6)) clamped to [-127, 127], stored as the byte e + 127 in byte b
 * of q_scale[t, h]; q_packed[t, h, j] = E2M1(q[t, h, 2j] / 2^e) | E2M1(q[t, h,
 * 2j + 1] / 2^e) << 4 with E2M1 rounding to nearest (ties to the even code,
 * saturating at 6, keeping the sign of zero); w_out[t, h] = weights[t, h] *
 * weight_scale (FP32). Heads H <= h < padded_heads get zeros in all three. */
#define SMLA_DTYPE_BF16 1
#define SMLA_DTYPE_F32 2

typedef struct smla_mxfp4_shape {
    int32_t tokens;       /* T */
    int32_t heads;        /* H */
    int32_t padded_heads; /* P >= H */
    int32_t head_dim;     /* 128 */
    int32_t q_dtype;      /* SMLA_DTYPE_BF16 or SMLA_DTYPE_F32 */
    int32_t reserved;     /* 0 */
    int64_t q_stride_token, q_stride_head; /* q elements (multiples of 8); values contiguous */
    int64_t w_stride_token;                /* float elements of `weights`; heads contiguous */
    int64_t packed_stride_token;           /* bytes of q_packed (multiple of 8); heads contiguous, 64 bytes each */
    int64_t scale_stride_token;            /* int32 elements of q_scale; heads contiguous */
    int64_t w_out_stride_token;            /* float elements of w_out; heads contiguous */
} smla_mxfp4_shape;

/* Quantises the indexer query.
 *   q          device, [T, H, 128] of q_dtype, 16-byte aligned.
 *   weights    device, float [T, H].
 *   q_packed   device, uint8 [T, P, 64], 8-byte aligned.
 *   q_scale    device, int32 [T, P].
 *   w_out      device, float [T, P].
 * Every buffer belongs to the caller; nothing is allocated. Launched with
 * programmatic dependent launch; captureable in a CUDA graph.
 * Errors: SMLA_EINVAL (null buffers, negative sizes or strides, misalignment),
 * SMLA_EUNSUPPORTED (head_dim != 128, unknown dtype, tokens * padded_heads
 * within 2^10 of 2^31) before any launch;
 * SMLA_ECUDA when the launch fails. */
int smla_mxfp4_q_quant(const smla_mxfp4_shape* shape, const void* q, const float* weights, float weight_scale,
                       void* q_packed, int32_t* q_scale, float* w_out, void* stream);

/* ---------------------------------------------------- value projection + gate
 * The step after the merge, after the Kimi K3.1 `mla/dcp` page (DcpValue,
 * after the merged rows): each merged latent row is projected by its head's
 * W_UV to 128 values and gated by a sigmoid. For token t < T, head h < H and
 * value v < 128:
 *   acc = sum over j < 512 of latent[t, h, j] * w_uv[h, j, v]  (BF16 x BF16, FP32 accumulation)
 *   out[t, h*128 + v] = BF16(float(BF16(acc)) * 1 / (1 + exp(-gate[t, h*128 + v])))
 * and out[t, h*128 + v] = +0.0 when lens is given and lens[t] <= 0. */
typedef struct smla_value_shape {
    int32_t tokens;   /* T */
    int32_t heads;    /* H */
    int32_t reserved[2];
    int64_t latent_stride_token, latent_stride_head; /* BF16 elements, positive multiples of 8; latents contiguous */
    int64_t gate_stride_token;                       /* BF16 elements (multiple of 8); H*128 contiguous */
    int64_t out_stride_token;                        /* BF16 elements (multiple of 8); H*128 contiguous */
} smla_value_shape;

/* Projects and gates.
 *   latent  device, BF16 [T, H, 512] (the merged rows), 16-byte aligned.
 *   w_uv    device, BF16 [H, 512, 128], contiguous, 16-byte aligned.
 *   gate    device, BF16 [T, H*128], 16-byte aligned.
 *   lens    device, int32 [T], or NULL (every token live).
 *   out     device, BF16 [T, H*128], 16-byte aligned.
 * Every buffer belongs to the caller; nothing is allocated. Launched with
 * programmatic dependent launch; captureable in a CUDA graph. A bounded wait
 * that gives up sets SMLA_DEV_TIMEOUT in the device error word.
 * Errors: SMLA_EINVAL (null buffers, negative sizes, latent strides not
 * positive multiples of 8, gate or out token strides below H*128 or not
 * multiples of 8, misalignment), SMLA_EUNSUPPORTED (T above
 * 65535 * 64 or H above 65535, no tensor-map encoder) before any launch;
 * SMLA_ECUDA when the launch fails. T = 0 or H = 0 launches nothing. */
int smla_value_gate(const smla_value_shape* shape, const void* latent, const void* w_uv, const void* gate,
                    const int32_t* lens, void* out, void* stream);

/* The merge and the projection in one pass, as the page's owner runs them
 * (DcpValue: the LSE merge of the partial sets into shared memory, then W_UV
 * and the gate): for each (token, head) the row smla_merge would write, kept
 * on chip, then the projection and gate of smla_value_gate. out equals
 * smla_value_gate of smla_merge's out bit for bit. */
typedef struct smla_merge_value_shape {
    int32_t sources;  /* S partial sets (0: every row is empty) */
    int32_t tokens;   /* T */
    int32_t heads;    /* H */
    int32_t reserved; /* 0 */
    /* BF16 elements between consecutive sources / tokens / heads of `parts`
     * (non-negative multiples of 8; the 512 latents of a row are contiguous) */
    int64_t part_stride_source, part_stride_token, part_stride_head;
    /* float elements between consecutive sources / tokens of `lses` (heads contiguous) */
    int64_t lse_stride_source, lse_stride_token;
    int64_t gate_stride_token; /* BF16 elements (multiple of 8, >= H*128); H*128 contiguous */
    int64_t out_stride_token;  /* BF16 elements (multiple of 8, >= H*128); H*128 contiguous */
} smla_merge_value_shape;

/* Merges, projects and gates.
 *   parts   device, BF16 [S, T, H, 512] at the shape's strides, 16-byte aligned.
 *   lses    device, float [S, T, H] base-2 LSEs at the shape's strides.
 *   lens    device, int32 [T] counts (<= 0: the token is empty), or NULL.
 *   w_uv    device, BF16 [H, 512, 128], contiguous, 16-byte aligned.
 *   gate    device, BF16 [T, H*128], 16-byte aligned.
 *   out     device, BF16 [T, H*128], 16-byte aligned; must not overlap the inputs.
 * Every buffer belongs to the caller; nothing is allocated. Launched with
 * programmatic dependent launch; captureable in a CUDA graph. A bounded wait
 * that gives up sets SMLA_DEV_TIMEOUT in the device error word.
 * Errors: SMLA_EINVAL (null buffers, negative sizes or strides, misaligned
 * rows, gate or out token strides below H*128 or not multiples of 8),
 * SMLA_EUNSUPPORTED (S above 64, T above 65535 * 64 or H above 65535, no
 * tensor-map encoder) before any launch; SMLA_ECUDA when the launch fails.
 * T = 0 or H = 0 launches nothing. */
int smla_merge_value(const smla_merge_value_shape* shape, const void* parts, const float* lses,
                     const int32_t* lens, const void* w_uv, const void* gate, void* out, void* stream);

/* ------------------------------------------------------------------------
 * Decode over fp8_ds_mla cache rows (Kimi K3.1 dsa_indexer_mxfp4 page,
 * mxfp4_fused_prologue: mla_cache [num_blocks, block_size, 656] bytes, filled
 * with [kv_c_normed | k_pe] and viewed as FP8, float32 and BF16). The page
 * prints no row layout; this library reads a 656-byte row as bytes 0..511 the
 * E4M3 codes of the 512 latents, bytes 512..527 four little-endian FP32
 * scales (scale b covers latents 128 b .. 128 b + 127), bytes 528..655 the 64
 * rope values as little-endian BF16. Latent j is dec(code_j) * s_(j / 128).
 * The attention is smla_decode's with K the 576 values of a row and V its 512
 * latents; the row scales take the place of k_scale. */
typedef struct smla_ds_mla_shape {
    int32_t tokens;     /* T >= 0 */
    int32_t heads;      /* H: a positive multiple of 32, <= 1024 */
    int32_t width;      /* W >= 0 */
    int32_t num_pools;  /* 1 or 2 */
    int32_t pool_split; /* columns < pool_split read pool 0 (num_pools == 2) */
    int32_t head_tile;  /* heads per CTA: 0 lets the library choose, 32, or 64 (H a multiple of 64) */
    int64_t q_stride_token, q_stride_head;       /* q_latent: bytes, multiples of 16; head stride >= 512 */
    int64_t rope_stride_token, rope_stride_head; /* q_rope: BF16 elements, multiples of 8; head stride >= 64 */
    int64_t idx_stride_token;                    /* int32 elements, >= W */
    int64_t out_stride_token, out_stride_head;   /* BF16 elements, even; head stride >= 512 */
    int64_t lse_stride_token;                    /* float elements */
} smla_ds_mla_shape;

/* Sparse MLA decode over fp8_ds_mla rows.
 *   q_latent  device, E4M3 [T, H, 512] at the shape's byte strides, 16-byte aligned.
 *   q_rope    device, BF16 [T, H, 64] at the shape's element strides, 16-byte aligned.
 *   kv_pools  host array of num_pools descriptors: rows of row_bytes = 656,
 *             data 16-byte aligned in device memory.
 *   indices, lens, sinks, lse, stream: as for smla_decode.
 *   bmm1_scale  multiplies the dot products (> 0); bmm2_scale multiplies the
 *             output (the row scales replace k_scale).
 *   out       device, BF16 [T, H, 512].
 * One CTA per (token, 32 or 64 heads: smla_ds_mla_head_tile), no key split;
 * launched with programmatic dependent launch; captureable in a CUDA graph
 * (no allocation, no synchronisation). Both head tiles compute the same
 * arithmetic in the same order. Errors: SMLA_EINVAL / SMLA_EUNSUPPORTED before anything is
 * launched, SMLA_ECUDA when the launch fails; an index beyond its pool and a
 * wait that timed out set bits in the device error word. */
int smla_decode_ds_mla(const smla_ds_mla_shape* shape, const void* q_latent, const void* q_rope,
                       const smla_pool* kv_pools, const int32_t* indices, const int32_t* lens, const float* sinks,
                       float bmm1_scale, float bmm2_scale, void* out, float* lse, void* stream);

/* The heads per CTA smla_decode_ds_mla takes for `shape` on a device of
 * `num_sms` SMs (<= 0: the current device's count): shape->head_tile when it
 * is 32 or 64; with 0, 64 where H is a multiple of 64 and the 64-head grid
 * (T x H / 64 CTAs) takes fewer waves of the SMs than the 32-head grid, else
 * 32. Returns 32, 64, SMLA_EINVAL (a shape smla_decode_ds_mla rejects for
 * its heads or head_tile) or SMLA_ECUDA (no device to query). */
int smla_ds_mla_head_tile(const smla_ds_mla_shape* shape, int num_sms);

/* Reads and clears the current device's error word (SMLA_DEV_* bits) in
 * stream order, without synchronising the device: a one-thread kernel on
 * `stream` (a cudaStream_t, NULL: the legacy default stream) exchanges the
 * word for zero once the work queued before it on that stream has finished,
 * its value is copied to `bits` (host) and only `stream` is waited for.
 * Concurrent reads from several host threads are serialised on the host (one
 * staging word per device). Not captureable: SMLA_EINVAL on a stream that is
 * capturing, or for a NULL `bits`; SMLA_ECUDA when a launch, the copy or the
 * wait fails. This library has no counterpart on the pages; it replaces a
 * device-wide synchronisation in callers that keep other streams busy. */
int smla_read_device_error(void* stream, int32_t* bits);

/* Reads and clears the current device's error word after synchronising the
 * whole device (every stream). Returns SMLA_OK, SMLA_EINVAL (NULL `bits`) or
 * SMLA_ECUDA. */
int smla_device_error(int32_t* bits);

/* Self-test of the bounded waits every kernel of this library uses: launches
 * one warp on `stream` that waits on an mbarrier expecting one arrival, with
 * the waits' own code and a limit of `limit_ns` nanoseconds. With `arrive`
 * set, the warp arrives itself and the wait succeeds; with `arrive` zero
 * nothing arrives, the wait gives up after about `limit_ns` and the kernel
 * sets SMLA_DEV_TIMEOUT in the error word and returns, leaving the context
 * usable. No counterpart on the pages. Errors: SMLA_EINVAL for `limit_ns`
 * outside [1000, 1e9]; SMLA_ECUDA when the launch fails. */
int smla_selftest_bounded_wait(int arrive, int64_t limit_ns, void* stream);

/* A static string for a return code. */
const char* smla_error_string(int code);

/* The last CUDA error code seen by this thread (0 if none). */
int smla_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int smla_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SMLA_H */
