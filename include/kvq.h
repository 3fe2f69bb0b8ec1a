/*
 * kvq.h -- C ABI of libkvq: low-bit KV-cache append/quantize and fused
 * dequantize-and-attend decode for one GPU (NVIDIA GB300, sm_103a).
 *
 * The method (sources, by page title and section):
 *  - "KVTuner" review, observation 2 and "Intra-Layer KV Cache Quantization
 *    Precision Pair Pruning" / "KV Cache quantization (Online)": K is quantized
 *    per channel (asymmetric min/scale), each layer keeps its own static
 *    (K bits, V bits) pair from KV8, K8V4, KV4, K4V2, KV2.
 *  - KVQuant (arXiv 2401.18079), abstract and "technical approach": per-channel
 *    K, pre-RoPE K (RoPE applied after dequantization), non-uniform per-layer
 *    datatypes, per-vector dense-and-sparse outliers (~1 %), fused kernels.
 *  - InnerQ (arXiv 2602.23200), "Methodology" 1-5: V grouped along the hidden
 *    dimension (groups of 64 channels) with one min/scale per group, scales
 *    loaded once and reused by every element of the group, fp16 windows for
 *    the most recent and the sink tokens, one fused dequant + GEMV pass.
 *  - "Hadamard rotation-based 2-bit quantization for KV cache compression",
 *    TL;DR and "section details": V rotated by a Hadamard matrix, then uniform
 *    2-bit; the inverse rotation is applied once after the attention sum.
 *
 * Conventions shared by every entry point
 *  - All device pointers are plain CUDA device addresses; the caller owns all
 *    memory.  The library never allocates, frees or synchronises, and keeps
 *    no state between calls: everything is a pure function of the config and
 *    the token counts passed in.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are returned before anything is
 *    launched.  A failed launch returns KVQ_ERR_CUDA.  No C++ exception
 *    crosses the ABI.
 *  - fp16 is IEEE binary16 passed as 16-bit words (`uint16_t`).
 *  - A "stream" of the cache is one (batch row b, KV head h) pair,
 *    s = b * n_kv_heads + h.  Query head hq reads KV head hq / (Hq / Hkv).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stdint.h>

/* The library is built with hidden symbol visibility: only the calls below
 * are exported (so that two builds loaded into one process do not bind to
 * each other's internal symbols). */
#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the type behind cudaStream_t */
typedef struct CUstream_st *kvq_stream_t;

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = -1, /* null pointer, bad size, bad token count      */
    KVQ_ERR_UNSUPPORTED = -2, /* valid but not built: head_dim, bits, groups  */
    KVQ_ERR_CAPACITY = -3,    /* tokens beyond max_tokens                      */
    KVQ_ERR_WORKSPACE = -4,   /* workspace missing or too small                */
    KVQ_ERR_CUDA = -5         /* a CUDA launch or runtime call failed          */
} kvq_status;

/* Per-layer cache configuration.  A model with per-layer bit pairs simply
 * uses one kvq_config per layer ("KVTuner" review, online application of
 * the offline-chosen pairs). */
typedef struct kvq_config {
    int32_t batch;            /* B >= 1                                        */
    int32_t n_q_heads;        /* Hq, a multiple of n_kv_heads                  */
    int32_t n_kv_heads;       /* Hkv >= 1                                      */
    int32_t head_dim;         /* d; 128 is the supported value                 */
    int32_t max_tokens;       /* capacity of every sequence, >= 1              */
    int32_t k_bits;           /* 2, 4, 8: uniform per-channel K; 3: non-uniform
                                 per-token K codes; 16: plain fp16 cache (then
                                 v_bits must be 16 too)                        */
    int32_t v_bits;           /* 2, 4, 8: uniform per-token V over groups of
                                 v_group_channels; 3: non-uniform; 16: fp16    */
    int32_t k_group_tokens;   /* G_K: tokens per K group; 32 is supported      */
    int32_t v_group_channels; /* G_V: channels per V group: 32, 64 or 128      */
    int32_t n_sink;           /* S: first S tokens stay fp16 (attention sinks) */
    int32_t n_recent;         /* R: at least R most recent tokens stay fp16    */
    int32_t v_hadamard;       /* 1: rotate V by Hn = H/sqrt(d) before quantizing
                                 (uniform or non-uniform V); the decode applies
                                 Hn once to the summed quantized part          */
    int32_t k_pre_rope;       /* 1: K is cached before RoPE; the decode applies
                                 RoPE (rotate-half pairs (i, i+d/2), angle
                                 t * rope_theta^(-2i/d) at position t) after
                                 dequantization.  q is always passed already
                                 rotated for its own position.                 */
    float rope_theta;         /* RoPE base, e.g. 10000                         */
    int32_t outliers_per_vector; /* non-uniform mode: k fp16 outliers kept per
                                 token vector (0..8)                           */
    float k_lut[8];           /* non-uniform K levels, strictly increasing,
                                 fp16-representable                            */
    float v_lut[8];           /* non-uniform V levels                          */
    float softmax_scale;      /* 0 selects 1/sqrt(d)                           */
    int32_t split_tokens;     /* decode: quantized tokens per split-K chunk
                                 (multiple of G_K); 0 selects automatically    */
    int32_t position_offset;  /* absolute position of the cache's first token
                                 (0 for a whole context; the first token of a
                                 context shard, see kvq_context_shard): RoPE
                                 after dequantization rotates the key at
                                 position_offset + t.  >= 0, and
                                 position_offset + max_tokens < 2^31           */
    /* InnerQ (InnerQ summary, "Key Contributions" and "Methodology" 1-4): */
    int32_t k_group_channels; /* 0: K per channel over k_group_tokens tokens;
                                 64: K per token in groups of 64 channels along
                                 the hidden dimension (uniform 2/4/8-bit K,
                                 64-channel V groups, no pre-RoPE K)           */
    int32_t hybrid_groups;    /* 1: every uniform K and V group codes itself
                                 symmetrically when its mean lies within half an
                                 asymmetric step of zero,
                                 |mean| * 2^(b+1) <= max - min (mean in exact
                                 fp64): scale = max|x| / (2^(b-1) - 1), code =
                                 clamp(rint(x / scale), -(2^(b-1)-1), 2^(b-1)-1)
                                 + 2^(b-1), stored min = -2^(b-1) * fp16(scale)
                                 (so dequantization is unchanged); otherwise
                                 asymmetric.  0: always asymmetric.            */
    int32_t k_channel_norm;   /* 1 (with k_group_channels 64): per-channel key
                                 normalisation: the first append into an empty
                                 cache sets n_c = the smallest power of two
                                 >= max |K_c| over its tokens (1 for a zero
                                 channel); quantized keys are coded as K / n_c
                                 and the decode multiplies q by n_c.  Sinks and
                                 the fp16 window stay raw.                     */
    /* Per-head (K, V) bits (RateQuant summary, "Methodology" 3-4: per-head
     * allocation, K and V separate): a layer whose KV heads use different
     * pairs is held as one cache per distinct pair, each covering a subset
     * of the layer's heads; n_kv_heads / n_q_heads are the subset's counts. */
    int32_t kv_heads_total;   /* the layer's KV heads (0: n_kv_heads).  k_new,
                                 v_new are [B][kv_heads_total][n_new][d]; q,
                                 out and lse are [B][kv_heads_total *
                                 (n_q_heads / n_kv_heads)][...]; only this
                                 cache's heads are read and written            */
    const int32_t *kv_head_index; /* host array of n_kv_heads distinct layer
                                 KV-head indices (< kv_heads_total, at most 256
                                 entries) that this cache holds, in its stream
                                 order; NULL: heads 0 .. n_kv_heads - 1.  Read
                                 during each call only.                        */
    int32_t sm_budget;        /* decode: spread this cache's work over at most
                                 this many SMs (0: all).  The caches of one
                                 layer's distinct pairs, each given a share,
                                 can then be decoded side by side on separate
                                 CUDA streams (each with its own workspace).   */
} kvq_config;

/* Window rule.  For a sequence holding T tokens:
 *   positions [0, min(S, T))           sinks, fp16
 *   positions [S, S + Nq)              quantized, Nq = G_K * floor((T-S-R)/G_K)
 *                                      (0 when T - S - R <= 0)
 *   positions [S + Nq, T)              fp16 recent window, W tokens, R <= W < R+G_K
 *                                      once T >= S + R
 * Appending tokens one at a time flushes exactly one G_K group whenever the
 * window reaches R + G_K tokens, which gives the same Nq as one bulk append.
 * fp16 mode (bits 16) quantizes nothing: every token is a window token. */

typedef struct kvq_region {
    uint64_t offset; /* byte offset inside the layer buffer (256-byte aligned) */
    uint64_t bytes;  /* size in bytes (0 if the region is unused)              */
} kvq_region;

/* Byte layout of one layer buffer.  NS = batch * n_kv_heads streams,
 * Qcap = G_K * floor(max(0, max_tokens - S - R) / G_K) quantized-token slots,
 * Gcap = Qcap / G_K, RING = R + G_K window slots (max_tokens in fp16 mode),
 * KROW = d * k_bits / 8, VROW = d * v_bits / 8 bytes per packed row.
 * Quantized token index i = t - S for position t.
 *
 *  k_codes   [NS][Qcap][KROW] u8   packed K row of token i: code of channel c at
 *                                  bits [b*c, b*c+b) of the row's little-endian
 *                                  bitstream (bit 0 = LSB of byte 0)
 *  k_scales  uniform K:  [NS][Gcap][d] {min, scale} fp16 pairs (min first), one
 *                        per channel per G_K-token group
 *            InnerQ K (k_group_channels 64): [NS][Qcap][d/64] {min, scale}, one
 *                        per token per 64-channel group
 *            non-uniform K: [NS][Qcap] {min, s} fp16 pairs, one per token
 *  v_codes   [NS][Qcap][VROW] u8   packed V row of token i (rotated domain when
 *                                  v_hadamard)
 *  v_scales  uniform V:  [NS][Qcap][d/G_V] {min, scale} fp16 pairs
 *            non-uniform V: [NS][Qcap] {min, s} fp16 pairs
 *  k_sink, v_sink [NS][S][d] fp16  sink tokens
 *  k_ring, v_ring [NS][RING][d] fp16  window tokens; position t lives in slot
 *                                  (t - S) mod RING (slot t in fp16 mode); V is
 *                                  stored unrotated
 *  k_norm   [NS][d] f32            InnerQ key normalisation n_c (k_channel_norm)
 *  k_csr_rowptr [NS][Qcap+1] i32, k_csr_col [NS][Qcap*k] u8,
 *  k_csr_val [NS][Qcap*k] fp16     non-uniform K outliers as CSR over token rows
 *                                  (rowptr counts from 0 per stream; columns
 *                                  ascend within a row); same for v_csr_*
 *
 * Uniform quantizer (per group of n values, b bits, fp32 arithmetic, RN):
 *   scale = (max - min) / (2^b - 1); code = clamp(rint((x - min)/scale), 0, 2^b-1);
 *   stored min = fp16(min) (exact), scale = fp16_RN(scale); a constant group
 *   stores scale 0 and codes 0.  Dequantized value: min + code * scale.
 * Non-uniform quantizer (one token vector): the k largest |x| (ties -> lower
 *   channel) are kept as fp16 outliers with code 0; over the rest,
 *   s = (max - min)/(L7 - L0), u = (x - min)/s,
 *   code = #{i : u > (L_i + L_{i+1})*0.5 - L0}; value = min + s*(L_code - L0).
 * Hadamard: v' = fp16_RN(fp32(1/sqrt(d)) * FWHT_fp32(v)), butterfly stages of
 *   width 1, 2, ..., d/2, (a, b) -> (a + b, a - b).
 */
typedef struct kvq_layout {
    kvq_region k_codes, k_scales, v_codes, v_scales;
    kvq_region k_sink, v_sink, k_ring, v_ring;
    kvq_region k_csr_rowptr, k_csr_col, k_csr_val;
    kvq_region v_csr_rowptr, v_csr_col, v_csr_val;
    uint64_t layer_bytes;     /* bytes of one layer buffer                     */
    uint64_t workspace_bytes; /* decode scratch needed for any T <= max_tokens  */
    int32_t max_splits;       /* upper bound on decode splits per stream        */
    int32_t ring_slots;       /* RING                                           */
    int32_t q_cap;            /* Qcap                                           */
    kvq_region k_norm;        /* InnerQ key normalisation (0 bytes if unused)   */
    kvq_region rows;          /* a ragged append's per-row counts (2 KB)        */
} kvq_layout;

/* kvq_layout_query -- host only, no CUDA call.
 * Fills *out with the region offsets/sizes of one layer buffer, the layer
 * buffer size and the decode workspace size for `cfg`.
 * Returns KVQ_ERR_INVALID_ARG for null pointers or inconsistent sizes,
 * KVQ_ERR_UNSUPPORTED for combinations the kernels are not built for. */
KVQ_API kvq_status kvq_layout_query(const kvq_config *cfg, kvq_layout *out);

/* kvq_append -- write n_new tokens per sequence into the cache.
 * ("KVTuner" review, online quantization at the fixed per-layer pair;
 *  InnerQ Methodology 1-4; KVQuant per-channel / pre-RoPE K, NUQ, outliers;
 *  Hadamard write-up: rotate V, then quantize.)
 *   layer_buf     device, layer_bytes, laid out as kvq_layout describes; the
 *                 caller zero-fills it once before the first append (not
 *                 required for correctness of quantized data, only so that
 *                 unused bytes are defined)
 *   tokens_before number of tokens each sequence held before this call
 *   k_new, v_new  device fp16 [B][Hkv][n_new][d], K before RoPE when
 *                 k_pre_rope, otherwise as the model produced it
 *   n_new         >= 1; tokens_before + n_new <= max_tokens
 * Tokens that fall in the sink or window regions are copied as fp16; every
 * time the window reaches R + G_K tokens its oldest G_K tokens are quantized
 * (for a bulk prefill, all groups at once).  Launches one quantize kernel when
 * groups are flushed, then one copy kernel for the fp16 tokens.
 * Errors: KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CAPACITY,
 * KVQ_ERR_CUDA. */
KVQ_API kvq_status kvq_append(const kvq_config *cfg, void *layer_buf, int32_t tokens_before,
                      const uint16_t *k_new, const uint16_t *v_new, int32_t n_new,
                      kvq_stream_t stream);

/* kvq_decode_attn -- one decode step of attention over the cache.
 * (KVQuant fused low-bit mat-vec kernels; InnerQ Methodology 3 and 5: fused
 *  group dequant + GEMV with scales reused across the group; Hadamard
 *  write-up: inverse rotation after the attention sum; KVQuant pre-RoPE K.)
 *   layer_buf  device, as written by kvq_append
 *   tokens     T, 1 <= T <= max_tokens: the sequence length to attend over
 *   q          device fp16 [B][Hq][d]
 *   out        device fp16 [B][Hq][d]: softmax(scale * q K^T) V
 *   lse        device f32 [B][Hq] natural-log log-sum-exp of the scaled
 *              logits, or NULL
 *   workspace  device scratch of ws_bytes >= layout.workspace_bytes; its
 *              first NS 32-bit words are split counters that must be zero
 *              before the first call (zero the whole workspace once); every
 *              call leaves them zero again.  Calls that share a workspace
 *              must not overlap on the GPU.
 * One kernel launch.  The cache is cut into pieces that are each streamed
 * once: contiguous ranges of 32-token groups and fp16 tokens per warp in the
 * persistent tensor-core kernel (uniform K/V with 64-channel V groups, or
 * the fp16 cache), or per-CTA splits in the split kernel (NUQ, pre-RoPE K,
 * other V group sizes).  Whichever piece of a stream finishes last merges
 * the stream's partial results by log-sum-exp and applies the inverse
 * Hadamard rotation to the quantized part.
 * Errors: KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CAPACITY,
 * KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA. */
KVQ_API kvq_status kvq_decode_attn(const kvq_config *cfg, const void *layer_buf, int32_t tokens,
                           const uint16_t *q, uint16_t *out, float *lse,
                           void *workspace, uint64_t ws_bytes, kvq_stream_t stream);

/* The split-kernel plan for `tokens` on the host: splits per stream (CTAs
 * per stream of the split-K kernel) and how many of them cover quantized
 * groups; host only, for measurement.  With split_tokens = 0 the decode
 * itself may raise the quantized splits (up to 64) so that its grid fills
 * whole waves of the kernel's resident CTAs on the device it runs on. */
KVQ_API kvq_status kvq_decode_plan(const kvq_config *cfg, int32_t tokens, int32_t *splits_per_stream,
                           int32_t *quantized_splits);

/* Which decode kernel kvq_decode_attn launches for `tokens` (host only, for
 * measurement and tests): *persistent = 1 for the persistent tensor-core
 * kernel (uniform 2/4/8-bit K and V with 64-channel V groups and no pre-RoPE
 * K, or the fp16 cache), 0 for the split-K kernel (non-uniform codes,
 * pre-RoPE K, 32- or 128-channel V groups).  *gq_slots = query-head slots per
 * KV head the kernel is instantiated for (1, 2, 4 or 8).
 * Errors: KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_CAPACITY. */
KVQ_API kvq_status kvq_decode_path(const kvq_config *cfg, int32_t tokens, int32_t *persistent, int32_t *gq_slots);

/* kvq_append_ragged -- kvq_append for sequences of different lengths.
 * The pages attend one context length per call; a batch of sequences at
 * different positions (requests that started at different times, prompts
 * of different lengths) takes this call instead.  Batch row b appends
 * n_new[b] tokens after tokens_before[b] (0 = empty row; n_new[b] = 0 leaves
 * the row as it is); each row follows the same window rule as kvq_append.
 *   tokens_before, n_new  host int32 [batch]; tokens_before[b] >= 0,
 *                         0 <= n_new[b] <= n_stride,
 *                         tokens_before[b] + n_new[b] <= max_tokens
 *   k_new, v_new          device fp16 [B][Hkv][n_stride][d]: row b's tokens
 *                         are the first n_new[b] of its n_stride slots
 *   n_stride              >= 1, the inputs' token dimension
 * InnerQ key normalisation (k_channel_norm) is fixed per row by the row's
 * first append into its empty cache (tokens_before[b] = 0).  The per-row
 * counts are copied into the layer buffer's `rows` region (a small kernel
 * on `stream`) for the append kernels that follow.
 * Errors: as kvq_append; KVQ_ERR_UNSUPPORTED when batch > 256. */
KVQ_API kvq_status kvq_append_ragged(const kvq_config *cfg, void *layer_buf, const int32_t *tokens_before,
                             const int32_t *n_new, const uint16_t *k_new, const uint16_t *v_new,
                             int32_t n_stride, kvq_stream_t stream);

/* kvq_decode_attn_ragged -- kvq_decode_attn for sequences of different
 * lengths: batch row b attends over its own tokens[b] tokens.
 *   tokens     host int32 [batch], 1 <= tokens[b] <= max_tokens
 *   workspace  always required, ws_bytes >= layout.workspace_bytes: with
 *              more than 16 rows the row tables are copied into its end (a
 *              small kernel on `stream`); up to 16 rows they travel in the
 *              launch parameters
 *   other arguments as kvq_decode_attn.
 * Runs the kernel kvq_decode_attn would: the persistent kernel lays every
 * stream's own work items end to end and cuts them into equal ranges;
 * the split-K kernel is planned for the longest row (a stream's splits past
 * its own tokens contribute nothing).
 * Errors: as kvq_decode_attn; KVQ_ERR_UNSUPPORTED when batch > 256. */
KVQ_API kvq_status kvq_decode_attn_ragged(const kvq_config *cfg, const void *layer_buf, const int32_t *tokens,
                                  const uint16_t *q, uint16_t *out, float *lse,
                                  void *workspace, uint64_t ws_bytes, kvq_stream_t stream);

/* kvq_decode_attn_noalloc -- kvq_decode_attn without a caller workspace.
 * The pages have no counterpart: this exists for callers that cannot
 * allocate device memory where they decode (a pool that owns all device
 * memory, a host framework that forbids allocations on its hot path, a
 * real-time loop).  The split-K scratch is a fixed 8 MiB array inside the
 * library, held on every GPU that loads it until the process exits.
 *   Arguments as kvq_decode_attn, minus workspace/ws_bytes.
 *   No cudaMalloc/cudaFree or other allocating call; the split counters are
 *   cleared with cudaMemsetAsync on `stream` before the launch.
 *   The array's device address is looked up (cudaGetSymbolAddress, that
 *   device current) on every call whose stream is not being captured; a call
 *   during stream capture reuses the last address looked up on its device.
 *   So make one call on each device before any stream capture (and again
 *   after a cudaDeviceReset, which may move the array).
 *   All calls share the array: calls that overlap on the GPU race; serialise
 *   them.
 *   The split kernel's splits are widened to the device's SMs as in
 *   kvq_decode_attn when the partials fit the array, else the host plan
 *   (kvq_decode_plan) is used as is.
 * Errors: as kvq_decode_attn; KVQ_ERR_WORKSPACE when this call's scratch
 * (split counters + per-split partials) would exceed 8 MiB. */
KVQ_API kvq_status kvq_decode_attn_noalloc(const kvq_config *cfg, const void *layer_buf, int32_t tokens,
                                   const uint16_t *q, uint16_t *out, float *lse,
                                   kvq_stream_t stream);

/* kvq_fit_nuq_lut -- fit the 8 levels of a non-uniform (3-bit) table to
 * calibration vectors: unweighted Lloyd iterations (KVQuant summary,
 * "technical approach": non-uniform per-layer datatypes computed offline;
 * the sensitivity weighting needs a model's gradients and is not done).
 * Every dense value of a vector is placed in its vector's dense range as the
 * encoder maps it -- the `outliers` largest |x| removed (ties to the lower
 * channel), u = RN((x - min) / (max - min)) in fp32 -- on a grid of 2^-16,
 * p = rint(u * 2^16) in [0, 2^16]; a vector with a constant dense part gives
 * no value.  Lloyd starts from l_i = i * 2^16 / 7, holds l_0 = 0 and
 * l_7 = 2^16 (every vector's min and max sit there), assigns every p to the
 * level it is nearest to (p > (l_i + l_{i+1}) / 2 moves it up; a tie stays
 * down, as in the encoder) and moves l_1..l_6 to the mean of their values
 * (exact integer sums, one fp64 division; an empty level stays), until an
 * update changes nothing or max_iters updates were made.  The table is
 * lut_out[i] = fp16_RN(l_i / 2^16) in [0, 1] (the encoder is invariant to
 * an affine map of the table).
 *   x          device fp16 [n_vectors][head_dim], 8-byte aligned (head_dim 128)
 *   outliers   0..8: per-vector outliers left out, as kvq_config's
 *              outliers_per_vector
 *   hadamard   1: rotate each vector by Hn first, as the encoder does for a
 *              Hadamard-rotated V
 *   workspace  device scratch of >= KVQ_NUQ_FIT_WORKSPACE_BYTES, 8-byte
 *              aligned (its contents need not be zero)
 *   lut_out    device f32 [8]
 *   info_out   device int32 [1] or NULL: the updates made, or -1 when the
 *              rounded levels are not strictly increasing (the table is then
 *              not usable)
 * Three launches on `stream` (a memset and two kernels).  Errors:
 * KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA. */
#define KVQ_NUQ_FIT_WORKSPACE_BYTES (3ull * 65538ull * 8ull)
KVQ_API kvq_status kvq_fit_nuq_lut(const uint16_t *x, int64_t n_vectors, int32_t head_dim, int32_t outliers,
                           int32_t hadamard, int32_t max_iters, void *workspace, uint64_t ws_bytes,
                           float *lut_out, int32_t *info_out, kvq_stream_t stream);

/* Per-head (K, V) bit allocation (RateQuant summary, "Methodology" 1-4).
 *
 * kvq_measure_distortion -- the mean squared error of this cache's uniform
 * quantizers at `bits` (2, 4 or 8, for K and V alike) on calibration tokens,
 * per KV head of the layer, K and V separately (the "distortion
 * calibration" of RateQuant, here of this quantizer):
 *   k, v      device fp16 [B][kv_heads_total][n_tokens][d], 16-byte aligned
 *   K         per channel over the whole 32-token blocks of the n_tokens (or,
 *             with k_group_channels 64, per token over 64-channel groups of
 *             the keys divided by the per-channel normalisation of these
 *             tokens when k_channel_norm is set); V per token over
 *             v_group_channels groups, rotated first when v_hadamard; the
 *             config's hybrid_groups; x^ = min + code * scale from the stored
 *             fp16 pair; errors in fp64 (the normalised keys' errors scaled
 *             back by n_c)
 *   workspace device, >= B * n_kv_heads * d * 4 bytes when k_channel_norm
 *             (else may be NULL)
 *   mse_out   device f64 [kv_heads_total][2]: {D_K, D_V} averaged over the
 *             batch rows and tokens
 * cfg's k_bits / v_bits are ignored (bits applies); non-uniform and fp16
 * configs are not supported.  Errors: KVQ_ERR_INVALID_ARG,
 * KVQ_ERR_UNSUPPORTED, KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA. */
KVQ_API kvq_status kvq_measure_distortion(const kvq_config *cfg, const uint16_t *k, const uint16_t *v, int32_t n_tokens,
                                  int32_t bits, void *workspace, uint64_t ws_bytes, double *mse_out,
                                  kvq_stream_t stream);

/* kvq_rate_allocate -- host only.  For n components (typically 2 per KV
 * head: K and V) with measured distortions distortion[i][0..2] at 2, 4 and
 * 8 bits (all > 0, falling), fits D_i(b) = alpha_i * beta_i^-b by least
 * squares in ln D (beta_i must exceed 1), and allocates total_bits bits
 * (>= 2 n) by the greedy marginal-gain rule on the ladder 2 -> 4 -> 8:
 * every component starts at 2 bits, and while a step fits the remaining
 * budget the one with the largest w_i (D_i(b) - D_i(b')) / (b' - b) is taken
 * (ties to the lower index).  weights (sensitivities w_i) may be NULL (all
 * 1).  bits_out[n] gets 2, 4 or 8; alpha_out, beta_out and waterfill_out
 * (the continuous reverse water-filling optimum b_i with sum b_i =
 * total_bits, from w_i alpha_i ln(beta_i) beta_i^-b_i equal for all i) may
 * be NULL.  Errors: KVQ_ERR_INVALID_ARG. */
KVQ_API kvq_status kvq_rate_allocate(int32_t n, const double *distortion, const double *weights, int32_t total_bits,
                             int32_t *bits_out, double *alpha_out, double *beta_out, double *waterfill_out);

/* Context-parallel decode (KVQuant summary, abstract and main results: a
 * 10M-token context on an 8-GPU system).  The context of every sequence is
 * cut into n_shards contiguous shards at quantized-group boundaries, each
 * held by its own cache (one per GPU): shard 0 keeps the S sink tokens, the
 * last shard the fp16 recent window, every shard an equal share (+-1) of
 * the Nq / G_K quantized groups (fp16 cache: of the 32-token blocks).  The
 * union of the shards' caches holds exactly the groups, scales, sinks and
 * window of one cache of the whole context, so decoding every shard with
 * the same query and merging the results by log-sum-exp (kvq_merge_attn)
 * gives the attention over the whole context.  Appended tokens go to the
 * last shard.
 *
 * kvq_context_shard -- host only.  For a context of `tokens` tokens (at the
 * time the shards are filled), fills *shard_cfg (cfg with n_sink = S on
 * shard 0 and 0 elsewhere, n_recent = R on the last shard and 0 elsewhere,
 * position_offset = cfg->position_offset + *first_token, max_tokens = the
 * shard's tokens, or what is left of cfg->max_tokens on the last shard),
 * *first_token and *shard_tokens (0 for a shard that holds no token: it
 * takes part in the merge as an empty part, lse = -inf, and is not decoded).
 * Errors: KVQ_ERR_INVALID_ARG (n_shards < 1 or > 65536, shard out of range,
 * tokens < 1), KVQ_ERR_CAPACITY, and the config errors of kvq_layout_query. */
KVQ_API kvq_status kvq_context_shard(const kvq_config *cfg, int32_t tokens, int32_t n_shards, int32_t shard,
                             kvq_config *shard_cfg, int32_t *first_token, int32_t *shard_tokens);

/* kvq_merge_attn -- attention over the union of n_parts disjoint parts of a
 * context from each part's normalised output and log-sum-exp (the decode's
 * out and lse):  lse = log sum_r exp(lse_r),  out = sum_r exp(lse_r - lse) out_r.
 * (The same merge the decode applies to its own split partials.)
 *   outs     device fp16 [n_parts][rows][head_dim]
 *   lses     device f32  [n_parts][rows], natural log; -inf marks an empty part
 *   out      device fp16 [rows][head_dim] (may not alias outs)
 *   lse_out  device f32  [rows] or NULL (-inf where every part is empty; out
 *            is then 0)
 * rows = batch * n_q_heads; head_dim = 128.  One launch, fp32 arithmetic.
 * Errors: KVQ_ERR_INVALID_ARG (n_parts < 1, rows < 0, null or misaligned
 * pointers), KVQ_ERR_UNSUPPORTED (head_dim), KVQ_ERR_CUDA. */
KVQ_API kvq_status kvq_merge_attn(int32_t n_parts, int64_t rows, int32_t head_dim, const uint16_t *outs,
                          const float *lses, uint16_t *out, float *lse_out, kvq_stream_t stream);

/* Static string naming a status code. */
KVQ_API const char *kvq_status_string(kvq_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
