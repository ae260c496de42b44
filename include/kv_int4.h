/*
 * kv_int4.h -- C ABI of the INT4 per-(token, head) KV-cache library for NVIDIA GB300 (sm_103a).
 *
 * Two operations, both asynchronous on the caller's CUDA stream, and the pairs of the INT8
 * comparator and of the INT2 Lloyd-Max mode:
 *
 *   kv_int4_write            rotate, quantise and pack new K/V head vectors into a paged cache;
 *   kv_int4_paged_attention  causal attention of queries over that cache (decode, split-KV
 *                            segments, chunked prefill);
 *   kv_int8_write            the INT8 per-(token, head) comparator's cache write;
 *   kv_int8_paged_attention  decode attention over the INT8 comparator's cache;
 *   kv_int2_write            the INT2 per-(token, head) Lloyd-Max cache write;
 *   kv_int2_paged_attention  decode attention over the INT2 cache.
 *
 * The caller owns every buffer.  The library never allocates device or host memory: the
 * attention's split-KV partials live in a caller-provided workspace whose size
 * kv_int4_attention_workspace_bytes() reports.  All pointers are DEVICE pointers unless a
 * comment says otherwise, and must stay valid until the stream reaches the launched work.
 *
 * Errors: every entry point validates its arguments on the host and returns a status without
 * launching anything when they are wrong.  Problems only visible on the device (a slot or block
 * id past the end of the cache, a query chunk longer than its sequence, a sign that is not
 * +-1, a pipeline wait that ran out of time) never trap: the element is skipped, and a counter
 * in a device-resident status array is incremented (kv_int4_read_device_status).
 *
 * The method (page titles and sections of the sources):
 *  - "[Feature] Triton INT4 / INT2 per-token-head KV cache quantization" (vLLM PR #40633),
 *    description: random Hadamard pre-rotation, asymmetric 4-bit codes with one fp32 scale per
 *    (token, head), the 4-bit zero-point hidden in the low 4 mantissa bits of that scale, the
 *    asymmetry corrected on the score side, packed K/V read with split dot products;
 *    review notes: head size must be a power of two, quantise with the truncated scale.
 *  - "PR #40835 report", get_kv_cache_shape: cache shape
 *    (num_blocks, 2, block_size, num_kv_heads, head_size / 2 + 4), uint8.
 *  - "tests/quantization/test_per_token_kv_cache.py": the write call
 *    (key, value, caches, slot_mapping; slot < 0 = padding, skipped) and the unified-attention
 *    call (q, cache, cu_seqlens_q, seqused_k, max_seqlen_q, max_seqlen_k, softmax_scale,
 *    causal=True, block_table, split-KV segment buffers).
 */
#ifndef KV_INT4_H
#define KV_INT4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* kv_int4_stream_t;

typedef enum {
    KV_INT4_OK = 0,
    KV_INT4_EINVAL = 1,        /* null pointer, negative or inconsistent size                  */
    KV_INT4_EUNSUPPORTED = 2,  /* head size, block size, head grouping or dtype not built        */
    KV_INT4_EALIGN = 3,        /* a pointer is not 16-byte aligned                               */
    KV_INT4_EWORKSPACE = 4,    /* workspace missing or smaller than the reported size            */
    KV_INT4_ECUDA = 5          /* a CUDA runtime or driver call failed (launch, attribute, ...)  */
} kv_int4_status;

typedef enum { KV_INT4_F16 = 0, KV_INT4_BF16 = 1, KV_INT4_F32 = 2 } kv_int4_dtype;

/* Indices into the device status array (kv_int4_read_device_status). */
enum {
    KV_INT4_STAT_SLOT_OUT_OF_RANGE = 0,  /* write: slot >= num_blocks * block_size (row skipped)      */
    KV_INT4_STAT_BLOCK_OUT_OF_RANGE = 1, /* attention: block id outside [0, num_blocks) (block skipped) */
    KV_INT4_STAT_BAD_SEQUENCE = 2,       /* attention: query chunk longer than its sequence, or a
                                            sequence longer than its block table                        */
    KV_INT4_STAT_WAIT_TIMEOUT = 3,       /* a pipeline wait gave up; the CTA's output is not valid      */
    KV_INT4_STAT_BAD_SIGN = 4,           /* a rotation sign that is not exactly +1.0f or -1.0f           */
    KV_INT4_STAT_COUNT = 8
};

/* Bytes of one cached (token, head) row: head_size/2 bytes of codes, then the fp32 scale word. */
int32_t kv_int4_row_bytes(int32_t head_size);

/*
 * kv_int4_write -- encode num_tokens new K and V head vectors into the paged cache.
 *
 * For every token t with slot = slot_mapping[t] >= 0, every kv head h, and plane p (0 = K, 1 = V)
 * with x = the input vector upcast exactly to fp32:
 *   1. y = c * H_d * (D x): D = diag(rht_signs), H_d the natural-order (Sylvester) Walsh-Hadamard
 *      matrix, c = fp32(1/sqrt(head_size)); butterflies at strides 1, 2, ..., head_size/2 in fp32
 *      round-to-nearest-even, then one multiply by c per element;
 *   2. s = max(fp32((max y - min y) / 15), 1e-6); s' = s with the low 4 mantissa bits cleared;
 *   3. zp = clamp(rint(fp32(-min y / s')), 0, 15);
 *   4. code_i = clamp(nearest-even integer of the exact value y_i * fp32(1/s') + zp, 0, 15);
 *   5. row byte j = code_{2j} | code_{2j+1} << 4 (j < head_size/2), then the 32-bit word
 *      bits(s') | zp little-endian, stored at cache[slot / block_size][p][slot % block_size][h].
 * The bytes written are bit-exact with that definition.
 *
 * k, v          [num_tokens, num_kv_heads, head_size] contiguous, dtype F16 or BF16; 16-B aligned.
 * slot_mapping  [num_tokens] int64; < 0 = padding token (skipped); >= num_blocks*block_size is
 *               skipped and counted (KV_INT4_STAT_SLOT_OUT_OF_RANGE).
 * rht_signs     [head_size] float, each exactly +1.0f or -1.0f (only the sign bit is used; other
 *               values are counted as KV_INT4_STAT_BAD_SIGN).  The same vector must be passed to
 *               kv_int4_paged_attention.
 * cache         (num_blocks, 2, block_size, num_kv_heads, head_size/2 + 4) uint8, 16-B aligned.
 * Supported: head_size in {64, 128}; block_size 16; num_kv_heads in 1..64.
 * num_tokens == 0 launches nothing and returns KV_INT4_OK.
 */
kv_int4_status kv_int4_write(const void* k, const void* v, kv_int4_dtype dtype, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_size, const int64_t* slot_mapping,
                             const float* rht_signs, uint8_t* cache, int64_t num_blocks,
                             int32_t block_size, kv_int4_stream_t stream);

/*
 * INT8 per-(token, head) comparator rows: head_size int8 codes, then the fp32 scale word
 * (head_size + 4 bytes; "PR #40835 report", get_kv_cache_shape for the non-INT4 per-token-head
 * modes).
 */
int32_t kv_int8_row_bytes(int32_t head_size);

/*
 * kv_int8_write -- the INT8 per-(token, head) cache write, the comparator the pages measure the
 * INT4 mode against ("tests/quantization/test_per_token_kv_cache.py", INT8_CONFIG and
 * _quantize_per_token_head_ref; the round-half-away fix of the INT8 reshape kernel in
 * "[Feature] Triton INT4 / INT2 per-token-head KV cache quantization").  No rotation and no
 * zero-point: per (token, kv head, plane) vector x,
 *   s = max(fp32(max|x_i| / 127), 1e-6), r = fp32(1 / s),
 *   q_i = clamp(trunc(fp32(fp32(x_i * r) + (x_i * r >= 0 ? 0.5 : -0.5))), -128, 127),
 * stored as q_0 .. q_{d-1} (two's complement) then the little-endian bits of s, at
 * cache[slot / 16][plane][slot % 16][head] of a (num_blocks, 2, 16, num_kv_heads, head_size + 4)
 * uint8 cache.  Arguments, validation, skipped slots and error behaviour as kv_int4_write (there
 * are no signs).
 */
kv_int4_status kv_int8_write(const void* k, const void* v, kv_int4_dtype dtype, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_size, const int64_t* slot_mapping,
                             uint8_t* cache, int64_t num_blocks, int32_t block_size,
                             kv_int4_stream_t stream);

/*
 * INT2 Lloyd-Max rows: head_size / 4 code bytes (four 2-bit codes each), then the fp32 scale word
 * (head_size / 4 + 4 bytes).
 */
int32_t kv_int2_row_bytes(int32_t head_size);

/*
 * kv_int2_write -- the INT2 per-(token, head) cache write ("[Feature] Triton INT4 / INT2
 * per-token-head KV cache quantization", description: four 2-bit values per byte, Hadamard
 * pre-rotation over the head dimension, dequantisation by a lookup of one of 4 Lloyd-Max centroids
 * fitted over N(0, 1)).  The page fixes neither the centroids nor the scale; this library takes:
 *   y = c * H_d * (D x) exactly as kv_int4_write (same rht_signs, same fp32 butterfly order);
 *   sigma = max(fp32 sqrt(fp32(sum y_i^2) / d), 1e-6), the fp32 squares summed by folding the
 *     vector in halves (a_i + a_{i + d/2}, then + a_{i + d/4}, ..., then a_0 + a_1);
 *   r = fp32(1 / sigma); z_i = fp32(y_i * r);
 *   code_i = [z_i >= -t] + [z_i >= 0] + [z_i >= t], standing for -b, -a, a, b, where a = 0.45278,
 *     b = 1.51042, t = (a + b) / 2 = 0.98160 are the outputs and threshold of the 4-level
 *     Lloyd-Max quantiser of N(0, 1) (J. Max, 1960), each rounded to fp32;
 * stored as head_size / 4 bytes (element 4j + k in bits 2k, 2k + 1 of byte j) then the
 * little-endian bits of sigma, at cache[slot / 16][plane][slot % 16][head] of a
 * (num_blocks, 2, 16, num_kv_heads, head_size / 4 + 4) uint8 cache.  A reader reconstructs
 * y_hat_i = sigma * centroid(code_i) and x_hat = the inverse rotation of y_hat.  Arguments,
 * validation, skipped slots and error behaviour as kv_int4_write.
 */
kv_int4_status kv_int2_write(const void* k, const void* v, kv_int4_dtype dtype, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_size, const int64_t* slot_mapping,
                             const float* rht_signs, uint8_t* cache, int64_t num_blocks,
                             int32_t block_size, kv_int4_stream_t stream);

/*
 * Bytes of workspace kv_int4_paged_attention needs for these sizes (same arguments as the
 * attention call; segment_len 0 = the library's choice).  It holds each sequence's first
 * segment index and, per split-KV segment (at most num_seqs * ceil(max_seq_len / segment_len) of
 * them), eight warps' partial outputs (head_size * 32 bytes each, twice that when
 * num_q_heads = 8 * num_kv_heads) and (max, sum) pairs.  Returns 0 when the arguments are invalid
 * or num_seqs is 0.
 */
size_t kv_int4_attention_workspace_bytes(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                         int32_t num_seqs, int32_t max_seq_len, int32_t segment_len);

/*
 * The KV-token length of one split-KV segment that kv_int4_paged_attention uses for these sizes
 * (segment_len 0 = the library's choice: about four segments per resident CTA over
 * num_seqs * max_seq_len tokens, a multiple of 32 in 32..4096; otherwise segment_len itself).
 * 0 if invalid.
 */
int32_t kv_int4_attention_segment_len(int32_t num_seqs, int32_t max_seq_len, int32_t segment_len);

/*
 * kv_int4_paged_attention -- causal attention over the INT4 cache.
 *
 * Sequence b has seq_lens[b] cached tokens (this step's tokens already written) and the query
 * rows query_start_loc[b] .. query_start_loc[b+1]-1 (like cu_seqlens_q); its t-th query sits at
 * position seq_lens[b] - q_len_b + t and sees keys 0 .. that position.  Query head g reads kv
 * head g / (num_q_heads / num_kv_heads).  With x_K, x_V the cached rows decoded as
 * (code - zp) * s' and un-rotated, out = softmax(softmax_scale * q . x_K) x_V.
 *
 * Computation: Q is rotated once (q' = R q); scores are dot products of q' with the raw codes
 * in the rotated domain, the zero-point is subtracted from the codes and the scale s' applied per
 * key; an online softmax accumulates P V in the rotated domain and the result is un-rotated
 * (out = R^T o).  Sequences with one query token take the decode path: their contexts are cut
 * into segments of segment_len tokens (segment k of a sequence holds its tokens
 * [k segment_len, (k+1) segment_len)), a grid of about two CTAs per SM walks the batch's segments
 * in runs balanced by cache blocks, each segment writes a (max, sum, output) partial, and a
 * combine step merges each sequence's partials in an order fixed by that sequence's segment count
 * alone.  A segment's arithmetic does not
 * depend on the rest of the batch, so for a fixed segment_len a sequence's output is the same
 * alone or in any batch.  Sequences with more than one query token take the chunked-prefill
 * kernel.
 *
 * q                [num_q_tokens, num_q_heads, head_size], q_dtype F16 or BF16, 16-B aligned.
 * cache            as written by kv_int4_write.
 * block_tables     [num_seqs, max_blocks_per_seq] int32.
 * seq_lens         [num_seqs] int32; query_start_loc [num_seqs + 1] int32 (cumulative).
 * max_query_len    host int: max over b of q_len_b (1 for a pure decode batch).
 * max_seq_len      host int: >= max over b of seq_lens[b]; sizes the workspace.  Longer decode
 *                  contexts are clamped to it (and counted as bad metadata).
 * rht_signs        the vector passed to kv_int4_write.
 * segment_len      KV tokens per split-KV segment, a multiple of 16; 0 = library's choice.
 * out              [num_q_tokens, num_q_heads, head_size], out_dtype F16, BF16 or F32.
 * workspace        >= kv_int4_attention_workspace_bytes(...) bytes, 16-B aligned.  Overlapping
 *                  calls must not share a workspace.
 * Supported: head_size in {64, 128}; block_size 16; num_kv_heads in {1, 2, 4, 8};
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}.  An empty context (seq_len 0) yields zeros.
 */
kv_int4_status kv_int4_paged_attention(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                       int32_t num_q_heads, const uint8_t* cache,
                                       int64_t num_blocks, int32_t num_kv_heads,
                                       int32_t head_size, int32_t block_size,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, const int32_t* query_start_loc,
                                       int32_t num_seqs, int32_t max_query_len,
                                       int32_t max_seq_len, float softmax_scale,
                                       const float* rht_signs, int32_t segment_len, void* out,
                                       kv_int4_dtype out_dtype, void* workspace,
                                       size_t workspace_bytes, kv_int4_stream_t stream);

/*
 * kv_int4_paged_attention_ex -- kv_int4_paged_attention with the unified-attention interface's
 * options ("tests/quantization/test_per_token_kv_cache.py", the window_size and softcap arguments
 * of unified_attention; the PR #40633 description lists sliding window, softcap, ALiBi and qq_bias
 * among the helpers the packed read path shares).  On the scaled logit s_j = softmax_scale *
 * q . x_K,j of key j for a query at position pos, the t-th query of a chunk whose first query sits
 * at position c = seq_len - q_len, in this order:
 *   softcap > 0            s_j <- softcap * tanh(s_j / softcap)
 *   alibi_slopes != NULL   s_j <- s_j + alibi_slopes[g] * (j - pos), g the query head
 *   qq_bias != NULL        s_j <- s_j + qq_bias[t * qq_bias_stride + (j - c)] for c <= j
 *                          (j - c < qq_bias_stride; keys before the chunk take no bias)
 *   window_left >= 0       key j is visible only if pos - j <= window_left (besides j <= pos)
 * options NULL, or window_left < 0, softcap 0, alibi_slopes NULL and qq_bias NULL: exactly
 * kv_int4_paged_attention.  alibi_slopes: DEVICE fp32 [num_q_heads]; qq_bias: DEVICE fp32, row t at
 * qq_bias + t * qq_bias_stride, at least max_query_len rows (one matrix for every sequence and
 * head; the query-to-query bias reading of the page's "qq_bias"), a -inf entry masks its key.
 * Returns KV_INT4_EINVAL for a negative or non-finite softcap or a qq_bias_stride below
 * max_query_len; everything else as kv_int4_paged_attention (same workspace).  The options are
 * read at the call.
 */
typedef struct {
    int32_t window_left;        /* < 0: no window */
    float softcap;              /* 0: none */
    const float* alibi_slopes;  /* NULL: none */
    const float* qq_bias;       /* NULL: none */
    int32_t qq_bias_stride;     /* elements per qq_bias row, >= max_query_len */
} kv_int4_attn_options;

kv_int4_status kv_int4_paged_attention_ex(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                          int32_t num_q_heads, const uint8_t* cache,
                                          int64_t num_blocks, int32_t num_kv_heads,
                                          int32_t head_size, int32_t block_size,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* seq_lens, const int32_t* query_start_loc,
                                          int32_t num_seqs, int32_t max_query_len,
                                          int32_t max_seq_len, float softmax_scale,
                                          const float* rht_signs, int32_t segment_len, void* out,
                                          kv_int4_dtype out_dtype, void* workspace,
                                          size_t workspace_bytes, kv_int4_stream_t stream,
                                          const kv_int4_attn_options* options);

/*
 * kv_int8_paged_attention -- decode attention over the INT8 comparator's cache (as written by
 * kv_int8_write), the read side of the comparison the pages make between the INT4 mode and INT8
 * per-(token, head) quantisation ("PR #40835 report", summary; "tests/quantization/
 * test_per_token_kv_cache.py", INT8_CONFIG and _quantize_per_token_head_ref).
 *
 * Every sequence must have exactly one query token (max_query_len 1; a larger value returns
 * KV_INT4_EUNSUPPORTED and launches nothing).  With x_K, x_V the cached rows decoded as code * s
 * (no rotation, no zero-point), out = softmax(softmax_scale * q . x_K) x_V.  The computation is the
 * decode path of kv_int4_paged_attention with INT8 rows: the same split-KV segments, the same
 * segment-length rule and workspace size (kv_int4_attention_workspace_bytes with these arguments),
 * the same partials and combine, the query and the output not rotated.  Arguments, alignment,
 * supported sizes, clamping and error behaviour as kv_int4_paged_attention, without rht_signs.
 */
kv_int4_status kv_int8_paged_attention(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                       int32_t num_q_heads, const uint8_t* cache,
                                       int64_t num_blocks, int32_t num_kv_heads,
                                       int32_t head_size, int32_t block_size,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, const int32_t* query_start_loc,
                                       int32_t num_seqs, int32_t max_query_len,
                                       int32_t max_seq_len, float softmax_scale,
                                       int32_t segment_len, void* out, kv_int4_dtype out_dtype,
                                       void* workspace, size_t workspace_bytes,
                                       kv_int4_stream_t stream);

/*
 * kv_int2_paged_attention -- decode attention over the INT2 Lloyd-Max cache (as written by
 * kv_int2_write with the same rht_signs).  Every sequence must have exactly one query token
 * (max_query_len 1; a larger value returns KV_INT4_EUNSUPPORTED and launches nothing).  With x_K,
 * x_V the cached rows decoded as the inverse rotation of sigma * centroid(code),
 * out = softmax(softmax_scale * q . x_K) x_V.  The computation is the decode path of
 * kv_int4_paged_attention with INT2 rows: the query rotated as for INT4, the scores and P.V taken
 * on the rotated codes through the centroid table (held as fp16: 0.45288 and 1.5107, a relative
 * error of at most 2.3e-4 per centroid), the output un-rotated; the same split-KV segments,
 * segment-length rule, workspace size (kv_int4_attention_workspace_bytes with these arguments),
 * partials and combine.  Arguments, alignment, supported sizes, clamping and error behaviour as
 * kv_int4_paged_attention.
 */
kv_int4_status kv_int2_paged_attention(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                       int32_t num_q_heads, const uint8_t* cache,
                                       int64_t num_blocks, int32_t num_kv_heads,
                                       int32_t head_size, int32_t block_size,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, const int32_t* query_start_loc,
                                       int32_t num_seqs, int32_t max_query_len,
                                       int32_t max_seq_len, float softmax_scale,
                                       const float* rht_signs, int32_t segment_len, void* out,
                                       kv_int4_dtype out_dtype, void* workspace,
                                       size_t workspace_bytes, kv_int4_stream_t stream);

/*
 * kv_int4_paged_attention_noalloc -- the same attention for callers that cannot allocate device
 * memory.  (The pages have no counterpart: this entry point is an addition of this library.)
 *
 * Some callers cannot provide the workspace kv_int4_paged_attention asks for: a serving engine
 * that hands all free device memory to its KV cache at start-up and keeps no allocator on the
 * decode path, a plugin host that forbids device allocation after initialisation, or a decode loop
 * that cannot afford cudaMalloc's implicit device-wide synchronisation.  This variant takes the
 * same arguments minus the workspace and keeps its workspace in a fixed scratch array of
 * KV_INT4_NOALLOC_SCRATCH_BYTES bytes that lives in the library's own device memory (allocated
 * when the library is loaded, held by every GPU that loads it until the process exits).  It calls
 * no cudaMalloc, cudaFree or allocating library routine.
 *
 * Segment length: an explicit segment_len is used as given.  With segment_len 0 the call takes the
 * library's usual choice (kv_int4_attention_segment_len) when its workspace fits the scratch array;
 * otherwise it raises the segment length in steps of 32 tokens, up to 4096, to the first value whose
 * kv_int4_attention_workspace_bytes() fits, and computes exactly what kv_int4_paged_attention computes
 * with that segment_len.  Returns KV_INT4_EWORKSPACE, launching nothing, when the workspace for an
 * explicit segment_len, or for 4096, exceeds KV_INT4_NOALLOC_SCRATCH_BYTES (use a larger
 * segment_len, or the regular entry point).  The first call on a device looks up the scratch
 * array's device address (a runtime call that does not touch any stream); make that first call
 * before any stream capture.
 * Every call shares the one array and it keeps the last call's contents; nothing in it needs to
 * start at zero, because each call writes every partial it later reads.  Calls that overlap on the
 * GPU (different streams, or different host threads on one device) race on the array: serialise
 * them.
 */
#define KV_INT4_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

kv_int4_status kv_int4_paged_attention_noalloc(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                               int32_t num_q_heads, const uint8_t* cache,
                                               int64_t num_blocks, int32_t num_kv_heads,
                                               int32_t head_size, int32_t block_size,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* seq_lens, const int32_t* query_start_loc,
                                               int32_t num_seqs, int32_t max_query_len,
                                               int32_t max_seq_len, float softmax_scale,
                                               const float* rht_signs, int32_t segment_len, void* out,
                                               kv_int4_dtype out_dtype, kv_int4_stream_t stream);

/*
 * kv_int4_paged_attention_noalloc_ex -- the no-allocation attention with the options of
 * kv_int4_paged_attention_ex (options NULL: exactly kv_int4_paged_attention_noalloc).  Segment
 * length, scratch array and error behaviour as kv_int4_paged_attention_noalloc; the options as
 * kv_int4_paged_attention_ex.
 */
kv_int4_status kv_int4_paged_attention_noalloc_ex(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                                  int32_t num_q_heads, const uint8_t* cache,
                                                  int64_t num_blocks, int32_t num_kv_heads,
                                                  int32_t head_size, int32_t block_size,
                                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                  const int32_t* seq_lens, const int32_t* query_start_loc,
                                                  int32_t num_seqs, int32_t max_query_len,
                                                  int32_t max_seq_len, float softmax_scale,
                                                  const float* rht_signs, int32_t segment_len, void* out,
                                                  kv_int4_dtype out_dtype, kv_int4_stream_t stream,
                                                  const kv_int4_attn_options* options);

/*
 * Copy the current device's status counters (KV_INT4_STAT_COUNT uint32 values) to the HOST array
 * counts.  Synchronises the stream first.  The counters keep counting until cleared.
 */
kv_int4_status kv_int4_read_device_status(uint32_t* counts, kv_int4_stream_t stream);

/* Zero the current device's status counters (asynchronous on the stream). */
kv_int4_status kv_int4_clear_device_status(kv_int4_stream_t stream);

/*
 * Diagnostic of the bounded-wait machinery: launches one CTA that waits on a shared-memory barrier
 * nothing will ever complete and gives up after timeout_ns (clamped to 1 s), recording the give-up
 * as KV_INT4_STAT_WAIT_TIMEOUT exactly as the pipelined kernels do.  The device stays usable.
 */
kv_int4_status kv_int4_selftest_wait_timeout(uint64_t timeout_ns, kv_int4_stream_t stream);

/* Static description of a status code (never NULL). */
const char* kv_int4_status_string(kv_int4_status status);

#ifdef __cplusplus
}
#endif

#endif /* KV_INT4_H */
