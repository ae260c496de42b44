// Internal declarations shared by the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace kvi4 {

constexpr int kBlockSize = 16;   // tokens per cache block
constexpr int kPrefillRows = 128;   // query rows (tokens x q heads of one kv head) per prefill CTA

// Upper bound of every pipeline wait inside a kernel (ns).  A wait that runs out records
// KV_INT4_STAT_WAIT_TIMEOUT and the kernel winds down instead of spinning forever.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

enum class DType : int { F16 = 0, BF16 = 1, F32 = 2 };

struct WriteParams {
    const void* k;
    const void* v;
    const int64_t* slots;
    const float* signs;
    uint8_t* cache;
    uint32_t* status;
    int64_t num_tokens;
    int64_t num_slots;  // num_blocks * block_size
    int H;
    float c;            // fp32(1 / sqrt(head_size))
};

struct AttnParams {
    const void* q;
    const uint8_t* cache;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* qsl;       // query_start_loc
    const float* signs;
    void* out;
    int32_t* ws_meta;         // [num_seqs + 1] first split-KV unit of each sequence (exclusive prefix)
    int32_t* ws_ptile;        // [num_seqs + 1] first prefill query tile of each sequence (exclusive
                              // prefix, written by the walker's CTA 0 when pf_tiles_cap > 0)
    uint32_t* ws_q;           // [num_seqs, qrec_words] rotated-query records of the decode sequences
    float* ws_po;             // [units, 8 warps, po_floats] unnormalised partial outputs (fragment order)
    float* ws_pml;            // [units, 8 warps, 8 columns, 2] partial (max in log2 units, sum)
    uint32_t* status;
    int64_t num_blocks;
    int64_t num_q_tokens;
    int num_seqs;
    int max_query_len;
    int H;                    // kv heads
    int G;                    // q heads per kv head
    int Hq;
    int max_blocks_per_seq;
    int seg_len;              // decode split-KV segment (unit) length in tokens, a multiple of 16
    int len_cap;              // decode context lengths are clamped to this (max_seq_len, block table)
    int pf_tiles_cap;         // > 0: the prefill grid covers this many query tiles per kv head (a
                              // bound on the batch's total) through ws_ptile; 0: one grid slice per
                              // sequence (few empty slices, no lookup)
    int combine_warps;        // combine warps per (sequence, kv head): a power of two, 1..16
    int qrec_words;           // 32-bit words of one rotated-query record
    uint32_t seg_rcp;         // floor(2^32 / seg_len), for fast_div
    uint32_t segb_rcp;        // floor(2^32 / (seg_len / 16)) (all ones for 1)
    int wph_shift;            // log2(8 / H): consumer warps per kv head
    float softmax_scale;
    float c;                  // fp32(1 / sqrt(head_size))
    // options of the unified-attention interface, on the scaled logit s of key j at query position
    // pos, in log2 units (x = s log2 e): x <- C tanh(x / C), x <- x + slope log2e (j - pos),
    // x <- x + qq_bias[pos - c][j - c] log2e for the keys j >= c of the query chunk (c its first
    // position), key visible only if pos - j <= window_left
    int opts;                 // kOptWindow | kOptSoftcap | kOptAlibi | kOptQQ
    int window_left;
    float cap_l2;             // C = softcap log2 e
    float inv_cap_l2;         // 1 / C
    const float* alibi;       // [Hq] slopes (natural-log units)
    const float* qq_bias;     // [rows >= max_query_len][qq_stride] (natural-log units)
    int qq_stride;            // elements per row, >= max_query_len
};
constexpr int kOptWindow = 1, kOptSoftcap = 2, kOptAlibi = 4, kOptQQ = 8;

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_write(const WriteParams& p, int head_size, DType dt, cudaStream_t stream);
// INT8 per-(token, head) comparator rows (D codes + fp32 scale); p.signs and p.c are not used.
cudaError_t launch_write_int8(const WriteParams& p, int head_size, DType dt, cudaStream_t stream);
// INT2 Lloyd-Max rows (D/4 code bytes + the fp32 RMS scale) after the INT4 mode's rotation.
cudaError_t launch_write_int2(const WriteParams& p, int head_size, DType dt, cudaStream_t stream);
// Decode path: query rotation, the split-KV segment walker, and the combine that finishes every
// decode sequence.  num_ctas is the walker's grid (decode_grid_size).
// bits: 4 for the INT4 cache, 8 for the INT8 comparator's cache (no rotation, no zero-points), 2 for
// the INT2 Lloyd-Max cache (rotated, centroids, no zero-points)
cudaError_t launch_decode(const AttnParams& p, int head_size, int num_ctas, DType q_dt, DType out_dt,
                          cudaStream_t stream, int bits);
// the INT8 and INT2 instantiations of the decode path (launch_decode calls them for bits 8 and 2)
cudaError_t launch_decode_int8(const AttnParams& p, int head_size, int num_ctas, DType q_dt, DType out_dt,
                               cudaStream_t stream);
cudaError_t launch_decode_int2(const AttnParams& p, int head_size, int num_ctas, DType q_dt, DType out_dt,
                               cudaStream_t stream);
int decode_grid_size(int64_t max_weight_total, int64_t max_units);
constexpr int kDecodeMaxUnits = 256;   // split-KV units one walker CTA may own

// Rotated-query record of one decode sequence (32-bit words): per kv head, 32-dimension group and
// lane the 4 (8 when G == 8) fp16x2 words that lane feeds to the score mma, then the Hq logit
// factors and the Hq sums of the stored query halves (each padded to a multiple of 4).
inline constexpr uint32_t decode_qrec_words(int D, int H, int G) {
    return (uint32_t)H * (uint32_t)D * (G == 8 ? 8u : 4u) + 2u * (((uint32_t)(H * G) + 3u) & ~3u);
}
// One warp's unnormalised partial output of one split-KV unit of the decode path: D/16 row tiles
// x 16 (32 when G == 8) lanes x 4 accumulators (shared by the host's workspace layout and the
// kernels).
inline constexpr uint32_t decode_po_floats(int D, int G) { return (uint32_t)(D / 16) * (G == 8 ? 32u : 16u) * 4u; }

cudaError_t launch_prefill(const AttnParams& p, int head_size, int max_query_len, DType q_dt, DType out_dt,
                           cudaStream_t stream);
// The prefill kernel instantiated with the logit options (p.opts != 0); launch_prefill calls it.
cudaError_t launch_prefill_opts(const AttnParams& p, int head_size, int max_query_len, DType q_dt, DType out_dt,
                                cudaStream_t stream);

int num_sms();

// floor(2^32 / d) for 1 <= d (all ones for d = 1): the multiplier fast_div expects.
inline uint32_t div_rcp(uint32_t d) { return d <= 1 ? 0xFFFFFFFFu : (uint32_t)((1ull << 32) / d); }

// Opt a kernel in to `bytes` of dynamic shared memory, once per device (so that launches issued
// under stream capture contain nothing but the launch itself).
// Host threads may launch concurrently: the per-device record is atomic (two threads that both see
// it short set the same attributes, which is harmless).
template <auto Kern>
cudaError_t opt_in_smem(size_t bytes) {
    static std::atomic<size_t> done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (done[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    // prefer the largest shared-memory carve-out, so that several CTAs fit on an SM
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(Kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) {
        size_t prev = done[dev].load(std::memory_order_relaxed);
        while (prev < bytes && !done[dev].compare_exchange_weak(prev, bytes, std::memory_order_release)) {
        }
    }
    return e;
}

}  // namespace kvi4
