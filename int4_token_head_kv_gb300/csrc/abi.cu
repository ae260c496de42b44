// The C ABI declared in include/kv_int4.h: argument validation on the host, the device status
// counters, the split-KV segment policy, and kernel launches on the caller's stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/kv_int4.h"
#include "device.cuh"
#include "internal.h"

namespace kvi4 {

// Device status counters (KV_INT4_STAT_*): module-scope device memory, one copy per device that
// loads the library.  Kernels add to them; the host reads and clears them through the ABI.
__device__ uint32_t g_status[KV_INT4_STAT_COUNT];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

uint32_t* status_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<uint32_t*>(ptr);
    }
    return g_status_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype_16(kv_int4_dtype d) { return d == KV_INT4_F16 || d == KV_INT4_BF16; }

bool is_pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

kv_int4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KV_INT4_OK : KV_INT4_ECUDA; }

}  // namespace

int num_sms() {
    const int dev = current_device();
    if (dev < 0) return 152;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

namespace {

// One thread waits on an mbarrier that expects an arrival nobody makes.
__global__ void wait_timeout_kernel(uint32_t* status, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0, timeout_ns)) count_status(status, KV_INT4_STAT_WAIT_TIMEOUT);
    }
}

}  // namespace

}  // namespace kvi4

using namespace kvi4;

extern "C" {

int32_t kv_int4_row_bytes(int32_t head_size) { return head_size > 0 ? head_size / 2 + 4 : 0; }

const char* kv_int4_status_string(kv_int4_status s) {
    switch (s) {
        case KV_INT4_OK: return "ok";
        case KV_INT4_EINVAL: return "invalid argument (null pointer, negative or inconsistent size)";
        case KV_INT4_EUNSUPPORTED: return "unsupported head size, block size, head grouping or dtype";
        case KV_INT4_EALIGN: return "pointer not 16-byte aligned";
        case KV_INT4_EWORKSPACE: return "workspace missing or too small";
        case KV_INT4_ECUDA: return "CUDA call failed";
    }
    return "unknown status";
}

kv_int4_status kv_int4_write(const void* k, const void* v, kv_int4_dtype dtype, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_size, const int64_t* slot_mapping,
                             const float* rht_signs, uint8_t* cache, int64_t num_blocks, int32_t block_size,
                             kv_int4_stream_t stream) {
    if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0) return KV_INT4_EINVAL;
    if (head_size != 64 && head_size != 128) return KV_INT4_EUNSUPPORTED;
    if (block_size != kBlockSize || num_kv_heads > 64 || !valid_dtype_16(dtype)) return KV_INT4_EUNSUPPORTED;
    if (num_tokens == 0) return KV_INT4_OK;
    if (num_tokens * num_kv_heads * 2 >= (int64_t)1 << 31) return KV_INT4_EUNSUPPORTED;   // 32-bit vector index
    if (!k || !v || !slot_mapping || !rht_signs || !cache) return KV_INT4_EINVAL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(cache)) return KV_INT4_EALIGN;
    WriteParams p;
    p.k = k;
    p.v = v;
    p.slots = slot_mapping;
    p.signs = rht_signs;
    p.cache = cache;
    p.status = status_ptr();
    p.num_tokens = num_tokens;
    p.num_slots = num_blocks * block_size;
    p.H = num_kv_heads;
    p.c = (float)(1.0 / std::sqrt((double)head_size));
    return from_cuda(launch_write(p, head_size, dtype == KV_INT4_BF16 ? DType::BF16 : DType::F16,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kv_int8_row_bytes(int32_t head_size) { return head_size > 0 ? head_size + 4 : 0; }

kv_int4_status kv_int8_write(const void* k, const void* v, kv_int4_dtype dtype, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_size, const int64_t* slot_mapping, uint8_t* cache,
                             int64_t num_blocks, int32_t block_size, kv_int4_stream_t stream) {
    if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0) return KV_INT4_EINVAL;
    if (head_size != 64 && head_size != 128) return KV_INT4_EUNSUPPORTED;
    if (block_size != kBlockSize || num_kv_heads > 64 || !valid_dtype_16(dtype)) return KV_INT4_EUNSUPPORTED;
    if (num_tokens == 0) return KV_INT4_OK;
    if (num_tokens * num_kv_heads * 2 >= (int64_t)1 << 31) return KV_INT4_EUNSUPPORTED;   // 32-bit vector index
    if (!k || !v || !slot_mapping || !cache) return KV_INT4_EINVAL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(cache)) return KV_INT4_EALIGN;
    WriteParams p;
    p.k = k;
    p.v = v;
    p.slots = slot_mapping;
    p.signs = nullptr;
    p.cache = cache;
    p.status = status_ptr();
    p.num_tokens = num_tokens;
    p.num_slots = num_blocks * block_size;
    p.H = num_kv_heads;
    p.c = 1.0f;
    return from_cuda(launch_write_int8(p, head_size, dtype == KV_INT4_BF16 ? DType::BF16 : DType::F16,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kv_int2_row_bytes(int32_t head_size) { return head_size > 0 ? head_size / 4 + 4 : 0; }

kv_int4_status kv_int2_write(const void* k, const void* v, kv_int4_dtype dtype, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_size, const int64_t* slot_mapping,
                             const float* rht_signs, uint8_t* cache, int64_t num_blocks, int32_t block_size,
                             kv_int4_stream_t stream) {
    if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0) return KV_INT4_EINVAL;
    if (head_size != 64 && head_size != 128) return KV_INT4_EUNSUPPORTED;
    if (block_size != kBlockSize || num_kv_heads > 64 || !valid_dtype_16(dtype)) return KV_INT4_EUNSUPPORTED;
    if (num_tokens == 0) return KV_INT4_OK;
    if (num_tokens * num_kv_heads * 2 >= (int64_t)1 << 31) return KV_INT4_EUNSUPPORTED;   // 32-bit vector index
    if (!k || !v || !slot_mapping || !rht_signs || !cache) return KV_INT4_EINVAL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(cache)) return KV_INT4_EALIGN;
    WriteParams p;
    p.k = k;
    p.v = v;
    p.slots = slot_mapping;
    p.signs = rht_signs;
    p.cache = cache;
    p.status = status_ptr();
    p.num_tokens = num_tokens;
    p.num_slots = num_blocks * block_size;
    p.H = num_kv_heads;
    p.c = (float)(1.0 / std::sqrt((double)head_size));
    return from_cuda(launch_write_int2(p, head_size, dtype == KV_INT4_BF16 ? DType::BF16 : DType::F16,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kv_int4_attention_segment_len(int32_t num_seqs, int32_t max_seq_len, int32_t segment_len) {
    if (num_seqs < 0 || max_seq_len < 0 || segment_len < 0) return 0;
    if (segment_len > 0) return (segment_len % kBlockSize == 0) ? segment_len : 0;
    // About four segments per walker CTA (two per SM) over the largest batch these sizes allow: finer
    // segments balance the block split better but every segment costs a partial to write and to
    // merge.  A multiple of 32 tokens (whole block pairs), 32..4096.
    const int64_t ctas = 2ll * num_sms();
    const int64_t work = (int64_t)num_seqs * (int64_t)max_seq_len;
    int64_t seg = (work + 4 * ctas - 1) / (4 * ctas);
    seg = ((seg + 31) / 32) * 32;
    if (seg < 32) seg = 32;
    if (seg > 4096) seg = 4096;
    return (int32_t)seg;
}

}  // extern "C"

namespace {

// Workspace of the decode path, in 256-byte-aligned regions:
//   meta  [num_seqs + 1] int32             first unit of each sequence
//   ptile [num_seqs + 1] int32             first prefill query tile of each sequence
//   q     [num_seqs, qrec_words]           rotated-query records
//   po    [units, 8, po_floats]            unnormalised partial outputs
//   pml   [units, 8, 16] fp32              partial (max, sum) per column
// units <= num_seqs * ceil(max_seq_len / segment_len).
struct WsLayout {
    size_t meta, ptile, q, po, pml, total;
    int64_t records;   // most partial records of one (sequence, kv head)
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool ws_layout(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t num_seqs, int32_t max_seq_len,
               int32_t seg, WsLayout* w) {
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_size <= 0 || seg <= 0)
        return false;
    const int G = num_q_heads / num_kv_heads;
    const int64_t seg_per_seq = ((int64_t)max_seq_len + seg - 1) / seg;
    const int64_t max_units = (int64_t)num_seqs * seg_per_seq;
    w->records = seg_per_seq * (8 / num_kv_heads);
    w->meta = 0;
    w->ptile = align256((size_t)(num_seqs + 1) * 4);
    w->q = w->ptile + align256((size_t)(num_seqs + 1) * 4);
    w->po = w->q + align256((size_t)num_seqs * decode_qrec_words(head_size, num_kv_heads, G) * 4);
    w->pml = w->po + align256((size_t)max_units * 8 * decode_po_floats(head_size, G) * 4);
    w->total = w->pml + (size_t)max_units * 8 * 16 * 4;
    return true;
}

kv_int4_status paged_attention_impl(int bits, const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                       int32_t num_q_heads, const uint8_t* cache, int64_t num_blocks,
                                       int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
                                       int32_t max_query_len, int32_t max_seq_len, float softmax_scale,
                                       const float* rht_signs, int32_t segment_len, void* out,
                                       kv_int4_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                       kv_int4_stream_t stream, const kv_int4_attn_options* options) {
    if (num_q_tokens < 0 || num_seqs < 0 || num_blocks < 0 || max_query_len < 0 || max_seq_len < 0 ||
        max_blocks_per_seq < 0 || segment_len < 0)
        return KV_INT4_EINVAL;
    if (head_size != 64 && head_size != 128) return KV_INT4_EUNSUPPORTED;
    if (block_size != kBlockSize) return KV_INT4_EUNSUPPORTED;
    if (!is_pow2_in(num_kv_heads, 1, 8) || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return KV_INT4_EUNSUPPORTED;
    const int G = num_q_heads / num_kv_heads;
    if (!is_pow2_in(G, 1, 8)) return KV_INT4_EUNSUPPORTED;
    if (!valid_dtype_16(q_dtype) || !(valid_dtype_16(out_dtype) || out_dtype == KV_INT4_F32))
        return KV_INT4_EUNSUPPORTED;
    if (segment_len % kBlockSize != 0 || num_seqs > 65535) return KV_INT4_EUNSUPPORTED;
    if (!(softmax_scale == softmax_scale)) return KV_INT4_EINVAL;
    if (options && !(options->softcap >= 0.0f && options->softcap <= 3.0e38f)) return KV_INT4_EINVAL;
    if (options && options->qq_bias && options->qq_bias_stride < std::max(1, max_query_len)) return KV_INT4_EINVAL;
    if (num_q_tokens == 0 || num_seqs == 0) return KV_INT4_OK;
    if (!q || !cache || !block_tables || !seq_lens || !query_start_loc || (bits != 8 && !rht_signs) || !out)
        return KV_INT4_EINVAL;
    if (bits != 4 && max_query_len > 1) return KV_INT4_EUNSUPPORTED;   // the INT8 and INT2 modes decode only
    if (max_query_len < 1 || max_blocks_per_seq < 1) return KV_INT4_EINVAL;
    if (!aligned16(q) || !aligned16(out) || !aligned16(cache)) return KV_INT4_EALIGN;

    const int32_t seg = kv_int4_attention_segment_len(num_seqs, max_seq_len, segment_len);
    if (seg <= 0) return KV_INT4_EINVAL;
    const int64_t len_cap = std::min<int64_t>(max_seq_len, (int64_t)max_blocks_per_seq * kBlockSize);
    const int64_t max_blocks_total = (int64_t)num_seqs * ((len_cap + kBlockSize - 1) / kBlockSize);
    if (max_blocks_total >= ((int64_t)1 << 31)) return KV_INT4_EUNSUPPORTED;   // 32-bit block positions
    WsLayout w;
    if (!ws_layout(num_q_heads, num_kv_heads, head_size, num_seqs, max_seq_len, seg, &w)) return KV_INT4_EINVAL;
    if (workspace == nullptr || workspace_bytes < w.total) return KV_INT4_EWORKSPACE;
    if (!aligned16(workspace)) return KV_INT4_EALIGN;

    AttnParams p;
    p.q = q;
    p.cache = cache;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.qsl = query_start_loc;
    p.signs = rht_signs;
    p.out = out;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.ws_meta = reinterpret_cast<int32_t*>(ws + w.meta);
    p.ws_ptile = reinterpret_cast<int32_t*>(ws + w.ptile);
    p.ws_q = reinterpret_cast<uint32_t*>(ws + w.q);
    p.qrec_words = (int)decode_qrec_words(head_size, num_kv_heads, G);
    p.ws_po = reinterpret_cast<float*>(ws + w.po);
    p.ws_pml = reinterpret_cast<float*>(ws + w.pml);
    {   // warps per (sequence, kv head) in the combine: about one per four records, 1..16
        int cw = 1;
        while (cw < 16 && (int64_t)cw * 4 < w.records) cw <<= 1;
        p.combine_warps = cw;
    }
    p.seg_rcp = div_rcp((uint32_t)seg);
    p.segb_rcp = div_rcp((uint32_t)(seg / kBlockSize));
    p.wph_shift = num_kv_heads == 8 ? 0 : num_kv_heads == 4 ? 1 : num_kv_heads == 2 ? 2 : 3;
    p.status = status_ptr();
    p.num_blocks = num_blocks;
    p.num_q_tokens = num_q_tokens;
    p.num_seqs = num_seqs;
    p.max_query_len = max_query_len;
    p.H = num_kv_heads;
    p.G = G;
    p.Hq = num_q_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.seg_len = seg;
    p.len_cap = (int)len_cap;
    {   // prefill grid: at most num_q_tokens / 2 sequences have two or more queries, and their
        // tiles of BQ tokens cover at most num_q_tokens queries.  When one grid slice per sequence
        // is not much larger than that bound, it needs no tile lookup and is taken.
        const int64_t bq = 128 / G;
        const int64_t per_seq = ((int64_t)max_query_len + bq - 1) / bq;
        const int64_t npf = std::min<int64_t>(num_seqs, num_q_tokens / 2);
        const int64_t bound = std::max<int64_t>(1, std::min((num_q_tokens + npf * (bq - 1)) / bq, npf * per_seq));
        const int64_t sliced = (int64_t)num_seqs * per_seq;
        p.pf_tiles_cap = (sliced <= bound + bound / 4 || bound > (1 << 24)) ? 0 : (int)bound;
    }
    p.softmax_scale = softmax_scale;
    p.c = (float)(1.0 / std::sqrt((double)head_size));
    p.opts = 0;
    p.window_left = -1;
    p.cap_l2 = 0.0f;
    p.inv_cap_l2 = 0.0f;
    p.alibi = nullptr;
    p.qq_bias = nullptr;
    p.qq_stride = 0;
    if (options) {
        if (options->window_left >= 0) {
            p.opts |= kOptWindow;
            p.window_left = options->window_left;
        }
        if (options->softcap > 0.0f) {
            p.opts |= kOptSoftcap;
            p.cap_l2 = (float)((double)options->softcap * 1.4426950408889634);
            p.inv_cap_l2 = 1.0f / p.cap_l2;
        }
        if (options->alibi_slopes) {
            p.opts |= kOptAlibi;
            p.alibi = options->alibi_slopes;
        }
        if (options->qq_bias) {
            p.opts |= kOptQQ;
            p.qq_bias = options->qq_bias;
            p.qq_stride = options->qq_bias_stride;
        }
    }

    const int64_t max_units = (int64_t)num_seqs * (((int64_t)max_seq_len + seg - 1) / seg);
    // balance weight bound: the blocks, plus at most one padded unit per sequence
    const int ctas = decode_grid_size(max_blocks_total + (int64_t)num_seqs * (seg / kBlockSize), max_units);
    const DType qd = q_dtype == KV_INT4_BF16 ? DType::BF16 : DType::F16;
    const DType od = out_dtype == KV_INT4_BF16 ? DType::BF16 : (out_dtype == KV_INT4_F16 ? DType::F16 : DType::F32);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_decode(p, head_size, ctas, qd, od, s, bits);
    if (e == cudaSuccess && bits == 4 && max_query_len > 1) e = launch_prefill(p, head_size, max_query_len, qd, od, s);
    return from_cuda(e);
}

}  // namespace

extern "C" {

size_t kv_int4_attention_workspace_bytes(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                         int32_t num_seqs, int32_t max_seq_len, int32_t segment_len) {
    if (num_seqs <= 0 || max_seq_len < 0) return 0;
    const int32_t seg = kv_int4_attention_segment_len(num_seqs, max_seq_len, segment_len);
    WsLayout w;
    if (!ws_layout(num_q_heads, num_kv_heads, head_size, num_seqs, max_seq_len, seg, &w)) return 0;
    return w.total;
}

kv_int4_status kv_int4_paged_attention(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                       int32_t num_q_heads, const uint8_t* cache, int64_t num_blocks,
                                       int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
                                       int32_t max_query_len, int32_t max_seq_len, float softmax_scale,
                                       const float* rht_signs, int32_t segment_len, void* out,
                                       kv_int4_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                       kv_int4_stream_t stream) {
    return paged_attention_impl(4, q, q_dtype, num_q_tokens, num_q_heads, cache, num_blocks, num_kv_heads, head_size,
                                block_size, block_tables, max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                                max_query_len, max_seq_len, softmax_scale, rht_signs, segment_len, out, out_dtype,
                                workspace, workspace_bytes, stream, nullptr);
}

kv_int4_status kv_int4_paged_attention_ex(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                          int32_t num_q_heads, const uint8_t* cache, int64_t num_blocks,
                                          int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
                                          int32_t max_query_len, int32_t max_seq_len, float softmax_scale,
                                          const float* rht_signs, int32_t segment_len, void* out,
                                          kv_int4_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                          kv_int4_stream_t stream, const kv_int4_attn_options* options) {
    return paged_attention_impl(4, q, q_dtype, num_q_tokens, num_q_heads, cache, num_blocks, num_kv_heads, head_size,
                                block_size, block_tables, max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                                max_query_len, max_seq_len, softmax_scale, rht_signs, segment_len, out, out_dtype,
                                workspace, workspace_bytes, stream, options);
}

kv_int4_status kv_int8_paged_attention(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                       int32_t num_q_heads, const uint8_t* cache, int64_t num_blocks,
                                       int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
                                       int32_t max_query_len, int32_t max_seq_len, float softmax_scale,
                                       int32_t segment_len, void* out, kv_int4_dtype out_dtype, void* workspace,
                                       size_t workspace_bytes, kv_int4_stream_t stream) {
    return paged_attention_impl(8, q, q_dtype, num_q_tokens, num_q_heads, cache, num_blocks, num_kv_heads, head_size,
                                block_size, block_tables, max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                                max_query_len, max_seq_len, softmax_scale, nullptr, segment_len, out, out_dtype,
                                workspace, workspace_bytes, stream, nullptr);
}

kv_int4_status kv_int2_paged_attention(const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens,
                                       int32_t num_q_heads, const uint8_t* cache, int64_t num_blocks,
                                       int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
                                       int32_t max_query_len, int32_t max_seq_len, float softmax_scale,
                                       const float* rht_signs, int32_t segment_len, void* out,
                                       kv_int4_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                       kv_int4_stream_t stream) {
    return paged_attention_impl(2, q, q_dtype, num_q_tokens, num_q_heads, cache, num_blocks, num_kv_heads, head_size,
                                block_size, block_tables, max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                                max_query_len, max_seq_len, softmax_scale, rht_signs, segment_len, out, out_dtype,
                                workspace, workspace_bytes, stream, nullptr);
}

kv_int4_status kv_int4_selftest_wait_timeout(uint64_t timeout_ns, kv_int4_stream_t stream) {
    uint32_t* ptr = status_ptr();
    if (!ptr) return KV_INT4_ECUDA;
    if (timeout_ns > 1000000000ull) timeout_ns = 1000000000ull;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ptr, timeout_ns);
    return from_cuda(cudaGetLastError());
}

kv_int4_status kv_int4_read_device_status(uint32_t* counts, kv_int4_stream_t stream) {
    if (!counts) return KV_INT4_EINVAL;
    uint32_t* ptr = status_ptr();
    if (!ptr) return KV_INT4_ECUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return KV_INT4_ECUDA;
    return from_cuda(cudaMemcpy(counts, ptr, sizeof(uint32_t) * KV_INT4_STAT_COUNT, cudaMemcpyDeviceToHost));
}

kv_int4_status kv_int4_clear_device_status(kv_int4_stream_t stream) {
    uint32_t* ptr = status_ptr();
    if (!ptr) return KV_INT4_ECUDA;
    return from_cuda(cudaMemsetAsync(ptr, 0, sizeof(uint32_t) * KV_INT4_STAT_COUNT,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
