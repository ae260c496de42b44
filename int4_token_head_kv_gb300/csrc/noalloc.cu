// kv_int4_paged_attention_noalloc: the paged attention with its split-KV scratch in a fixed
// module-scope device array instead of a caller-provided workspace, for callers that cannot
// allocate device memory.  The array is device memory of the library itself; in host code its
// name only denotes a host-side stand-in, so the host looks up its device address once per device
// and passes that address on, like any caller's workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kv_int4.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KV_INT4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device with that
// device current; nullptr when the lookup fails.
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch[dev] = ptr;
    }
    return g_scratch[dev];
}

// Segment length that keeps the workspace within the scratch array.  An explicit segment_len is
// used as given.  For segment_len 0 the library's usual choice is kept when it fits; otherwise the
// segment grows in steps of 32 tokens (whole block pairs, as the library's own choice) up to 4096
// until the workspace fits.  Returns 0 when nothing fits.
int32_t scratch_segment_len(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t num_seqs,
                            int32_t max_seq_len, int32_t segment_len, size_t* need) {
    *need = kv_int4_attention_workspace_bytes(num_q_heads, num_kv_heads, head_size, num_seqs, max_seq_len,
                                              segment_len);
    if (segment_len != 0 || *need <= KV_INT4_NOALLOC_SCRATCH_BYTES) return segment_len;
    int32_t seg = kv_int4_attention_segment_len(num_seqs, max_seq_len, 0);
    while (seg > 0 && seg < 4096) {
        seg = seg + 32 > 4096 ? 4096 : seg + 32;
        *need = kv_int4_attention_workspace_bytes(num_q_heads, num_kv_heads, head_size, num_seqs, max_seq_len, seg);
        if (*need <= KV_INT4_NOALLOC_SCRATCH_BYTES) return seg;
    }
    return 0;
}

}  // namespace

extern "C" kv_int4_status kv_int4_paged_attention_noalloc_ex(
    const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens, int32_t num_q_heads, const uint8_t* cache,
    int64_t num_blocks, int32_t num_kv_heads, int32_t head_size, int32_t block_size, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
    int32_t max_query_len, int32_t max_seq_len, float softmax_scale, const float* rht_signs, int32_t segment_len,
    void* out, kv_int4_dtype out_dtype, kv_int4_stream_t stream, const kv_int4_attn_options* options) {
    size_t need = 0;
    const int32_t seg = scratch_segment_len(num_q_heads, num_kv_heads, head_size, num_seqs, max_seq_len,
                                            segment_len, &need);
    if (need > KV_INT4_NOALLOC_SCRATCH_BYTES) return KV_INT4_EWORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = scratch_address();
        if (scratch == nullptr) return KV_INT4_ECUDA;
    }
    return kv_int4_paged_attention_ex(q, q_dtype, num_q_tokens, num_q_heads, cache, num_blocks, num_kv_heads,
                                      head_size, block_size, block_tables, max_blocks_per_seq, seq_lens,
                                      query_start_loc, num_seqs, max_query_len, max_seq_len, softmax_scale, rht_signs,
                                      seg, out, out_dtype, scratch,
                                      need > 0 ? (size_t)KV_INT4_NOALLOC_SCRATCH_BYTES : 0, stream, options);
}

extern "C" kv_int4_status kv_int4_paged_attention_noalloc(
    const void* q, kv_int4_dtype q_dtype, int64_t num_q_tokens, int32_t num_q_heads, const uint8_t* cache,
    int64_t num_blocks, int32_t num_kv_heads, int32_t head_size, int32_t block_size, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
    int32_t max_query_len, int32_t max_seq_len, float softmax_scale, const float* rht_signs, int32_t segment_len,
    void* out, kv_int4_dtype out_dtype, kv_int4_stream_t stream) {
    return kv_int4_paged_attention_noalloc_ex(q, q_dtype, num_q_tokens, num_q_heads, cache, num_blocks, num_kv_heads,
                                              head_size, block_size, block_tables, max_blocks_per_seq, seq_lens,
                                              query_start_loc, num_seqs, max_query_len, max_seq_len, softmax_scale,
                                              rht_signs, segment_len, out, out_dtype, stream, nullptr);
}
