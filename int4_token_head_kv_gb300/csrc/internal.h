// Internal declarations shared by the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvi4 {

constexpr int kBlockSize = 16;   // tokens per cache block

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
    float* ws_o;              // [num_q_tokens, Hq, nseg_max, D] partial outputs (not normalised)
    float* ws_ml;             // [num_q_tokens, Hq, nseg_max, 2] partial (max in log2 units, sum)
    uint32_t* status;
    int64_t num_blocks;
    int64_t num_q_tokens;
    int num_seqs;
    int max_query_len;
    int H;                    // kv heads
    int G;                    // q heads per kv head
    int Hq;
    int max_blocks_per_seq;
    int seg_len;              // decode split-KV segment length (tokens, multiple of 16)
    int nseg_max;
    float softmax_scale;
    float c;                  // fp32(1 / sqrt(head_size))
};

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_write(const WriteParams& p, int head_size, DType dt, cudaStream_t stream);
cudaError_t launch_decode(const AttnParams& p, int head_size, DType q_dt, DType out_dt, cudaStream_t stream);
cudaError_t launch_combine(const AttnParams& p, int head_size, DType out_dt, cudaStream_t stream);
cudaError_t launch_prefill(const AttnParams& p, int head_size, int max_query_len, DType q_dt, DType out_dt,
                           cudaStream_t stream);

int num_sms();

// Opt a kernel in to `bytes` of dynamic shared memory, once per device (so that launches issued
// under stream capture contain nothing but the launch itself).
template <auto Kern>
cudaError_t opt_in_smem(size_t bytes) {
    static size_t done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (done[dev] >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    // prefer the largest shared-memory carve-out, so that several CTAs fit on an SM
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(Kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) done[dev] = bytes;
    return e;
}

}  // namespace kvi4
