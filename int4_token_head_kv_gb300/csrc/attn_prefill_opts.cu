// The chunked-prefill kernel with the logit options of the unified-attention interface (sliding
// window, softcap, ALiBi), in a translation unit of its own so that both flavours compile in parallel.
#include "attn_prefill.cuh"

namespace kvi4 {

cudaError_t launch_prefill_opts(const AttnParams& p, int head_size, int max_query_len, DType q_dt, DType out_dt,
                                cudaStream_t stream) {
    return launch_prefill_all<true>(p, head_size, max_query_len, q_dt, out_dt, stream);
}

}  // namespace kvi4
