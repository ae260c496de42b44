// The chunked-prefill kernel without logit options, and the entry that picks the flavour.
#include "attn_prefill.cuh"

namespace kvi4 {

cudaError_t launch_prefill(const AttnParams& p, int head_size, int max_query_len, DType q_dt, DType out_dt,
                           cudaStream_t stream) {
    if (p.opts != 0) return launch_prefill_opts(p, head_size, max_query_len, q_dt, out_dt, stream);
    return launch_prefill_all<false>(p, head_size, max_query_len, q_dt, out_dt, stream);
}

}  // namespace kvi4
