// The decode path over the INT8 comparator's cache (no rotation, no zero-points).
#include "attn_decode.cuh"

namespace kvi4 {

cudaError_t launch_decode_int8(const AttnParams& p, int head_size, int num_ctas, DType q_dt, DType out_dt,
                               cudaStream_t stream) {
    return launch_decode_mode<8>(p, head_size, num_ctas, q_dt, out_dt, stream);
}

}  // namespace kvi4
