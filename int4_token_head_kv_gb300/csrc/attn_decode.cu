// The decode path over the INT4 cache, the grid-size rule, and the entry that picks the cache mode.
#include "attn_decode.cuh"

namespace kvi4 {

int decode_grid_size(int64_t max_weight_total, int64_t max_units) {
    int64_t n = 2ll * num_sms();
    if (n > max_units) n = max_units;
    // a share of weight w holds at most w + 2 unit starts (every unit weighs at least one block)
    const int64_t need = (max_weight_total + kMaxUnits - 3) / (kMaxUnits - 2);
    if (n < need) n = need;
    if (n < 1) n = 1;
    return n > 0x7FFFFFFF ? 0x7FFFFFFF : (int)n;
}

cudaError_t launch_decode(const AttnParams& p, int head_size, int num_ctas, DType q_dt, DType out_dt,
                          cudaStream_t stream, int bits) {
    if (bits == 8) return launch_decode_int8(p, head_size, num_ctas, q_dt, out_dt, stream);
    if (bits == 2) return launch_decode_int2(p, head_size, num_ctas, q_dt, out_dt, stream);
    return launch_decode_mode<4>(p, head_size, num_ctas, q_dt, out_dt, stream);
}

}  // namespace kvi4
