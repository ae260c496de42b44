// Pieces shared by the decode and prefill attention kernels over the INT4 cache.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device.cuh"

namespace kvi4 {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1.0e30f;   // "no key seen yet" running max (finite, so exp2 never sees inf - inf)

template <typename T>
__device__ __forceinline__ float load_elem(const void* base, int64_t i);
template <>
__device__ __forceinline__ float load_elem<__half>(const void* base, int64_t i) {
    return __half2float(static_cast<const __half*>(base)[i]);
}
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const void* base, int64_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

template <typename T>
__device__ __forceinline__ void store_elem(void* base, int64_t i, float x);
template <>
__device__ __forceinline__ void store_elem<__half>(void* base, int64_t i, float x) {
    static_cast<__half*>(base)[i] = __float2half_rn(x);
}
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(void* base, int64_t i, float x) {
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ void store_elem<float>(void* base, int64_t i, float x) {
    static_cast<float*>(base)[i] = x;
}

// The attention options on one visible key's logit x (log2 units) for a query at position pos and
// key j: softcap C tanh(x / C) (tanh(y) = 1 - 2 / (e^{2y} + 1)), then the ALiBi bias
// slope_l2 (j - pos), then the query-to-query bias of the keys in the query chunk (cs: position of
// the chunk's first query), then the window (-inf when pos - j > window_left).  Masked keys stay -inf.
__device__ __forceinline__ float apply_opts(float x, int j, int pos, float slope_l2, const AttnParams& p, int cs) {
    if (!(x > -INFINITY)) return x;
    if (p.opts & kOptSoftcap) {
        const float e = fast_exp2(2.0f * kLog2e * (x * p.inv_cap_l2));   // e^{2y}, y = x / C
        x = p.cap_l2 * (1.0f - 2.0f / (e + 1.0f));
    }
    if (p.opts & kOptAlibi) x = fmaf(slope_l2, (float)(j - pos), x);
    if (p.opts & kOptQQ) {
        const int u = j - cs, r = pos - cs;   // key and query indices in the chunk (r < max_query_len)
        if (u >= 0 && u < p.qq_stride && r >= 0) x = fmaf(__ldg(p.qq_bias + (int64_t)r * p.qq_stride + u), kLog2e, x);
    }
    if ((p.opts & kOptWindow) && pos - j > p.window_left) x = -INFINITY;
    return x;
}

// Walsh-Hadamard transform (unnormalised, natural order) of a D-vector spread over a warp:
// lane l holds x[k] = v[l + 32 k].  Strides below 32 pair lanes, larger strides pair slots.
template <int D>
__device__ __forceinline__ void warp_fwht(float (&x)[D / 32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
            const float o = __shfl_xor_sync(0xffffffffu, x[k], h);
            x[k] = (lane & h) ? (o - x[k]) : (x[k] + o);
        }
    }
#pragma unroll
    for (int h = 1; h < D / 32; h <<= 1) {
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
            if (k & h) continue;
            const float a = x[k], b = x[k + h];
            x[k] = a + b;
            x[k + h] = a - b;
        }
    }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Power-of-two prescale that brings max|x| into [2^14, 2^15), so the fp16 copy of the rotated
// query neither overflows nor loses precision to subnormals.  Returns the exponent e (x * 2^e).
__device__ __forceinline__ int prescale_exponent(float maxabs) {
    if (!(maxabs > 0.0f)) return 0;
    const int ex = (int)((__float_as_uint(maxabs) >> 23) & 0xFF) - 127;
    int e = 14 - ex;
    return e < -100 ? -100 : (e > 100 ? 100 : e);
}

__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Walsh-Hadamard transform of NB vectors of one warp at once (vector k: lane l holds
// x[k][j] = v_k[l + 32 j]).  The butterfly stages of the NB vectors interleave, so the warp pays
// one chain of shuffle latencies instead of NB.
template <int D, int NB>
__device__ __forceinline__ void warp_fwht_batch(float (&x)[NB][D / 32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int k = 0; k < NB; ++k) {
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const float o = __shfl_xor_sync(0xffffffffu, x[k][j], h);
                x[k][j] = (lane & h) ? (o - x[k][j]) : (x[k][j] + o);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < NB; ++k) {
#pragma unroll
        for (int h = 1; h < D / 32; h <<= 1) {
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                if (j & h) continue;
                const float a = x[k][j], b = x[k][j + h];
                x[k][j] = a + b;
                x[k][j + h] = a - b;
            }
        }
    }
}

// fp32 pair -> (hi, lo) fp16x2 pairs with hi + lo ~ the pair to about 22 bits.
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_f16x2(a, b);
    const __half2 h = *reinterpret_cast<const __half2*>(&hi);
    const float2 hf = __half22float2(h);
    lo = pack_f16x2(a - hf.x, b - hf.y);
}

// fp32 -> (hi, lo) fp16 halves of one value in one register (hi in the low 16 bits), hi + lo ~ x
// to about 22 bits.
__device__ __forceinline__ uint32_t hi_lo_f16x2(float x) {
    const __half hi = __float2half_rn(x);
    const __half lo = __float2half_rn(x - __half2float(hi));
    return (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
}

// Un-rotate an accumulated output vector held by a warp (lane l: x[k] = o[l + 32 k]) and store it:
// out = c * D * H_d * (o * inv_l).
template <int D, typename OT>
__device__ __forceinline__ void unrotate_store(float (&x)[D / 32], float inv_l, const float* sgn, float c, void* out,
                                               int64_t ooff) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) x[k] *= inv_l;
    warp_fwht<D>(x);
#pragma unroll
    for (int k = 0; k < D / 32; ++k) store_elem<OT>(out, ooff + lane + 32 * k, x[k] * c * sgn[lane + 32 * k]);
}

}  // namespace kvi4
