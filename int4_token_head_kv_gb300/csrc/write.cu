// Cache write of the INT4 per-(token, head) KV cache: random Hadamard rotation, asymmetric 4-bit
// quantisation with the zero-point hidden in the scale's low mantissa bits, nibble packing and a
// paged store ("[Feature] Triton INT4 / INT2 per-token-head KV cache quantization", description;
// "PR #40835 report", get_kv_cache_shape).
//
// One thread encodes one (token, head, plane) vector entirely in registers.  Every arithmetic step
// is an explicit round-to-nearest-even operation (intrinsics or packed fp32x2 PTX), so the bytes
// are bit-exact with the definition in kv_int4.h regardless of how the compiler schedules them:
//   butterflies at strides 1, 2, ..., D/2 (fixed order) -> multiply by c -> min/max ->
//   s = (max - min) / 15 floored at 1e-6 -> s' = s with the low 4 mantissa bits cleared ->
//   zp = clamp(rint(-min / s'), 0, 15) -> code = clamp(N(y * (1/s') + zp), 0, 15).
// The last step uses one fused multiply-add against 1.5 * 2^23 + zp: the sum lands in
// [2^23, 2^24) where the fp32 spacing is 1, so the single rounding of the FMA is exactly the
// nearest-even integer of the real value y * r + zp, and the code sits in the low mantissa bits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device.cuh"

namespace kvi4 {
namespace {

constexpr int kWriteThreads = 128;
constexpr float kRoundMagic = 12582912.0f;        // 1.5 * 2^23
constexpr uint32_t kRoundMagicBits = 0x4B400000u;

// Upcast a pair of 16-bit floats (low half = even element) to fp32, exactly.
template <typename T>
__device__ __forceinline__ float2 upcast_pair(uint32_t w);

template <>
__device__ __forceinline__ float2 upcast_pair<__nv_bfloat16>(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

template <>
__device__ __forceinline__ float2 upcast_pair<__half>(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

template <int D, typename T>
__global__ void __launch_bounds__(kWriteThreads) write_kernel(const __grid_constant__ WriteParams p) {
    using Gm = Geo<D>;
    // Sign flips as XOR masks on pairs of 16-bit inputs (the sign bit is bit 15 of each half in
    // both fp16 and bf16).
    __shared__ uint32_t sign_mask[D / 2];
    for (int j = threadIdx.x; j < D / 2; j += blockDim.x) {
        const float s0 = p.signs[2 * j], s1 = p.signs[2 * j + 1];
        sign_mask[j] = ((__float_as_uint(s0) >> 31) << 15) | ((__float_as_uint(s1) >> 31) << 31);
        if (blockIdx.x == 0 && ((fabsf(s0) != 1.0f) || (fabsf(s1) != 1.0f))) count_status(p.status, 4);
    }
    __syncthreads();

    const int H = p.H;
    const int64_t nvec = p.num_tokens * H * 2;
    for (int64_t vi = (int64_t)blockIdx.x * kWriteThreads + threadIdx.x; vi < nvec;
         vi += (int64_t)gridDim.x * kWriteThreads) {
        // vi = (t * 2 + plane) * H + h: a warp writes whole contiguous (token, plane) rows
        const int h = (int)(vi % H);
        const int64_t tp = vi / H;
        const int plane = (int)(tp & 1);
        const int64_t t = tp >> 1;
        const int64_t slot = __ldg(p.slots + t);
        if (slot < 0) continue;
        if (slot >= p.num_slots) {
            if (plane == 0 && h == 0) count_status(p.status, 0);
            continue;
        }

        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(plane ? p.v : p.k) +
                                                          (t * H + h) * D);
        float u[D];
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 q = __ldg(src + c);
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = c * 4 + e;
                const float2 x = upcast_pair<T>(w4[e] ^ sign_mask[j]);
                // stride-1 butterfly straight from the pair
                u[2 * j] = __fadd_rn(x.x, x.y);
                u[2 * j + 1] = __fsub_rn(x.x, x.y);
            }
        }
        // strides 2 .. D/2, two lanes at a time
#pragma unroll
        for (int hs = 2; hs < D; hs <<= 1) {
#pragma unroll
            for (int i = 0; i < D; i += 2) {
                if (i & hs) continue;
                const float2 a = make_float2(u[i], u[i + 1]);
                const float2 b = make_float2(u[i + hs], u[i + hs + 1]);
                const float2 s = add_f32x2(a, b);
                const float2 d = sub_f32x2(a, b);
                u[i] = s.x;
                u[i + 1] = s.y;
                u[i + hs] = d.x;
                u[i + hs + 1] = d.y;
            }
        }
        const float2 c2 = make_float2(p.c, p.c);
#pragma unroll
        for (int i = 0; i < D; i += 2) {
            const float2 y = mul_f32x2(make_float2(u[i], u[i + 1]), c2);
            u[i] = y.x;
            u[i + 1] = y.y;
        }
        // min / max over the rotated vector (exact)
        float mx0 = u[0], mx1 = u[1], mn0 = u[0], mn1 = u[1];
#pragma unroll
        for (int i = 2; i < D; i += 4) {
            mx0 = max3(mx0, u[i], u[i + 1]);
            mn0 = min3(mn0, u[i], u[i + 1]);
            if (i + 3 < D) {
                mx1 = max3(mx1, u[i + 2], u[i + 3]);
                mn1 = min3(mn1, u[i + 2], u[i + 3]);
            }
        }
        const float mx = fmaxf(mx0, mx1), mn = fminf(mn0, mn1);
        float s = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
        if (!(s >= 1e-6f)) s = 1e-6f;
        const uint32_t sb = __float_as_uint(s) & 0xFFFFFFF0u;
        const float sp = __uint_as_float(sb);
        const float zr = rintf(__fdiv_rn(-mn, sp));
        const uint32_t zp = zr < 0.0f ? 0u : (zr > 15.0f ? 15u : (uint32_t)zr);
        const float r = __frcp_rn(sp);
        const float zpm = kRoundMagic + (float)zp;   // exact
        // The map y -> RN(y * r + zpm) is monotone, so the codes of min and max bound all codes:
        // clamping is needed only when one of them falls outside [0, 15].
        const float lo = __fmaf_rn(mn, r, zpm), hi = __fmaf_rn(mx, r, zpm);
        const bool clamp = !(lo >= kRoundMagic && hi <= kRoundMagic + 15.0f);
        const float2 r2 = make_float2(r, r), z2 = make_float2(zpm, zpm);

        uint32_t words[Gm::KW];
#pragma unroll
        for (int wi = 0; wi < Gm::KW; ++wi) {
            uint32_t acc = 0;
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                float2 f = fma_f32x2(make_float2(u[wi * 8 + k], u[wi * 8 + k + 1]), r2, z2);
                if (clamp) {
                    f.x = fminf(fmaxf(f.x, kRoundMagic), kRoundMagic + 15.0f);
                    f.y = fminf(fmaxf(f.y, kRoundMagic), kRoundMagic + 15.0f);
                }
                acc += (__float_as_uint(f.x) << (4 * k)) + (__float_as_uint(f.y) << (4 * k + 4));
            }
            // each term carried kRoundMagicBits << 4k; their sum modulo 2^32 is 0x3F400000
            words[wi] = acc - 0x3F400000u;
        }

        const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
        uint32_t* row = reinterpret_cast<uint32_t*>(p.cache + (((blk * 2 + plane) * kBlockSize + off) * H + h) * Gm::RB);
#pragma unroll
        for (int wi = 0; wi < Gm::KW; ++wi) row[wi] = words[wi];
        row[Gm::KW] = sb | zp;
    }
    (void)kRoundMagicBits;
}

template <int D, typename T>
cudaError_t launch_write_t(const WriteParams& p, cudaStream_t stream) {
    const int64_t nvec = p.num_tokens * p.H * 2;
    int64_t blocks = (nvec + kWriteThreads - 1) / kWriteThreads;
    const int64_t cap = (int64_t)num_sms() * 64;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    write_kernel<D, T><<<(unsigned)blocks, kWriteThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_write(const WriteParams& p, int head_size, DType dt, cudaStream_t stream) {
    if (head_size == 128) {
        return dt == DType::BF16 ? launch_write_t<128, __nv_bfloat16>(p, stream) : launch_write_t<128, __half>(p, stream);
    }
    return dt == DType::BF16 ? launch_write_t<64, __nv_bfloat16>(p, stream) : launch_write_t<64, __half>(p, stream);
}

}  // namespace kvi4
