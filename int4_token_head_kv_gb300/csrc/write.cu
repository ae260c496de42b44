// Cache write of the INT4 per-(token, head) KV cache: random Hadamard rotation, asymmetric 4-bit
// quantisation with the zero-point hidden in the scale's low mantissa bits, nibble packing and a
// paged store ("[Feature] Triton INT4 / INT2 per-token-head KV cache quantization", description;
// "PR #40835 report", get_kv_cache_shape).
//
// Two threads (a lane pair) encode one (token, head, plane) vector in registers.  Every arithmetic
// step is an explicit round-to-nearest-even operation (intrinsics, packed fp32x2 builtins, or a
// mixed-precision FMA that reads a bf16 input in place: fp32 result, one rounding), so the bytes
// are bit-exact with the definition in kv_int4.h regardless of how the compiler schedules them:
//   butterflies at strides 1, 2, ..., D/2 (fixed order) -> multiply by c -> min/max ->
//   s = (max - min) / 15 floored at 1e-6 -> s' = s with the low 4 mantissa bits cleared ->
//   zp = clamp(rint(-min / s'), 0, 15) -> code = clamp(N(y * (1/s') + zp), 0, 15).
// The last step uses one fused multiply-add against 1.5 * 2^23 + zp: the sum lands in
// [2^23, 2^24) where the fp32 spacing is 1, so the single rounding of the FMA is exactly the
// nearest-even integer of the real value y * r + zp, and the code sits in the low mantissa bits.
//
// The lane pair splits the vector by the parity of the element index after the stride-1
// butterflies: thread t keeps elements 2m + t.  Each thread forms its own stride-1 outputs straight
// from the inputs (a + b for t = 0, a - b for t = 1), and every later stride pairs two elements of
// the same parity, so the rest of the rotation needs no exchange.  Only the min/max and the code
// bytes (whose two nibbles come from the two threads) cross the pair.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

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

// Sign tables of the half-vector encoder (shared memory, built once per CTA):
//   xmask[t][m]  XOR mask for input pair m and element parity t: bit 31 = sign of element 2m + 1
//                times (t ? -1 : +1); bit 15 = sign of element 2m for fp16 inputs (bf16 inputs take
//                it from esign[]);
//   esign[k + i] (k a multiple of 4) the signs of elements 2m and 2m + 2 as bf16 +-1.0 (low, high
//                half), m = k + 2(i & 1) in the first half of the pairs (i < 2) or the second
//                (i >= 2, m + D/4): one 16-byte load gives the even signs of pairs k .. k + 3 of both.
template <int D>
struct WriteSigns {
    uint32_t xmask[2][D / 2];
    uint32_t esign[D / 4];
};

// RN(a * b + c) with a the low bf16 half of a2, b the low (HI_B false) or high bf16 half of b2 and c
// fp32, in one mixed-precision FMA: the bf16 operands are read in place, with no upcast.  With b =
// +-1 the product is exact and the one rounding is that of the fp32 sum.
template <bool HI_B>
__device__ __forceinline__ float fma_bf16_lo(uint32_t a2, uint32_t b2, float c) {
    float d;
    if constexpr (!HI_B)
        asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2; fma.rn.f32.bf16 %0, al, bl, %3; }"
            : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    else
        asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2; fma.rn.f32.bf16 %0, al, bh, %3; }"
            : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    return d;
}

// One thread's half of a rotated vector.  row: the vector's D/2 input pairs (pair m = elements 2m,
// 2m + 1, low half first) in shared memory; t: this thread's element parity.  With Q = D/4, thread t
// ends with P[k] = (y_{2k+t}, y_{2(k+Q)+t}) in a register pair.  A butterfly at stride 2s (s < Q) of
// the element index pairs local m with m + s, i.e. P[k] with P[k + s] lane by lane; the stride D/2
// pairs the two lanes of P[k].
template <int D, typename T>
__device__ __forceinline__ void rotate_half(const uint32_t* row, const WriteSigns<D>& sg, int t, float c,
                                            float2 (&P)[D / 4]) {
    constexpr int Q = D / 4;
    const uint32_t* xm = sg.xmask[t];
    // stride 1: u_{2m+t} = a_m + (t ? -1 : 1) b_m, (a_m, b_m) = the sign-flipped input pair m
#pragma unroll
    for (int k = 0; k < Q; k += 4) {
        const uint4 lo = *reinterpret_cast<const uint4*>(row + k);
        const uint4 hi = *reinterpret_cast<const uint4*>(row + k + Q);
        const uint4 mlo = *reinterpret_cast<const uint4*>(xm + k);
        const uint4 mhi = *reinterpret_cast<const uint4*>(xm + k + Q);
        const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w}, wh[4] = {hi.x, hi.y, hi.z, hi.w};
        const uint32_t ml[4] = {mlo.x, mlo.y, mlo.z, mlo.w}, mh[4] = {mhi.x, mhi.y, mhi.z, mhi.w};
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            // odd element: its sign (and the parity's -1) by XOR while masking out the even half (one
            // logic op); even element: read in place by a mixed-precision FMA with its bf16 sign
            const uint4 es = *reinterpret_cast<const uint4*>(sg.esign + k);
            auto odd = [](uint32_t w, uint32_t m) { return __uint_as_float((w ^ m) & 0xFFFF0000u); };
            P[k] = make_float2(fma_bf16_lo<false>(wl[0], es.x, odd(wl[0], ml[0])),
                               fma_bf16_lo<false>(wh[0], es.z, odd(wh[0], mh[0])));
            P[k + 1] = make_float2(fma_bf16_lo<true>(wl[1], es.x, odd(wl[1], ml[1])),
                                   fma_bf16_lo<true>(wh[1], es.z, odd(wh[1], mh[1])));
            P[k + 2] = make_float2(fma_bf16_lo<false>(wl[2], es.y, odd(wl[2], ml[2])),
                                   fma_bf16_lo<false>(wh[2], es.w, odd(wh[2], mh[2])));
            P[k + 3] = make_float2(fma_bf16_lo<true>(wl[3], es.y, odd(wl[3], ml[3])),
                                   fma_bf16_lo<true>(wh[3], es.w, odd(wh[3], mh[3])));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 xa = upcast_pair<T>(wl[e] ^ ml[e]);
                const float2 xb = upcast_pair<T>(wh[e] ^ mh[e]);
                P[k + e] = add_f32x2(make_float2(xa.x, xb.x), make_float2(xa.y, xb.y));
            }
        }
    }
    // strides 2, 4, ..., D/4 of the element index
#pragma unroll
    for (int st = 1; st < Q; st <<= 1) {
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            if (k & st) continue;
            const float2 a = P[k], b = P[k + st];
            P[k] = add_f32x2(a, b);
            P[k + st] = sub_f32x2(a, b);
        }
    }
    // stride D/2, then the normalisation
    const float2 c2 = make_float2(c, c);
#pragma unroll
    for (int k = 0; k < Q; ++k)
        P[k] = mul_f32x2(make_float2(__fadd_rn(P[k].x, P[k].y), __fsub_rn(P[k].x, P[k].y)), c2);
}

// One thread's half of an INT4 vector: the rotation, then the Q/4 code words this thread stores
// (t = 0: words 0 .. Q/4 - 1; t = 1: words Q/4 .. Q/2 - 1) and the scale word.
template <int D, typename T>
__device__ __forceinline__ void encode_half(const uint32_t* row, const WriteSigns<D>& sg, int t, float c,
                                            uint32_t (&out)[D / 16 + 1]) {
    constexpr int Q = D / 4;
    float2 P[Q];
    rotate_half<D, T>(row, sg, t, c, P);
    // min / max over the rotated vector (exact): this half, then the other
    float mx0 = P[0].x, mx1 = P[0].y, mn0 = P[0].x, mn1 = P[0].y;
#pragma unroll
    for (int k = 1; k < Q; k += 2) {
        mx0 = max3(mx0, P[k].x, P[k].y);
        mn0 = min3(mn0, P[k].x, P[k].y);
        if (k + 1 < Q) {
            mx1 = max3(mx1, P[k + 1].x, P[k + 1].y);
            mn1 = min3(mn1, P[k + 1].x, P[k + 1].y);
        }
    }
    float mx = fmaxf(mx0, mx1), mn = fminf(mn0, mn1);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
    float s = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    if (!(s >= 1e-6f)) s = 1e-6f;
    const uint32_t sb = __float_as_uint(s) & 0xFFFFFFF0u;
    const float sp = __uint_as_float(sb);
    const float zr = rintf(__fdiv_rn(-mn, sp));
    const uint32_t zp = zr < 0.0f ? 0u : (zr > 15.0f ? 15u : (uint32_t)zr);
    const float r = __frcp_rn(sp);
    const float zpm = kRoundMagic + (float)zp;   // exact
    // The map y -> RN(y * r + zpm) is monotone, so the codes of min and max bound all codes:
    // clamping is needed only when one of them falls outside [0, 15] (rare: a one-signed vector),
    // and clamping codes already in range changes nothing, so the warp clamps all or none.
    const float lo = __fmaf_rn(mn, r, zpm), hi = __fmaf_rn(mx, r, zpm);
    const bool clamp = __any_sync(0xffffffffu, !(lo >= kRoundMagic && hi <= kRoundMagic + 15.0f));
    const float2 r2 = make_float2(r, r), z2 = make_float2(zpm, zpm);
    float2 f[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) f[k] = fma_f32x2(P[k], r2, z2);
    if (clamp) {
#pragma unroll
        for (int k = 0; k < Q; ++k) {
            f[k].x = fminf(fmaxf(f[k].x, kRoundMagic), kRoundMagic + 15.0f);
            f[k].y = fminf(fmaxf(f[k].y, kRoundMagic), kRoundMagic + 15.0f);
        }
    }
    // Element 2m + t is the nibble 4t of row byte m, byte m % 4 of word m / 4: f[k].x (m = k) goes
    // to word k / 4, f[k].y (m = k + Q) to word Q / 4 + k / 4.  A code's float has bits
    // 0x4B400000 + code; four of them at bytes 0..3 (multiply-adds) sum to 0x8B400000 + the codes
    // (mod 2^32), and the word is then moved up by 4t nibble bits: (sum - 0x8B400000) * 16^t.
    const uint32_t mul = t ? 16u : 1u;
    const uint32_t cst = t ? 0x4C000000u : 0x74C00000u;   // -(0x8B400000 * 16^t) mod 2^32
    uint32_t xw[Q / 4], yw[Q / 4];
#pragma unroll
    for (int w = 0; w < Q / 4; ++w) {
        const float2* g = f + 4 * w;
        const uint32_t ax = __float_as_uint(g[0].x) + __float_as_uint(g[1].x) * 256u +
                            __float_as_uint(g[2].x) * 65536u + __float_as_uint(g[3].x) * 16777216u;
        const uint32_t ay = __float_as_uint(g[0].y) + __float_as_uint(g[1].y) * 256u +
                            __float_as_uint(g[2].y) * 65536u + __float_as_uint(g[3].y) * 16777216u;
        xw[w] = ax * mul + cst;
        yw[w] = ay * mul + cst;
    }
    // thread 0 finishes the first half of the row's words, thread 1 the second: each sends the
    // other the nibbles it holds of the other's words
#pragma unroll
    for (int w = 0; w < Q / 4; ++w) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, t ? xw[w] : yw[w], 1);
        out[w] = (t ? yw[w] : xw[w]) | other;
    }
    out[Q / 4] = sb | zp;
}

// INT2 Lloyd-Max mode ("[Feature] Triton INT4 / INT2 per-token-head KV cache quantization",
// description: four 2-bit codes per byte, Hadamard pre-rotation, centroids of the 4-level Lloyd-Max
// quantiser of N(0, 1)).  After the INT4 mode's rotation, per vector:
//   sigma = max(sqrt(fp32(sum y_i^2) / D), 1e-6), the sum of the fp32 squares folded in halves
//   (a_i + a_{i + D/2}, then + a_{i + D/4}, ...); r = fp32(1 / sigma); z_i = fp32(y_i * r);
//   code_i = [z_i >= -t] + [z_i >= 0] + [z_i >= t]   (codes 0..3 stand for -b, -a, a, b)
// stored as D/4 bytes (element 4j + k in bits 2k of byte j), then the bits of sigma.
// Lloyd-Max outputs a, b and threshold t = (a + b) / 2 of N(0, 1) (J. Max, 1960), fp32-rounded.
constexpr float kLmA = 0x1.cfa592p-2f;    // 0.45278
constexpr float kLmB = 0x1.82aabap+0f;    // 1.51042
constexpr float kLmT = 0x1.f6941ep-1f;    // 0.98160

// Thread t's half (elements of parity t): P[k] holds elements 2k + t and 2(k + Q) + t, so the fold
// strides D/2 .. 2 stay in the thread (P[k].x with P[k].y, then s[k] with s[k + h]) and the last
// (elements 0 and 1) pairs the two threads.  Element 2m + t is field 2(m & 1) + t of byte m >> 1:
// the .x elements fill bytes 0 .. Q/2 - 1 (words 0 .. Q/8 - 1), the .y elements the rest.
template <int D, typename T>
__device__ __forceinline__ void encode_half_int2(const uint32_t* row, const WriteSigns<D>& sg, int t, float c,
                                                 uint32_t (&out)[D / 32 + 1]) {
    constexpr int Q = D / 4;
    float2 P[Q];
    rotate_half<D, T>(row, sg, t, c, P);
    float sq[Q];
#pragma unroll
    for (int k = 0; k < Q; ++k) sq[k] = __fadd_rn(__fmul_rn(P[k].x, P[k].x), __fmul_rn(P[k].y, P[k].y));
#pragma unroll
    for (int h = Q / 2; h >= 1; h >>= 1) {
#pragma unroll
        for (int k = 0; k < h; ++k) sq[k] = __fadd_rn(sq[k], sq[k + h]);
    }
    const float sum = __fadd_rn(sq[0], __shfl_xor_sync(0xffffffffu, sq[0], 1));
    float sigma = __fsqrt_rn(__fmul_rn(sum, 1.0f / (float)D));   // the power-of-two product is exact
    if (!(sigma >= 1e-6f)) sigma = 1e-6f;
    const float r = __frcp_rn(sigma);
    // two codes per element pair m = 2j, 2j + 1 of a byte: fields t and 2 + t
    auto code = [&](float y) -> uint32_t {
        const float z = __fmul_rn(y, r);
        return (uint32_t)(z >= -kLmT) + (uint32_t)(z >= 0.0f) + (uint32_t)(z >= kLmT);
    };
    uint32_t xw[Q / 8], yw[Q / 8];
#pragma unroll
    for (int w = 0; w < Q / 8; ++w) {
        uint32_t ax = 0, ay = 0;
#pragma unroll
        for (int by = 0; by < 4; ++by) {
            const int m = 2 * (4 * w + by);   // the byte's first element pair index
            ax |= (code(P[m].x) | (code(P[m + 1].x) << 4)) << (8 * by);
            ay |= (code(P[m].y) | (code(P[m + 1].y) << 4)) << (8 * by);
        }
        const uint32_t sh = 2u * (uint32_t)t;
        xw[w] = ax << sh;
        yw[w] = ay << sh;
    }
#pragma unroll
    for (int w = 0; w < Q / 8; ++w) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, t ? xw[w] : yw[w], 1);
        out[w] = (t ? yw[w] : xw[w]) | other;
    }
    out[Q / 8] = __float_as_uint(sigma);
    (void)kLmA;
    (void)kLmB;
}

// INT8 per-(token, head) comparator ("tests/quantization/test_per_token_kv_cache.py",
// _quantize_per_token_head_ref with INT8_CONFIG; rounding as in the INT8 reshape-kernel fix of
// "[Feature] Triton INT4 / INT2 per-token-head KV cache quantization"): no rotation, no zero-point,
//   s = max(fp32(max|x| / 127), 1e-6); r = fp32(1 / s);
//   q = clamp(trunc(fp32(fp32(x * r) + (x * r >= 0 ? 0.5 : -0.5))), -128, 127),
// stored as D two's-complement bytes then the bits of s.
template <int D, typename T>
__device__ __forceinline__ void load_vector_raw(const uint4* src, float (&u)[D]) {
#pragma unroll
    for (int cc = 0; cc < D / 8; ++cc) {
        const uint4 q = src[cc];
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = upcast_pair<T>(w4[e]);
            u[2 * (cc * 4 + e)] = x.x;
            u[2 * (cc * 4 + e) + 1] = x.y;
        }
    }
}

template <int D>
__device__ __forceinline__ void encode_vector_int8(const float (&u)[D], uint32_t (&words)[D / 4 + 1]) {
    float a0 = fabsf(u[0]), a1 = fabsf(u[1]);
#pragma unroll
    for (int i = 2; i < D; i += 4) {
        a0 = max3(a0, fabsf(u[i]), fabsf(u[i + 1]));
        if (i + 3 < D) a1 = max3(a1, fabsf(u[i + 2]), fabsf(u[i + 3]));
    }
    float s = __fdiv_rn(fmaxf(a0, a1), 127.0f);
    if (!(s >= 1e-6f)) s = 1e-6f;
    const float r = __frcp_rn(s);
#pragma unroll
    for (int wi = 0; wi < D / 4; ++wi) {
        uint32_t w = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float v = __fmul_rn(u[wi * 4 + k], r);
            int c = __float2int_rz(__fadd_rn(v, v >= 0.0f ? 0.5f : -0.5f));
            c = c < -128 ? -128 : (c > 127 ? 127 : c);
            w |= ((uint32_t)c & 0xFFu) << (8 * k);
        }
        words[wi] = w;
    }
    words[D / 4] = __float_as_uint(s);
}

// Work split: vectors are numbered v = (t * 2 + plane) * H + h, so H consecutive vectors are one
// (token, plane) row group, contiguous in the cache.  Each warp owns tiles of TV consecutive vectors
// (TV = 32 / threads per vector: 16 for INT4, 32 for INT8) and works through them on its own (no
// CTA-wide barriers): it prefetches the next tile's inputs, one bulk async copy of 2D bytes per
// vector completing on the buffer's mbarrier, into one of two padded shared-memory buffers (row
// stride 2D + 16 bytes, so the 16-byte reads of 8 neighbouring rows hit distinct banks), encodes the
// current tile, stages the encoded rows in the buffer it just read, and writes each row group with
// one bulk async store (when H divides TV and a group is a multiple of 16 bytes; otherwise each
// thread stores its own words).
constexpr int kWriteWarps = kWriteThreads / 32;

template <int D, int TV>
struct WriteSmem {
    static constexpr int kRowPad = 2 * D + 16;
    static constexpr int kBuf = TV * kRowPad;                   // one tile of inputs
    static constexpr int kPerWarp = 2 * kBuf;
    static constexpr int kBars = kWriteWarps * kPerWarp;        // two mbarriers per warp
    static constexpr int kBytes = kBars + kWriteWarps * 2 * 8 + (int)sizeof(WriteSigns<D>);
};


__device__ __forceinline__ void bulk_store_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Vector index -> (row of K/V, plane) with 32-bit arithmetic; shifts when H is a power of two.
struct VecIndex {
    uint32_t H, hmask;
    int hshift;   // -1: H is not a power of two
    __device__ __forceinline__ void split(uint32_t v, uint32_t& token, uint32_t& h, uint32_t& plane) const {
        uint32_t tp;
        if (hshift >= 0) {
            h = v & hmask;
            tp = v >> hshift;
        } else {
            tp = v / H;
            h = v - tp * H;
        }
        plane = tp & 1u;
        token = tp >> 1;
    }
};

// BITS: 4 the INT4 cache, 8 the INT8 comparator, 2 the INT2 Lloyd-Max mode.
template <int BITS>
struct WriteShape {
    static constexpr int kTpv = BITS == 8 ? 1 : 2;          // threads per vector
    static constexpr int kTileVecs = 32 / kTpv;             // vectors per warp tile
    static constexpr int kMinBlocks = BITS == 8 ? 3 : 5;    // resident CTAs per SM (register budget)
};

template <int D, typename T, int BITS>
__global__ void __launch_bounds__(kWriteThreads, WriteShape<BITS>::kMinBlocks)
    write_kernel(const __grid_constant__ WriteParams p) {
    using Gm = Geo<D>;
    using Sh = WriteShape<BITS>;
    constexpr bool INT8 = BITS == 8;
    constexpr int TPV = Sh::kTpv, TV = Sh::kTileVecs;
    constexpr int RB = INT8 ? D + 4 : (BITS == 2 ? D / 4 + 4 : Gm::RB);   // cache row bytes
    constexpr int NW = RB / 4 - 1;                                       // code words per row (then the scale)
    constexpr int OW = INT8 ? NW + 1 : NW / 2 + 1;   // words one thread stores (the last: the scale word)
    using Sm = WriteSmem<D, TV>;
    extern __shared__ __align__(128) uint8_t smem[];
    // Launched as a programmatic dependent: wait for the previous kernel of the stream (it may
    // produce K, V or the slots), then let the next kernel start its own set-up.
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vl = lane / TPV, part = lane % TPV;   // this thread's vector of the tile and its part
    uint8_t* wbuf = smem + warp * Sm::kPerWarp;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::kBars) + warp * 2;   // this warp's [buffer]
    WriteSigns<D>& sgn = *reinterpret_cast<WriteSigns<D>*>(smem + Sm::kBars + kWriteWarps * 2 * 8);
    if (lane == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    for (int j = tid; j < (INT8 ? 0 : D / 2); j += kWriteThreads) {   // INT8 rows take no signs
        const float s0 = p.signs[2 * j], s1 = p.signs[2 * j + 1];
        // bf16 takes the even sign in the FMA (its mask flips only the odd element); fp16 in the XOR
        const uint32_t m = ((std::is_same<T, __nv_bfloat16>::value ? 0u : (__float_as_uint(s0) >> 31)) << 15) |
                           ((__float_as_uint(s1) >> 31) << 31);
        sgn.xmask[0][j] = m;
        sgn.xmask[1][j] = m ^ 0x80000000u;
        if ((j & 1) == 0) {   // the bf16 signs of elements 2j and 2j + 2
            const float s2 = p.signs[2 * j + 2];
            const int kk = j % (D / 4), half = j / (D / 4);
            sgn.esign[(kk & ~3) + ((kk >> 1) & 1) + 2 * half] =
                (s0 < 0.0f ? 0xBF80u : 0x3F80u) | ((s2 < 0.0f ? 0xBF80u : 0x3F80u) << 16);
        }
        if (blockIdx.x == 0 && ((fabsf(s0) != 1.0f) || (fabsf(s1) != 1.0f))) count_status(p.status, 4);
    }
    __syncthreads();

    const uint32_t H = (uint32_t)p.H;
    VecIndex vx;
    vx.H = H;
    vx.hmask = H - 1;
    vx.hshift = (H & (H - 1)) == 0 ? __ffs(H) - 1 : -1;
    const uint32_t nvec = (uint32_t)(p.num_tokens * H * 2);
    const uint32_t ntiles = (nvec + TV - 1) / TV;
    const uint32_t gwarp = blockIdx.x * kWriteWarps + warp, nwarps = gridDim.x * kWriteWarps;
    const uint32_t group_bytes = H * RB;
    const bool grouped = vx.hshift >= 0 && H <= (uint32_t)TV && (group_bytes % 16) == 0;
    const uint8_t* kin = static_cast<const uint8_t*>(p.k);
    const uint8_t* vin = static_cast<const uint8_t*>(p.v);

    // lane i < TV copies vector i of the tile (2D bytes) into row i of the buffer
    auto prefetch = [&](uint32_t tile, uint8_t* buf, uint64_t* bar) {
        const uint32_t v0 = tile * TV;
        const uint32_t live_vecs = min((uint32_t)TV, nvec - v0);
        if (lane == 0) mbar_arrive_expect_tx(bar, live_vecs * (uint32_t)(D * 2));
        __syncwarp();
        if ((uint32_t)lane < live_vecs) {
            uint32_t tok, h, pl;
            vx.split(v0 + lane, tok, h, pl);
            bulk_copy_g2s(buf + lane * Sm::kRowPad, (pl ? vin : kin) + (uint64_t)(tok * H + h) * (D * 2), D * 2, bar,
                          policy_evict_first());
        }
    };

    uint32_t tile = gwarp;
    int it = 0;
    bool waited_out = false;
    if (tile < ntiles) prefetch(tile, wbuf, &bars[0]);
    for (; tile < ntiles; tile += nwarps, ++it) {
        uint8_t* cur = wbuf + (it & 1) * Sm::kBuf;
        uint8_t* nxt = wbuf + ((it + 1) & 1) * Sm::kBuf;
        // the other buffer was last an output stage: its bulk stores must have read it
        if (grouped) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
        if (tile + nwarps < ntiles) prefetch(tile + nwarps, nxt, &bars[(it + 1) & 1]);
        // this tile's rows: use (it >> 1) of buffer it & 1
        if (__any_sync(0xffffffffu, !mbar_wait(&bars[it & 1], (uint32_t)(it >> 1) & 1u))) {
            if (lane == 0) count_status(p.status, 3);
            waited_out = true;
            break;
        }
        const uint32_t v = tile * TV + vl;
        const bool live = v < nvec;
        uint32_t words[OW];
        if constexpr (INT8) {
            float u[D];
            if (live) load_vector_raw<D, T>(reinterpret_cast<const uint4*>(cur + vl * Sm::kRowPad), u);
            __syncwarp();   // the tile's inputs are in registers; its buffer becomes the output stage
            if (live) encode_vector_int8<D>(u, words);
        } else {
            // every lane runs the encoder (it exchanges values within the lane pair); a vector past
            // the end reads row 0, which every tile holds, and its words are discarded
            const uint32_t* in = reinterpret_cast<const uint32_t*>(cur + (live ? vl : 0) * Sm::kRowPad);
            if constexpr (BITS == 2) encode_half_int2<D, T>(in, sgn, part, p.c, words);
            else encode_half<D, T>(in, sgn, part, p.c, words);
            __syncwarp();   // the tile's inputs are consumed; its buffer becomes the output stage
        }
        // this thread's words of the row: all of them (INT8), or the first / second half of the code
        // words (INT4 / INT2 parts 0 / 1; part 1 also the scale word)
        const int w0 = INT8 ? 0 : part * (NW / 2);
        const int nw = INT8 ? OW : (part ? OW : OW - 1);
        uint32_t tok = 0, h = 0, pl = 0;
        if (live) vx.split(v, tok, h, pl);
        if (grouped) {
            uint32_t* orow = reinterpret_cast<uint32_t*>(cur + vl * RB) + w0;
            if (live) {
#pragma unroll
                for (int wi = 0; wi < OW; ++wi)
                    if (wi < nw) orow[wi] = words[wi];
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // staged rows -> bulk store
            __syncwarp();
            // the first thread of each row group stores the whole group
            if (live && h == 0 && part == 0) {
                const int64_t slot = __ldg(p.slots + tok);
                if (slot >= p.num_slots) {
                    if (pl == 0) count_status(p.status, 0);
                } else if (slot >= 0) {
                    const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
                    bulk_store_s2g(p.cache + ((blk * 2 + pl) * kBlockSize + off) * (int64_t)group_bytes,
                                   cur + vl * RB, group_bytes);
                }
            }
        } else if (live) {
            const int64_t slot = __ldg(p.slots + tok);
            if (slot >= p.num_slots) {
                if (pl == 0 && h == 0 && part == 0) count_status(p.status, 0);
            } else if (slot >= 0) {
                const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
                uint32_t* row =
                    reinterpret_cast<uint32_t*>(p.cache + (((blk * 2 + pl) * kBlockSize + off) * H + h) * RB) + w0;
#pragma unroll
                for (int wi = 0; wi < OW; ++wi)
                    if (wi < nw) row[wi] = words[wi];
            }
        }
    }
    if (waited_out && tile + nwarps < ntiles) {   // let the copy in flight land before the warp exits
        (void)mbar_wait(&bars[(it + 1) & 1], (uint32_t)((it + 1) >> 1) & 1u);
    }
    if (grouped) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    (void)kRoundMagicBits;
}

template <int D, typename T, int BITS>
cudaError_t launch_write_t(const WriteParams& p, cudaStream_t stream) {
    using Sh = WriteShape<BITS>;
    using Sm = WriteSmem<D, Sh::kTileVecs>;
    const int64_t ntiles = (p.num_tokens * p.H * 2 + Sh::kTileVecs - 1) / Sh::kTileVecs;
    int64_t blocks = (ntiles + kWriteWarps - 1) / kWriteWarps;
    const int64_t cap = (int64_t)num_sms() * Sh::kMinBlocks;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaError_t err = opt_in_smem<write_kernel<D, T, BITS>>(Sm::kBytes);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kWriteThreads);
    cfg.dynamicSmemBytes = Sm::kBytes;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, write_kernel<D, T, BITS>, p);
}

}  // namespace

namespace {
template <int BITS>
cudaError_t launch_write_mode(const WriteParams& p, int head_size, DType dt, cudaStream_t stream) {
    if (head_size == 128) {
        return dt == DType::BF16 ? launch_write_t<128, __nv_bfloat16, BITS>(p, stream)
                                 : launch_write_t<128, __half, BITS>(p, stream);
    }
    return dt == DType::BF16 ? launch_write_t<64, __nv_bfloat16, BITS>(p, stream)
                             : launch_write_t<64, __half, BITS>(p, stream);
}
}  // namespace

cudaError_t launch_write(const WriteParams& p, int head_size, DType dt, cudaStream_t stream) {
    return launch_write_mode<4>(p, head_size, dt, stream);
}

cudaError_t launch_write_int8(const WriteParams& p, int head_size, DType dt, cudaStream_t stream) {
    return launch_write_mode<8>(p, head_size, dt, stream);
}

cudaError_t launch_write_int2(const WriteParams& p, int head_size, DType dt, cudaStream_t stream) {
    return launch_write_mode<2>(p, head_size, dt, stream);
}

}  // namespace kvi4
