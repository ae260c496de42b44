// Device-side building blocks shared by the kernels of the INT4 per-(token, head) KV cache:
// inline-PTX wrappers (mbarrier, bulk async copy, packed fp32x2 arithmetic, mma.sync, movmatrix)
// and the nibble -> fp16 unpacking used by both attention kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace kvi4 {

// Row geometry of one cached (token, head) vector.
template <int D>
struct Geo {
    static constexpr int RB = D / 2 + 4;   // bytes: D/2 code bytes + fp32 scale word
    static constexpr int RW = RB / 4;      // 32-bit words per row
    static constexpr int KW = D / 8;       // code words per row (8 nibbles each)
    static constexpr int KSTEPS = D / 16;  // k-steps of a 16-deep mma over the head dimension
    static constexpr int KWPT = KW / 4;    // code words one thread of a quad reads per row
    static constexpr int MT = D / 16;      // 16-row tiles covering the head dimension
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// n / d for n < 2^31 with rcp = floor(2^32 / d) (all ones for d = 1): the high product is n / d
// or one less, and one comparison fixes it.
__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint32_t d, uint32_t rcp) {
    uint32_t q = __umulhi(n, rcp);
    if (n - q * d >= d) ++q;
    return q;
}

__device__ __forceinline__ void count_status(uint32_t* status, int which) {
    if (status != nullptr) atomicAdd(status + which, 1u);
}

// ------------------------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the phase with the given parity (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase completes or about
// hint_ns pass, instead of spinning (a spinning warp takes issue slots from its neighbours).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; give up after timeout_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns = kWaitTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

// 16-byte asynchronous copy global -> shared (not allocated in L1); a dead copy writes zeros and
// reads nothing.  dst and src 16-byte aligned.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool live) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(live ? 16 : 0)
                 : "memory");
}

// One arrival on the mbarrier once every asynchronous copy this thread issued so far has landed
// (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 1-D bulk copy global -> shared, completion signalled on an mbarrier (transaction bytes).
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Bring [src, src + bytes) into L2 (no completion to wait for).  16-byte aligned, bytes a multiple
// of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------ programmatic dependent launch
// A kernel launched with the programmatic-serialization attribute may start while the previous
// kernel of the stream is still running; griddep_wait() blocks until that kernel has completed and
// its memory is visible.  Without the attribute both are no-ops.

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// -------------------------------------------------------------------- packed fp32 (sm_100+)
// Each lane of the pair is an independent IEEE round-to-nearest-even operation, so results are
// bit-identical to two scalar operations.  The compiler builtins keep the pair in a register pair
// (no packing moves around each operation).  a - b is fma(b, -1, a): the product is exact, so the
// one rounding is that of a - b.

__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) { return __fadd2_rn(a, b); }

__device__ __forceinline__ float2 sub_f32x2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a); }

__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ------------------------------------------------------------------------ tensor-core helpers

// D = A(16x16, row) * B(16x8, col) + D, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 b16 matrix held in mma fragment layout (row = lane/4, cols 2*(lane%4), +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// RN(a * b + c): a the low (HI_A false) or high fp16 half of a2, b the low fp16 half of b2, c fp32,
// in one mixed-precision FMA that reads the fp16 operands in place (exact upcasts, one rounding).
template <bool HI_A>
__device__ __forceinline__ float fma_f16_f32(uint32_t a2, uint32_t b2, float c) {
    float d;
    if constexpr (!HI_A)
        asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2; fma.rn.f32.f16 %0, al, bl, %3; }"
            : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    else
        asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2; fma.rn.f32.f16 %0, ah, bl, %3; }"
            : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ----------------------------------------------------------------------- nibble unpacking
//
// A 32-bit word holds 8 codes e0..e7 (e0 in bits 0-3, e1 in bits 4-7, ...).  OR-ing a nibble
// into the mantissa of fp16 1024.0 (0x6400) gives exactly 1024 + n (the mantissa unit at that
// exponent is 1); a nibble shifted up by 4 gives 1024 + 16 n.  Subtracting 1024 + zp, or
// scaling by 1/16 and subtracting 64 + zp, leaves code - zp exactly as fp16.

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// fp16 (1024 + zp) and -(64 + zp) for a zero-point 0..15
__device__ __forceinline__ uint32_t zp_lo_half(uint32_t zp) { return 0x6400u + zp; }
__device__ __forceinline__ uint32_t zp_hi_half(uint32_t zp) { return 0xD400u + (zp << 4); }

// Word w (8 codes) with per-half zero points -> 4 fp16x2 values holding code - zp:
//   o[0] = (e0, e4), o[1] = (e1, e5), o[2] = (e2, e6), o[3] = (e3, e7)   (low half, high half)
// zlo / zhi: the two halves' zp_lo_half / zp_hi_half packed into a 32-bit pair.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t zlo, uint32_t zhi, uint32_t (&o)[4]) {
    constexpr uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u, kExp = 0x64006400u, kSixteenth = 0x2C002C00u;
    const uint32_t w8 = w >> 8;
    o[0] = hsub2(lop3_and_or(w, kLo, kExp), zlo);
    o[1] = hfma2(lop3_and_or(w, kHi, kExp), kSixteenth, zhi);
    o[2] = hsub2(lop3_and_or(w8, kLo, kExp), zlo);
    o[3] = hfma2(lop3_and_or(w8, kHi, kExp), kSixteenth, zhi);
}

// Two rows' words (token a, token b) -> 8 fp16x2 values (a.e_i - zp_a, b.e_i - zp_b), i = 0..7.
__device__ __forceinline__ void unpack_word_pair(uint32_t wa, uint32_t wb, uint32_t zlo, uint32_t zhi,
                                                 uint32_t (&o)[8]) {
    uint32_t lo[4], hi[4];
    unpack_word(prmt(wa, wb, 0x5410u), zlo, zhi, lo);
    unpack_word(prmt(wa, wb, 0x7632u), zlo, zhi, hi);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[i] = lo[i];
        o[4 + i] = hi[i];
    }
}

// The same 8 nibbles with no offset to remove: a masked nibble is already an exact fp16 number, the
// subnormal n 2^-24 (low nibbles) or 16 n 2^-24 = n 2^-20 (high nibbles).  The caller folds the 2^24
// and the extra 16 of the odd dimensions (the high nibbles) into the other operand and the results.
// Pairs as unpack_word: o[0] = dims (0, 4), o[1] = (1, 5) x 16, o[2] = (2, 6), o[3] = (3, 7) x 16.
__device__ __forceinline__ void unpack_word_sub(uint32_t w, uint32_t (&o)[4]) {
    const uint32_t w8 = w >> 8;
    o[0] = w & 0x000F000Fu;
    o[1] = w & 0x00F000F0u;
    o[2] = w8 & 0x000F000Fu;
    o[3] = w8 & 0x00F000F0u;
}

// ----------------------------------------------------------------------- int8 code unpacking
// Four int8 codes of a word as offset binary x + 128 (the sign bit flipped) under the fp16 exponent
// byte 0x64 give 1024 + x + 128 exactly; subtracting 1152 leaves x.
constexpr uint32_t kI8Exp = 0x64646464u, kI8Flip = 0x80808080u, kI8Bias = 0x64806480u;   // (1152, 1152)

// Dimensions 0..3 (word w0) and 4..7 (word w1) of a row as fp16 pairs (0, 1), (2, 3), (4, 5), (6, 7).
__device__ __forceinline__ void unpack_i8(uint32_t w0, uint32_t w1, uint32_t (&o)[4]) {
    const uint32_t u0 = w0 ^ kI8Flip, u1 = w1 ^ kI8Flip;
    o[0] = hsub2(prmt(u0, kI8Exp, 0x5140u), kI8Bias);
    o[1] = hsub2(prmt(u0, kI8Exp, 0x7362u), kI8Bias);
    o[2] = hsub2(prmt(u1, kI8Exp, 0x5140u), kI8Bias);
    o[3] = hsub2(prmt(u1, kI8Exp, 0x7362u), kI8Bias);
}

// The same eight dimensions of two rows a and b: o[i] = (a's dimension i, b's dimension i).
__device__ __forceinline__ void unpack_i8_pair(uint32_t a0, uint32_t a1, uint32_t b0, uint32_t b1, uint32_t (&o)[8]) {
    const uint32_t m[4] = {prmt(a0 ^ kI8Flip, b0 ^ kI8Flip, 0x5140u), prmt(a0 ^ kI8Flip, b0 ^ kI8Flip, 0x7362u),
                           prmt(a1 ^ kI8Flip, b1 ^ kI8Flip, 0x5140u), prmt(a1 ^ kI8Flip, b1 ^ kI8Flip, 0x7362u)};
#pragma unroll
    for (int k = 0; k < 4; ++k) {   // m[k] = (a_2k, b_2k, a_2k+1, b_2k+1)
        o[2 * k] = hsub2(prmt(m[k], kI8Exp, 0x4140u), kI8Bias);
        o[2 * k + 1] = hsub2(prmt(m[k], kI8Exp, 0x4342u), kI8Bias);
    }
}

// ----------------------------------------------------------------------- int2 centroid lookup
// The INT2 mode's Lloyd-Max outputs -b, -a, a, b of N(0, 1) (codes 0..3; a = 0.45278, b = 1.51042,
// J. Max 1960) as fp16 (0x3E0B = 1.5107, 0x373F = 0.45288), laid out as a byte table for prmt: code
// c sits at bytes 2c, 2c + 1 of (kU2Lo, kU2Hi).
constexpr uint32_t kU2Lo = 0xB73FBE0Bu;   // (-b, -a)
constexpr uint32_t kU2Hi = 0x3E0B373Fu;   // (a, b)

// Selectors of field k of all four bytes of x at once: byte b of the result is the selector pair
// (2c, 2c + 1) of that byte's code c, so its low half looks up bytes 0 and 1, its high half bytes
// 2 and 3 (no carries cross a byte: 0x22 c + 0x10 <= 0x76).
__device__ __forceinline__ uint32_t u2_selectors(uint32_t x, int k) {
    return ((x >> (2 * k)) & 0x03030303u) * 0x22u + 0x10101010u;
}

// One 16-bit group h -> its 4 fp16 pairs (dim k, dim k + 4), one selector per pair.
__device__ __forceinline__ void unpack_u2(uint32_t h, uint32_t (&o)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = prmt(kU2Lo, kU2Hi, u2_selectors(h, k));
}

// Two 16-bit groups packed in x (group a in the low half, b in the high half; dims 0..3 of a group
// in its byte 0, 4..7 in its byte 1, dim 4j + k at bits 2k of byte j) -> 4 fp16 pairs each, (dim k,
// dim k + 4), k = 0..3: the order unpack_word gives INT4 nibbles.
__device__ __forceinline__ void unpack_u2_x2(uint32_t x, uint32_t (&oa)[4], uint32_t (&ob)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t s = u2_selectors(x, k);
        oa[k] = prmt(kU2Lo, kU2Hi, s);
        ob[k] = prmt(kU2Lo, kU2Hi, s >> 16);
    }
}

// The same 8 dims of two rows a and b (16-bit groups ha, hb): o[i] = (a's dim i, b's dim i).
__device__ __forceinline__ void unpack_u2_pair(uint32_t ha, uint32_t hb, uint32_t (&o)[8]) {
    const uint32_t y = prmt(ha, hb, 0x5140u);   // a.byte 0, b.byte 0, a.byte 1, b.byte 1
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t s = u2_selectors(y, k);
        o[k] = prmt(kU2Lo, kU2Hi, s);
        o[4 + k] = prmt(kU2Lo, kU2Hi, s >> 16);
    }
}

// Token order inside a 16-token block used by the attention kernels: mma row / key index r maps
// to token tau(r) = ((r & 7) >> 1) + 4 * (r & 1) + 8 * (r >> 3).  It makes the four rows a thread
// reads for P.V (tokens t, t+4, t+8, t+12 of lane quad t) fall in distinct shared-memory banks.
__host__ __device__ __forceinline__ constexpr int block_token(int r) {
    return ((r & 7) >> 1) + 4 * (r & 1) + 8 * (r >> 3);
}

}  // namespace kvi4
