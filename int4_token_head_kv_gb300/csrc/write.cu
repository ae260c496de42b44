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

// load_vector: D 16-bit inputs (D/2 little-endian pairs) -> fp32 after the sign flips (XOR masks on
// the pairs: bit 15 of each half is the sign in fp16 and bf16) and the stride-1 butterflies.
// encode_vector: the remaining butterflies, normalisation, scale / zero-point and codes; output
// the D/8 code words and the scale word of the cache row.
template <int D, typename T>
__device__ __forceinline__ void load_vector(const uint4* src, const uint32_t* sign_mask, float (&u)[D]) {
#pragma unroll
    for (int cc = 0; cc < D / 8; ++cc) {
        const uint4 q = src[cc];
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = cc * 4 + e;
            const float2 x = upcast_pair<T>(w4[e] ^ sign_mask[j]);
            // stride-1 butterfly straight from the pair
            u[2 * j] = __fadd_rn(x.x, x.y);
            u[2 * j + 1] = __fsub_rn(x.x, x.y);
        }
    }
}

template <int D>
__device__ __forceinline__ void encode_vector(float (&u)[D], float c, uint32_t (&words)[Geo<D>::KW + 1]) {
    using Gm = Geo<D>;
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
    const float2 c2 = make_float2(c, c);
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
    words[Gm::KW] = sb | zp;
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
// (token, plane) row group, contiguous in the cache.  Each warp owns tiles of 32 consecutive
// vectors and works through them on its own (no CTA-wide barriers): it prefetches the next tile's
// inputs, one bulk async copy of 2D bytes per lane (its vector) completing on the buffer's
// mbarrier, into one of two padded shared-memory buffers
// (row stride 2D + 16 bytes, so the 16-byte reads of 8 neighbouring rows hit distinct banks),
// encodes the current tile with one vector per lane, stages the encoded rows in the buffer it just
// read, and writes each row group with one bulk async store (when H divides 32 and a group is a
// multiple of 16 bytes; otherwise each lane stores its own row).
constexpr int kWarpVecs = 32;
constexpr int kWriteWarps = kWriteThreads / 32;

template <int D>
struct WriteSmem {
    static constexpr int kRowPad = 2 * D + 16;
    static constexpr int kBuf = kWarpVecs * kRowPad;            // one tile of inputs
    static constexpr int kPerWarp = 2 * kBuf;
    static constexpr int kBars = kWriteWarps * kPerWarp;        // two mbarriers per warp
    static constexpr int kBytes = kBars + kWriteWarps * 2 * 8 + (D / 2) * 4;
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

template <int D, typename T, bool INT8>
__global__ void __launch_bounds__(kWriteThreads, 3) write_kernel(const __grid_constant__ WriteParams p) {
    using Gm = Geo<D>;
    constexpr int RB = INT8 ? D + 4 : Gm::RB;       // cache row bytes
    constexpr int NW = INT8 ? D / 4 : Gm::KW;       // code words per row (then the scale word)
    using Sm = WriteSmem<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    // Launched as a programmatic dependent: wait for the previous kernel of the stream (it may
    // produce K, V or the slots), then let the next kernel start its own set-up.
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* wbuf = smem + warp * Sm::kPerWarp;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::kBars) + warp * 2;   // this warp's [buffer]
    uint32_t* sign_mask = reinterpret_cast<uint32_t*>(smem + Sm::kBars + kWriteWarps * 2 * 8);
    if (lane == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    for (int j = tid; j < (INT8 ? 0 : D / 2); j += kWriteThreads) {   // INT8 rows take no signs
        const float s0 = p.signs[2 * j], s1 = p.signs[2 * j + 1];
        sign_mask[j] = ((__float_as_uint(s0) >> 31) << 15) | ((__float_as_uint(s1) >> 31) << 31);
        if (blockIdx.x == 0 && ((fabsf(s0) != 1.0f) || (fabsf(s1) != 1.0f))) count_status(p.status, 4);
    }
    __syncthreads();

    const uint32_t H = (uint32_t)p.H;
    VecIndex vx;
    vx.H = H;
    vx.hmask = H - 1;
    vx.hshift = (H & (H - 1)) == 0 ? __ffs(H) - 1 : -1;
    const uint32_t nvec = (uint32_t)(p.num_tokens * H * 2);
    const uint32_t ntiles = (nvec + kWarpVecs - 1) / kWarpVecs;
    const uint32_t gwarp = blockIdx.x * kWriteWarps + warp, nwarps = gridDim.x * kWriteWarps;
    const uint32_t group_bytes = H * RB;
    const bool grouped = vx.hshift >= 0 && H <= (uint32_t)kWarpVecs && (group_bytes % 16) == 0;
    const uint8_t* kin = static_cast<const uint8_t*>(p.k);
    const uint8_t* vin = static_cast<const uint8_t*>(p.v);

    // lane copies its vector of the tile (2D bytes) into row lane of the buffer
    auto prefetch = [&](uint32_t tile, uint8_t* buf, uint64_t* bar) {
        const uint32_t v0 = tile * kWarpVecs;
        const uint32_t live_vecs = min((uint32_t)kWarpVecs, nvec - v0);
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
        const uint32_t v = tile * kWarpVecs + lane;
        const bool live = v < nvec;
        float u[D];
        uint32_t words[NW + 1];
        if constexpr (INT8) {
            if (live) load_vector_raw<D, T>(reinterpret_cast<const uint4*>(cur + lane * Sm::kRowPad), u);
            __syncwarp();   // the tile's inputs are in registers; its buffer becomes the output stage
            if (live) encode_vector_int8<D>(u, words);
        } else {
            if (live) load_vector<D, T>(reinterpret_cast<const uint4*>(cur + lane * Sm::kRowPad), sign_mask, u);
            __syncwarp();   // the tile's inputs are in registers; its buffer becomes the output stage
            if (live) encode_vector<D>(u, p.c, words);
        }
        uint32_t tok = 0, h = 0, pl = 0;
        if (live) vx.split(v, tok, h, pl);
        if (grouped) {
            uint32_t* orow = reinterpret_cast<uint32_t*>(cur + lane * RB);
            if (live) {
#pragma unroll
                for (int wi = 0; wi <= NW; ++wi) orow[wi] = words[wi];
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // staged rows -> bulk store
            __syncwarp();
            // the first lane of each row group stores the whole group
            if (live && h == 0) {
                const int64_t slot = __ldg(p.slots + tok);
                if (slot >= p.num_slots) {
                    if (pl == 0) count_status(p.status, 0);
                } else if (slot >= 0) {
                    const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
                    bulk_store_s2g(p.cache + ((blk * 2 + pl) * kBlockSize + off) * (int64_t)group_bytes,
                                   cur + lane * RB, group_bytes);
                }
            }
        } else if (live) {
            const int64_t slot = __ldg(p.slots + tok);
            if (slot >= p.num_slots) {
                if (pl == 0 && h == 0) count_status(p.status, 0);
            } else if (slot >= 0) {
                const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
                uint32_t* row = reinterpret_cast<uint32_t*>(p.cache + (((blk * 2 + pl) * kBlockSize + off) * H + h) * RB);
#pragma unroll
                for (int wi = 0; wi <= NW; ++wi) row[wi] = words[wi];
            }
        }
    }
    if (waited_out && tile + nwarps < ntiles) {   // let the copy in flight land before the warp exits
        (void)mbar_wait(&bars[(it + 1) & 1], (uint32_t)((it + 1) >> 1) & 1u);
    }
    if (grouped) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    (void)kRoundMagicBits;
}

template <int D, typename T, bool INT8>
cudaError_t launch_write_t(const WriteParams& p, cudaStream_t stream) {
    using Sm = WriteSmem<D>;
    const int64_t ntiles = (p.num_tokens * p.H * 2 + kWarpVecs - 1) / kWarpVecs;
    int64_t blocks = (ntiles + kWriteWarps - 1) / kWriteWarps;
    const int64_t cap = (int64_t)num_sms() * 3;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaError_t err = opt_in_smem<write_kernel<D, T, INT8>>(Sm::kBytes);
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
    return cudaLaunchKernelEx(&cfg, write_kernel<D, T, INT8>, p);
}

}  // namespace

namespace {
template <bool INT8>
cudaError_t launch_write_mode(const WriteParams& p, int head_size, DType dt, cudaStream_t stream) {
    if (head_size == 128) {
        return dt == DType::BF16 ? launch_write_t<128, __nv_bfloat16, INT8>(p, stream)
                                 : launch_write_t<128, __half, INT8>(p, stream);
    }
    return dt == DType::BF16 ? launch_write_t<64, __nv_bfloat16, INT8>(p, stream)
                             : launch_write_t<64, __half, INT8>(p, stream);
}
}  // namespace

cudaError_t launch_write(const WriteParams& p, int head_size, DType dt, cudaStream_t stream) {
    return launch_write_mode<false>(p, head_size, dt, stream);
}

cudaError_t launch_write_int8(const WriteParams& p, int head_size, DType dt, cudaStream_t stream) {
    return launch_write_mode<true>(p, head_size, dt, stream);
}

}  // namespace kvi4
