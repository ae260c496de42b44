// Chunked-prefill attention over the INT4 cache: sequences with more than one query token
// ("[Feature] Triton INT4 / INT2 per-token-head KV cache quantization", packed read path;
// causal queries at positions seq_len - q_len + t as in the unified-attention call of
// test_triton_unified_attention_per_token_head_scale), on the fifth-generation tensor cores.
//
// One CTA per (query tile, kv head, sequence): 128 rows = (128 / G) query tokens x G query heads
// of that kv head.  The CTA walks the key tiles its rows can see (causal), 128 keys per tile:
//   S = Q' (K - zp)^T   tcgen05.mma, A = the rotated, power-of-two-prescaled queries as fp16
//                       high + low halves (two MMAs per k-step) held in tensor memory, B = the
//                       tile's keys dequantised to exact fp16 (code - zp) in shared memory
//                       (K-major, 128-byte swizzle); S accumulates in fp32 in tensor memory
//   online softmax     per row: logit = S * s'_K * alpha, causal mask, a reference maximum that
//                       moves only on jumps of more than 2^8; P_w = p * s'_V * 2^-E as fp16
//                       written back over S (E: a reference exponent of the V scales)
//   O += P_w (V - zp)  tcgen05.mma, A = P_w from tensor memory, B = the values dequantised to
//                       fp16 in shared memory (the same row layout as K, read MN-major); O stays
//                       in tensor memory for the whole key range
// and un-rotates its rows at the end.
//
// Warp roles (384 threads): warps 0-7 own the rows (warp w reads tensor-memory lanes
// 32 (w % 4) .. + 31, the lower or upper half of the key columns for w < 4 or w >= 4), rotate the
// queries and run the softmax and the epilogue; warps 8-11 load the packed codes of the next key
// tile (one key per thread, registers double-buffered) and dequantise them into the shared-memory
// tile pair of its parity.  Warp 8 also allocates tensor memory, and its first thread issues every
// MMA after dequantising its key of each tile: S of tile j once the tile is in shared memory, then
// P.V of tile j - 1 once its weights are in tensor memory (the double-buffered hand-offs impose
// that order anyway).
// Tensor memory (512 columns): Q' high, Q' low, two S buffers (S of tile j + 1 is computed while
// the softmax of tile j runs), O.  Hand-offs go through mbarriers (tcgen05.commit for the MMAs);
// every wait is bounded and a wait that gives up is counted and winds the CTA down.
#include "attn_common.cuh"

namespace kvi4 {
namespace {

constexpr int kPfRows = 128;                  // query rows per CTA (the MMA M)
constexpr int kPfKeys = 128;                  // keys per tile (the S MMA N, the P.V MMA K)
constexpr int kPfSoftmaxWarps = 8;
constexpr int kPfDequantWarps = 4;
constexpr int kPfMmaWarp = kPfSoftmaxWarps;   // the first dequantisation warp
constexpr int kPfThreads = (kPfSoftmaxWarps + kPfDequantWarps) * 32;
constexpr int kPfSoftmaxThreads = kPfSoftmaxWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kPfLazyMax = 8.0f;            // log2 units the row's reference maximum may trail
constexpr uint32_t kPfLazyExp = 4;            // binades the V exponent reference may trail

// Shared-memory layout (bytes from a 1024-aligned base).  A fp16 tile is 128 keys x D dims as
// D/64 chunks of [128 rows x 128 B], 128-byte swizzled: [K tile 0][V tile 0][K tile 1][V tile 1].
// Before the first tile the query halves are staged over tiles 1 (rows of D + 8 halves), and after
// the last the fp32 output rows over tiles 0-1 (rows of D + 4 floats).
template <int D>
struct PfLayout {
    static constexpr uint32_t kTile = (D / 64) * kPfKeys * 128;
    static constexpr uint32_t kQStride = D + 8;                                   // halves per staged row
    static constexpr uint32_t kQStage = 2u * kPfRows * kQStride * 2;              // high + low
    static constexpr uint32_t kOStride = D + 4;                                   // floats per staged row
    static constexpr uint32_t kMisc = ((4 * kTile > 2 * kTile + kQStage ? 4 * kTile : 2 * kTile + kQStage) +
                                       1023u) & ~1023u;
    static_assert(kPfRows * kOStride * 4 <= 4 * kTile, "output staging");
    // misc region
    static constexpr uint32_t kSk = kMisc;                           // [2][128] f32 key scales s'_K
    static constexpr uint32_t kSv = kSk + 2 * kPfKeys * 4;           // [2][128] V scale words
    static constexpr uint32_t kEblk = kSv + 2 * kPfKeys * 4;         // [2][4] per-warp max V exponent
    static constexpr uint32_t kRowMax = kEblk + 2 * 4 * 4;           // [2 tiles][2 halves][128] f32
    static constexpr uint32_t kRowL = kRowMax + 2 * 2 * kPfRows * 4;  // [2][128] f32
    static constexpr uint32_t kAlpha = kRowL + 2 * kPfRows * 4;      // [128] f32
    static constexpr uint32_t kSigns = kAlpha + kPfRows * 4;         // [D] f32
    static constexpr uint32_t kBars = (kSigns + D * 4 + 7u) & ~7u;   // mbarriers
    // kv_full[2], pv_done[2], s_full[2], p_full[2], q_ready, flush, rows[2], q_stage, epi[2]
    static constexpr int kNumBars = 2 + 2 + 2 + 2 + 1 + 1 + 2 + 1 + 2;
    static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
    static constexpr uint32_t kFlags = kTmemSlot + 4;
    static constexpr uint32_t kBytes = kFlags + 4 + 1024;            // + alignment slack
};

// tensor-memory columns
template <int D>
struct PfTmem {
    static constexpr uint32_t kQh = 0, kQl = D / 2, kS0 = D, kS1 = D + kPfKeys, kO = D + 2 * kPfKeys;
    static_assert(kO + D <= kTmemCols, "tensor memory");
};

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: fp32 accumulator, fp16 A and B, M = 128, N = n, B K-major
// (b_mn = 0) or MN-major (b_mn = 1), A K-major.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t n, uint32_t b_mn) {
    return (1u << 4) | (b_mn << 16) | ((n >> 3) << 17) | ((uint32_t)(kPfRows >> 4) << 24);
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit tensor-memory columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r in a [rows x 128 B] block with the 128-byte
// swizzle the tensor-core descriptors expect: the chunk index is XOR-ed with r mod 8.
__device__ __forceinline__ uint32_t swz128(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

// Eight codes of one word (dims 8w .. 8w+7) as fp16 (code - zp) in dimension order.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, uint32_t zp) {
    const uint32_t zl = zp_lo_half(zp) * 0x10001u, zh = zp_hi_half(zp) * 0x10001u;
    uint32_t o[4];
    unpack_word(w, zl, zh, o);   // (e0,e4) (e1,e5) (e2,e6) (e3,e7)
    return make_uint4(prmt(o[0], o[1], 0x5410u), prmt(o[2], o[3], 0x5410u), prmt(o[0], o[1], 0x7632u),
                      prmt(o[2], o[3], 0x7632u));
}

template <int D, typename QT, typename OT>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ AttnParams p) {
    using Gm = Geo<D>;
    using Ly = PfLayout<D>;
    using Tm = PfTmem<D>;
    constexpr int KSTEPS = D / 16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- the CTA's rows; everything up to the barrier set-up exits uniformly
    const int ntile = (int)(gridDim.x / (unsigned)p.H);
    const int qtile = ntile - 1 - (int)(blockIdx.x / (unsigned)p.H), h = (int)(blockIdx.x % (unsigned)p.H);
    const int seq = blockIdx.z;
    const int q0 = __ldg(p.qsl + seq);
    const int qlen = __ldg(p.qsl + seq + 1) - q0;
    if (qlen <= 1) return;   // decode sequences (and empty ones) are not this kernel's
    if (q0 < 0 || (int64_t)q0 + qlen > p.num_q_tokens || qlen > p.max_query_len) {
        if (qtile == 0 && h == 0 && threadIdx.x == 0) count_status(p.status, 2);
        if (q0 < 0 || (int64_t)q0 + qlen > p.num_q_tokens) return;
    }
    const int G = p.G, Hq = p.Hq, H = p.H;
    const int BQ = kPfRows / G;
    const int qt0 = qtile * BQ;
    if (qt0 >= qlen) return;
    int L = __ldg(p.seq_lens + seq);
    // the same context cap as the decode path (max_seq_len and the block table), counted as bad metadata
    if (L > p.len_cap || qlen > L) {
        if (qtile == 0 && h == 0 && threadIdx.x == 0) count_status(p.status, 2);
        L = min(L, p.len_cap);
    }
    const int pos0 = L - qlen;   // position of query token 0
    const int cta_lim = min(pos0 + min(qlen - 1, qt0 + BQ - 1), L - 1);   // last key any row sees
    const int nkt = cta_lim >= 0 ? cta_lim / kPfKeys + 1 : 0;

    float* sk = reinterpret_cast<float*>(smem + Ly::kSk);
    uint32_t* sv = reinterpret_cast<uint32_t*>(smem + Ly::kSv);
    uint32_t* eblkw = reinterpret_cast<uint32_t*>(smem + Ly::kEblk);
    float* rowmax = reinterpret_cast<float*>(smem + Ly::kRowMax);
    float* rowl = reinterpret_cast<float*>(smem + Ly::kRowL);
    float* alpha = reinterpret_cast<float*>(smem + Ly::kAlpha);
    float* sgn = reinterpret_cast<float*>(smem + Ly::kSigns);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::kBars);
    uint64_t* kv_full = bars;        // [2] dequantised tile ready (128 arrivals)
    uint64_t* pv_done = bars + 2;    // [2] P.V of the tile done (commit): its tiles and S buffer free
    uint64_t* s_full = bars + 4;     // [2] S of the tile in tensor memory (commit)
    uint64_t* p_full = bars + 6;     // [2] P of the tile in tensor memory (256 arrivals)
    uint64_t* q_ready = bars + 8;    // queries in tensor memory, staging free (256 arrivals)
    uint64_t* flush = bars + 9;      // the MMA thread's last commit (teardown)
    // barriers among the 256 row threads (bounded waits, unlike a hardware named barrier): the
    // row-maximum exchange of tiles of each parity, the query staging, the epilogue's two steps
    uint64_t* rows_sync = bars + 10;
    uint64_t* q_stage = bars + 12;
    uint64_t* epi = bars + 13;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kFlags);

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&kv_full[b], kPfDequantWarps * 32);
            mbar_init(&pv_done[b], 1);
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], kPfSoftmaxThreads);
        }
        mbar_init(q_ready, kPfSoftmaxThreads);
        mbar_init(flush, 1);
        for (int i = 0; i < 5; ++i) mbar_init(&rows_sync[i], kPfSoftmaxThreads);   // rows_sync[2], q_stage, epi[2]
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < D; i += blockDim.x) sgn[i] = p.signs[i] < 0.0f ? -1.0f : 1.0f;
    if (warp == kPfMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    uint8_t* tiles = smem;   // [K0][V0][K1][V1]
    auto ktile = [&](int b) { return tiles + (uint32_t)b * 2u * Ly::kTile; };
    auto vtile = [&](int b) { return tiles + (uint32_t)b * 2u * Ly::kTile + Ly::kTile; };
    // a wait that runs out counts once and winds the CTA down
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar, parity)) return true;
        if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) count_status(p.status, 3);
        return false;
    };
    // all 256 row threads meet (warp-uniform result)
    auto rows_meet = [&](uint64_t* bar, uint32_t parity) -> bool {
        mbar_arrive(bar);
        return __all_sync(0xffffffffu, wait(bar, parity));
    };

    if (warp < kPfSoftmaxWarps) {
        // ================================================================ rows: softmax + epilogue
        const int r = 32 * (warp & 3) + lane, hf = warp >> 2;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        __half* qs_hi = reinterpret_cast<__half*>(ktile(1));
        __half* qs_lo = qs_hi + kPfRows * Ly::kQStride;
        // ---- rotate the queries: warp w the rows 16 w .. 16 w + 15 (lanes across dimensions)
        for (int i = 0; i < kPfRows / kPfSoftmaxWarps; ++i) {
            const int R = warp * (kPfRows / kPfSoftmaxWarps) + i;
            const int qt = qt0 + R / G, gg = R % G;
            if (nkt > 0 && qt < qlen) {
                const float a = rotate_query<D, QT>(p.q, ((int64_t)(q0 + qt) * Hq + h * G + gg) * D, sgn,
                                                    qs_hi + R * Ly::kQStride, qs_lo + R * Ly::kQStride, p.c,
                                                    p.softmax_scale);
                if (lane == 0) alpha[R] = a;
            } else {
                for (int k = lane; k < D; k += 32) qs_hi[R * Ly::kQStride + k] = qs_lo[R * Ly::kQStride + k] = __float2half(0.0f);
                if (lane == 0) alpha[R] = 0.0f;
            }
        }
        bool ok = rows_meet(q_stage, 0);
        // ---- this thread's half of its row into tensor memory (high, then low halves)
        if (ok) {
            constexpr int kWords = D / 4;   // 32-bit words of a half row
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint32_t* src = reinterpret_cast<const uint32_t*>((part ? qs_lo : qs_hi) + r * Ly::kQStride) +
                                      hf * kWords;
                uint32_t w[kWords];
#pragma unroll
                for (int j = 0; j < kWords; j += 4) {
                    const uint4 v = *reinterpret_cast<const uint4*>(src + j);
                    w[j] = v.x;
                    w[j + 1] = v.y;
                    w[j + 2] = v.z;
                    w[j + 3] = v.w;
                }
                const uint32_t ta = tmem + lane_base + (part ? Tm::kQl : Tm::kQh) + hf * kWords;
                if constexpr (kWords == 32) {
                    tmem_st32(ta, w);
                } else {
#pragma unroll
                    for (int c0 = 0; c0 < kWords; c0 += 16) tmem_st16(ta + c0, w + c0);
                }
            }
            tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(q_ready);
        const float al = alpha[r];
        const int qt_r = qt0 + r / G;
        const int pos_r = qt_r < qlen ? pos0 + qt_r : -1;   // last visible key of this row
        float m = kNegBig, l = 0.0f;
        uint32_t E = 0;   // reference biased exponent of the V scales

        for (int j = 0; j < nkt && ok; ++j) {
            const int b = j & 1;
            const uint32_t ph = (uint32_t)(j >> 1) & 1u;
            ok = wait(&s_full[b], ph) && wait(&kv_full[b], ph);
            if (__any_sync(0xffffffffu, !ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t scol = (b ? Tm::kS1 : Tm::kS0) + (uint32_t)hf * 64u;
            uint32_t s[64];
            tmem_ld32(tmem + lane_base + scol, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
            tmem_ld32(tmem + lane_base + scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
            tmem_ld_wait();
            const int key0 = j * kPfKeys + hf * 64;
            const float* skb = sk + b * kPfKeys + hf * 64;
            float bm = -INFINITY;
            const bool full = key0 + 63 <= pos_r;   // no causal mask in this half-tile
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(skb + c);
                const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool vis = kk[e] > 0.0f && (full || key0 + c + e <= pos_r);
                    const float x = vis ? __uint_as_float(s[c + e]) * kk[e] * al : -INFINITY;
                    s[c + e] = __float_as_uint(x);
                    bm = fmaxf(bm, x);
                }
            }
            float* rm = rowmax + (b * 2) * kPfRows;
            rm[hf * kPfRows + r] = bm;
            if (!rows_meet(&rows_sync[b], ph)) {
                ok = false;
                break;
            }
            bm = fmaxf(bm, rm[(1 - hf) * kPfRows + r]);
            // reference maximum and V exponent (the same decisions in both halves of a row; E in
            // every row, from the tile's per-warp maxima)
            const bool up = bm > m + kPfLazyMax;
            const float fm = up ? fast_exp2(m - bm) : 1.0f;
            if (up) m = bm;
            const uint32_t* eb4 = eblkw + b * 4;
            const uint32_t eb = max(max(eb4[0], eb4[1]), max(eb4[2], eb4[3]));
            float fe = 1.0f;
            if (eb > E + kPfLazyExp || (E == 0u && eb > 0u)) {
                fe = (E == 0u || eb - E > 126u) ? 0.0f : __uint_as_float((127u + E - eb) << 23);
                E = eb;
            }
            l *= fm;
            const float f = fm * fe;
            if (j > 0 && __any_sync(0xffffffffu, f != 1.0f)) {
                // O must hold P.V of the previous tile before it is rescaled
                ok = wait(&pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u);
                if (__any_sync(0xffffffffu, !ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 16) {
                    uint32_t o[16];
                    tmem_ld16(tmem + lane_base + Tm::kO + hf * (D / 2) + c0, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                    tmem_st16(tmem + lane_base + Tm::kO + hf * (D / 2) + c0, o);
                }
                tmem_st_wait();
            }
            // weights w = p * s'_V * 2^-E as fp16 pairs, written over this half's first 32 S columns
            const float wsc = __uint_as_float((254u - E) << 23);   // 2^(127 - E)
            const uint32_t* svb = sv + b * kPfKeys + hf * 64;
            float ls = 0.0f;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t pw[16];
#pragma unroll
                for (int c = c0; c < c0 + 32; c += 4) {
                    const uint4 v4 = *reinterpret_cast<const uint4*>(svb + c);
                    const uint32_t vv[4] = {v4.x, v4.y, v4.z, v4.w};
                    float w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float pr = fast_exp2(__uint_as_float(s[c + e]) - m);
                        ls += pr;
                        w[e] = pr * (__uint_as_float(vv[e] & 0xFFFFFFF0u) * wsc);
                    }
                    pw[(c - c0) / 2] = pack_f16x2(w[0], w[1]);
                    pw[(c - c0) / 2 + 1] = pack_f16x2(w[2], w[3]);
                }
                tmem_st16(tmem + lane_base + scol + c0 / 2, pw);
            }
            l += ls;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[b]);
        }
        // ---- epilogue: O / l, scaled back by 2^(E - 127), staged, un-rotated
        if (ok && nkt > 0) ok = wait(&pv_done[(nkt - 1) & 1], (uint32_t)((nkt - 1) >> 1) & 1u);
        tc_fence_after();
        rowl[hf * kPfRows + r] = l;
        ok = rows_meet(&epi[0], 0) && ok;
        const bool good = __all_sync(0xffffffffu, ok) && nkt > 0;
        const float lt = l + rowl[(1 - hf) * kPfRows + r];
        const float es = E ? __uint_as_float(E << 23) : 0.0f;
        const float sc = lt > 0.0f ? es / lt : 0.0f;
        float* ostage = reinterpret_cast<float*>(tiles);
        if (good) {
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + Tm::kO + hf * (D / 2) + c0, o);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) ostage[r * Ly::kOStride + hf * (D / 2) + c0 + e] = __uint_as_float(o[e]) * sc;
            }
        } else {
            for (int e = 0; e < D / 2; ++e) ostage[r * Ly::kOStride + hf * (D / 2) + e] = 0.0f;
        }
        if (!rows_meet(&epi[1], 0)) ok = false;
        for (int i = 0; i < kPfRows / kPfSoftmaxWarps && ok; ++i) {
            const int R = warp * (kPfRows / kPfSoftmaxWarps) + i;
            const int qt = qt0 + R / G, gg = R % G;
            if (qt >= qlen) continue;
            float xv[D / 32];
#pragma unroll
            for (int k = 0; k < D / 32; ++k) xv[k] = ostage[R * Ly::kOStride + lane + 32 * k];
            unrotate_store<D, OT>(xv, 1.0f, sgn, p.c, p.out, ((int64_t)(q0 + qt) * Hq + h * G + gg) * D);
        }
    } else {
        // ================================================================ dequantisation of key tiles
        const int k = threadIdx.x - kPfSoftmaxThreads;   // this thread's key of every tile
        const bool issuer = k == 0;                        // warp 8, lane 0: also issues the MMAs
        const int32_t* table = p.block_tables + (int64_t)seq * p.max_blocks_per_seq;
        constexpr int NW = Gm::KW + 1;                    // words of a row: codes, then the scale word
        constexpr uint32_t idS = idesc_f16(kPfKeys, 0), idPV = idesc_f16(D, 1);
        uint32_t cur[2][NW], nxt[2][NW];
        bool cur_ok = false, nxt_ok = false;
        auto fetch = [&](int j, uint32_t (&w)[2][NW], bool& okk) {
            const int key = j * kPfKeys + k;
            okk = false;
            if (key <= cta_lim) {
                const int blk = __ldg(table + key / kBlockSize);
                if (blk >= 0 && (int64_t)blk < p.num_blocks) {
                    okk = true;
#pragma unroll
                    for (int pl = 0; pl < 2; ++pl) {
                        const uint32_t* row = reinterpret_cast<const uint32_t*>(
                            p.cache + (((int64_t)blk * 2 + pl) * kBlockSize + key % kBlockSize) * H * Gm::RB +
                            (int64_t)h * Gm::RB);
#pragma unroll
                        for (int i = 0; i < NW; ++i) w[pl][i] = __ldg(row + i);
                    }
                } else if (key % kBlockSize == 0) {
                    count_status(p.status, 1);
                }
            }
        };
        // the MMA issue of P.V for tile t (issuer thread only)
        auto issue_pv = [&](int t) -> bool {
            const int b = t & 1;
            if (!wait(&p_full[b], (uint32_t)(t >> 1) & 1u)) return false;
            tc_fence_after();
            const uint32_t pcol = tmem + (b ? Tm::kS1 : Tm::kS0);
            const uint32_t vb = smem_u32(vtile(b));
#pragma unroll
            for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                const uint32_t a = pcol + (kk < 4 ? 8u * kk : 64u + 8u * (kk - 4));
                const uint64_t bd = smem_desc_sw128(vb + (uint32_t)kk * 16u * 128u, kPfKeys * 128u, 1024u);
                mma_ts(tmem + Tm::kO, a, bd, idPV, t > 0 || kk > 0);
            }
            mma_commit(&pv_done[b]);
            return true;
        };
        if (nkt > 0) fetch(0, cur, cur_ok);
        bool ok = true;
        for (int j = 0; j < nkt && ok; ++j) {
            const int b = j & 1;
            if (j == 1) ok = wait(q_ready, 0);                           // the query staging sat on tiles 1
            if (ok && j >= 2) ok = wait(&pv_done[b], (uint32_t)((j - 2) >> 1) & 1u);   // tiles b free
            if (!__all_sync(0xffffffffu, ok)) break;
            if (j + 1 < nkt) fetch(j + 1, nxt, nxt_ok);
            uint8_t* kt = ktile(b);
            uint8_t* vt = vtile(b);
#pragma unroll
            for (int pl = 0; pl < 2; ++pl) {
                uint8_t* t = pl ? vt : kt;
                const uint32_t zp = cur[pl][Gm::KW] & 15u;
#pragma unroll
                for (int w = 0; w < Gm::KW; ++w) {
                    const uint4 v = cur_ok ? dequant_word(cur[pl][w], zp) : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(t + (uint32_t)(w / 8) * (kPfKeys * 128u) + swz128((uint32_t)k, (uint32_t)(w % 8))) = v;
                }
            }
            sk[b * kPfKeys + k] = cur_ok ? __uint_as_float(cur[0][Gm::KW] & 0xFFFFFFF0u) : 0.0f;
            const uint32_t vsw = cur_ok ? cur[1][Gm::KW] : 0u;
            sv[b * kPfKeys + k] = vsw;
            const uint32_t wmax = __reduce_max_sync(0xffffffffu, vsw);   // positive floats order like their bits
            if (lane == 0) eblkw[b * 4 + (warp - kPfSoftmaxWarps)] = (wmax >> 23) & 0xFFu;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor core reads
            mbar_arrive(&kv_full[b]);
#pragma unroll
            for (int pl = 0; pl < 2; ++pl)
#pragma unroll
                for (int i = 0; i < NW; ++i) cur[pl][i] = nxt[pl][i];
            cur_ok = nxt_ok;
            if (issuer) {
                // S of tile j (its S buffer was last read by P.V of tile j - 2, waited for above)
                bool mok = (j > 0 || wait(q_ready, 0)) && wait(&kv_full[b], (uint32_t)(j >> 1) & 1u);
                if (mok) {
                    tc_fence_after();
                    const uint32_t sd = tmem + (b ? Tm::kS1 : Tm::kS0);
                    const uint32_t kb = smem_u32(kt);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
#pragma unroll
                        for (int kk = 0; kk < KSTEPS; ++kk) {
                            const uint64_t bd = smem_desc_sw128(
                                kb + (uint32_t)(kk / 4) * (kPfKeys * 128u) + (uint32_t)(kk % 4) * 32u, 16u, 1024u);
                            mma_ts(sd, tmem + (half ? Tm::kQl : Tm::kQh) + 8u * kk, bd, idS, half > 0 || kk > 0);
                        }
                    }
                    mma_commit(&s_full[b]);
                    if (j >= 1) mok = issue_pv(j - 1);
                }
                ok = mok;
            }
            __syncwarp();
        }
        if (issuer) {
            if (ok && nkt > 0) issue_pv(nkt - 1);
            // every MMA issued has completed before the CTA tears tensor memory down
            mma_commit(flush);
            (void)mbar_wait(flush, 0);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPfMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

template <int D, typename QT, typename OT>
cudaError_t launch_prefill_t(const AttnParams& p, int max_query_len, cudaStream_t stream) {
    const size_t smem = PfLayout<D>::kBytes;
    cudaError_t err = opt_in_smem<prefill_kernel<D, QT, OT>>(smem);
    if (err != cudaSuccess) return err;
    const int BQ = kPfRows / p.G;
    dim3 grid((unsigned)(((max_query_len + BQ - 1) / BQ) * p.H), 1, p.num_seqs);
    prefill_kernel<D, QT, OT><<<grid, kPfThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int D, typename QT>
cudaError_t prefill_by_out(const AttnParams& p, int mql, DType out_dt, cudaStream_t s) {
    switch (out_dt) {
        case DType::F16: return launch_prefill_t<D, QT, __half>(p, mql, s);
        case DType::BF16: return launch_prefill_t<D, QT, __nv_bfloat16>(p, mql, s);
        default: return launch_prefill_t<D, QT, float>(p, mql, s);
    }
}

}  // namespace

cudaError_t launch_prefill(const AttnParams& p, int head_size, int max_query_len, DType q_dt, DType out_dt,
                           cudaStream_t stream) {
    if (head_size == 128)
        return q_dt == DType::BF16 ? prefill_by_out<128, __nv_bfloat16>(p, max_query_len, out_dt, stream)
                                   : prefill_by_out<128, __half>(p, max_query_len, out_dt, stream);
    return q_dt == DType::BF16 ? prefill_by_out<64, __nv_bfloat16>(p, max_query_len, out_dt, stream)
                               : prefill_by_out<64, __half>(p, max_query_len, out_dt, stream);
}

}  // namespace kvi4
