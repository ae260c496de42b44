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
//   online softmax     per row: logit = S * s'_K * k0 * 2^-e (k0 = c * scale * log2(e), e the
//                       row's query prescale), causal mask on the diagonal tiles, a reference
//                       maximum m that moves only on jumps of more than 2^8; the weights
//                       P_w = 2^(logit - m + 127 - E) * s'_V (one FMA before exp2; E a reference
//                       exponent of the V scales) as fp16 written back over S, and their sum l'
//                       carries the same 2^(127 - E), so out = O / l' without it
//   O += P_w (V - zp)  tcgen05.mma, A = P_w from tensor memory, B = the values dequantised to
//                       fp16 in shared memory (K's row layout, rows in the key order the weights
//                       are laid out in, read MN-major); O stays in tensor memory for the whole
//                       key range
// and un-rotates its rows at the end.
//
// Warp roles (480 threads): warps 0-7 own the rows, rotate the queries and run the softmax and
// the epilogue (warp w the 16 rows 32 (w % 4) + 16 (w / 4) .. + 15, read in the 16-lane
// tensor-memory layout, so that a row's four threads meet by shuffles); warps 13-14 stage the
// packed K and V rows of the coming key tiles in shared memory with asynchronous copies, four
// tiles ahead; warps 8-11 dequantise a staged tile (one key per thread) into the fp16 K and V
// tiles of its parity, each half once the MMA that read it before is done; warp 12 allocates
// tensor memory and one of its threads issues every MMA, S or P.V, whichever is ready.
// Dimension order: a tile row holds each code word's eight dimensions in the order the nibble
// unpacking yields them (8w + 0, 4, 1, 5, 2, 6, 3, 7), so the dequantisation needs no permutes;
// Q' is stored in tensor memory in the same order (the contraction over dimensions does not care),
// and the epilogue puts O's columns back in dimension order.
// Tensor memory (512 columns): Q' high, Q' low, two S buffers (S of tile j + 1 is computed while
// the softmax of tile j runs), O.  Hand-offs go through mbarriers (tcgen05.commit for the MMAs);
// every wait is bounded and a wait that gives up is counted and winds the CTA down.
// The kernel is a template on OPTS (window / softcap / ALiBi on the logits): attn_prefill.cu
// instantiates it without them, attn_prefill_opts.cu with them, so that the default kernel carries
// none of their code.
#pragma once

#include <cudaTypedefs.h>

#include <type_traits>

#include "attn_common.cuh"

namespace kvi4 {
namespace {

constexpr int kPfRows = kPrefillRows;         // query rows per CTA (the MMA M)
constexpr int kPfKeys = 128;                  // keys per tile (the S MMA N, the P.V MMA K)
constexpr int kPfPairs = 2;                   // fp16 K/V tile pairs in shared memory
constexpr int kPfKRing = 4;                   // key-tile records (K scales, "K converted") in flight
constexpr int kPfRawStages = 4;               // packed key tiles staged ahead of their conversion
constexpr int kPfSoftmaxWarps = 8;
constexpr int kPfDequantWarps = 4;
constexpr int kPfMmaWarp = kPfSoftmaxWarps + kPfDequantWarps;
constexpr int kPfLoadWarps = 2;               // one per plane (K, V)
constexpr int kPfThreads = (kPfMmaWarp + 1 + kPfLoadWarps) * 32;
constexpr int kPfSoftmaxThreads = kPfSoftmaxWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kPfLazyMax = 8.0f;            // log2 units the row's reference maximum may trail
constexpr uint32_t kPfLazyExp = 4;            // binades the V exponent reference may trail

// Shared-memory layout (bytes from a 1024-aligned base).  A fp16 tile is 128 keys x D dims as
// D/64 chunks of [128 rows x 128 B], 128-byte swizzled; kPfPairs K/V tile pairs (key tile j uses
// pair j % kPfPairs): [K 0][V 0][K 1][V 1].  Before the first tile pair 1 holds the CTA's query rows
// (K 1, the same layout) and the rotation matrix (V 1), and after the last the fp32 output rows sit
// over pairs 0-1 (rows of D + 4 floats).  Then kPfRawStages staging buffers of packed rows as the cache holds them,
// [plane][128 keys][kWindow words] (key tile j in stage j % kPfRawStages): a row of D/8 + 1 words
// arrives with the 16-byte-aligned window of cache bytes around it, at its own word offset 0..3.
template <int D>
struct PfLayout {
    static constexpr uint32_t kTile = (D / 64) * kPfKeys * 128;
    static constexpr uint32_t kOStride = D + 4;                                   // floats per staged row
    static constexpr uint32_t kMisc = 2 * kPfPairs * kTile;
    static_assert((D / 64) * D * 128 <= kTile, "rotation matrix staging");
    static_assert(kPfRows * kOStride * 4 <= 4 * kTile, "output staging");
    static constexpr uint32_t kRowWords = D / 8 + 1;                              // packed row: codes + scale
    static constexpr uint32_t kChunks = (kRowWords + 3 + 3) / 4;                  // 16-byte chunks of a window
    static constexpr uint32_t kWindow = 4 * kChunks;
    static constexpr uint32_t kRawStage = 2u * kPfKeys * kWindow * 4;
    static constexpr uint32_t kRaw = kMisc;
    // misc region
    static constexpr uint32_t kSk = kRaw + kPfRawStages * kRawStage;    // [kring][128] f32 s'_K * k0 (0: no key)
    static constexpr uint32_t kDeadF = kSk + kPfKRing * kPfKeys * 4;  // [kring][4] u32: a dequantising warp saw a key with no row
    static constexpr uint32_t kSv = kDeadF + kPfKRing * 4 * 4;       // [pairs][128] f32 s'_V
    static constexpr uint32_t kEblk = kSv + kPfPairs * kPfKeys * 4;  // [pairs][4] per-warp max V exponent
    static constexpr uint32_t kSigns = kEblk + kPfPairs * 4 * 4;     // [D] f32
    static constexpr uint32_t kSignBits = kSigns + D * 4;            // [D / 32] u32: bit j of word i: sign 32 i + j < 0
    static constexpr uint32_t kBars = (kSignBits + D / 8 + 7u) & ~7u;   // mbarriers
    // k_full[kring], k_free[pairs], v_full[pairs], v_free[pairs], pv_done[2], s_full[2], p_full[2], q_ready,
    // flush, q_tma, rot_in, rot_done, epi, raw_full[stages], raw_free[stages]
    static constexpr int kNumBars = kPfKRing + 3 * kPfPairs + 2 + 2 + 2 + 1 + 1 + 3 + 1 + 2 * kPfRawStages;
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
// the same with bf16 A and B
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n, uint32_t b_mn) {
    return idesc_f16(n, b_mn) | (1u << 7) | (1u << 10);
}

// A and B both from shared memory (descriptors), D in tensor memory
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)acc)
        : "memory");
}

// Tiled 3-D tensor copy global -> shared: the tensor map's box at (x, y, z), completion signalled on
// the mbarrier (transaction bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// position in a group of 16 contraction slots that the 16-lane tensor-memory layout gives the
// value of column p (a thread's column pair 8i + 2t, + 1 is stored as word 8 (i / 2) + 2t + i % 2)
// four words of fp16 (one = 0x3C00) or bf16 (one = 0x3F80) +-1: element j is negative where bit j of
// neg8 is set (element 2e in the low half of word e)
__device__ __forceinline__ void pm1_words(uint32_t neg8, uint32_t one, uint32_t (&w)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
        w[e] = (one * 0x10001u) | (((neg8 >> (2 * e)) & 1u) << 15) | (((neg8 >> (2 * e + 1)) & 1u) << 31);
}
// the dimension a tile column holds: each group of 8 in the order 0, 4, 1, 5, 2, 6, 3, 7
__host__ __device__ constexpr int dim_of_column(int c) { return (c & ~7) + ((c & 7) >> 1) + 4 * (c & 1); }
__host__ __device__ constexpr int slot_of_column(int p) {
    return (p & ~15) + 4 * ((p >> 1) & 3) + 2 * ((p >> 3) & 1) + (p & 1);
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



// 16 lanes x 256 bits, four times along the columns (16 registers): thread i = 4 g + t gets, for
// repetition c, r[4c] = (lane g, column 8c + 2t), r[4c + 1] = (g, 8c + 2t + 1), r[4c + 2] = (g + 8,
// 8c + 2t), r[4c + 3] = (g + 8, 8c + 2t + 1), lanes counted from the address's lane.
__device__ __forceinline__ void tmem_ld_q4(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// the same layout, one repetition (4 registers)
__device__ __forceinline__ void tmem_ld_q1(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_q1(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3])
                 : "memory");
}
// the same layout, eight repetitions (32 registers)
__device__ __forceinline__ void tmem_ld_q8(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }


// Byte offset of 16-byte chunk c (0..7) of row r in a [rows x 128 B] block with the 128-byte
// swizzle the tensor-core descriptors expect: the chunk index is XOR-ed with r mod 8.
__device__ __forceinline__ uint32_t swz128(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

// TILED: the grid covers the batch's prefill query tiles through the walker's tile index (a batch
// of many decode sequences); otherwise one grid slice per sequence.  Separate instantiations keep the
// per-sequence grid's indices plain block coordinates.
template <int D, typename QT, typename OT, bool OPTS, bool TILED>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap qmap) {
    using Gm = Geo<D>;
    using Ly = PfLayout<D>;
    using Tm = PfTmem<D>;
    constexpr int KSTEPS = D / 16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- the CTA's rows; everything up to the barrier set-up exits uniformly.  A sequence's
    // tiles run in descending order, so its longest rows start first.  Two grids:
    //  * pf_tiles_cap > 0: tile v of the batch's prefill query tiles (ws_ptile: each sequence's
    //    first tile), found by a 32-way search in each warp;
    //  * otherwise one grid slice (blockIdx.z) per sequence, ntile tiles each.
    const int v = (int)(blockIdx.x / (unsigned)p.H), h = (int)(blockIdx.x % (unsigned)p.H);
    int seq, qtile;
    if constexpr (TILED) {
        const int32_t* ptile = p.ws_ptile;
        int lo = 0, hi = p.num_seqs + 1;   // ptile[lo] <= v < ptile[hi], ptile[num_seqs + 1] = infinity
        while (hi - lo > 1) {
            const int step = (hi - lo + 31) / 32;
            const int idx = lo + step * lane;
            const unsigned le = __ballot_sync(0xffffffffu, idx < hi && __ldg(ptile + idx) <= v);
            lo += step * (31 - __clz(le));   // lane 0 (ptile[lo] <= v) is always set
            hi = min(hi, lo + step);
        }
        if (lo >= p.num_seqs) return;   // past the batch's last tile (ptile[num_seqs] = the total)
        seq = lo;
        qtile = __ldg(ptile + seq + 1) - 1 - v;
    } else {
        seq = blockIdx.z;
        qtile = (int)(gridDim.x / (unsigned)p.H) - 1 - v;
    }
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
    float* sv = reinterpret_cast<float*>(smem + Ly::kSv);
    uint32_t* eblkw = reinterpret_cast<uint32_t*>(smem + Ly::kEblk);
    float* sgn = reinterpret_cast<float*>(smem + Ly::kSigns);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::kBars);
    // The K and V halves of a tile pair live apart: K tile j is free once S of tile j is done, V tile
    // j once its P.V is.  "K converted" is kept per key tile mod kPfKRing so that no record is
    // overwritten before the rows of its tile have read it (tile j + 4 waits for S of tile j + 2,
    // which waits for P.V of tile j).
    uint64_t* k_full = bars;                    // [kring] K tile and scales of tile j (128 arrivals)
    uint64_t* k_free = k_full + kPfKRing;       // [pairs] K tile j % 2 read by S of tile j (commit)
    uint64_t* v_full = k_free + kPfPairs;       // [pairs] V tile and scales of tile j (128 arrivals)
    uint64_t* v_free = v_full + kPfPairs;       // [pairs] V tile j % 2 read by P.V of tile j (commit)
    uint64_t* pv_done = v_free + kPfPairs;      // [2] P.V of tile j done (commit): S buffer j % 2 and O free
    uint64_t* s_full = pv_done + 2;             // [2] S of the tile in tensor memory (commit)
    uint64_t* p_full = s_full + 2;              // [2] P of the tile in tensor memory (256 arrivals)
    uint64_t* q_ready = p_full + 2;             // queries in tensor memory, staging free (256 arrivals)
    uint64_t* flush = q_ready + 1;              // the MMA thread's last commit (teardown)
    uint64_t* q_tma = flush + 1;                // the CTA's query rows in shared memory (bytes)
    uint64_t* rot_in = q_tma + 1;               // the rotation matrix in shared memory (256 arrivals)
    uint64_t* rot_done = rot_in + 1;            // the rotated queries in tensor memory (commit)
    // the 256 row threads meet (a bounded wait, unlike a hardware named barrier) once the output
    // rows are staged
    uint64_t* epi = rot_done + 1;
    uint64_t* raw_full = epi + 1;            // [stages] packed rows of a key tile landed (64 lanes)
    uint64_t* raw_free = raw_full + kPfRawStages;   // [stages] that stage converted (128 arrivals)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kFlags);

    if (threadIdx.x == 0) {
        for (int b = 0; b < kPfKRing; ++b) mbar_init(&k_full[b], kPfDequantWarps * 32);
        for (int b = 0; b < kPfPairs; ++b) {
            mbar_init(&k_free[b], 1);
            mbar_init(&v_full[b], kPfDequantWarps * 32);
            mbar_init(&v_free[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&pv_done[b], 1);
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], kPfSoftmaxThreads);
        }
        mbar_init(q_ready, kPfSoftmaxThreads);
        mbar_init(flush, 1);
        mbar_init(q_tma, 1);
        mbar_init(rot_in, kPfSoftmaxThreads);
        mbar_init(rot_done, 1);
        mbar_init(epi, kPfSoftmaxThreads);
        for (int i = 0; i < kPfRawStages; ++i) {
            mbar_init(&raw_full[i], kPfLoadWarps * 32);
            mbar_init(&raw_free[i], kPfDequantWarps * 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    uint32_t* signbits = reinterpret_cast<uint32_t*>(smem + Ly::kSignBits);
    if (threadIdx.x < D) {   // whole warps (D is a multiple of 32)
        const bool neg = p.signs[threadIdx.x] < 0.0f;
        sgn[threadIdx.x] = neg ? -1.0f : 1.0f;
        const uint32_t m = __ballot_sync(0xffffffffu, neg);
        if (lane == 0) signbits[warp] = m;
    }
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
    // the row threads counted by the barrier meet (warp-uniform result)
    auto rows_meet = [&](uint64_t* bar, uint32_t parity) -> bool {
        mbar_arrive(bar);
        return __all_sync(0xffffffffu, wait(bar, parity));
    };

    if (warp < kPfSoftmaxWarps) {
        // ================================================================ rows: softmax + epilogue
        // Warp w owns the 16 rows 32 (w % 4) + 16 (w / 4) .. + 15 in the 16-lane tensor-memory
        // layout: thread (g, t) = (lane / 4, lane % 4) holds rows ra = rbase + g and rb = ra + 8 and,
        // of every group of 8 columns, columns 2t and 2t + 1; a row's maximum and sum meet over its
        // four threads by two shuffles.
        const int rbase = 32 * (warp & 3) + 16 * (warp >> 2);
        const int t4 = lane & 3;
        const int ra = rbase + (lane >> 2), rb = ra + 8;
        const uint32_t trow = tmem + ((uint32_t)rbase << 16);
        // ---- the rotation v = H_d (D q) as a matrix product on the tensor cores: the query rows
        // (loaded by the MMA thread) times B[p][k] = sign_k (-1)^popcount(n(p) & k), where row p of
        // B is the dimension n(p) whose value column p must hold for the query halves below to land
        // in the tiles' dimension order.  The entries are +-1, exact in the query type.
        {
            // row p = tid / (256 / D) of B, its chunks (8 inputs k each) split over 256 / D threads;
            // (-1)^popcount(n & k) = (-1)^popcount(n & 8 k8) (-1)^popcount(n & k % 8)
            constexpr int kRowChunks = D / 8, kThreadsPerRow = kPfSoftmaxThreads / D, kChunksPerThread = kRowChunks / kThreadsPerRow;
            uint8_t* qb = vtile(1);
            const uint32_t one = std::is_same<QT, __nv_bfloat16>::value ? 0x3F80u : 0x3C00u;
            const int prow = threadIdx.x / kThreadsPerRow;
            const int n = dim_of_column(slot_of_column(prow));
            uint32_t par8 = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) par8 |= ((uint32_t)__popc(n & j) & 1u) << j;
#pragma unroll
            for (int it = 0; it < kChunksPerThread; ++it) {
                const int k8 = (threadIdx.x % kThreadsPerRow) * kChunksPerThread + it;
                const uint32_t sb = (signbits[k8 / 4] >> (8 * (k8 % 4))) & 0xFFu;
                const uint32_t neg = par8 ^ sb ^ ((__popc(n & (8 * k8)) & 1) ? 0xFFu : 0u);
                uint32_t w[4];
                pm1_words(neg, one, w);
                *reinterpret_cast<uint4*>(qb + (uint32_t)(k8 / 8) * (uint32_t)(D * 128) + swz128((uint32_t)prow, (uint32_t)(k8 % 8))) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor core reads
            mbar_arrive(rot_in);
        }
        // ---- a power-of-two prescale 2^e bringing the row's max |v| into [2^14, 2^15), then fp16
        // high + low halves (qh + ql carries about 22 bits: a plain fp16 copy turns large keys into
        // logit errors a heavy-tailed cache shows) into tensor memory, where S's MMAs read them
        float rs_a = 1.0f, rs_b = 1.0f;   // 2^-e of each row
        bool ok = wait(rot_done, 0);
        if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            float v[D / 2];   // v[4i], v[4i + 1]: row a, columns 8i + 2t, + 1; v[4i + 2], v[4i + 3]: row b
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 64) tmem_ld_q8(trow + Tm::kS0 + c0, reinterpret_cast<uint32_t*>(v) + c0 / 2);
            tmem_ld_wait();
            float mxa = 0.0f, mxb = 0.0f;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                mxa = fmaxf(mxa, fmaxf(fabsf(v[4 * i]), fabsf(v[4 * i + 1])));
                mxb = fmaxf(mxb, fmaxf(fabsf(v[4 * i + 2]), fabsf(v[4 * i + 3])));
            }
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
            const int ea = prescale_exponent(mxa), eb = prescale_exponent(mxb);   // rows of zeros: 2^0
            const float sca = exp2i(ea), scb = exp2i(eb);
            rs_a = exp2i(-ea);
            rs_b = exp2i(-eb);
#pragma unroll
            for (int q = 0; q < D / 16; ++q) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = 2 * q + e;
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const float sc = rr ? scb : sca;
                        const float y0 = v[4 * i + 2 * rr] * sc, y1 = v[4 * i + 2 * rr + 1] * sc;
                        const __half h0 = __float2half_rn(y0), h1 = __float2half_rn(y1);
                        const __half l0 = __float2half_rn(y0 - __half2float(h0)), l1 = __float2half_rn(y1 - __half2float(h1));
                        hw[2 * rr + e] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                        lw[2 * rr + e] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
                    }
                }
                tmem_st_q1(trow + Tm::kQh + 8 * q, hw);
                tmem_st_q1(trow + Tm::kQl + 8 * q, lw);
            }
            tmem_st_wait();
        } else {
            ok = false;
        }
        tc_fence_before();
        mbar_arrive(q_ready);
        // ---- the key tiles
        const int qta = qt0 + ra / G, qtb = qt0 + rb / G;
        const int pos_a = qta < qlen ? pos0 + qta : -1, pos_b = qtb < qlen ? pos0 + qtb : -1;   // last visible key
        float m_a = kNegBig, m_b = kNegBig;     // reference maxima (log2 units)
        float l_a = 0.0f, l_b = 0.0f;           // this thread's part of the sums of 2^(127-E) p
        uint32_t E = 0;                         // reference biased exponent of the V scales (0: none yet)
        const uint32_t* deadf = reinterpret_cast<const uint32_t*>(smem + Ly::kDeadF);

        for (int j = 0; j < nkt && ok; ++j) {
            const int b = j & 1;
            const uint32_t ph = (uint32_t)(j >> 1) & 1u;
            const int kb = j % kPfPairs, kr = j % kPfKRing;
            ok = wait(&s_full[b], ph) && wait(&k_full[kr], (uint32_t)(j / kPfKRing) & 1u) &&
                 wait(&v_full[kb], (uint32_t)(j / kPfPairs) & 1u);
            if (__any_sync(0xffffffffu, !ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t scol = trow + (b ? Tm::kS1 : Tm::kS0);
            uint32_t s[64];   // s[4i], s[4i + 1]: row a, columns 8i + 2t, + 1; s[4i + 2], s[4i + 3]: row b
            tmem_ld_q8(scol, s);
            tmem_ld_q8(scol + 64, s + 32);
            tmem_ld_wait();
            // x = S * s'_K * k0 (0 scale: no key), masked; the row maxima
            const int key0 = j * kPfKeys;
            const float* skb = sk + kr * kPfKeys + 2 * t4;
            const bool clean = (deadf[kr * 4] | deadf[kr * 4 + 1] | deadf[kr * 4 + 2] | deadf[kr * 4 + 3]) == 0u &&
                               key0 + kPfKeys - 1 <= min(pos_a, pos_b);
            float bma = -INFINITY, bmb = -INFINITY;
            if (!OPTS && __all_sync(0xffffffffu, clean)) {   // every key live and visible to both rows
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 k2 = *reinterpret_cast<const float2*>(skb + 8 * i);
                    const float2 xa = mul_f32x2(make_float2(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1])), k2);
                    const float2 xb = mul_f32x2(make_float2(__uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3])), k2);
                    s[4 * i] = __float_as_uint(xa.x);
                    s[4 * i + 1] = __float_as_uint(xa.y);
                    s[4 * i + 2] = __float_as_uint(xb.x);
                    s[4 * i + 3] = __float_as_uint(xb.y);
                    bma = fmaxf(bma, fmaxf(xa.x, xa.y));
                    bmb = fmaxf(bmb, fmaxf(xb.x, xb.y));
                }
            } else if (OPTS) {
                // window / softcap / ALiBi on the log2 logit x rs, then back over rs (a power of two:
                // exact), so that the rest of the tile is the same as without options
                const float irs_a = 1.0f / rs_a, irs_b = 1.0f / rs_b;
                const float sla = (p.opts & kOptAlibi) ? __ldg(p.alibi + h * G + ra % G) * kLog2e : 0.0f;
                const float slb = (p.opts & kOptAlibi) ? __ldg(p.alibi + h * G + rb % G) * kLog2e : 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 k2 = *reinterpret_cast<const float2*>(skb + 8 * i);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float kk = e ? k2.y : k2.x;
                        const int key = key0 + 8 * i + 2 * t4 + e;
                        float xa = kk > 0.0f && key <= pos_a ? __uint_as_float(s[4 * i + e]) * kk : -INFINITY;
                        float xb = kk > 0.0f && key <= pos_b ? __uint_as_float(s[4 * i + 2 + e]) * kk : -INFINITY;
                        xa = apply_opts(xa * rs_a, key, pos_a, sla, p, pos0) * irs_a;
                        xb = apply_opts(xb * rs_b, key, pos_b, slb, p, pos0) * irs_b;
                        s[4 * i + e] = __float_as_uint(xa);
                        s[4 * i + 2 + e] = __float_as_uint(xb);
                        bma = fmaxf(bma, xa);
                        bmb = fmaxf(bmb, xb);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 k2 = *reinterpret_cast<const float2*>(skb + 8 * i);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float kk = e ? k2.y : k2.x;
                        const int key = key0 + 8 * i + 2 * t4 + e;
                        const float xa = kk > 0.0f && key <= pos_a ? __uint_as_float(s[4 * i + e]) * kk : -INFINITY;
                        const float xb = kk > 0.0f && key <= pos_b ? __uint_as_float(s[4 * i + 2 + e]) * kk : -INFINITY;
                        s[4 * i + e] = __float_as_uint(xa);
                        s[4 * i + 2 + e] = __float_as_uint(xb);
                        bma = fmaxf(bma, xa);
                        bmb = fmaxf(bmb, xb);
                    }
                }
            }
            bma = fmaxf(bma, __shfl_xor_sync(0xffffffffu, bma, 1));
            bmb = fmaxf(bmb, __shfl_xor_sync(0xffffffffu, bmb, 1));
            bma = fmaxf(bma, __shfl_xor_sync(0xffffffffu, bma, 2));
            bmb = fmaxf(bmb, __shfl_xor_sync(0xffffffffu, bmb, 2));
            // in log2 units (rs > 0: a power of two scales exactly); the four threads of a row take
            // the same decisions
            bma *= rs_a;
            bmb *= rs_b;
            const bool up_a = bma > m_a + kPfLazyMax, up_b = bmb > m_b + kPfLazyMax;
            const float fm_a = up_a ? fast_exp2(m_a - bma) : 1.0f, fm_b = up_b ? fast_exp2(m_b - bmb) : 1.0f;
            if (up_a) m_a = bma;
            if (up_b) m_b = bmb;
            const uint32_t* eb4 = eblkw + kb * 4;
            const uint32_t eb = max(max(eb4[0], eb4[1]), max(eb4[2], eb4[3]));
            const uint32_t Eeff = E ? E : 127u;
            float fe = 1.0f;
            if (E == 0u ? eb > 0u : eb > E + kPfLazyExp) {
                // rebase from 2^(127 - Eeff) to 2^(127 - eb); 0 when the jump underflows
                fe = eb > Eeff + 126u ? 0.0f : __uint_as_float((127u + Eeff - eb) << 23);
                E = eb;
            }
            const float f_a = fm_a * fe, f_b = fm_b * fe;
            l_a *= f_a;
            l_b *= f_b;
            if (j > 0 && __any_sync(0xffffffffu, f_a != 1.0f || f_b != 1.0f)) {
                // O must hold P.V of the previous tile before it is rescaled
                ok = wait(&pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u);
                if (__any_sync(0xffffffffu, !ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float2 fa2 = make_float2(f_a, f_a), fb2 = make_float2(f_b, f_b);
                // eight columns at a time: the scores stay in registers meanwhile
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 8) {
                    uint32_t o[4];
                    tmem_ld_q1(trow + Tm::kO + c0, o);
                    tmem_ld_wait();
                    const float2 oa = mul_f32x2(make_float2(__uint_as_float(o[0]), __uint_as_float(o[1])), fa2);
                    const float2 ob = mul_f32x2(make_float2(__uint_as_float(o[2]), __uint_as_float(o[3])), fb2);
                    o[0] = __float_as_uint(oa.x);
                    o[1] = __float_as_uint(oa.y);
                    o[2] = __float_as_uint(ob.x);
                    o[3] = __float_as_uint(ob.y);
                    tmem_st_q1(trow + Tm::kO + c0, o);
                }
                tmem_st_wait();
            }
            // p' = 2^(x rs - m + 127 - E), w = p' s'_V as fp16 pairs over the first 64 S columns: the
            // pair of columns 8i + 2t, + 1 goes to column 8 (i / 2) + 2t + i % 2 (the V tile holds its
            // rows in the matching order)
            const float eoff = (float)(127 - (int)(E ? E : 127u));
            const float2 rsa2 = make_float2(rs_a, rs_a), rsb2 = make_float2(rs_b, rs_b);
            const float2 moa2 = make_float2(eoff - m_a, eoff - m_a), mob2 = make_float2(eoff - m_b, eoff - m_b);
            const float* svb = sv + kb * kPfKeys + 2 * t4;
            float2 lsa = make_float2(0.0f, 0.0f), lsb = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t pw[4];
#pragma unroll
                for (int i = 2 * q; i < 2 * q + 2; ++i) {
                    const float2 v2 = *reinterpret_cast<const float2*>(svb + 8 * i);
                    const float2 ea = fma_f32x2(make_float2(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1])), rsa2, moa2);
                    const float2 eb2 = fma_f32x2(make_float2(__uint_as_float(s[4 * i + 2]), __uint_as_float(s[4 * i + 3])), rsb2, mob2);
                    const float2 pa = make_float2(fast_exp2(ea.x), fast_exp2(ea.y));
                    const float2 pb = make_float2(fast_exp2(eb2.x), fast_exp2(eb2.y));
                    lsa = add_f32x2(lsa, pa);
                    lsb = add_f32x2(lsb, pb);
                    const float2 wa = mul_f32x2(pa, v2), wb = mul_f32x2(pb, v2);
                    const int e = i & 1;
                    pw[e] = pack_f16x2(wa.x, wa.y);
                    pw[2 + e] = pack_f16x2(wb.x, wb.y);
                }
                tmem_st_q1(scol + 8 * q, pw);
            }
            l_a += lsa.x + lsa.y;
            l_b += lsb.x + lsb.y;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[b]);
        }
        // ---- epilogue: O / l' (the 2^(127 - E) of both cancels), staged in dimension order, un-rotated
        if (ok && nkt > 0) ok = wait(&pv_done[(nkt - 1) & 1], (uint32_t)((nkt - 1) >> 1) & 1u);
        tc_fence_after();
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
        // the last P.V is done, so nothing reads the tile pairs the staging below overwrites
        const bool good = __all_sync(0xffffffffu, ok) && nkt > 0;
        const float sc_a = l_a > 0.0f ? 1.0f / l_a : 0.0f, sc_b = l_b > 0.0f ? 1.0f / l_b : 0.0f;
        float* ost_a = reinterpret_cast<float*>(tiles) + ra * Ly::kOStride;
        float* ost_b = reinterpret_cast<float*>(tiles) + rb * Ly::kOStride;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[16];
            if (good) {
                tmem_ld_q4(trow + Tm::kO + c0, o);
                tmem_ld_wait();
            }
            // column 8w + j holds dimension 8w + (0, 4, 1, 5, 2, 6, 3, 7)[j]
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = c0 + 8 * i + 2 * t4 + e;
                    const int d = (c & ~7) + ((c & 1) << 2) + ((c & 7) >> 1);
                    ost_a[d] = good ? __uint_as_float(o[4 * i + e]) * sc_a : 0.0f;
                    ost_b[d] = good ? __uint_as_float(o[4 * i + 2 + e]) * sc_b : 0.0f;
                }
            }
        }
        if (!rows_meet(epi, 0)) ok = false;
        // un-rotation out = c D H x, four rows at a time (their butterfly chains interleave)
        const float* ost = reinterpret_cast<const float*>(tiles);
        constexpr int RPW = kPfRows / kPfSoftmaxWarps;
#pragma unroll 1
        for (int i0 = 0; i0 < RPW && ok; i0 += 4) {
            float xv[4][D / 32];
#pragma unroll
            for (int v = 0; v < 4; ++v)
#pragma unroll
                for (int k = 0; k < D / 32; ++k) xv[v][k] = ost[(warp * RPW + i0 + v) * Ly::kOStride + lane + 32 * k];
            warp_fwht_batch<D, 4>(xv);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int R = warp * RPW + i0 + v;
                const int qt = qt0 + R / G, gg = R % G;
                if (qt >= qlen) continue;
                const int64_t ooff = ((int64_t)(q0 + qt) * Hq + h * G + gg) * D;
#pragma unroll
                for (int k = 0; k < D / 32; ++k)
                    store_elem<OT>(p.out, ooff + lane + 32 * k, xv[v][k] * p.c * sgn[lane + 32 * k]);
            }
        }
    } else if (warp < kPfMmaWarp) {
        // ================================================================ dequantisation of key tiles
        const int k = threadIdx.x - kPfSoftmaxThreads;   // this thread's key of every tile
        constexpr int NW = Ly::kRowWords;                 // words of a row: codes, then the scale word
        const float k0 = p.c * p.softmax_scale * kLog2e;  // raw score -> log2 logit, before 2^-e
        // word offset of this key's rows in their windows: rows of token slot r start at byte
        // (r H + h) (D/2 + 4) of a block plane, the cache and its block and plane strides are
        // multiples of 16 bytes, and D/2 + 4 is 4 mod 16
        const int row_off = ((k % kBlockSize) * H + h) & 3;
        // the V tile row of this key: the weights of S columns 16 q + 8 e + 2 t + b sit at
        // contraction position 16 q + 4 t + 2 e + b (the 16-lane tensor-memory layout they are
        // written in)
        const uint32_t vrow = (uint32_t)slot_of_column(k);
        for (int j = 0; j < nkt; ++j) {
            const int kb = j % kPfPairs, st = j % kPfRawStages;
            bool ok = wait(&raw_full[st], (uint32_t)(j / kPfRawStages) & 1u);
            if (!__all_sync(0xffffffffu, ok)) break;
            // this key's K and V windows (16-byte loads; lanes k..k+7 hit eight distinct 16-byte bank
            // groups), then the row's words from its offset; a key the loaders skipped (none, or
            // past the CTA's last key) reads as zero words: scale 0
            const uint4* win4 = reinterpret_cast<const uint4*>(smem + Ly::kRaw + st * Ly::kRawStage) + k * Ly::kChunks;
            uint32_t kw[2][NW];
#pragma unroll
            for (int pl = 0; pl < 2; ++pl) {
                uint32_t wv[Ly::kWindow];
#pragma unroll
                for (int c = 0; c < (int)Ly::kChunks; ++c) {
                    const uint4 v = win4[pl * kPfKeys * Ly::kChunks + c];
                    wv[4 * c] = v.x;
                    wv[4 * c + 1] = v.y;
                    wv[4 * c + 2] = v.z;
                    wv[4 * c + 3] = v.w;
                }
#pragma unroll
                for (int w = 0; w < NW + 1; ++w) wv[w] = (row_off & 2) ? wv[w + 2] : wv[w];
#pragma unroll
                for (int w = 0; w < NW; ++w) kw[pl][w] = (row_off & 1) ? wv[w + 1] : wv[w];
            }
            mbar_arrive(&raw_free[st]);
            // K half, then V half, each once its tile is free (K: S of tile j - 2 done, V: its P.V)
#pragma unroll
            for (int pl = 0; pl < 2; ++pl) {
                ok = !(j == 1 && pl == 0) || wait(q_ready, 0);        // the query staging sat on pair 1
                if (ok && j >= kPfPairs) ok = wait(pl ? &v_free[kb] : &k_free[kb], (uint32_t)(j / kPfPairs - 1) & 1u);
                if (!__all_sync(0xffffffffu, ok)) break;
                uint8_t* t = pl ? vtile(kb) : ktile(kb);
                const uint32_t trow = pl ? vrow : (uint32_t)k;
                const uint32_t zp = kw[pl][Gm::KW] & 15u;
                const uint32_t zl = zp_lo_half(zp) * 0x10001u, zh = zp_hi_half(zp) * 0x10001u;
#pragma unroll
                for (int w = 0; w < Gm::KW; ++w) {
                    // code - zp of dimensions 8w + (0, 4), (1, 5), (2, 6), (3, 7): the tile order
                    uint32_t o[4];
                    unpack_word(kw[pl][w], zl, zh, o);
                    *reinterpret_cast<uint4*>(t + (uint32_t)(w / 8) * (kPfKeys * 128u) + swz128(trow, (uint32_t)(w % 8))) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
                if (pl == 0) {
                    sk[(j % kPfKRing) * kPfKeys + k] = __uint_as_float(kw[0][Gm::KW] & 0xFFFFFFF0u) * k0;
                    const uint32_t nodead = __ballot_sync(0xffffffffu, kw[0][Gm::KW] == 0u);
                    if (lane == 0)
                        reinterpret_cast<uint32_t*>(smem + Ly::kDeadF)[(j % kPfKRing) * 4 + (warp - kPfSoftmaxWarps)] = nodead;
                } else {
                    const uint32_t vsw = kw[1][Gm::KW];
                    sv[kb * kPfKeys + k] = __uint_as_float(vsw & 0xFFFFFFF0u);
                    const uint32_t wmax = __reduce_max_sync(0xffffffffu, vsw);   // positive floats order like their bits
                    if (lane == 0) eblkw[kb * 4 + (warp - kPfSoftmaxWarps)] = (wmax >> 23) & 0xFFu;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor core reads
                mbar_arrive(pl ? &v_full[kb] : &k_full[j % kPfKRing]);
            }
            if (!ok) break;
        }
    } else if (warp > kPfMmaWarp) {
        // ================================================================ loads of packed rows
        // Loader warp l copies plane l (K or V) of each key tile into its staging buffer with 16-byte
        // asynchronous copies of each row's aligned window: copy t of a lane moves chunk
        // i = lane + 32 t of the tile's plane in (key, chunk) order, which is also the staging
        // order.  Keys past the CTA's last key, or in a block the table does not name, are
        // zero-filled (scale word 0: no key).  A window never leaves the cache: the cache starts on
        // a 16-byte boundary (the entry point checks) and its size is a multiple of 16 bytes.
        constexpr int C = Ly::kChunks;
        constexpr int kCopies = kPfKeys * C / 32;
        static_assert(kPfKeys * C % 32 == 0, "whole copies per lane");
        const int pl = warp - kPfMmaWarp - 1;
        const int32_t* table = p.block_tables + (int64_t)seq * p.max_blocks_per_seq;
        const int64_t tok_stride = (int64_t)H * Gm::RB, blk_stride = 2 * kBlockSize * tok_stride;
        // the plane of block 0; a row's window is at blk * blk_stride + ((h RB + r tok_stride) & ~15)
        const uint8_t* base = p.cache + (int64_t)pl * kBlockSize * tok_stride;
        // copy t of this lane, the same for every tile: its key (bits 24..30) and its window chunk's
        // byte offset from the block's plane (bits 0..23)
        uint32_t cp[kCopies];
#pragma unroll
        for (int t = 0; t < kCopies; ++t) {
            const int i = lane + 32 * t, key = i / C, c = i - key * C;
            const uint32_t row = (uint32_t)h * (uint32_t)Gm::RB + (uint32_t)(key % kBlockSize) * (uint32_t)tok_stride;
            cp[t] = ((uint32_t)key << 24) | ((row & ~15u) + 16u * (uint32_t)c);
        }
        // lane b < 8: the table entry of keys 16 b .. 16 b + 15 of tile j (-1: no such key); loaded
        // one tile ahead and only checked when used, so that the load is never waited for
        auto lookup = [&](int j) -> int {
            return lane < kPfKeys / kBlockSize && j * kPfKeys + lane * kBlockSize <= cta_lim
                       ? __ldg(table + j * (kPfKeys / kBlockSize) + lane)
                       : -1;
        };
        int blk_next = nkt > 0 ? lookup(0) : -1;
        bool ok = true;
        for (int j = 0; j < nkt && ok; ++j) {
            const int st = j % kPfRawStages;
            if (j >= kPfRawStages) ok = wait(&raw_free[st], (uint32_t)(j / kPfRawStages - 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) break;
            int blkv = blk_next;
            if (j + 1 < nkt) blk_next = lookup(j + 1);
            if (blkv != -1 && (blkv < 0 || (int64_t)blkv >= p.num_blocks)) {   // a block the table does not name
                if (pl == 0) count_status(p.status, 1);
                blkv = -1;
            }
            const uint32_t dst = smem_u32(smem + Ly::kRaw + st * Ly::kRawStage) + (uint32_t)(pl * kPfKeys * C * 16);
            const int key_lim = cta_lim - j * kPfKeys;    // last key of this tile the CTA sees
#pragma unroll
            for (int t = 0; t < kCopies; ++t) {
                const int key = (int)(cp[t] >> 24);
                const int blk = __shfl_sync(0xffffffffu, blkv, key / kBlockSize);
                const bool live = blk >= 0 && key <= key_lim;
                const uint8_t* src = base + (int64_t)(live ? blk : 0) * blk_stride + (cp[t] & 0xFFFFFFu);
                cp_async16_zfill(dst + 16u * (uint32_t)(lane + 32 * t), src, live);
            }
            cp_async_arrive_noinc(&raw_full[st]);
        }
        cp_async_wait_all();   // no copy outlives the CTA
    } else if (lane == 0) {
        // ================================================================ the MMA issuer
        // Issues whichever is ready next: S of tile js (its tile pair dequantised, its S buffer read
        // by P.V of tile js - 2) or P.V of tile jp (its weights in tensor memory).  S runs at most
        // two tiles ahead of P.V.  The issuer polls without sleeping: a suspended issuer would add
        // its wake-up to every hand-off on the critical path.
        constexpr uint32_t idS = idesc_f16(kPfKeys, 0), idPV = idesc_f16(D, 1);
        // the CTA's query rows (token qt0 + R / G, head h G + R % G for row R) into pair 1's K tile,
        // then their rotation into S buffer 0
        {
            mbar_arrive_expect_tx(q_tma, Ly::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tma_load_3d(ktile(1) + c * (kPfRows * 128), &qmap, 64 * c, h * G, q0 + qt0, q_tma);
            bool rok = wait(q_tma, 0) && wait(rot_in, 0);
            if (rok) {
                tc_fence_after();
                constexpr uint32_t idR = std::is_same<QT, __nv_bfloat16>::value ? idesc_bf16(D, 0) : idesc_f16(D, 0);
                const uint32_t qa = smem_u32(ktile(1)), qb = smem_u32(vtile(1));
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const uint64_t ad = smem_desc_sw128(qa + (uint32_t)(kk / 4) * (kPfRows * 128u) + (uint32_t)(kk % 4) * 32u, 16u, 1024u);
                    const uint64_t bd = smem_desc_sw128(qb + (uint32_t)(kk / 4) * (uint32_t)(D * 128) + (uint32_t)(kk % 4) * 32u, 16u, 1024u);
                    mma_ss(tmem + Tm::kS0, ad, bd, idR, kk > 0);
                }
                mma_commit(rot_done);
            }
        }
        auto issue_s = [&](int j) {
            const uint32_t sd = tmem + ((j & 1) ? Tm::kS1 : Tm::kS0);
            const uint32_t kbase = smem_u32(ktile(j % kPfPairs));
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const uint64_t bd = smem_desc_sw128(
                        kbase + (uint32_t)(kk / 4) * (kPfKeys * 128u) + (uint32_t)(kk % 4) * 32u, 16u, 1024u);
                    mma_ts(sd, tmem + (half ? Tm::kQl : Tm::kQh) + 8u * kk, bd, idS, half > 0 || kk > 0);
                }
            }
            mma_commit(&s_full[j & 1]);
            mma_commit(&k_free[j % kPfPairs]);
        };
        auto issue_pv = [&](int t) {
            const uint32_t pcol = tmem + ((t & 1) ? Tm::kS1 : Tm::kS0);
            const uint32_t vb = smem_u32(vtile(t % kPfPairs));
#pragma unroll
            for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                const uint32_t a = pcol + 8u * kk;   // P of keys 16 kk .. 16 kk + 15 (in contraction order)
                const uint64_t bd = smem_desc_sw128(vb + (uint32_t)kk * 16u * 128u, kPfKeys * 128u, 1024u);
                mma_ts(tmem + Tm::kO, a, bd, idPV, t > 0 || kk > 0);
            }
            mma_commit(&pv_done[t & 1]);
            mma_commit(&v_free[t % kPfPairs]);
        };
        bool ok = nkt == 0 || wait(q_ready, 0);
        int js = 0, jp = 0;
        uint64_t t0 = global_timer_ns();
        while (ok && jp < nkt) {
            bool did = false;
            if (js < nkt && js < jp + 2 && mbar_test_wait(&k_full[js % kPfKRing], (uint32_t)(js / kPfKRing) & 1u) &&
                (js < 2 || mbar_test_wait(&pv_done[js & 1], (uint32_t)((js - 2) >> 1) & 1u))) {
                tc_fence_after();
                issue_s(js++);
                did = true;
            }
            if (jp < js && mbar_test_wait(&p_full[jp & 1], (uint32_t)(jp >> 1) & 1u)) {
                tc_fence_after();
                issue_pv(jp++);
                did = true;
            }
            if (did) {
                t0 = global_timer_ns();
            } else {
                if (*abort_flag) {
                    ok = false;
                } else if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                    if (atomicExch(const_cast<int*>(abort_flag), 1) == 0) count_status(p.status, 3);
                    ok = false;
                }
            }
        }
        // every MMA issued has completed before the CTA tears tensor memory down
        mma_commit(flush);
        (void)mbar_wait(flush, 0);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPfMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

// cuTensorMapEncodeTiled from the driver, looked up once
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::atomic<void*> fn{nullptr};
    void* f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || f == nullptr)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// The queries as a 3-D tensor [token][q head][D] of QT, read in boxes of [128 / G tokens][G heads]
// [64 dims] with the 128-byte swizzle the MMA descriptors expect.  Tokens past the last read as 0.
template <int D, typename QT>
cudaError_t query_map(const AttnParams& p, CUtensorMap* map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.num_q_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * sizeof(QT), (cuuint64_t)p.Hq * D * sizeof(QT)};
    const cuuint32_t box[3] = {64u, (cuuint32_t)p.G, (cuuint32_t)(kPfRows / p.G)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(map,
                           std::is_same<QT, __nv_bfloat16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           3, const_cast<void*>(static_cast<const void*>(p.q)), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, typename QT, typename OT, bool OPTS, bool TILED>
cudaError_t launch_prefill_grid(const AttnParams& p, int max_query_len, cudaStream_t stream) {
    const size_t smem = PfLayout<D>::kBytes;
    cudaError_t err = opt_in_smem<prefill_kernel<D, QT, OT, OPTS, TILED>>(smem);
    if (err != cudaSuccess) return err;
    if (p.num_q_tokens <= 0 || kPfRows % p.G != 0) return cudaErrorInvalidValue;
    CUtensorMap qmap;
    err = query_map<D, QT>(p, &qmap);
    if (err != cudaSuccess) return err;
    const int BQ = kPfRows / p.G;
    const dim3 grid = TILED ? dim3((unsigned)p.pf_tiles_cap * (unsigned)p.H)   // the walker's tile index
                            : dim3((unsigned)(((max_query_len + BQ - 1) / BQ) * p.H), 1, p.num_seqs);
    prefill_kernel<D, QT, OT, OPTS, TILED><<<grid, kPfThreads, smem, stream>>>(p, qmap);
    return cudaGetLastError();
}

template <int D, typename QT, typename OT, bool OPTS>
cudaError_t launch_prefill_t(const AttnParams& p, int max_query_len, cudaStream_t stream) {
    return p.pf_tiles_cap > 0 ? launch_prefill_grid<D, QT, OT, OPTS, true>(p, max_query_len, stream)
                              : launch_prefill_grid<D, QT, OT, OPTS, false>(p, max_query_len, stream);
}

template <int D, typename QT, bool OPTS>
cudaError_t prefill_by_out(const AttnParams& p, int mql, DType out_dt, cudaStream_t s) {
    switch (out_dt) {
        case DType::F16: return launch_prefill_t<D, QT, __half, OPTS>(p, mql, s);
        case DType::BF16: return launch_prefill_t<D, QT, __nv_bfloat16, OPTS>(p, mql, s);
        default: return launch_prefill_t<D, QT, float, OPTS>(p, mql, s);
    }
}

// Every (head size, query type, output type) instantiation of one OPTS flavour.
template <bool OPTS>
cudaError_t launch_prefill_all(const AttnParams& p, int head_size, int max_query_len, DType q_dt, DType out_dt,
                               cudaStream_t stream) {
    if (head_size == 128)
        return q_dt == DType::BF16 ? prefill_by_out<128, __nv_bfloat16, OPTS>(p, max_query_len, out_dt, stream)
                                   : prefill_by_out<128, __half, OPTS>(p, max_query_len, out_dt, stream);
    return q_dt == DType::BF16 ? prefill_by_out<64, __nv_bfloat16, OPTS>(p, max_query_len, out_dt, stream)
                               : prefill_by_out<64, __half, OPTS>(p, max_query_len, out_dt, stream);
}

}  // namespace
}  // namespace kvi4
