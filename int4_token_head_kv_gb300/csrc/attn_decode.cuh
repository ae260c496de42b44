// Decode attention over the INT4 cache (one query token per sequence), as split-KV segments.
//
// Method ("[Feature] Triton INT4 / INT2 per-token-head KV cache quantization", description of the
// packed read path): Q is rotated with the same random Hadamard transform as K and V, scores are
// dot products of the rotated query with the raw 4-bit codes, the asymmetry (zero-point) is
// corrected per key and the per-key scale applied, an online softmax accumulates P V in the
// rotated domain, and the output is un-rotated.  Long contexts are split into segments whose
// (max, sum, accumulator) partials are combined afterwards ("3D" segment reduction of the
// unified-attention interface, test_triton_unified_attention_per_token_head_scale).
//
// GB300 design, three launches per call:
//  0. qrot_kernel rotates each decode query once (v = H_d D q, power-of-two prescale, fp16 high +
//     low halves laid out as the score mma's B fragments, the per-head logit factor and sum(q')).
//     It only reads the queries, so it may run while the cache write that precedes it finishes.
//  1. decode_kernel walks split-KV units.  Unit sigma of sequence b is its KV tokens
//     [sigma S, (sigma + 1) S), S = seg_len.  A fixed grid of about two CTAs per SM takes
//     contiguous runs of units, balanced by cache blocks (CTA c owns the units that start in
//     [c W / n, (c + 1) W / n) of the batch's W decode blocks, a sequence's partial last unit
//     counting as a whole one when the sequence has several), and every unit writes
//     its own (max, sum, unnormalised output) partial.  A unit's arithmetic does not depend on
//     the CTA that runs it, so a sequence's output does not depend on the rest of the batch.
//  2. combine_kernel merges the units of each sequence in a fixed order and un-rotates.
//
// Walker CTA:
//  * All kv heads of a 16-token block are one contiguous, 16-byte-aligned region (K plane then V
//    plane, 2 * 16 * H * (D/2+4) bytes) streamed through a shared-memory ring (5 stages, 4 with
//    eight query heads per kv head) by 1-D bulk async copies (cp.async.bulk + mbarrier
//    transaction counts, L2 evict-first).  The ring runs across unit boundaries.  There is no
//    producer warp: the CTA's block ids are staged in shared memory up front (and its first
//    blocks prefetched into L2 while the previous kernels finish), thread 0 issues the first
//    copies, and the last consumer warp to finish with a stage issues its next block.  The
//    rotated-query record of each run of units of one sequence arrives the same way.
//  * Eight consumer warps: warp w owns kv head w % H (and every (8/H)-th block pair when H < 8).
//    Split-dot scores over the even and odd nibble streams: each K code word is masked into its
//    nibbles as exact fp16 subnormals with no offset (even codes e 2^-24, odd codes 16 o 2^-24:
//    one logic op per pair), and S^T[16 tokens x 8 columns] = Codes[16 x D] . Q'^T comes from
//    mma.sync m16n8k16; the query record carries the odd dimensions divided by 16, the logit factor
//    times 2^24 and sum(Q') over 2^24, so the zero-point is removed per key with the sum(Q') * zp
//    correction on the same scale.  (The tensor cores accumulate products of subnormal operands
//    with a few bits less precision, measured about 1e-6 of the sum of |terms| against the query's
//    operands; an offset left in the operands, such as 1024 + e, would cost about 8 bits, which
//    heavy-tailed caches expose.)
//  * P^T is transposed in registers (movmatrix) into the B operand of O^T[D x 8] += Codes_V^T P^T.
//    The V codes are exact fp16 integers (even codes through fp16 1024 + e, odd codes through
//    1024 + 16 e, both brought back by one constant fp16x2 operation): against weights whose
//    magnitudes span many binades, subnormal code operands would lose about 7 bits.
//    V's per-key scale is folded into P (w = p * s'_V * 2^-E, E a running max exponent, so the
//    fp16 weights never overflow); w and Q' are carried as fp16 high + low halves.  V's
//    zero-points leave O through sum(w zp), kept per column alongside O.
//
// The kernels are templates on the cache mode (BITS 4: INT4; 8: the INT8 comparator; 2: the INT2
// Lloyd-Max mode), each instantiated in a translation unit of its own (attn_decode.cu,
// attn_decode_int8.cu, attn_decode_int2.cu) so that the three compile in parallel.
#pragma once

#include "attn_common.cuh"

namespace kvi4 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = kConsumerWarps * 32;   // no producer warp: see the refill rule below
constexpr int kMaxStages = 8;                         // ring slots the state area has room for
constexpr int kMaxUnits = kDecodeMaxUnits;            // units per CTA (the host sizes the grid so)
constexpr int kTableWin = 256;                        // block ids of a CTA staged in shared memory
constexpr uint32_t kSmemPerSm = 233472;               // 228 KB of shared memory per SM
constexpr uint32_t kSmemPerCtaReserved = 1024;

constexpr int kMaxHead = 128;
// unpack_word operands that turn V codes into exact fp16 integers: lo nibbles 1024 + e - 1024,
// hi nibbles (1024 + 16 e) / 16 - 64
constexpr uint32_t kCodeLo = 0x64006400u;   // (1024, 1024)
constexpr uint32_t kCodeHi = 0xD400D400u;   // (-64, -64)
constexpr float kLazyMax = 8.0f;     // log2 units the running maximum may fall behind a block's
constexpr uint32_t kLazyExp = 4;     // binades the V exponent reference may fall behind a V scale

// Cached rows: BITS = 4 is the INT4 cache (D/2 code bytes, then the scale word with the zero-point
// in its low nibble), BITS = 8 the INT8 comparator (D int8 codes, then the fp32 scale), BITS = 2 the
// INT2 Lloyd-Max mode (D/4 code bytes, then the fp32 scale).  INT4 and INT2 rows are rotated.
template <int D, int BITS>
struct RowGeo {
    static constexpr int RB = D * BITS / 8 + 4;   // bytes per row
    static constexpr int SW = D * BITS / 32;      // index of the scale word
};

// Ring depth: 5 stages with up to 4 query heads per kv head, 4 with 8 (whose query records are
// twice as large), so that two CTAs fit an SM; INT8 blocks are twice as large, 2 stages; INT2
// blocks about half as large, 8 stages (two CTAs of 8 kv heads still fit an SM).
template <bool WIDE, int BITS>
struct WalkerShape {
    static constexpr int kStages = BITS == 8 ? 2 : BITS == 2 ? 8 : (WIDE ? 4 : 5);
};

struct DecodeSmem {
    uint32_t stage_bytes;   // one block (K + V planes)
    uint32_t qrec_bytes;    // one sequence's rotated-query record
    uint32_t nq;            // query buffers (2 when two CTAs still fit an SM, else 1)
    uint32_t q_off;
    uint32_t state_off;     // barriers, counters, unit list, block-table window
    uint32_t total;
};

constexpr uint32_t kStateBytes = kMaxStages * 8u + 2u * 8u    // ring and query barriers
                                 + kConsumerWarps * 8u        // scan scratch
                                 + (kMaxStages + 4u + kMaxStages + 4u + 8u) * 4u   // valid, flags, refill counters, info
                                 + kMaxUnits * 16u            // units
                                 + 3u * kMaxUnits * 4u        // unit start blocks, run starts, run query rows
                                 + kTableWin * 4u             // block-table window
                                 + kMaxHead * 4u;             // signs

template <int D, bool WIDE, int BITS>
__host__ __device__ inline DecodeSmem decode_smem_layout(int H, int Hq) {
    using Sh = WalkerShape<WIDE, BITS>;
    DecodeSmem s;
    s.stage_bytes = 2u * kBlockSize * (uint32_t)H * RowGeo<D, BITS>::RB;
    s.qrec_bytes = decode_qrec_words(D, H, Hq / H) * 4u;
    s.q_off = (Sh::kStages * s.stage_bytes + 127u) & ~127u;
    s.nq = 2;
    for (;;) {
        s.state_off = (s.q_off + s.nq * s.qrec_bytes + 127u) & ~127u;
        s.total = s.state_off + ((kStateBytes + 127u) & ~127u);
        if (s.nq == 1 || 2u * (s.total + kSmemPerCtaReserved) <= kSmemPerSm) break;
        s.nq = 1;
    }
    return s;
}

// Exclusive prefix sum over the CTA's 256 threads (all threads must call it); *total gets the sum.
__device__ __forceinline__ unsigned long long block_exclusive_scan(unsigned long long v, unsigned long long* wsum,
                                                                   unsigned long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    unsigned long long before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        const unsigned long long s = wsum[w];
        before += (w < warp) ? s : 0ull;
        all += s;
    }
    __syncthreads();
    *total = all;
    return before + x - v;
}

// The low nibble of a word as an exact float: 2^23 + n - 2^23 (one logic op and one add).
__device__ __forceinline__ float nibble_to_float(uint32_t w) {
    return __uint_as_float(0x4B000000u | (w & 15u)) - 8388608.0f;
}

__device__ __forceinline__ uint32_t pack_halves(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// ------------------------------------------------------------------ 0. query rotation

// One CTA per sequence; only decode sequences (one query token) are rotated.  Record of a sequence
// (32-bit words): for kv head h, 32-dimension group j and lane, the QW fp16x2 words that lane feeds
// to the score mma; then alpha[Hq rounded up to 4] (raw score -> log2-domain logit, before the
// key's scale) and qsum[Hq rounded up to 4] (sum of the stored high + low halves of each vector).
template <int D, bool WIDE, int BITS, typename QT>
__global__ void __launch_bounds__(256) qrot_kernel(const __grid_constant__ AttnParams p) {
    constexpr int QW = WIDE ? 8 : 4, KWPT = D / 32;
    extern __shared__ __align__(128) uint8_t smem[];
    griddep_launch_dependents();   // the walker's set-up reads only metadata
    const int seq = blockIdx.x;
    const int q0 = __ldg(p.qsl + seq);
    const bool decode = __ldg(p.qsl + seq + 1) - q0 == 1 && q0 >= 0 && (int64_t)q0 < p.num_q_tokens;
    if (decode) {   // uniform over the CTA
        const int H = p.H, G = p.G, Hq = p.Hq, Hq4 = (Hq + 3) & ~3;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        float* sgn = reinterpret_cast<float*>(smem);
        float* alpha = sgn + D;
        float* qsum = alpha + Hq4;
        __half* qh = reinterpret_cast<__half*>(qsum + Hq4);
        __half* ql = qh + Hq * D;
        // INT8 queries are not rotated (sign +1, no transform, no 1/sqrt(d) of the transform)
        for (int i = threadIdx.x; i < D; i += blockDim.x) sgn[i] = BITS != 8 && p.signs[i] < 0.0f ? -1.0f : 1.0f;
        __syncthreads();
        const float lsc = (BITS != 8 ? p.c : 1.0f) * p.softmax_scale * kLog2e;
        for (int v0 = warp; v0 < Hq; v0 += 4 * 8) {   // four vectors per warp at a time
            float x[4][D / 32];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int v = v0 + 8 * k;
#pragma unroll
                for (int j = 0; j < D / 32; ++j)
                    x[k][j] = v < Hq ? load_elem<QT>(p.q, ((int64_t)q0 * Hq + v) * D + lane + 32 * j) * sgn[lane + 32 * j]
                                     : 0.0f;
            }
            // v = H_d D q; a power-of-two prescale brings max|v| into [2^14, 2^15) for the halves
            if constexpr (BITS != 8) warp_fwht_batch<D, 4>(x);
            float mx[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mx[k] = 0.0f;
#pragma unroll
                for (int j = 0; j < D / 32; ++j) mx[k] = fmaxf(mx[k], fabsf(x[k][j]));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int k = 0; k < 4; ++k) mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], off));
            }
            float sum[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int v = v0 + 8 * k;
                const int e = prescale_exponent(mx[k]);
                const float sc = exp2i(e);
                sum[k] = 0.0f;
#pragma unroll
                for (int j = 0; j < D / 32; ++j) {
                    const float y = x[k][j] * sc;
                    const __half hi = __float2half_rn(y);
                    const __half lo = __float2half_rn(y - __half2float(hi));
                    sum[k] += __half2float(hi) + __half2float(lo);
                    if (v < Hq) {
                        qh[v * D + lane + 32 * j] = hi;
                        ql[v * D + lane + 32 * j] = lo;
                    }
                }
                if (lane == 0 && v < Hq) alpha[v] = lsc * exp2i(-e);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int k = 0; k < 4; ++k) sum[k] += __shfl_xor_sync(0xffffffffu, sum[k], off);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (lane == 0 && v0 + 8 * k < Hq) qsum[v0 + 8 * k] = sum[k];
        }
        __syncthreads();
        // Score-mma B fragments.  Lane (g, t) of kv head h's warp feeds, for the group W = t + 4 j of
        // dims 8W .. 8W+7 of a key row, the pairs (8W+2hh, 8W+2hh+4) and (8W+2hh+1, 8W+2hh+5) of its
        // column's vector, hh = 0, 1 (the order of the unpacked nibbles); with INT8 codes the pairs
        // (8W+4hh, 8W+4hh+1) and (8W+4hh+2, 8W+4hh+3).  INT2 groups unpack in the INT4 order.  Columns: G == 8, head g (high halves; the low
        // halves follow as a second tile); otherwise head g >> 1, the high half for even g and the
        // low half for odd g.
        uint32_t* rec = p.ws_q + (size_t)seq * p.qrec_words;
        for (int idx = threadIdx.x; idx < H * KWPT * 32; idx += blockDim.x) {
            const int ln = idx & 31, j = (idx >> 5) % KWPT, h = idx / (32 * KWPT);
            const int g = ln >> 2, t = ln & 3;
            const int head = WIDE ? g : (g >> 1);
            const bool live = head < G;
            const int vrow = (h * G + (live ? head : 0)) * D;
            const __half* qv = (WIDE || (g & 1) == 0 ? qh : ql) + vrow;
            const __half* qv2 = ql + vrow;
            const int W = t + 4 * j;
            uint32_t w[QW];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int d0 = BITS != 8 ? 8 * W + 2 * hh : 8 * W + 4 * hh;
                const int s1 = BITS != 8 ? 4 : 1, s2 = BITS != 8 ? 1 : 2;   // second of a pair; next pair
                // INT4: the odd dimensions meet high nibbles, which unpack as 16 x their code
                const __half od = __float2half(BITS == 4 ? 0.0625f : 1.0f);
                w[2 * hh] = live ? pack_halves(qv[d0], qv[d0 + s1]) : 0u;
                w[2 * hh + 1] = live ? pack_halves(__hmul(qv[d0 + s2], od), __hmul(qv[d0 + s2 + s1], od)) : 0u;
                if constexpr (WIDE) {
                    w[4 + 2 * hh] = live ? pack_halves(qv2[d0], qv2[d0 + s1]) : 0u;
                    w[5 + 2 * hh] = live ? pack_halves(__hmul(qv2[d0 + s2], od), __hmul(qv2[d0 + s2 + s1], od)) : 0u;
                }
            }
            uint4* dst = reinterpret_cast<uint4*>(rec) + (size_t)idx * (QW / 4);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            if constexpr (WIDE) dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        float* ralpha = reinterpret_cast<float*>(rec + (size_t)H * D * QW);
        for (int v = threadIdx.x; v < Hq4; v += blockDim.x) {
            ralpha[v] = v < Hq ? alpha[v] : 0.0f;
            ralpha[Hq4 + v] = v < Hq ? qsum[v] : 0.0f;
        }
    }
    // Complete only after the previous kernel of the stream (the cache write, typically) has:
    // whoever waits for this kernel then also sees that kernel's results.
    griddep_wait();
}

// ------------------------------------------------------------------ 1. split-KV unit walker

// OPTS: the call has window / softcap / ALiBi options (a separate instantiation, so that the plain
// path carries none of their registers)
template <int D, bool WIDE, int BITS, bool OPTS>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_kernel(const __grid_constant__ AttnParams p) {
    using Gm = Geo<D>;
    using Rw = RowGeo<D, BITS>;
    constexpr int QW = WIDE ? 8 : 4;      // fragment words per lane per 32-dimension group
    constexpr int NLS = WIDE ? 32 : 16;
    constexpr int kStages = WalkerShape<WIDE, BITS>::kStages;
    constexpr uint32_t PO = decode_po_floats(D, WIDE ? 8 : 1);
    extern __shared__ __align__(128) uint8_t smem[];
    const int H = p.H, G = p.G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const DecodeSmem lay = decode_smem_layout<D, WIDE, BITS>(H, p.Hq);
    const int nq = (int)lay.nq;
    uint8_t* ring = smem;
    uint8_t* qbuf = smem + lay.q_off;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.state_off);
    uint64_t* qfull = full + kMaxStages;
    unsigned long long* wsum = reinterpret_cast<unsigned long long*>(qfull + 2);
    int* valid = reinterpret_cast<int*>(wsum + kConsumerWarps);
    int* flags = valid + kMaxStages;   // [0] a wait gave up, [1] blocks issued, [2] query rows issued
    int* released = flags + 4;         // per stage: consumer warps done with its current block
    int* qreleased = released + kMaxStages;   // per query buffer: consumer warps done reading it
    int* info = qreleased + 4;
    int4* units = reinterpret_cast<int4*>(info + 8);     // (seq, first block in seq, global unit, tokens)
    int* ustart = reinterpret_cast<int*>(units + kMaxUnits);   // first block, in the batch's block order
    int* run_first = ustart + kMaxUnits;                 // first unit of each run of one sequence
    int* run_seq = run_first + kMaxUnits;                // that sequence
    int* tbl = run_seq + kMaxUnits;                      // block ids of the CTA's first kTableWin blocks

    // Launched as a programmatic dependent (of the cache write, typically): everything up to
    // griddep_wait() below reads only the host-provided metadata (query_start_loc, seq_lens, block
    // tables, signs) and writes only shared memory.  The combine may be scheduled right away: it
    // waits for this grid before reading anything, and its CTAs become resident as walker CTAs
    // retire.
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0;
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qfull[s], 1);
            qreleased[s] = 0;
        }
        for (int s = 0; s < 4; ++s) flags[s] = 0;
        fence_mbar_init();
    }

    // ---- the batch's decode units: each thread scans a contiguous slice of the sequences
    const int N = p.num_seqs, S = p.seg_len, SB = S / kBlockSize;
    const int per = (N + kDecodeThreads - 1) / kDecodeThreads;
    const int b0 = min(N, (int)threadIdx.x * per), b1 = min(N, b0 + per);
    // (decode context length or 0, query row) of sequence b from its metadata
    auto decode_of = [&](int q0, int q1, int L, bool count) -> int2 {
        if (q1 - q0 != 1) return make_int2(0, 0);
        if (q0 < 0 || (int64_t)q0 >= p.num_q_tokens) {
            if (count) count_status(p.status, 2);
            return make_int2(0, 0);
        }
        if (L > p.len_cap) {   // longer than max_seq_len or than its block table
            if (count) count_status(p.status, 2);
            L = p.len_cap;
        }
        return make_int2(max(L, 0), q0);
    };
    // Stage (L, q0) of every sequence in shared memory (the ring is idle until the first copy).
    // Thread t's i-th sequence t * per + i sits at entry i * 256 + t, so the passes below read
    // consecutive words across a warp; a batch too large for it reads global memory per pass.
    int2* meta = reinterpret_cast<int2*>(smem);
    const bool staged = (uint32_t)per * kDecodeThreads * 8u <= lay.state_off;
    if (staged) {
        for (int i0 = 0; i0 < per; i0 += 4) {
            int q0[4], q1[4], L[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int b = min(b0 + i0 + k, N - 1);
                q0[k] = __ldg(p.qsl + b);
                q1[k] = __ldg(p.qsl + b + 1);
                L[k] = __ldg(p.seq_lens + b);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (b0 + i0 + k < b1)
                    meta[(i0 + k) * kDecodeThreads + threadIdx.x] = decode_of(q0[k], q1[k], L[k], blockIdx.x == 0);
            }
        }
    }
    __syncthreads();
    // (L, q0) of this thread's i-th sequence, and of any sequence b
    auto own_info = [&](int i, bool count) -> int2 {
        if (staged) return meta[i * kDecodeThreads + threadIdx.x];
        const int b = b0 + i;
        return decode_of(__ldg(p.qsl + b), __ldg(p.qsl + b + 1), __ldg(p.seq_lens + b), count);
    };
    auto seq_info = [&](int b) -> int2 {
        if (staged) return meta[(b % per) * kDecodeThreads + b / per];
        return decode_of(__ldg(p.qsl + b), __ldg(p.qsl + b + 1), __ldg(p.seq_lens + b), false);
    };
    // Balance weight of a sequence: its blocks, except that the last (partial) unit of a sequence
    // with several units weighs a whole unit.  A CTA's share then rarely ends with two whole
    // units after a short tail unit (a common 2.5-unit overload when shares hold about two units).
    auto weight_of = [&](uint32_t nblk, uint32_t nseg) -> uint32_t {
        return nseg > 1u ? nseg * (uint32_t)SB : nblk;
    };
    uint32_t my_units = 0, my_blocks = 0, my_weight = 0;
    for (int b = b0; b < b1; ++b) {
        const int L = own_info(b - b0, blockIdx.x == 0).x;
        const uint32_t nseg = fast_div((uint32_t)(L + S - 1), (uint32_t)S, p.seg_rcp);
        const uint32_t nblk = (uint32_t)((L + kBlockSize - 1) / kBlockSize);
        my_units += nseg;
        my_blocks += nblk;
        my_weight += weight_of(nblk, nseg);
    }
    unsigned long long tot, wtot;
    const unsigned long long pre =
        block_exclusive_scan(((unsigned long long)my_blocks << 32) | my_units, wsum, &tot);
    const uint32_t wb_t = (uint32_t)block_exclusive_scan(my_weight, wsum, &wtot);
    const uint32_t U = (uint32_t)tot, Wt = (uint32_t)wtot;
    const uint32_t ub_t = (uint32_t)pre, bb_t = (uint32_t)(pre >> 32);

    // This CTA's share of the batch's weight, [f(c), f(c+1)) with f(c) = c Wt / n in fp32: any
    // monotone f with f(0) = 0 and f(n) = Wt splits it exactly, and every CTA evaluates the
    // shared boundary the same way.  Then the units that start inside it (unit k of a sequence
    // starts at its weight offset + k SB).
    const float per_cta = (float)Wt / (float)gridDim.x;
    auto boundary = [&](uint32_t c) -> uint32_t {
        if (c >= gridDim.x) return Wt;
        const uint32_t f = (uint32_t)((float)c * per_cta);
        return f < Wt ? f : Wt;
    };
    const uint32_t A = boundary(blockIdx.x), E = boundary(blockIdx.x + 1);
    auto units_before = [&](uint32_t X, uint32_t bb, uint32_t nseg) -> uint32_t {
        if (X <= bb) return 0u;
        const uint32_t k = fast_div(X - bb + SB - 1, (uint32_t)SB, p.segb_rcp);
        return k < nseg ? k : nseg;
    };
    uint32_t below_a = 0, below_e = 0;
    {
        uint32_t wb = wb_t;
        for (int b = b0; b < b1; ++b) {
            const int L = own_info(b - b0, false).x;
            const uint32_t nseg = fast_div((uint32_t)(L + S - 1), (uint32_t)S, p.seg_rcp);
            const uint32_t nblk = (uint32_t)((L + kBlockSize - 1) / kBlockSize);
            below_a += units_before(A, wb, nseg);
            below_e += units_before(E, wb, nseg);
            wb += weight_of(nblk, nseg);
        }
    }
    unsigned long long lohi;
    block_exclusive_scan(((unsigned long long)below_e << 32) | below_a, wsum, &lohi);
    const uint32_t u_lo = (uint32_t)lohi;
    int nunits = (int)((uint32_t)(lohi >> 32) - u_lo);
    if (nunits > kMaxUnits) {   // cannot happen for a grid the host sized; never overrun the list
        if (threadIdx.x == 0) count_status(p.status, 2);
        nunits = kMaxUnits;
    }
    {
        uint32_t bb = bb_t, ub = ub_t;
        for (int b = b0; b < b1 && ub < u_lo + (uint32_t)nunits; ++b) {
            const int L = own_info(b - b0, false).x;
            const int nseg = (int)fast_div((uint32_t)(L + S - 1), (uint32_t)S, p.seg_rcp);
            const int nblk = (L + kBlockSize - 1) / kBlockSize;
            const int64_t lo_rel = (int64_t)u_lo - ub, hi_rel = (int64_t)u_lo + nunits - ub;
            const int64_t s_lo = lo_rel > 0 ? lo_rel : 0;
            const int64_t s_hi = hi_rel < nseg ? hi_rel : nseg;
            for (int64_t sg = s_lo; sg < s_hi; ++sg) {
                const int j = (int)(ub + sg - u_lo);
                units[j] = make_int4(b, (int)sg * SB, (int)(ub + sg), min(S, L - (int)sg * S));
                ustart[j] = (int)(bb + sg * SB);
            }
            bb += (uint32_t)nblk;
            ub += (uint32_t)nseg;
        }
    }
    __syncthreads();
    // runs of consecutive units of one sequence share a rotated-query record
    unsigned long long nruns_ll;
    {
        const int j = threadIdx.x;
        const bool first = j < nunits && (j == 0 || units[j].x != units[j - 1].x);
        const int r = (int)block_exclusive_scan(first ? 1ull : 0ull, wsum, &nruns_ll);
        if (first) {
            run_first[r] = j;
            run_seq[r] = units[j].x;
        }
    }
    const int nruns = (int)nruns_ll;
    const int Bs = nunits > 0 ? ustart[0] : 0;
    const int nb_cta = nunits > 0 ? ustart[nunits - 1] - Bs + (units[nunits - 1].w + kBlockSize - 1) / kBlockSize : 0;

    // block id of the CTA's i-th block (the unit holding it, then its block table entry)
    auto block_id = [&](int i) -> int {
        int lo = 0, hi = nunits - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ustart[mid] - Bs <= i) lo = mid;
            else hi = mid - 1;
        }
        const int4 u = units[lo];
        return __ldg(p.block_tables + (int64_t)u.x * p.max_blocks_per_seq + u.y + (i - (ustart[lo] - Bs)));
    };
    for (int i = threadIdx.x; i < min(nb_cta, kTableWin); i += kDecodeThreads) tbl[i] = block_id(i);
    __syncthreads();

    const uint32_t stage_bytes = lay.stage_bytes, qrec_bytes = lay.qrec_bytes;
    // Ring refill rule: block i goes to stage i % kStages.  The first kStages blocks are issued up
    // front; afterwards the LAST consumer warp to finish with block i (counted in released[])
    // issues block i + kStages into the same stage, so no warp ever blocks waiting to refill.
    auto produce = [&](int i) {
        const int st = i % kStages;
        const int blk = i < kTableWin ? tbl[i] : block_id(i);
        const bool ok = blk >= 0 && (int64_t)blk < p.num_blocks;
        valid[st] = ok ? 1 : 0;
        atomicMax(&flags[1], i + 1);
        if (ok) {
            mbar_arrive_expect_tx(&full[st], stage_bytes);
            bulk_copy_g2s(ring + (size_t)st * stage_bytes, p.cache + (int64_t)blk * stage_bytes, stage_bytes,
                          &full[st], policy_evict_first());
        } else {
            count_status(p.status, 1);
            mbar_arrive(&full[st]);
        }
    };
    // The query record of run r goes to buffer r % nq, refilled the same way once every warp has
    // read it.
    auto produce_q = [&](int r) {
        const int qs = r & (nq - 1);
        atomicMax(&flags[2], r + 1);
        mbar_arrive_expect_tx(&qfull[qs], qrec_bytes);
        bulk_copy_g2s(qbuf + (size_t)qs * qrec_bytes, p.ws_q + (size_t)run_seq[r] * p.qrec_words, qrec_bytes,
                      &qfull[qs], policy_evict_first());
    };
    // Warm L2 with the first blocks while the previous kernels finish: the copies issued after the
    // wait then hit L2.  (A block the cache write is still updating is safe to prefetch: the copy
    // after the wait reads L2, where that write lands.)
    if (threadIdx.x < min(nb_cta, kStages)) {
        const int blk = tbl[threadIdx.x];
        if (blk >= 0 && (int64_t)blk < p.num_blocks) bulk_prefetch_l2(p.cache + (int64_t)blk * stage_bytes, stage_bytes);
    }
    griddep_wait();   // the query records, and through them the cache, come from earlier kernels
    if (blockIdx.x == 0 && p.max_query_len > 1 && p.pf_tiles_cap > 0) {
        // The prefill's tile index: sequence b's first query tile among the batch's prefill tiles
        // (tiles of 128 / G tokens over its first min(q_len, max_query_len) queries; none for q_len
        // <= 1).  Clamped to the grid the host launches, which bounds the total from the query
        // count; a batch past it (inconsistent metadata) is counted.
        const int bq = kPrefillRows / G;
        auto tiles_of = [&](int b) -> uint32_t {
            const int ql = __ldg(p.qsl + b + 1) - __ldg(p.qsl + b);
            return ql > 1 ? (uint32_t)((min(ql, p.max_query_len) + bq - 1) / bq) : 0u;
        };
        uint32_t mine = 0;
        for (int b = b0; b < b1; ++b) mine += tiles_of(b);
        unsigned long long total;
        uint32_t t = (uint32_t)block_exclusive_scan(mine, wsum, &total);
        const uint32_t cap = (uint32_t)p.pf_tiles_cap;
        for (int b = b0; b < b1; ++b) {
            p.ws_ptile[b] = (int)min(t, cap);
            t += tiles_of(b);
        }
        if (threadIdx.x == 0) {
            p.ws_ptile[N] = (int)min((uint32_t)total, cap);
            if (total > cap) count_status(p.status, 2);
        }
    }
    if (blockIdx.x == 0) {   // the combine's sequence index
        uint32_t ub = ub_t;
        for (int b = b0; b < b1; ++b) {
            p.ws_meta[b] = (int)ub;
            ub += fast_div((uint32_t)(own_info(b - b0, false).x + S - 1), (uint32_t)S, p.seg_rcp);
        }
        if (threadIdx.x == 0) p.ws_meta[N] = (int)U;
    }
    if (threadIdx.x == 0) {   // the first query rows, then the first blocks
        for (int r = 0; r < min(nq, nruns); ++r) produce_q(r);
        for (int i = 0; i < min(kStages, nb_cta); ++i) produce(i);
    }

    float o[Gm::MT][4];
    float m0 = kNegBig, m1 = kNegBig, l0 = 0.0f, l1 = 0.0f;
    uint32_t eref = 0;   // running max biased exponent of V scales seen in the unit
    const int g = lane >> 2, t = lane & 3;
    const int h = warp & (H - 1);
    const int wph = 1 << p.wph_shift;
    const int sub = warp >> (3 - p.wph_shift);
    const int tk0 = block_token(g), tk1 = block_token(g + 8);
    // Score columns (the mma N dimension, 8 wide).  WIDE (8 query heads per kv head): column n is
    // head n, with a second 8-wide tile carrying the low halves; lane quad t holds heads 2t, 2t+1.
    // Otherwise column 2n carries the high half of head n and column 2n + 1 its low half, so the
    // split costs no extra mma, and lane quad t holds head t with both halves (their sum is local;
    // m1, l1, al1, qs1 and WZ1 are then unused).  The weights of P.V take the same columns.
    const int hb = WIDE ? 2 * t : t;
    uint32_t qb[Gm::KSTEPS][WIDE ? 4 : 2];
    float al0 = 0.0f, al1 = 0.0f;     // logit factor of heads hb, hb + 1
    float qs0 = 0.0f, qs1 = 0.0f;     // sum(Q') of those heads (high + low halves as stored)
    float sl0 = 0.0f, sl1 = 0.0f;     // their ALiBi slopes in log2 units
    float WZ0 = 0.0f, WZ1 = 0.0f;     // sum(w zp) per head
    int run = -1, prev_seq = -1;
    bool stop = false;

    for (int j = 0; j < nunits && !stop; ++j) {
        const int4 u = units[j];
        if (u.x != prev_seq) {   // a new sequence: its rotated-query record from the buffer
            prev_seq = u.x;
            ++run;
            const int qs = run & (nq - 1);
            const bool qok = mbar_wait(&qfull[qs], (uint32_t)(run >> (nq - 1)) & 1u);
            if (__any_sync(0xffffffffu, !qok)) {   // warp-uniform
                if (lane == 0) {
                    count_status(p.status, 3);
                    atomicExch(flags, 1);
                }
                break;
            }
            const uint8_t* rec = qbuf + (size_t)qs * qrec_bytes;
            const uint4* fr = reinterpret_cast<const uint4*>(rec) + ((size_t)h * Gm::KWPT * 32 + lane) * (QW / 4);
#pragma unroll
            for (int k = 0; k < Gm::KWPT; ++k) {
                const uint4 a = fr[k * 32 * (QW / 4)];
                qb[2 * k][0] = a.x;
                qb[2 * k][1] = a.y;
                qb[2 * k + 1][0] = a.z;
                qb[2 * k + 1][1] = a.w;
                if constexpr (WIDE) {
                    const uint4 b = fr[k * 32 * (QW / 4) + 1];
                    qb[2 * k][2] = b.x;
                    qb[2 * k][3] = b.y;
                    qb[2 * k + 1][2] = b.z;
                    qb[2 * k + 1][3] = b.w;
                }
            }
            const float* alpha = reinterpret_cast<const float*>(rec) + (size_t)H * D * QW;
            const float* qsum = alpha + ((p.Hq + 3) & ~3);
            al0 = (hb < G) ? alpha[h * G + hb] : 0.0f;
            al1 = (WIDE && hb + 1 < G) ? alpha[h * G + hb + 1] : 0.0f;
            qs0 = (hb < G) ? qsum[h * G + hb] : 0.0f;
            qs1 = (WIDE && hb + 1 < G) ? qsum[h * G + hb + 1] : 0.0f;
            if constexpr (BITS == 4) {   // the scores come out over 2^24 (subnormal code operands)
                al0 *= 16777216.0f;
                al1 *= 16777216.0f;
                qs0 *= 0x1.0p-24f;
                qs1 *= 0x1.0p-24f;
            }
            if constexpr (OPTS) {
                const bool alibi = (p.opts & kOptAlibi) != 0;
                sl0 = alibi && hb < G ? __ldg(p.alibi + h * G + hb) * kLog2e : 0.0f;
                sl1 = alibi && WIDE && hb + 1 < G ? __ldg(p.alibi + h * G + hb + 1) * kLog2e : 0.0f;
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();   // this warp's reads of the buffer come before the count
                // the counter wraps to 0 on the last warp's increment
                if (atomicInc(reinterpret_cast<unsigned*>(&qreleased[qs]), kConsumerWarps - 1) == kConsumerWarps - 1) {
                    __threadfence_block();
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    if (run + nq < nruns && !*(volatile int*)flags) produce_q(run + nq);
                }
            }
        }

#pragma unroll
        for (int i = 0; i < Gm::MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
        m0 = kNegBig;
        m1 = kNegBig;
        l0 = 0.0f;
        l1 = 0.0f;
        WZ0 = WZ1 = 0.0f;
        eref = 0;
        const int li0 = ustart[j] - Bs;
        // the decode query's position (the staged metadata is gone: the ring has overwritten it)
        const int posd = OPTS ? min(__ldg(p.seq_lens + u.x), p.len_cap) - 1 : 0;
        const int nbu = (u.w + kBlockSize - 1) / kBlockSize;

        // Two blocks (32 tokens) per iteration: their score chains, one softmax update and their
        // P.V products interleave, which gives each warp independent work to overlap latencies.
        for (int k = 0; k < nbu; k += 2) {
            const int i = li0 + k;
            const int npair = min(2, nbu - k);
            int st[2];
            bool ok[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) st[b] = (i + b) % kStages;
            bool timed_out = false;
            for (int b = 0; b < npair; ++b) {
                if (!mbar_wait(&full[st[b]], (uint32_t)((i + b) / kStages) & 1u)) timed_out = true;
            }
            if (__any_sync(0xffffffffu, timed_out)) {   // warp-uniform
                if (lane == 0) {
                    count_status(p.status, 3);
                    atomicExch(flags, 1);
                }
                stop = true;
                break;
            }
#pragma unroll
            for (int b = 0; b < 2; ++b) ok[b] = b < npair && valid[st[b]];
            if (((k >> 1) & (wph - 1)) == sub && (ok[0] || ok[1])) {
                const uint8_t* kp[2];
                const uint8_t* vp[2];
                float x[2][4];
                uint32_t vs0[2], vs1[2];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    kp[b] = ring + (size_t)st[b] * stage_bytes;
                    vp[b] = kp[b] + (size_t)kBlockSize * H * Rw::RB;
                }
                // ---- scores Codes_K Q'^T for both blocks, high and low halves of Q'
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const uint32_t* kr0 = reinterpret_cast<const uint32_t*>(kp[b] + (tk0 * H + h) * Rw::RB);
                    const uint32_t* kr1 = reinterpret_cast<const uint32_t*>(kp[b] + (tk1 * H + h) * Rw::RB);
                    const uint32_t ks0 = kr0[Rw::SW], ks1 = kr1[Rw::SW];
                    // two independent accumulation chains per block: the high- and low-half tiles
                    // when G = 8, the two halves of each code word otherwise
                    float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    float c2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    if (ok[b]) {
                        uint32_t nx0[4], nx1[4];   // INT2: the next group's operands, unpacked with this one
                        (void)nx0;
                        (void)nx1;
#pragma unroll
                        for (int q = 0; q < Gm::KWPT; ++q) {
                            uint32_t a0[4], a1[4];
                            if constexpr (BITS == 4) {
                                unpack_word_sub(kr0[t + 4 * q], a0);
                                unpack_word_sub(kr1[t + 4 * q], a1);
                            } else if constexpr (BITS == 2 && WIDE) {   // 16-bit groups of 8 dims
                                unpack_u2(reinterpret_cast<const uint16_t*>(kr0)[t + 4 * q], a0);
                                unpack_u2(reinterpret_cast<const uint16_t*>(kr1)[t + 4 * q], a1);
                            } else if constexpr (BITS == 2) {
                                // two groups at a time, t + 4q and t + 4q + 4 (with eight query heads
                                // per kv head the extra registers would spill)
                                if ((q & 1) == 0) {
                                    const uint16_t* g0 = reinterpret_cast<const uint16_t*>(kr0) + t + 4 * q;
                                    const uint16_t* g1 = reinterpret_cast<const uint16_t*>(kr1) + t + 4 * q;
                                    unpack_u2_x2((uint32_t)g0[0] | ((uint32_t)g0[4] << 16), a0, nx0);
                                    unpack_u2_x2((uint32_t)g1[0] | ((uint32_t)g1[4] << 16), a1, nx1);
                                } else {
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        a0[e] = nx0[e];
                                        a1[e] = nx1[e];
                                    }
                                }
                            } else {
                                unpack_i8(kr0[2 * (t + 4 * q)], kr0[2 * (t + 4 * q) + 1], a0);
                                unpack_i8(kr1[2 * (t + 4 * q)], kr1[2 * (t + 4 * q) + 1], a1);
                            }
                            if constexpr (WIDE) {
                                mma_f16_16816(c, a0[0], a1[0], a0[1], a1[1], qb[2 * q][0], qb[2 * q][1]);
                                mma_f16_16816(c, a0[2], a1[2], a0[3], a1[3], qb[2 * q + 1][0], qb[2 * q + 1][1]);
                                mma_f16_16816(c2, a0[0], a1[0], a0[1], a1[1], qb[2 * q][2], qb[2 * q][3]);
                                mma_f16_16816(c2, a0[2], a1[2], a0[3], a1[3], qb[2 * q + 1][2], qb[2 * q + 1][3]);
                            } else {
                                mma_f16_16816(c, a0[0], a1[0], a0[1], a1[1], qb[2 * q][0], qb[2 * q][1]);
                                mma_f16_16816(c2, a0[2], a1[2], a0[3], a1[3], qb[2 * q + 1][0], qb[2 * q + 1][1]);
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) c[e] += c2[e];
                    const int tb = (k + b) * kBlockSize;   // token offset of this block in the unit
                    const bool v0 = ok[b] && tb + tk0 < u.w, v1 = ok[b] && tb + tk1 < u.w;
                    constexpr uint32_t kScaleMask = BITS == 4 ? 0xFFFFFFF0u : 0xFFFFFFFFu;   // INT8 / INT2: plain fp32
                    const float sk0 = __uint_as_float(ks0 & kScaleMask), sk1 = __uint_as_float(ks1 & kScaleMask);
                    // score = S - zp sum(Q'), then the key's scale and the logit factor (INT8 / INT2: no zp)
                    const float zk0 = BITS == 4 ? nibble_to_float(ks0) : 0.0f, zk1 = BITS == 4 ? nibble_to_float(ks1) : 0.0f;
                    if constexpr (WIDE) {   // x = (token tk0: heads hb, hb+1; token tk1: heads hb, hb+1)
                        x[b][0] = v0 ? fmaf(-zk0, qs0, c[0]) * sk0 * al0 : -INFINITY;
                        x[b][1] = v0 ? fmaf(-zk0, qs1, c[1]) * sk0 * al1 : -INFINITY;
                        x[b][2] = v1 ? fmaf(-zk1, qs0, c[2]) * sk1 * al0 : -INFINITY;
                        x[b][3] = v1 ? fmaf(-zk1, qs1, c[3]) * sk1 * al1 : -INFINITY;
                    } else {   // x[0] = token tk0, x[2] = token tk1 (head hb; high + low columns)
                        x[b][0] = v0 ? fmaf(-zk0, qs0, c[0] + c[1]) * sk0 * al0 : -INFINITY;
                        x[b][2] = v1 ? fmaf(-zk1, qs0, c[2] + c[3]) * sk1 * al0 : -INFINITY;
                        x[b][1] = x[b][3] = -INFINITY;
                    }
                    if constexpr (OPTS) {   // window / softcap / ALiBi
                        const int jb = u.y * kBlockSize + tb;   // position of this block's first token
                        x[b][0] = apply_opts(x[b][0], jb + tk0, posd, sl0, p, posd);
                        x[b][2] = apply_opts(x[b][2], jb + tk1, posd, sl0, p, posd);
                        if constexpr (WIDE) {
                            x[b][1] = apply_opts(x[b][1], jb + tk0, posd, sl1, p, posd);
                            x[b][3] = apply_opts(x[b][3], jb + tk1, posd, sl1, p, posd);
                        }
                    }
                    const uint32_t* vg0 = reinterpret_cast<const uint32_t*>(vp[b] + (tk0 * H + h) * Rw::RB);
                    const uint32_t* vg1 = reinterpret_cast<const uint32_t*>(vp[b] + (tk1 * H + h) * Rw::RB);
                    vs0[b] = v0 ? vg0[Rw::SW] : 0u;   // invisible tokens: scale word 0 (exponent 0, weight 0)
                    vs1[b] = v1 ? vg1[Rw::SW] : 0u;
                }
                // ---- one online-softmax update for heads hb (, hb+1) over the 32 tokens
                float bm0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
                float bm1 = WIDE ? fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3])) : kNegBig;
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                    if constexpr (WIDE) bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
                }
                // The reference maximum moves only when a block's maximum passes it by more than
                // kLazyMax (log2 units): the weights then stay below 2^kLazyMax and most updates need
                // no rescaling of O (the softmax is the same for any reference).
                const bool up0 = bm0 > m0 + kLazyMax, up1 = bm1 > m1 + kLazyMax;
                const float mn0 = up0 ? bm0 : m0, mn1 = up1 ? bm1 : m1;
                const float r0 = up0 ? fast_exp2(m0 - mn0) : 1.0f, r1 = up1 ? fast_exp2(m1 - mn1) : 1.0f;
                float pr[2][4];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    pr[b][0] = fast_exp2(x[b][0] - mn0);
                    pr[b][2] = fast_exp2(x[b][2] - mn0);
                    pr[b][1] = WIDE ? fast_exp2(x[b][1] - mn1) : 0.0f;
                    pr[b][3] = WIDE ? fast_exp2(x[b][3] - mn1) : 0.0f;
                }
                m0 = mn0;
                m1 = mn1;
                l0 = l0 * r0 + ((pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]));
                if constexpr (WIDE) l1 = l1 * r1 + ((pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]));
                // ---- V scales: exponent reference so the fp16 weights stay in range
                // scale words are positive floats (zero for invisible tokens): their bit patterns order
                // like the values, so the largest word carries the largest exponent
                const uint32_t wmax = max(max(vs0[0], vs1[0]), max(vs0[1], vs1[1]));
                const uint32_t eblk = (__reduce_max_sync(0xffffffffu, wmax) >> 23) & 0xFFu;
                // The exponent reference moves only when a V scale passes it by more than kLazyExp
                // binades (the fp16 weights then stay below 2^(kLazyMax + kLazyExp + 1)).
                float escale = 1.0f;
                if (eblk > eref + kLazyExp || (eref == 0u && eblk > 0u)) {
                    // 2^(eref - eblk); 0 when nothing was accumulated yet or the jump underflows
                    escale = (eref == 0u || eblk - eref > 126u) ? 0.0f : __uint_as_float((127u + eref - eblk) << 23);
                    eref = eblk;
                }
                // (one head per lane when !WIDE: its high- and low-weight columns scale alike)
                const float f0 = r0 * escale, f1 = (WIDE ? r1 : r0) * escale;
                if (__any_sync(0xffffffffu, f0 != 1.0f || f1 != 1.0f)) {
#pragma unroll
                    for (int mt = 0; mt < Gm::MT; ++mt) {
                        o[mt][0] *= f0;
                        o[mt][1] *= f1;
                        o[mt][2] *= f0;
                        o[mt][3] *= f1;
                    }
                    WZ0 *= f0;
                    WZ1 *= f1;
                }
                const float wsc = __uint_as_float((254u - eref) << 23);   // 2^(127 - eref)
                // ---- O^T += Codes_V^T P^T for both blocks
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    if (!ok[b]) continue;
                    constexpr uint32_t kVMask = BITS == 4 ? 0xFFFFFFF0u : 0xFFFFFFFFu;
                    const float sv0 = __uint_as_float(vs0[b] & kVMask) * wsc;
                    const float sv1 = __uint_as_float(vs1[b] & kVMask) * wsc;
                    // weights w = p * s'_V * 2^-E (invisible tokens: 0)
                    const float wa0 = pr[b][0] * sv0, wa1 = pr[b][1] * sv0;   // token tk0
                    const float wb0 = pr[b][2] * sv1, wb1 = pr[b][3] * sv1;   // token tk1
                    uint32_t bb0, bb1;
                    if constexpr (WIDE) {
                        // All eight columns are heads: plain fp16 weights (they are not exponentiated
                        // again, so their 11 bits cost each term at most 2^-11 relative).  sum(w zp)
                        // takes the same rounded weights: the codes' mean is far from zero, so the
                        // rounding errors cancel only against the zero-points they were made with.
                        const uint32_t pa = pack_f16x2(wa0, wa1), pb = pack_f16x2(wb0, wb1);
                        if constexpr (BITS == 4) {
                            // mixed-precision FMAs read the weights in place; a masked zero-point
                            // nibble is the fp16 subnormal zp 2^-24, so WZ runs scaled by 2^-24.  The
                            // products are exact and at least 2^-48, so the scaling changes no
                            // rounding unless a rescale drives the sum below 2^-126.
                            const uint32_t zh0 = vs0[b] & 15u, zh1 = vs1[b] & 15u;
                            WZ0 = fma_f16_f32<false>(pa, zh0, fma_f16_f32<false>(pb, zh1, WZ0));
                            WZ1 = fma_f16_f32<true>(pa, zh0, fma_f16_f32<true>(pb, zh1, WZ1));
                        }
                        bb0 = movmatrix_trans(pa);
                        bb1 = movmatrix_trans(pb);
                    } else {
                        const float zv0 = BITS == 4 ? nibble_to_float(vs0[b]) : 0.0f;
                        const float zv1 = BITS == 4 ? nibble_to_float(vs1[b]) : 0.0f;
                        // head hb's weight as fp16 high (column 2t) + low (column 2t + 1) halves
                        WZ0 = fmaf(wa0, zv0, fmaf(wb0, zv1, WZ0));
                        bb0 = movmatrix_trans(hi_lo_f16x2(wa0));
                        bb1 = movmatrix_trans(hi_lo_f16x2(wb0));
                    }
                    const uint32_t* vr0 = reinterpret_cast<const uint32_t*>(vp[b] + ((t)*H + h) * Rw::RB);
                    const uint32_t* vr1 = reinterpret_cast<const uint32_t*>(vp[b] + ((t + 4) * H + h) * Rw::RB);
                    const uint32_t* vr2 = reinterpret_cast<const uint32_t*>(vp[b] + ((t + 8) * H + h) * Rw::RB);
                    const uint32_t* vr3 = reinterpret_cast<const uint32_t*>(vp[b] + ((t + 12) * H + h) * Rw::RB);
                    // dims 8G + i of two rows as fp16 pairs
                    auto dims8 = [&](const uint32_t* ra, const uint32_t* rb, int G8, uint32_t (&u)[8]) {
                        if constexpr (BITS == 4) unpack_word_pair(ra[G8], rb[G8], kCodeLo, kCodeHi, u);
                        else if constexpr (BITS == 2)
                            unpack_u2_pair(reinterpret_cast<const uint16_t*>(ra)[G8], reinterpret_cast<const uint16_t*>(rb)[G8], u);
                        else unpack_i8_pair(ra[2 * G8], ra[2 * G8 + 1], rb[2 * G8], rb[2 * G8 + 1], u);
                    };
                    if constexpr (D == 128) {
                        uint32_t ua[8], ubv[8], uc[8], ud[8];
                        dims8(vr0, vr1, g, ua);        // d = 8g + i, tokens t, t+4
                        dims8(vr0, vr1, g + 8, ubv);   // d = 64 + 8g + i
                        dims8(vr2, vr3, g, uc);        // tokens t+8, t+12
                        dims8(vr2, vr3, g + 8, ud);
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            mma_f16_16816(o[mt], ua[mt], ubv[mt], uc[mt], ud[mt], bb0, bb1);
                        }
                    } else {
                        uint32_t ua[8], uc[8];
                        dims8(vr0, vr1, g, ua);   // d = 8g + i
                        dims8(vr2, vr3, g, uc);
#pragma unroll
                        for (int mt = 0; mt < 4; ++mt) {
                            mma_f16_16816(o[mt], ua[mt], ua[4 + mt], uc[mt], uc[4 + mt], bb0, bb1);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();   // this warp's reads of the stages come before the counts
                for (int b = 0; b < npair; ++b) {
                    // the counter wraps to 0 on the last warp's increment
                    if (atomicInc(reinterpret_cast<unsigned*>(&released[st[b]]), kConsumerWarps - 1) ==
                        kConsumerWarps - 1) {
                        __threadfence_block();
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        if (i + b + kStages < nb_cta && !*(volatile int*)flags) produce(i + b + kStages);
                    }
                }
            }
        }
        if (stop) break;

        // ---- this warp's partial of unit j: (m, l) per head and O in fragment order, O scaled back
        // by 2^(E - 127).  Record slot (mt, ls) holds (row g: heads 2t', 2t'+1; row g + 8: the same
        // heads) for ls = 2g + t' (t' < 2) when !WIDE, (row g: heads 2t, 2t+1; row g+8: ...) for
        // ls = lane when WIDE; the (m, l) record of heads 2t', 2t'+1 sits at floats 4t' .. 4t'+3.
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            WZ0 += __shfl_xor_sync(0xffffffffu, WZ0, off);
            if constexpr (WIDE) {
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
                WZ1 += __shfl_xor_sync(0xffffffffu, WZ1, off);
            }
        }
        if constexpr (WIDE && BITS == 4) {   // sum(w zp) was carried scaled by 2^-24
            WZ0 *= 16777216.0f;
            WZ1 *= 16777216.0f;
        }
        const float es = eref ? __uint_as_float(eref << 23) : 0.0f;   // 2^(eref - 127)
        const size_t recn = (size_t)u.z * kConsumerWarps + warp;
        if constexpr (WIDE) {
            // O = sum(w code) - sum(w zp)
            float4* po = reinterpret_cast<float4*>(p.ws_po + recn * PO) + lane;
#pragma unroll
            for (int mt = 0; mt < Gm::MT; ++mt)
                po[mt * NLS] = make_float4((o[mt][0] - WZ0) * es, (o[mt][1] - WZ1) * es, (o[mt][2] - WZ0) * es,
                                           (o[mt][3] - WZ1) * es);
            if (g == 0) {
                float* ml = p.ws_pml + recn * 16 + 4 * t;
                ml[0] = m0;
                ml[1] = l0;
                ml[2] = m1;
                ml[3] = l1;
            }
        } else {
            // head t = high + low weight columns; lanes with even t take their neighbour's head
            float4* po = reinterpret_cast<float4*>(p.ws_po + recn * PO) + (g * 2 + (t >> 1));
#pragma unroll
            for (int mt = 0; mt < Gm::MT; ++mt) {
                const float a = (o[mt][0] + o[mt][1] - WZ0) * es, b = (o[mt][2] + o[mt][3] - WZ0) * es;
                const float a1 = __shfl_xor_sync(0xffffffffu, a, 1), b1 = __shfl_xor_sync(0xffffffffu, b, 1);
                if ((t & 1) == 0) po[mt * NLS] = make_float4(a, a1, b, b1);
            }
            const float m_n = __shfl_xor_sync(0xffffffffu, m0, 1), l_n = __shfl_xor_sync(0xffffffffu, l0, 1);
            if (g == 0 && (t & 1) == 0) {
                float* ml = p.ws_pml + recn * 16 + 2 * t;
                ml[0] = m0;
                ml[1] = l0;
                ml[2] = m_n;
                ml[3] = l_n;
            }
        }
    }

    // ---- a wait gave up: let every copy still in flight land before the CTA exits
    __syncthreads();
    if (threadIdx.x == 0 && flags[0]) {
        const int issued = flags[1];
        for (int i = max(0, issued - kStages); i < issued; ++i) mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u);
        const int qissued = flags[2];
        for (int r = max(0, qissued - nq); r < qissued; ++r) mbar_wait(&qfull[r & (nq - 1)], (uint32_t)(r >> (nq - 1)) & 1u);
    }
}

// ------------------------------------------------------------------ 2. combine

constexpr int kCombineWarps = 16;

// Dynamic shared memory of a combine CTA whose groups of W warps each own one (sequence, kv head).
template <int D, bool WIDE>
__host__ __device__ inline size_t combine_smem_bytes(int W, int G) {
    const int NT = Geo<D>::MT * (WIDE ? 32 : 16);
    return (size_t)kCombineWarps * NT * 16            // per-warp accumulator slots
           + (size_t)kCombineWarps * 4 * 16           // per-warp (m, l) of 8 columns
           + (size_t)(kCombineWarps / W) * G * (D + 4) * 4;   // normalised outputs per group
}

// A CTA of 16 warps in groups of W (a power of two, sized for the batch's longest sequence);
// group k owns (sequence, kv head) item blockIdx.x * 16 / W + k, a record being (segment, walker
// warp of that kv head).  The merge tree depends only on the item's own record count R, never on
// the batch: the records form nc = min(16, pow2 >= ceil(R / 4)) <= W contiguous chunks of
// ceil(R / nc); warp c folds chunk c in record order with an online rescaling, each lane owning
// the accumulator slots lane + 32 j of the fragment-ordered partials (whole 512-byte rows, so
// every load is coalesced, several records in flight), and the chunk states are then folded in
// chunk order through shared memory, normalised, and the G outputs un-rotated by the group's warps.
template <int D, bool WIDE, int BITS, typename OT>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const __grid_constant__ AttnParams p) {
    constexpr int NLS = WIDE ? 32 : 16;
    constexpr int NT = Geo<D>::MT * NLS;   // float4 slots of one record
    constexpr int SPL = NT / 32;           // slots per lane
    constexpr int UNR = WIDE ? 2 : 4;      // records in flight per lane
    constexpr int SO = D + 4;
    constexpr int kThreads = kCombineWarps * 32;
    __shared__ float sgn[D];
    __shared__ int wsum_c[kCombineWarps];
    __shared__ int first_unit[kThreads];   // batches of up to kThreads sequences: first unit of each
    extern __shared__ __align__(16) float4 cbuf[];
    float4* sacc = cbuf;                                   // [16 warps][NT]
    float4* sml = cbuf + kCombineWarps * NT;               // [16 warps][4]
    float* sout = reinterpret_cast<float*>(sml + kCombineWarps * 4);   // [groups][G][SO]
    // Up to the wait on the walker this kernel reads only host inputs, so it overlaps the walker's
    // last CTAs on the SMs they have left.
    if constexpr (BITS != 8)
        for (int i = threadIdx.x; i < D; i += blockDim.x) sgn[i] = p.signs[i] < 0.0f ? -1.0f : 1.0f;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // decode segments of sequence b (0 for other sequences), as the walker counts them
    auto segments_of = [&](int b) -> int {
        const int qb = __ldg(p.qsl + b);
        if (__ldg(p.qsl + b + 1) - qb != 1 || qb < 0 || (int64_t)qb >= p.num_q_tokens) return 0;
        const int L = min(max(__ldg(p.seq_lens + b), 0), p.len_cap);
        return (int)fast_div((uint32_t)(L + p.seg_len - 1), (uint32_t)p.seg_len, p.seg_rcp);
    };
    const bool local_first = p.num_seqs <= kThreads;   // else the walker's index in ws_meta
    if (local_first) {
        const int b = threadIdx.x;
        const int ns = b < p.num_seqs ? segments_of(b) : 0;
        int x = ns;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum_c[warp] = x;
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += wsum_c[w];
        first_unit[b] = before + x - ns;
    }
    const int W = p.combine_warps, grp = warp / W, sub = warp % W;
    const int H = p.H, G = p.G, Hq = p.Hq;
    const int64_t item = (int64_t)blockIdx.x * (kCombineWarps / W) + grp;
    const int h = (int)(item % H);
    const int seq = (int)(item / H);
    // Items past the batch, non-decode sequences and empty contexts do no merging, but every
    // thread reaches the barriers below.
    int nseg = 0, q0 = 0;
    bool active = seq < p.num_seqs;
    if (active) {
        q0 = __ldg(p.qsl + seq);
        active = __ldg(p.qsl + seq + 1) - q0 == 1 && q0 >= 0 && (int64_t)q0 < p.num_q_tokens;
    }
    if (active) {
        const int L = min(max(__ldg(p.seq_lens + seq), 0), p.len_cap);
        nseg = (int)fast_div((uint32_t)(L + p.seg_len - 1), (uint32_t)p.seg_len, p.seg_rcp);
    }
    const int64_t obase = ((int64_t)q0 * Hq + (int64_t)h * G) * D;
    const int ws = p.wph_shift;
    const int R = nseg << ws;
    __syncthreads();   // first_unit complete
    griddep_wait();
    griddep_launch_dependents();   // the next call's kernels may start their set-up
    const int ub = R > 0 ? (local_first ? first_unit[seq] : p.ws_meta[seq]) : 0;
    auto rec_of = [&](int r) -> size_t {
        return (size_t)(ub + (r >> ws)) * kConsumerWarps + h + (r & ((1 << ws) - 1)) * H;
    };
    const int tq = WIDE ? (lane & 3) : (lane & 1);   // this lane's columns: 2 tq, 2 tq + 1

    float m0 = kNegBig, m1 = kNegBig, l0 = 0.0f, l1 = 0.0f;
    float4 acc[SPL];
#pragma unroll
    for (int k = 0; k < SPL; ++k) acc[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    auto merge = [&](const float4& ml, const float4 (&ov)[SPL]) {
        const float n0 = fmaxf(m0, ml.x), n1 = fmaxf(m1, ml.z);
        const float a0 = fast_exp2(m0 - n0), b0 = fast_exp2(ml.x - n0);
        const float a1 = fast_exp2(m1 - n1), b1 = fast_exp2(ml.z - n1);
#pragma unroll
        for (int k = 0; k < SPL; ++k) {
            acc[k].x = acc[k].x * a0 + ov[k].x * b0;
            acc[k].z = acc[k].z * a0 + ov[k].z * b0;
            acc[k].y = acc[k].y * a1 + ov[k].y * b1;
            acc[k].w = acc[k].w * a1 + ov[k].w * b1;
        }
        l0 = l0 * a0 + ml.y * b0;
        l1 = l1 * a1 + ml.w * b1;
        m0 = n0;
        m1 = n1;
    };
    const float4* po = reinterpret_cast<const float4*>(p.ws_po);
    const float4* pml = reinterpret_cast<const float4*>(p.ws_pml);
    int nc = 1;
    while (nc < 16 && nc * 4 < R) nc <<= 1;
    const int K = (R + nc - 1) / nc;
    const int r_lo = sub < nc ? sub * K : R, r_hi = sub < nc ? min(R, (sub + 1) * K) : R;
    for (int r0 = r_lo; r0 < r_hi; r0 += UNR) {
        float4 ml[UNR], ov[UNR][SPL];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int r = r0 + u;
            const bool live = r < r_hi;
            const size_t rc = rec_of(live ? r : r0);
            ml[u] = live ? pml[rc * 4 + tq] : make_float4(kNegBig, 0.0f, kNegBig, 0.0f);
#pragma unroll
            for (int k = 0; k < SPL; ++k) ov[u][k] = live ? po[rc * NT + lane + 32 * k] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) merge(ml[u], ov[u]);
    }
    // the warps' states through shared memory; the group's threads then merge its slots
#pragma unroll
    for (int k = 0; k < SPL; ++k) sacc[warp * NT + lane + 32 * k] = acc[k];
    if (lane < (WIDE ? 4 : 2)) sml[warp * 4 + tq] = make_float4(m0, l0, m1, l1);
    __syncthreads();
    float* gout = sout + (size_t)grp * G * SO;
    if (R > 0) {
        const int w0 = grp * W;
        for (int slot = sub * 32 + lane; slot < NT; slot += W * 32) {
            const int mt = slot / NLS, ls = slot % NLS;
            const int sq = WIDE ? (ls & 3) : (ls & 1), gq = WIDE ? (ls >> 2) : (ls >> 1);
            float M0 = kNegBig, M1 = kNegBig;
            for (int w = 0; w < W; ++w) {
                M0 = fmaxf(M0, sml[(w0 + w) * 4 + sq].x);
                M1 = fmaxf(M1, sml[(w0 + w) * 4 + sq].z);
            }
            float L0 = 0.0f, L1 = 0.0f;
            float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int w = 0; w < W; ++w) {
                const float4 v = sml[(w0 + w) * 4 + sq], o = sacc[(w0 + w) * NT + slot];
                const float e0 = fast_exp2(v.x - M0), e1 = fast_exp2(v.z - M1);
                L0 += v.y * e0;
                L1 += v.w * e1;
                a.x += o.x * e0;
                a.z += o.z * e0;
                a.y += o.y * e1;
                a.w += o.w * e1;
            }
            const int c0 = 2 * sq, c1 = c0 + 1;
            const int dlo = 8 * gq + mt;
            const int dhi = (D == 128) ? 64 + 8 * gq + mt : 8 * gq + 4 + mt;
            if (c0 < G) {
                const float inv = L0 > 0.0f ? 1.0f / L0 : 0.0f;
                gout[c0 * SO + dlo] = a.x * inv;
                gout[c0 * SO + dhi] = a.z * inv;
            }
            if (c1 < G) {
                const float inv = L1 > 0.0f ? 1.0f / L1 : 0.0f;
                gout[c1 * SO + dlo] = a.y * inv;
                gout[c1 * SO + dhi] = a.w * inv;
            }
        }
    }
    __syncthreads();
    if (!active) return;
    if (R == 0) {   // empty context: zero output
        for (int i = sub * 32 + lane; i < G * D; i += W * 32) store_elem<OT>(p.out, obase + i, 0.0f);
        return;
    }
    for (int col = sub; col < G; col += W) {
        float x[D / 32];
#pragma unroll
        for (int k = 0; k < D / 32; ++k) x[k] = gout[col * SO + lane + 32 * k];
        if constexpr (BITS != 8) {
            unrotate_store<D, OT>(x, 1.0f, sgn, p.c, p.out, obase + (int64_t)col * D);
        } else {   // INT8: the output is not rotated
#pragma unroll
            for (int k = 0; k < D / 32; ++k) store_elem<OT>(p.out, obase + (int64_t)col * D + lane + 32 * k, x[k]);
        }
    }
}

// ------------------------------------------------------------------ launchers

template <int D, bool WIDE, int BITS, typename QT, typename OT>
cudaError_t launch_decode_t(const AttnParams& p, int num_ctas, cudaStream_t stream) {
    const DecodeSmem lay = decode_smem_layout<D, WIDE, BITS>(p.H, p.Hq);
    const bool opts = BITS == 4 && p.opts != 0;
    auto walker = opts ? decode_kernel<D, WIDE, BITS, BITS == 4> : decode_kernel<D, WIDE, BITS, false>;
    cudaError_t err = opts ? opt_in_smem<decode_kernel<D, WIDE, BITS, BITS == 4>>(lay.total)
                           : opt_in_smem<decode_kernel<D, WIDE, BITS, false>>(lay.total);
    if (err != cudaSuccess) return err;
    // All three kernels are programmatic dependents of their predecessor: each starts its set-up
    // while the previous kernel finishes and waits for it (griddep_wait) before touching its
    // results.
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    const size_t qsm = D * 4 + 2 * (size_t)((p.Hq + 3) & ~3) * 4 + 2 * (size_t)p.Hq * D * 2;
    cudaLaunchConfig_t qcfg = {};
    qcfg.gridDim = dim3((unsigned)p.num_seqs);
    qcfg.blockDim = dim3(256);
    qcfg.dynamicSmemBytes = qsm;
    qcfg.stream = stream;
    qcfg.attrs = &attr;
    qcfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&qcfg, qrot_kernel<D, WIDE, BITS, QT>, p);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t wcfg = {};
    wcfg.gridDim = dim3((unsigned)num_ctas);
    wcfg.blockDim = dim3(kDecodeThreads);
    wcfg.dynamicSmemBytes = lay.total;
    wcfg.stream = stream;
    wcfg.attrs = &attr;
    wcfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&wcfg, walker, p);
    if (err != cudaSuccess) return err;

    const int W = p.combine_warps;
    const int64_t items = (int64_t)p.num_seqs * p.H;
    const int64_t per_cta = kCombineWarps / W;
    const size_t csmem = combine_smem_bytes<D, WIDE>(W, p.G);
    err = opt_in_smem<combine_kernel<D, WIDE, BITS, OT>>(csmem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((items + per_cta - 1) / per_cta));
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.dynamicSmemBytes = csmem;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel<D, WIDE, BITS, OT>, p);
}

template <int D, bool WIDE, int BITS, typename QT>
cudaError_t decode_by_out(const AttnParams& p, int num_ctas, DType out_dt, cudaStream_t s) {
    switch (out_dt) {
        case DType::F16: return launch_decode_t<D, WIDE, BITS, QT, __half>(p, num_ctas, s);
        case DType::BF16: return launch_decode_t<D, WIDE, BITS, QT, __nv_bfloat16>(p, num_ctas, s);
        default: return launch_decode_t<D, WIDE, BITS, QT, float>(p, num_ctas, s);
    }
}

template <int D, bool WIDE, int BITS>
cudaError_t decode_by_q(const AttnParams& p, int num_ctas, DType q_dt, DType out_dt, cudaStream_t s) {
    return q_dt == DType::BF16 ? decode_by_out<D, WIDE, BITS, __nv_bfloat16>(p, num_ctas, out_dt, s)
                               : decode_by_out<D, WIDE, BITS, __half>(p, num_ctas, out_dt, s);
}

// Every (head size, grouping, query type, output type) instantiation of one cache mode.
template <int BITS>
cudaError_t launch_decode_mode(const AttnParams& p, int head_size, int num_ctas, DType q_dt, DType out_dt,
                               cudaStream_t stream) {
    const bool wide = p.G == 8;
    if (head_size == 128)
        return wide ? decode_by_q<128, true, BITS>(p, num_ctas, q_dt, out_dt, stream)
                    : decode_by_q<128, false, BITS>(p, num_ctas, q_dt, out_dt, stream);
    return wide ? decode_by_q<64, true, BITS>(p, num_ctas, q_dt, out_dt, stream)
                : decode_by_q<64, false, BITS>(p, num_ctas, q_dt, out_dt, stream);
}

}  // namespace
}  // namespace kvi4
