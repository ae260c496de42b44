// Decode attention over the INT4 cache (one query token per sequence), with split-KV segments.
//
// Method ("[Feature] Triton INT4 / INT2 per-token-head KV cache quantization", description of the
// packed read path): Q is rotated with the same random Hadamard transform as K and V, scores are
// dot products of the rotated query with the raw 4-bit codes, the asymmetry (zero-point) is
// corrected per key and the per-key scale applied, an online softmax accumulates P V in the
// rotated domain, and the output is un-rotated.  Long contexts are split into segments whose
// (max, sum, accumulator) partials are combined afterwards ("3D" segment reduction of the
// unified-attention interface, test_triton_unified_attention_per_token_head_scale).
//
// GB300 design:
//  * One CTA per (sequence, segment) covers ALL kv heads, so each 16-token block is one
//    contiguous 16-byte-aligned region (K plane then V plane, 2 * 16 * H * (D/2+4) bytes) that is
//    streamed into a 4-stage shared-memory ring with 1-D bulk async copies (cp.async.bulk +
//    mbarrier transaction counts, L2 evict-first).  There is no producer warp: the segment's block
//    ids are staged in shared memory up front, four lanes issue the first four copies, and the
//    last consumer warp to finish with a stage issues its next block.
//  * Eight consumer warps: warp w owns kv head w % H (and every (8/H)-th block when H < 8).
//    Scores S^T[16 tokens x 8 heads] = (K - zp)[16 x D] . Q'^T come from mma.sync m16n8k16 on
//    fp16 operands built straight from the packed bytes (codes and code - zp are exact in fp16);
//    the zero-point is subtracted while unpacking, which is the sum(Q) * zp correction folded in.
//  * P^T is transposed in registers (movmatrix) into the B operand of O^T[D x 8] += (V - zp)^T P^T.
//    V's per-key scale is folded into P (w = p * s'_V * 2^-E, E a running max exponent, so the fp16
//    weights never overflow).
#include "attn_common.cuh"

namespace kvi4 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = kConsumerWarps * 32;   // no producer warp: see the refill rule below
constexpr int kStages = 4;
constexpr int kTableWin = 512;   // block-table entries of a CTA's segment staged in shared memory

struct DecodeSmem {
    uint32_t stage_bytes;   // one block (K + V planes)
    uint32_t state_off;     // start of barriers etc. (after the ring / epilogue state overlay)
    uint32_t total;
};

template <int D>
__host__ __device__ inline DecodeSmem decode_smem_layout(int H, int Hq) {
    DecodeSmem s;
    s.stage_bytes = 2u * kBlockSize * (uint32_t)H * Geo<D>::RB;
    const uint32_t ring = kStages * s.stage_bytes;
    const uint32_t state = kConsumerWarps * 8u * D * 4u;
    s.state_off = ((ring > state ? ring : state) + 127u) & ~127u;
    const uint32_t tail = 2u * kStages * 8u      // full / empty barriers
                          + kStages * 4u + 16u     // valid flags, abort flag
                          + kStages * 4u + 16u     // refill counters
                          + kTableWin * 4u         // block-table window
                          + D * 4u                 // signs
                          + (uint32_t)Hq * 4u      // alpha
                          + 2u * kConsumerWarps * 8u * 4u  // per-warp (m, l)
                          + 2u * (uint32_t)Hq * D * 2u;  // rotated queries, fp16 hi and lo halves
    s.total = s.state_off + ((tail + 127u) & ~127u);
    return s;
}

template <int D, bool WIDE, typename QT, typename OT>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_kernel(const __grid_constant__ AttnParams p) {
    using Gm = Geo<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int seg = blockIdx.x, seq = blockIdx.y;
    const int q0 = __ldg(p.qsl + seq);
    if (__ldg(p.qsl + seq + 1) - q0 != 1) return;   // not a decode sequence
    if (q0 < 0 || (int64_t)q0 >= p.num_q_tokens) {
        if (seg == 0 && threadIdx.x == 0) count_status(p.status, 2);
        return;
    }
    const int H = p.H, G = p.G, Hq = p.Hq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int L = __ldg(p.seq_lens + seq);
    const int Lmax = min(p.max_blocks_per_seq * kBlockSize, p.nseg_max * p.seg_len);
    if (L > Lmax) {   // longer than its block table or than the max_seq_len the grid was sized for
        if (seg == 0 && threadIdx.x == 0) count_status(p.status, 2);
        L = Lmax;
    }
    if (L <= 0) {   // empty context: zero output
        if (seg == 0) {
            for (int i = threadIdx.x; i < Hq * D; i += blockDim.x) store_elem<OT>(p.out, (int64_t)q0 * Hq * D + i, 0.0f);
        }
        return;
    }
    const int S = p.seg_len;
    const int tok_begin = seg * S;
    if (tok_begin >= L) return;
    const int tok_end = min(L, tok_begin + S);
    const int nseg = (L + S - 1) / S;
    const int blk_first = tok_begin / kBlockSize;
    const int nblk = (tok_end + kBlockSize - 1) / kBlockSize - blk_first;

    const DecodeSmem lay = decode_smem_layout<D>(H, Hq);
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.state_off);
    int* valid = reinterpret_cast<int*>(full + 2 * kStages);
    int* abort_flag = valid + kStages;
    int* released = abort_flag + 4;    // per stage: consumer warps done with its current block
    int* tbl = released + kStages + 4;    // block ids of this segment's first kTableWin blocks
    float* sgn = reinterpret_cast<float*>(tbl + kTableWin);
    float* alpha = sgn + D;
    float* st_m = alpha + Hq;
    float* st_l = st_m + kConsumerWarps * 8;
    __half* qh = reinterpret_cast<__half*>(st_l + kConsumerWarps * 8);
    __half* ql = qh + Hq * D;
    float* st_o = reinterpret_cast<float*>(smem);   // epilogue overlay of the ring

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0;
        }
        abort_flag[0] = 0;
        abort_flag[1] = 0;   // blocks issued so far
        fence_mbar_init();
    }
    const int32_t* table = p.block_tables + (int64_t)seq * p.max_blocks_per_seq + blk_first;
    // one coalesced load of the segment's block ids, so that no ring refill waits on global memory
    for (int i = threadIdx.x; i < min(nblk, kTableWin); i += blockDim.x) tbl[i] = __ldg(table + i);
    for (int i = threadIdx.x; i < D; i += blockDim.x) sgn[i] = p.signs[i] < 0.0f ? -1.0f : 1.0f;
    __syncthreads();

    const uint8_t* seq_cache = p.cache;
    const uint32_t stage_bytes = lay.stage_bytes;
    // Ring refill rule: block i goes to stage i % kStages.  The first kStages blocks are issued up
    // front; afterwards the LAST consumer warp to finish with block i (counted in released[])
    // issues block i + kStages into the same stage, so no warp ever blocks waiting to refill.
    auto produce = [&](int i) {
        const int st = i % kStages;
        const int blk = i < kTableWin ? tbl[i] : __ldg(table + i);
        const bool ok = blk >= 0 && (int64_t)blk < p.num_blocks;
        valid[st] = ok ? 1 : 0;
        atomicMax(&abort_flag[1], i + 1);
        if (ok) {
            mbar_arrive_expect_tx(&full[st], stage_bytes);
            bulk_copy_g2s(ring + (size_t)st * stage_bytes, seq_cache + (int64_t)blk * stage_bytes, stage_bytes, &full[st],
                          policy_evict_first());
        } else {
            count_status(p.status, 1);
            mbar_arrive(&full[st]);
        }
    };
    if (threadIdx.x < min(kStages, nblk)) produce(threadIdx.x);   // the first copies, one lane each

    // Rotate this sequence's query (all Hq heads) into fp16 halves + per-head logit multiplier,
    // four vectors per warp at a time.
    for (int v0 = warp; v0 < Hq; v0 += 4 * kConsumerWarps) {
        int64_t rows[4];
        int slot[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int v = v0 + k * kConsumerWarps;
            rows[k] = v < Hq ? (int64_t)q0 * Hq + v : -1;
            slot[k] = v < Hq ? v : 0;
        }
        rotate_queries<D, QT, 4>(p.q, rows, slot, sgn, qh, ql, alpha, p.c, p.softmax_scale);
    }
    __syncthreads();

    // consumer state (lives across the role split so that the barriers below are uniform)
    float o[Gm::MT][4];
#pragma unroll
    for (int i = 0; i < Gm::MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m0 = kNegBig, m1 = kNegBig, l0 = 0.0f, l1 = 0.0f;
    uint32_t eref = 0;   // running max biased exponent of V scales seen so far
    const int g = lane >> 2, t = lane & 3;

    {
        // ------------------------------------------------------------------ consumers
        const int h = warp % H;
        const int wph = kConsumerWarps / H;
        const int sub = warp / H;
        const int tk0 = block_token(g), tk1 = block_token(g + 8);

        // Score columns (the mma N dimension, 8 wide).  WIDE (8 query heads per kv head): column n
        // is head n, with a second 8-wide tile carrying the low halves.  Otherwise columns 0-3
        // carry the high halves of heads 0-3 and columns 4-7 their low halves, so the split costs
        // no extra mma: lane quad t then holds heads hb, hb+1 with hb = 2 (t & 1).
        const int hb = WIDE ? 2 * t : 2 * (t & 1);
        uint32_t qb[Gm::KSTEPS][WIDE ? 4 : 2];
        {
            const int head = WIDE ? g : (g & 3);
            const bool live = head < G;
            const __half* qv = (WIDE || g < 4 ? qh : ql) + (h * G + (live ? head : 0)) * D;
            const __half* qv2 = ql + (h * G + (live ? head : 0)) * D;
            const __half z = __float2half(0.0f);
#pragma unroll
            for (int j = 0; j < Gm::KWPT; ++j) {
                const int W = t + 4 * j;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int d0 = 8 * W + 2 * hh;
                    __half2 b0 = live ? __halves2half2(qv[d0], qv[d0 + 4]) : __halves2half2(z, z);
                    __half2 b1 = live ? __halves2half2(qv[d0 + 1], qv[d0 + 5]) : __halves2half2(z, z);
                    qb[2 * j + hh][0] = *reinterpret_cast<uint32_t*>(&b0);
                    qb[2 * j + hh][1] = *reinterpret_cast<uint32_t*>(&b1);
                    if constexpr (WIDE) {
                        __half2 c0 = live ? __halves2half2(qv2[d0], qv2[d0 + 4]) : __halves2half2(z, z);
                        __half2 c1 = live ? __halves2half2(qv2[d0 + 1], qv2[d0 + 5]) : __halves2half2(z, z);
                        qb[2 * j + hh][2] = *reinterpret_cast<uint32_t*>(&c0);
                        qb[2 * j + hh][3] = *reinterpret_cast<uint32_t*>(&c1);
                    }
                }
            }
        }
        const float al0 = (hb < G) ? alpha[h * G + hb] : 0.0f;
        const float al1 = (hb + 1 < G) ? alpha[h * G + hb + 1] : 0.0f;
        const bool lo_lane = !WIDE && t >= 2;   // this lane's P columns carry low halves

        // Two blocks (32 tokens) per iteration: their score chains, one softmax update and their
        // P.V products interleave, which gives each warp independent work to overlap latencies.
        for (int i = 0; i < nblk; i += 2) {
            const int npair = min(2, nblk - i);
            int st[2];
            bool ok[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) st[b] = (i + b) % kStages;
            bool timed_out = false;
            for (int b = 0; b < npair; ++b) {
                if (!mbar_wait(&full[st[b]], ((i + b) / kStages) & 1)) timed_out = true;
            }
            if (timed_out) {
                if (lane == 0) {
                    count_status(p.status, 3);
                    atomicExch(abort_flag, 1);
                }
                break;
            }
#pragma unroll
            for (int b = 0; b < 2; ++b) ok[b] = b < npair && valid[st[b]];
            if (((i >> 1) % wph) == sub && (ok[0] || ok[1])) {
                const uint8_t* kp[2];
                const uint8_t* vp[2];
                int tokbase[2];
                float x[2][4];
                uint32_t vs0[2], vs1[2];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    kp[b] = ring + (size_t)st[b] * stage_bytes;
                    vp[b] = kp[b] + (size_t)kBlockSize * H * Gm::RB;
                    tokbase[b] = (blk_first + i + b) * kBlockSize;
                }
                // ---- S^T = (K - zp) Q'^T for both blocks, high and low halves of Q'
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const uint32_t* kr0 = reinterpret_cast<const uint32_t*>(kp[b] + (tk0 * H + h) * Gm::RB);
                    const uint32_t* kr1 = reinterpret_cast<const uint32_t*>(kp[b] + (tk1 * H + h) * Gm::RB);
                    const uint32_t ks0 = kr0[Gm::KW], ks1 = kr1[Gm::KW];
                    float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    float cl[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    if (ok[b]) {
                        const uint32_t z0l = zp_lo_half(ks0 & 15u), z0h = zp_hi_half(ks0 & 15u);
                        const uint32_t z1l = zp_lo_half(ks1 & 15u), z1h = zp_hi_half(ks1 & 15u);
                        const uint32_t zl0 = z0l | (z0l << 16), zh0 = z0h | (z0h << 16);
                        const uint32_t zl1 = z1l | (z1l << 16), zh1 = z1h | (z1h << 16);
#pragma unroll
                        for (int j = 0; j < Gm::KWPT; ++j) {
                            uint32_t a0[4], a1[4];
                            unpack_word(kr0[t + 4 * j], zl0, zh0, a0);
                            unpack_word(kr1[t + 4 * j], zl1, zh1, a1);
                            mma_f16_16816(c, a0[0], a1[0], a0[1], a1[1], qb[2 * j][0], qb[2 * j][1]);
                            mma_f16_16816(c, a0[2], a1[2], a0[3], a1[3], qb[2 * j + 1][0], qb[2 * j + 1][1]);
                            if constexpr (WIDE) {
                                mma_f16_16816(cl, a0[0], a1[0], a0[1], a1[1], qb[2 * j][2], qb[2 * j][3]);
                                mma_f16_16816(cl, a0[2], a1[2], a0[3], a1[3], qb[2 * j + 1][2], qb[2 * j + 1][3]);
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if constexpr (WIDE) c[e] += cl[e];
                        else c[e] += __shfl_xor_sync(0xffffffffu, c[e], 2);   // high + low columns
                    }
                    const bool v0 = ok[b] && tokbase[b] + tk0 < tok_end, v1 = ok[b] && tokbase[b] + tk1 < tok_end;
                    const float sk0 = __uint_as_float(ks0 & 0xFFFFFFF0u), sk1 = __uint_as_float(ks1 & 0xFFFFFFF0u);
                    x[b][0] = v0 ? c[0] * sk0 * al0 : -INFINITY;
                    x[b][1] = v0 ? c[1] * sk0 * al1 : -INFINITY;
                    x[b][2] = v1 ? c[2] * sk1 * al0 : -INFINITY;
                    x[b][3] = v1 ? c[3] * sk1 * al1 : -INFINITY;
                    const uint32_t* vg0 = reinterpret_cast<const uint32_t*>(vp[b] + (tk0 * H + h) * Gm::RB);
                    const uint32_t* vg1 = reinterpret_cast<const uint32_t*>(vp[b] + (tk1 * H + h) * Gm::RB);
                    vs0[b] = v0 ? vg0[Gm::KW] : 0u;   // invisible tokens: scale word 0 (exponent 0, weight 0)
                    vs1[b] = v1 ? vg1[Gm::KW] : 0u;
                }
                // ---- one online-softmax update for heads hb, hb+1 over the 32 tokens
                float bm0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
                float bm1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
                }
                const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
                const float r0 = fast_exp2(m0 - mn0), r1 = fast_exp2(m1 - mn1);
                float pr[2][4];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    pr[b][0] = fast_exp2(x[b][0] - mn0);
                    pr[b][1] = fast_exp2(x[b][1] - mn1);
                    pr[b][2] = fast_exp2(x[b][2] - mn0);
                    pr[b][3] = fast_exp2(x[b][3] - mn1);
                }
                m0 = mn0;
                m1 = mn1;
                l0 = l0 * r0 + ((pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]));
                l1 = l1 * r1 + ((pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]));
                // ---- V scales: exponent reference so the fp16 weights stay in range
                const uint32_t emax = max(max((vs0[0] >> 23) & 0xFFu, (vs1[0] >> 23) & 0xFFu),
                                          max((vs0[1] >> 23) & 0xFFu, (vs1[1] >> 23) & 0xFFu));
                const uint32_t eblk = __reduce_max_sync(0xffffffffu, emax);
                float escale = 1.0f;
                if (eblk > eref) {
                    // 2^(eref - eblk); 0 when nothing was accumulated yet or the jump underflows
                    escale = (eref == 0u || eblk - eref > 126u) ? 0.0f : __uint_as_float((127u + eref - eblk) << 23);
                    eref = eblk;
                }
                const float f0 = r0 * escale, f1 = r1 * escale;
                if (__any_sync(0xffffffffu, f0 != 1.0f || f1 != 1.0f)) {
#pragma unroll
                    for (int mt = 0; mt < Gm::MT; ++mt) {
                        o[mt][0] *= f0;
                        o[mt][1] *= f1;
                        o[mt][2] *= f0;
                        o[mt][3] *= f1;
                    }
                }
                const float wsc = __uint_as_float((254u - eref) << 23);   // 2^(127 - eref)
                // ---- O^T += (V - zp)^T P^T for both blocks
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    if (!ok[b]) continue;
                    const float sv0 = __uint_as_float(vs0[b] & 0xFFFFFFF0u) * wsc;
                    const float sv1 = __uint_as_float(vs1[b] & 0xFFFFFFF0u) * wsc;
                    // weights w = p * s'_V * 2^-E as fp16 high + low halves (invisible tokens: 0)
                    uint32_t xlo_h, xlo_l, xhi_h, xhi_l;
                    split_f16x2(pr[b][0] * sv0, pr[b][1] * sv0, xlo_h, xlo_l);
                    split_f16x2(pr[b][2] * sv1, pr[b][3] * sv1, xhi_h, xhi_l);
                    uint32_t b0, b1, b0l = 0, b1l = 0;
                    if constexpr (WIDE) {
                        b0 = movmatrix_trans(xlo_h);
                        b1 = movmatrix_trans(xhi_h);
                        b0l = movmatrix_trans(xlo_l);
                        b1l = movmatrix_trans(xhi_l);
                    } else {
                        b0 = movmatrix_trans(lo_lane ? xlo_l : xlo_h);
                        b1 = movmatrix_trans(lo_lane ? xhi_l : xhi_h);
                    }
                    const uint32_t* vr0 = reinterpret_cast<const uint32_t*>(vp[b] + ((t)*H + h) * Gm::RB);
                    const uint32_t* vr1 = reinterpret_cast<const uint32_t*>(vp[b] + ((t + 4) * H + h) * Gm::RB);
                    const uint32_t* vr2 = reinterpret_cast<const uint32_t*>(vp[b] + ((t + 8) * H + h) * Gm::RB);
                    const uint32_t* vr3 = reinterpret_cast<const uint32_t*>(vp[b] + ((t + 12) * H + h) * Gm::RB);
                    const uint32_t w0 = vr0[Gm::KW], w1 = vr1[Gm::KW], w2 = vr2[Gm::KW], w3 = vr3[Gm::KW];
                    const uint32_t zl01 = zp_lo_half(w0 & 15u) | (zp_lo_half(w1 & 15u) << 16);
                    const uint32_t zh01 = zp_hi_half(w0 & 15u) | (zp_hi_half(w1 & 15u) << 16);
                    const uint32_t zl23 = zp_lo_half(w2 & 15u) | (zp_lo_half(w3 & 15u) << 16);
                    const uint32_t zh23 = zp_hi_half(w2 & 15u) | (zp_hi_half(w3 & 15u) << 16);
                    if constexpr (D == 128) {
                        uint32_t ua[8], ub[8], uc[8], ud[8];
                        unpack_word_pair(vr0[g], vr1[g], zl01, zh01, ua);           // d = 8g + i, tokens t, t+4
                        unpack_word_pair(vr0[g + 8], vr1[g + 8], zl01, zh01, ub);   // d = 64 + 8g + i
                        unpack_word_pair(vr2[g], vr3[g], zl23, zh23, uc);           // tokens t+8, t+12
                        unpack_word_pair(vr2[g + 8], vr3[g + 8], zl23, zh23, ud);
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            mma_f16_16816(o[mt], ua[mt], ub[mt], uc[mt], ud[mt], b0, b1);
                            if constexpr (WIDE) mma_f16_16816(o[mt], ua[mt], ub[mt], uc[mt], ud[mt], b0l, b1l);
                        }
                    } else {
                        uint32_t ua[8], uc[8];
                        unpack_word_pair(vr0[g], vr1[g], zl01, zh01, ua);   // d = 8g + i
                        unpack_word_pair(vr2[g], vr3[g], zl23, zh23, uc);
#pragma unroll
                        for (int mt = 0; mt < 4; ++mt) {
                            mma_f16_16816(o[mt], ua[mt], ua[4 + mt], uc[mt], uc[4 + mt], b0, b1);
                            if constexpr (WIDE) mma_f16_16816(o[mt], ua[mt], ua[4 + mt], uc[mt], uc[4 + mt], b0l, b1l);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();   // this warp's reads of the stages come before the counts
                for (int b = 0; b < npair; ++b) {
                    if (atomicAdd(&released[st[b]], 1) == kConsumerWarps - 1) {
                        released[st[b]] = 0;
                        __threadfence_block();
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        if (i + b + kStages < nblk && !*(volatile int*)abort_flag) produce(i + b + kStages);
                    }
                }
            }
        }
    }
    // ---- per-warp state to shared memory, once the ring is drained
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag[0]) {
        // a wait gave up: let every copy still in flight land before the ring is reused
        const int issued = abort_flag[1];
        for (int i = max(0, issued - kStages); i < issued; ++i) mbar_wait(&full[i % kStages], (i / kStages) & 1);
    }
    __syncthreads();
    {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if constexpr (!WIDE) {
#pragma unroll
            for (int mt = 0; mt < Gm::MT; ++mt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][e] += __shfl_xor_sync(0xffffffffu, o[mt][e], 2);
            }
        }
        const int hb = WIDE ? 2 * t : 2 * (t & 1);
        const float es = eref ? __uint_as_float(eref << 23) : 0.0f;   // 2^(eref - 127)
        float* so = st_o + warp * 8 * D;
        if (WIDE || t < 2) {
#pragma unroll
            for (int mt = 0; mt < Gm::MT; ++mt) {
                const int dlo = 8 * g + mt;
                const int dhi = (D == 128) ? 64 + 8 * g + mt : 8 * g + 4 + mt;
                so[hb * D + dlo] = o[mt][0] * es;
                so[(hb + 1) * D + dlo] = o[mt][1] * es;
                so[hb * D + dhi] = o[mt][2] * es;
                so[(hb + 1) * D + dhi] = o[mt][3] * es;
            }
            if (g == 0) {
                st_m[warp * 8 + hb] = m0;
                st_m[warp * 8 + hb + 1] = m1;
                st_l[warp * 8 + hb] = l0;
                st_l[warp * 8 + hb + 1] = l1;
            }
        }
    }
    __syncthreads();

    // ---- merge the warps of each kv head, then finish (single segment) or store the partial;
    // four vectors per warp at a time
    const int wph = kConsumerWarps / H;
    for (int v0 = warp; v0 < Hq; v0 += 4 * kConsumerWarps) {
        float acc[4][D / 32], inv_l[4];
        int64_t ooff[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int v = v0 + k * kConsumerWarps;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) acc[k][j] = 0.0f;
            inv_l[k] = 0.0f;
            ooff[k] = -1;
            if (v >= Hq) continue;
            const int h = v / G, col = v % G;
            float M = kNegBig;
            for (int s = 0; s < wph; ++s) M = fmaxf(M, st_m[(h + s * H) * 8 + col]);
            float Lsum = 0.0f;
            for (int s = 0; s < wph; ++s) {
                const int w = h + s * H;
                const float wt = fast_exp2(st_m[w * 8 + col] - M);
                Lsum += wt * st_l[w * 8 + col];
#pragma unroll
                for (int j = 0; j < D / 32; ++j) acc[k][j] += wt * st_o[(w * 8 + col) * D + lane + 32 * j];
            }
            if (nseg == 1) {
                inv_l[k] = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
                ooff[k] = ((int64_t)q0 * Hq + v) * D;
            } else {
                const int64_t pi = ((int64_t)seq * Hq + v) * p.nseg_max + seg;
#pragma unroll
                for (int j = 0; j < D / 32; ++j) p.ws_o[pi * D + lane + 32 * j] = acc[k][j];
                if (lane == 0) {
                    p.ws_ml[pi * 2] = M;
                    p.ws_ml[pi * 2 + 1] = Lsum;
                }
            }
        }
        if (nseg == 1) unrotate_store_batch<D, OT, 4>(acc, inv_l, sgn, p.c, p.out, ooff);
    }
}

// Combine the per-segment partials of every decode sequence that spans more than one segment.
template <int D, typename OT>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttnParams p) {
    __shared__ float sgn[D];
    for (int i = threadIdx.x; i < D; i += blockDim.x) sgn[i] = p.signs[i] < 0.0f ? -1.0f : 1.0f;
    __syncthreads();
    const int seq = blockIdx.x;
    const int v = blockIdx.y * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (v >= p.Hq) return;
    const int q0 = __ldg(p.qsl + seq);
    if (__ldg(p.qsl + seq + 1) - q0 != 1) return;
    if (q0 < 0 || (int64_t)q0 >= p.num_q_tokens) return;
    const int L = min(__ldg(p.seq_lens + seq), min(p.max_blocks_per_seq * kBlockSize, p.nseg_max * p.seg_len));
    const int nseg = (L + p.seg_len - 1) / p.seg_len;
    if (nseg <= 1) return;
    const int64_t base = ((int64_t)seq * p.Hq + v) * p.nseg_max;
    // lanes run over segments: global max, per-segment weights and the weighted sum of l
    float M = kNegBig;
    for (int s0 = 0; s0 < nseg; s0 += 32) {
        const int s = s0 + lane;
        if (s < nseg) M = fmaxf(M, p.ws_ml[(base + s) * 2]);
    }
    M = warp_max(M);
    float Lpart = 0.0f;
    float acc[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) acc[k] = 0.0f;
    for (int s0 = 0; s0 < nseg; s0 += 32) {
        const int s = s0 + lane;
        const float wt = s < nseg ? fast_exp2(p.ws_ml[(base + s) * 2] - M) : 0.0f;
        if (s < nseg) Lpart += wt * p.ws_ml[(base + s) * 2 + 1];
        const int n = min(32, nseg - s0);
        // partial outputs of this group of segments: independent loads, four segments at a time
        for (int j0 = 0; j0 < n; j0 += 4) {
            float o4[4][D / 32], w4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u;
                w4[u] = __shfl_sync(0xffffffffu, wt, j & 31);
#pragma unroll
                for (int k = 0; k < D / 32; ++k)
                    o4[u][k] = j < n ? p.ws_o[(base + s0 + j) * D + lane + 32 * k] : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
#pragma unroll
                for (int k = 0; k < D / 32; ++k) acc[k] += w4[u] * o4[u][k];
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lpart += __shfl_xor_sync(0xffffffffu, Lpart, o);
    const float Lsum = Lpart;
    unrotate_store<D, OT>(acc, Lsum > 0.0f ? 1.0f / Lsum : 0.0f, sgn, p.c, p.out, ((int64_t)q0 * p.Hq + v) * D);
}

template <int D, typename QT, typename OT>
cudaError_t launch_decode_t(const AttnParams& p, cudaStream_t stream) {
    const DecodeSmem lay = decode_smem_layout<D>(p.H, p.Hq);
    const bool wide = p.G == 8;
    auto kern = wide ? decode_kernel<D, true, QT, OT> : decode_kernel<D, false, QT, OT>;
    cudaError_t err = wide ? opt_in_smem<decode_kernel<D, true, QT, OT>>(lay.total)
                           : opt_in_smem<decode_kernel<D, false, QT, OT>>(lay.total);
    if (err != cudaSuccess) return err;
    dim3 grid(p.nseg_max, p.num_seqs);
    kern<<<grid, kDecodeThreads, lay.total, stream>>>(p);
    return cudaGetLastError();
}

template <int D, typename OT>
cudaError_t launch_combine_t(const AttnParams& p, cudaStream_t stream) {
    dim3 grid(p.num_seqs, (p.Hq + 7) / 8);
    combine_kernel<D, OT><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D, typename QT>
cudaError_t decode_by_out(const AttnParams& p, DType out_dt, cudaStream_t s) {
    switch (out_dt) {
        case DType::F16: return launch_decode_t<D, QT, __half>(p, s);
        case DType::BF16: return launch_decode_t<D, QT, __nv_bfloat16>(p, s);
        default: return launch_decode_t<D, QT, float>(p, s);
    }
}

template <int D>
cudaError_t combine_by_out(const AttnParams& p, DType out_dt, cudaStream_t s) {
    switch (out_dt) {
        case DType::F16: return launch_combine_t<D, __half>(p, s);
        case DType::BF16: return launch_combine_t<D, __nv_bfloat16>(p, s);
        default: return launch_combine_t<D, float>(p, s);
    }
}

}  // namespace

cudaError_t launch_decode(const AttnParams& p, int head_size, DType q_dt, DType out_dt, cudaStream_t stream) {
    if (head_size == 128)
        return q_dt == DType::BF16 ? decode_by_out<128, __nv_bfloat16>(p, out_dt, stream)
                                   : decode_by_out<128, __half>(p, out_dt, stream);
    return q_dt == DType::BF16 ? decode_by_out<64, __nv_bfloat16>(p, out_dt, stream)
                               : decode_by_out<64, __half>(p, out_dt, stream);
}

cudaError_t launch_combine(const AttnParams& p, int head_size, DType out_dt, cudaStream_t stream) {
    return head_size == 128 ? combine_by_out<128>(p, out_dt, stream) : combine_by_out<64>(p, out_dt, stream);
}


}  // namespace kvi4
