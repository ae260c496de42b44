// Chunked-prefill attention over the INT4 cache: sequences with more than one query token
// ("[Feature] Triton INT4 / INT2 per-token-head KV cache quantization", packed read path;
// causal queries at positions seq_len - q_len + t as in the unified-attention call of
// test_triton_unified_attention_per_token_head_scale).
//
// One CTA per (query tile, kv head, sequence): 128 rows = (128 / G) query tokens x G query heads
// of that kv head, 16 rows per warp.  Each warp walks the key blocks its rows can see (causal),
// builds fp16 fragments of K - zp and V - zp directly from the packed bytes (read through L1, the
// next block prefetched into registers), and runs
//   S = Q' (K - zp)^T      mma.sync m16n8k16, Q' = rotated, power-of-two-prescaled queries as
//                          fp16 high + low halves (two mma per step)
//   online softmax with the per-key scale s'_K and the causal mask
//   O += P_w (V - zp)      P_w = p * s'_V * 2^-E as fp16 high + low halves, straight from S's
//                          accumulator registers
// and un-rotates its rows at the end.  The fragment layouts are the decode kernel's with the
// operand roles swapped (queries on the M side, keys on N).
#include "attn_common.cuh"

namespace kvi4 {
namespace {

constexpr int kPrefillWarps = 8;
constexpr int kPrefillThreads = kPrefillWarps * 32;
constexpr int kRows = kPrefillWarps * 16;

template <int D>
struct BlockWords {
    uint32_t k0[Geo<D>::KWPT], k1[Geo<D>::KWPT];   // code words of key rows tau(g), tau(g+8)
    uint32_t ks0, ks1;                             // their scale words
    uint32_t kc[4];                                // K scale words of tokens t, t+4, t+8, t+12
    uint32_t vw[4][D == 128 ? 2 : 1];              // V code words (g[, g+8]) of those tokens
    uint32_t vs[4];                                // their V scale words
    int ok;
};

template <int D>
__device__ __forceinline__ void load_block(BlockWords<D>& b, const uint8_t* cache, int64_t blk, int H, int h, int g,
                                           int t) {
    using Gm = Geo<D>;
    const int64_t plane_stride = (int64_t)kBlockSize * H * Gm::RB;
    const uint8_t* kp = cache + blk * 2 * plane_stride + (int64_t)h * Gm::RB;
    const uint8_t* vp = kp + plane_stride;
    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(kp + (int64_t)block_token(g) * H * Gm::RB);
    const uint32_t* r1 = reinterpret_cast<const uint32_t*>(kp + (int64_t)block_token(g + 8) * H * Gm::RB);
#pragma unroll
    for (int j = 0; j < Gm::KWPT; ++j) {
        b.k0[j] = __ldg(r0 + t + 4 * j);
        b.k1[j] = __ldg(r1 + t + 4 * j);
    }
    b.ks0 = __ldg(r0 + Gm::KW);
    b.ks1 = __ldg(r1 + Gm::KW);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int tok = t + 4 * c;
        const uint32_t* kr = reinterpret_cast<const uint32_t*>(kp + (int64_t)tok * H * Gm::RB);
        const uint32_t* vr = reinterpret_cast<const uint32_t*>(vp + (int64_t)tok * H * Gm::RB);
        b.kc[c] = __ldg(kr + Gm::KW);
        b.vs[c] = __ldg(vr + Gm::KW);
        b.vw[c][0] = __ldg(vr + g);
        if constexpr (D == 128) b.vw[c][1] = __ldg(vr + g + 8);
    }
}

template <int D, typename QT, typename OT>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_kernel(const __grid_constant__ AttnParams p) {
    using Gm = Geo<D>;
    constexpr int NT = 2 * Gm::MT;   // 8-wide output tiles over the head dimension
    extern __shared__ __align__(128) uint8_t smem[];
    const int qtile = blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
    const int q0 = __ldg(p.qsl + seq);
    const int qlen = __ldg(p.qsl + seq + 1) - q0;
    if (qlen <= 1) return;   // decode sequences (and empty ones) are not this kernel's
    if (q0 < 0 || (int64_t)q0 + qlen > p.num_q_tokens || qlen > p.max_query_len) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) count_status(p.status, 2);
        if (q0 < 0 || (int64_t)q0 + qlen > p.num_q_tokens) return;
    }
    const int G = p.G, Hq = p.Hq, H = p.H;
    const int BQ = kRows / G;
    const int qt0 = qtile * BQ;
    if (qt0 >= qlen) return;
    int L = __ldg(p.seq_lens + seq);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (L > p.max_blocks_per_seq * kBlockSize || qlen > L) {
        if (qtile == 0 && h == 0 && threadIdx.x == 0) count_status(p.status, 2);
        L = min(L, p.max_blocks_per_seq * kBlockSize);
    }
    const int pos0 = L - qlen;   // position of query token 0

    float* ostage = reinterpret_cast<float*>(smem);                         // [128][D] fp32 (epilogue)
    __half* qh = reinterpret_cast<__half*>(smem);                           // [128][D] fp16 (prologue)
    __half* ql = qh + kRows * D;                                            // [128][D] fp16 (prologue)
    uint4* qlf = reinterpret_cast<uint4*>(smem + (size_t)kRows * D * 4);    // [warps][KSTEPS][32] low-half A fragments
    float* alpha = reinterpret_cast<float*>(qlf + kPrefillWarps * Gm::KSTEPS * 32);   // [128]
    float* sgn = alpha + kRows;                                             // [D]
    for (int i = threadIdx.x; i < D; i += blockDim.x) sgn[i] = p.signs[i] < 0.0f ? -1.0f : 1.0f;
    __syncthreads();

    // ---- rotate this warp's 16 query rows
    for (int r = 0; r < 16; ++r) {
        const int R = warp * 16 + r;
        const int qt = qt0 + R / G, gg = R % G;
        if (qt < qlen) {
            const float a = rotate_query<D, QT>(p.q, ((int64_t)(q0 + qt) * Hq + h * G + gg) * D, sgn, qh + R * D,
                                                ql + R * D, p.c, p.softmax_scale);
            if (lane == 0) alpha[R] = a;
        } else {
            for (int k = lane; k < D; k += 32) qh[R * D + k] = ql[R * D + k] = __float2half(0.0f);
            if (lane == 0) alpha[R] = 0.0f;
        }
    }
    __syncwarp();
    const int g = lane >> 2, t = lane & 3;
    const int Rg = warp * 16 + g, Rg8 = Rg + 8;
    uint32_t qa[Gm::KSTEPS][4];
#pragma unroll
    for (int j = 0; j < Gm::KWPT; ++j) {
        const int W = t + 4 * j;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int d0 = 8 * W + 2 * hh;
            __half2 a0 = __halves2half2(qh[Rg * D + d0], qh[Rg * D + d0 + 4]);
            __half2 a1 = __halves2half2(qh[Rg8 * D + d0], qh[Rg8 * D + d0 + 4]);
            __half2 a2 = __halves2half2(qh[Rg * D + d0 + 1], qh[Rg * D + d0 + 5]);
            __half2 a3 = __halves2half2(qh[Rg8 * D + d0 + 1], qh[Rg8 * D + d0 + 5]);
            qa[2 * j + hh][0] = *reinterpret_cast<uint32_t*>(&a0);
            qa[2 * j + hh][1] = *reinterpret_cast<uint32_t*>(&a1);
            qa[2 * j + hh][2] = *reinterpret_cast<uint32_t*>(&a2);
            qa[2 * j + hh][3] = *reinterpret_cast<uint32_t*>(&a3);
            // the low halves go to a fragment-ordered area read once per k-step in the main loop
            __half2 l0 = __halves2half2(ql[Rg * D + d0], ql[Rg * D + d0 + 4]);
            __half2 l1 = __halves2half2(ql[Rg8 * D + d0], ql[Rg8 * D + d0 + 4]);
            __half2 l2 = __halves2half2(ql[Rg * D + d0 + 1], ql[Rg * D + d0 + 5]);
            __half2 l3 = __halves2half2(ql[Rg8 * D + d0 + 1], ql[Rg8 * D + d0 + 5]);
            qlf[(warp * Gm::KSTEPS + 2 * j + hh) * 32 + lane] =
                make_uint4(*reinterpret_cast<uint32_t*>(&l0), *reinterpret_cast<uint32_t*>(&l1),
                           *reinterpret_cast<uint32_t*>(&l2), *reinterpret_cast<uint32_t*>(&l3));
        }
    }
    const uint4* my_qlf = qlf + warp * Gm::KSTEPS * 32 + lane;
    const float al_g = alpha[Rg], al_g8 = alpha[Rg8];
    const int qt_g = qt0 + Rg / G, qt_g8 = qt0 + Rg8 / G;
    const int lim_g = qt_g < qlen ? pos0 + qt_g : -1;     // last visible key of each row
    const int lim_g8 = qt_g8 < qlen ? pos0 + qt_g8 : -1;
    __syncthreads();   // qh is dead from here on; the region becomes the output stage

    // keys this warp needs: up to the largest visible position among its rows
    const int last_qt = min(qlen - 1, qt0 + (warp * 16 + 15) / G);
    const int warp_lim = (qt0 + (warp * 16) / G < qlen) ? min(pos0 + last_qt, L - 1) : -1;
    const int nkb = warp_lim >= 0 ? warp_lim / kBlockSize + 1 : 0;

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_g = kNegBig, m_g8 = kNegBig, l_g = 0.0f, l_g8 = 0.0f;
    uint32_t eref = 0;
    const int32_t* table = p.block_tables + (int64_t)seq * p.max_blocks_per_seq;

    BlockWords<D> cur, nxt;
    auto fetch = [&](BlockWords<D>& b, int kb) {
        const int blk = __ldg(table + kb);
        b.ok = blk >= 0 && (int64_t)blk < p.num_blocks;
        if (b.ok) load_block<D>(b, p.cache, blk, H, h, g, t);
        else if (lane == 0) count_status(p.status, 1);
    };
    if (nkb > 0) fetch(cur, 0);
    for (int kb = 0; kb < nkb; ++kb) {
        if (kb + 1 < nkb) fetch(nxt, kb + 1);
        if (cur.ok) {
            // ---- S = Q' (K - zp)^T over 16 keys (two 8-key tiles)
            float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                const uint32_t z0l = zp_lo_half(cur.ks0 & 15u), z0h = zp_hi_half(cur.ks0 & 15u);
                const uint32_t z1l = zp_lo_half(cur.ks1 & 15u), z1h = zp_hi_half(cur.ks1 & 15u);
                const uint32_t zl0 = z0l | (z0l << 16), zh0 = z0h | (z0h << 16);
                const uint32_t zl1 = z1l | (z1l << 16), zh1 = z1h | (z1h << 16);
#pragma unroll
                for (int j = 0; j < Gm::KWPT; ++j) {
                    uint32_t b0[4], b1[4];
                    unpack_word(cur.k0[j], zl0, zh0, b0);
                    unpack_word(cur.k1[j], zl1, zh1, b1);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t* a = qa[2 * j + hh];
                        const uint4 al = my_qlf[(2 * j + hh) * 32];
                        mma_f16_16816(s[0], a[0], a[1], a[2], a[3], b0[2 * hh], b0[2 * hh + 1]);
                        mma_f16_16816(s[1], a[0], a[1], a[2], a[3], b1[2 * hh], b1[2 * hh + 1]);
                        mma_f16_16816(s[0], al.x, al.y, al.z, al.w, b0[2 * hh], b0[2 * hh + 1]);
                        mma_f16_16816(s[1], al.x, al.y, al.z, al.w, b1[2 * hh], b1[2 * hh + 1]);
                    }
                }
            }
            // ---- logits, causal mask, online softmax over rows g and g+8
            const int kbase = kb * kBlockSize;
            float x[2][4];
            float sk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) sk[c] = __uint_as_float(cur.kc[c] & 0xFFFFFFF0u);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int c = 2 * nt + e;            // key token t + 4c
                    const int key = kbase + t + 4 * c;
                    x[nt][e] = key <= lim_g ? s[nt][e] * sk[c] * al_g : -INFINITY;
                    x[nt][2 + e] = key <= lim_g8 ? s[nt][2 + e] * sk[c] * al_g8 : -INFINITY;
                }
            }
            float bm_g = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            float bm_g8 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                bm_g = fmaxf(bm_g, __shfl_xor_sync(0xffffffffu, bm_g, off));
                bm_g8 = fmaxf(bm_g8, __shfl_xor_sync(0xffffffffu, bm_g8, off));
            }
            const float mn_g = fmaxf(m_g, bm_g), mn_g8 = fmaxf(m_g8, bm_g8);
            const float r_g = fast_exp2(m_g - mn_g), r_g8 = fast_exp2(m_g8 - mn_g8);
            m_g = mn_g;
            m_g8 = mn_g8;
            float pr[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                pr[nt][0] = fast_exp2(x[nt][0] - mn_g);
                pr[nt][1] = fast_exp2(x[nt][1] - mn_g);
                pr[nt][2] = fast_exp2(x[nt][2] - mn_g8);
                pr[nt][3] = fast_exp2(x[nt][3] - mn_g8);
            }
            l_g = l_g * r_g + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
            l_g8 = l_g8 * r_g8 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
            // ---- V scale exponent reference (keys a row cannot see contribute nothing)
            uint32_t emax = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int key = kbase + t + 4 * c;
                if (key <= max(lim_g, lim_g8)) emax = max(emax, (cur.vs[c] >> 23) & 0xFFu);
            }
            const uint32_t eblk = __reduce_max_sync(0xffffffffu, emax);
            float escale = 1.0f;
            if (eblk > eref) {
                escale = (eref == 0u || eblk - eref > 126u) ? 0.0f : __uint_as_float((127u + eref - eblk) << 23);
                eref = eblk;
            }
            const float f_g = r_g * escale, f_g8 = r_g8 * escale;
            if (__any_sync(0xffffffffu, f_g != 1.0f || f_g8 != 1.0f)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    o[nt][0] *= f_g;
                    o[nt][1] *= f_g;
                    o[nt][2] *= f_g8;
                    o[nt][3] *= f_g8;
                }
            }
            const float wsc = __uint_as_float((254u - eref) << 23);
            // keys no row of this thread can see may sit in never-written slots: keep their
            // (possibly NaN) scale words out of the products
            float sv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                sv[c] = (kbase + t + 4 * c <= max(lim_g, lim_g8)) ? __uint_as_float(cur.vs[c] & 0xFFFFFFF0u) * wsc : 0.0f;
            // P_w as the A operand (C layout of two 8-key tiles == A layout of one 16-key tile)
            // (high and low fp16 halves, as for the queries)
            uint32_t pa0, pa1, pa2, pa3, pl0, pl1, pl2, pl3;
            split_f16x2(pr[0][0] * sv[0], pr[0][1] * sv[1], pa0, pl0);
            split_f16x2(pr[0][2] * sv[0], pr[0][3] * sv[1], pa1, pl1);
            split_f16x2(pr[1][0] * sv[2], pr[1][1] * sv[3], pa2, pl2);
            split_f16x2(pr[1][2] * sv[2], pr[1][3] * sv[3], pa3, pl3);
            // ---- O += P_w (V - zp)
            const uint32_t zl01 = zp_lo_half(cur.vs[0] & 15u) | (zp_lo_half(cur.vs[1] & 15u) << 16);
            const uint32_t zh01 = zp_hi_half(cur.vs[0] & 15u) | (zp_hi_half(cur.vs[1] & 15u) << 16);
            const uint32_t zl23 = zp_lo_half(cur.vs[2] & 15u) | (zp_lo_half(cur.vs[3] & 15u) << 16);
            const uint32_t zh23 = zp_hi_half(cur.vs[2] & 15u) | (zp_hi_half(cur.vs[3] & 15u) << 16);
            if constexpr (D == 128) {
                uint32_t ua[8], ub[8], uc[8], ud[8];
                unpack_word_pair(cur.vw[0][0], cur.vw[1][0], zl01, zh01, ua);   // d = 8g' + i, keys t, t+4
                unpack_word_pair(cur.vw[0][1], cur.vw[1][1], zl01, zh01, ub);   // d = 64 + 8g' + i
                unpack_word_pair(cur.vw[2][0], cur.vw[3][0], zl23, zh23, uc);   // keys t+8, t+12
                unpack_word_pair(cur.vw[2][1], cur.vw[3][1], zl23, zh23, ud);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    mma_f16_16816(o[i], pa0, pa1, pa2, pa3, ua[i], uc[i]);
                    mma_f16_16816(o[8 + i], pa0, pa1, pa2, pa3, ub[i], ud[i]);
                    mma_f16_16816(o[i], pl0, pl1, pl2, pl3, ua[i], uc[i]);
                    mma_f16_16816(o[8 + i], pl0, pl1, pl2, pl3, ub[i], ud[i]);
                }
            } else {
                uint32_t ua[8], uc[8];
                unpack_word_pair(cur.vw[0][0], cur.vw[1][0], zl01, zh01, ua);
                unpack_word_pair(cur.vw[2][0], cur.vw[3][0], zl23, zh23, uc);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    mma_f16_16816(o[i], pa0, pa1, pa2, pa3, ua[i], uc[i]);
                    mma_f16_16816(o[4 + i], pa0, pa1, pa2, pa3, ua[4 + i], uc[4 + i]);
                    mma_f16_16816(o[i], pl0, pl1, pl2, pl3, ua[i], uc[i]);
                    mma_f16_16816(o[4 + i], pl0, pl1, pl2, pl3, ua[4 + i], uc[4 + i]);
                }
            }
        }
        if (kb + 1 < nkb) cur = nxt;
    }

    // ---- epilogue: normalise, stage rows, un-rotate and store
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l_g += __shfl_xor_sync(0xffffffffu, l_g, off);
        l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, off);
    }
    const float es = eref ? __uint_as_float(eref << 23) : 0.0f;
    const float sc_g = l_g > 0.0f ? es / l_g : 0.0f, sc_g8 = l_g8 > 0.0f ? es / l_g8 : 0.0f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        // tile nt covers d = base + 8 n' for n' = 0..7 (base = mt or 64 + mt, D=64: mt or 4 + mt)
        const int mt = nt % Gm::MT, half = nt / Gm::MT;
        const int base = (D == 128) ? (half ? 64 + mt : mt) : (half ? 4 + mt : mt);
        const int d0 = base + 8 * (2 * t), d1 = base + 8 * (2 * t + 1);
        ostage[Rg * D + d0] = o[nt][0] * sc_g;
        ostage[Rg * D + d1] = o[nt][1] * sc_g;
        ostage[Rg8 * D + d0] = o[nt][2] * sc_g8;
        ostage[Rg8 * D + d1] = o[nt][3] * sc_g8;
    }
    __syncwarp();
    for (int r = 0; r < 16; ++r) {
        const int R = warp * 16 + r;
        const int qt = qt0 + R / G, gg = R % G;
        if (qt >= qlen) continue;
        float xv[D / 32];
#pragma unroll
        for (int k = 0; k < D / 32; ++k) xv[k] = ostage[R * D + lane + 32 * k];
        unrotate_store<D, OT>(xv, 1.0f, sgn, p.c, p.out, ((int64_t)(q0 + qt) * Hq + h * G + gg) * D);
    }
}

template <int D, typename QT, typename OT>
cudaError_t launch_prefill_t(const AttnParams& p, int max_query_len, cudaStream_t stream) {
    const size_t smem = (size_t)kRows * D * 4 + (size_t)kPrefillWarps * Geo<D>::KSTEPS * 32 * 16 + kRows * 4 + D * 4;
    auto kern = prefill_kernel<D, QT, OT>;
    cudaError_t err = opt_in_smem<prefill_kernel<D, QT, OT>>(smem);
    if (err != cudaSuccess) return err;
    const int BQ = kRows / p.G;
    dim3 grid((max_query_len + BQ - 1) / BQ, p.H, p.num_seqs);
    kern<<<grid, kPrefillThreads, smem, stream>>>(p);
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
