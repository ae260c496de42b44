// Chunked-prefill attention over the INT4 cache: sequences with more than one query token
// ("[Feature] Triton INT4 / INT2 per-token-head KV cache quantization", packed read path;
// causal queries at positions seq_len - q_len + t as in the unified-attention call of
// test_triton_unified_attention_per_token_head_scale).
//
// One CTA per (query tile, kv head, sequence): 128 rows = (128 / G) query tokens x G query heads
// of that kv head, 16 rows per warp.  The CTA walks the key blocks its rows can see (causal) once:
// all 256 threads dequantise a 16-token block into fp16 tiles K - zp and V - zp in shared memory
// (exact integers, natural dimension order, rows padded so that ldmatrix is bank-conflict free),
// double-buffered with one barrier per block, the codes of the block after next already in
// flight.  Each warp then runs, for its 16 rows,
//   S = Q' (K - zp)^T      mma.sync m16n8k16, B fragments by ldmatrix, Q' = rotated,
//                          power-of-two-prescaled queries as fp16 high + low halves
//   online softmax with the per-key scale s'_K and the causal mask
//   O += P_w (V - zp)      P_w = p * s'_V * 2^-E as fp16 high + low halves, straight from S's
//                          accumulator registers; V fragments by ldmatrix.trans
// and un-rotates its rows at the end.
#include "attn_common.cuh"

namespace kvi4 {
namespace {

constexpr int kPrefillWarps = 8;
constexpr int kPrefillThreads = kPrefillWarps * 32;
constexpr int kRows = kPrefillWarps * 16;

template <int D>
struct PrefillSmem {
    static constexpr int kTileStride = D + 8;                                 // halves per tile row
    static constexpr int kTileHalves = kBlockSize * kTileStride;              // one 16-token tile
    static constexpr size_t kStage = (size_t)kRows * D * 4;                   // q halves / output rows
    static constexpr size_t kQlf = (size_t)kPrefillWarps * (D / 16) * 32 * 16;
    static constexpr size_t kTiles = 2 * 2 * kTileHalves * 2;                 // [buf][plane] fp16 tiles
    static constexpr size_t kScales = 2 * 2 * kBlockSize * 4 + 16;            // [buf][plane] scale words + flags
    static constexpr size_t kBytes = kStage + kQlf + kTiles + kScales + kRows * 4 + D * 4;
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(row)));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(row)));
}

__device__ __forceinline__ uint32_t pack_h2(__half a, __half b) {
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

template <int D, typename QT, typename OT>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_kernel(const __grid_constant__ AttnParams p) {
    using Gm = Geo<D>;
    using Sm = PrefillSmem<D>;
    constexpr int NT = D / 8;          // 8-wide output tiles over the head dimension
    constexpr int KS = D / 16;         // 16-deep k-steps over the head dimension
    constexpr int TS = Sm::kTileStride;
    constexpr int WPP = kBlockSize * Gm::KW;   // code words of one plane of one block (one head)
    extern __shared__ __align__(128) uint8_t smem[];
    // blockIdx.x runs over (query tile, kv head) with the last (causally heaviest) tiles first, so
    // the light tiles fill the end of the schedule; blockIdx.z is the sequence.
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
    const int BQ = kRows / G;
    const int qt0 = qtile * BQ;
    if (qt0 >= qlen) return;
    int L = __ldg(p.seq_lens + seq);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the same context cap as the decode path (max_seq_len and the block table), counted as bad metadata
    if (L > p.len_cap || qlen > L) {
        if (qtile == 0 && h == 0 && threadIdx.x == 0) count_status(p.status, 2);
        L = min(L, p.len_cap);
    }
    const int pos0 = L - qlen;   // position of query token 0

    float* ostage = reinterpret_cast<float*>(smem);                               // [128][D] fp32 (epilogue)
    __half* qh = reinterpret_cast<__half*>(smem);                                 // [128][D] fp16 (prologue)
    __half* ql = qh + kRows * D;                                                  // [128][D] fp16 (prologue)
    uint4* qlf = reinterpret_cast<uint4*>(smem + Sm::kStage);                     // [warps][KS][32] low-half A fragments
    __half* tiles = reinterpret_cast<__half*>(smem + Sm::kStage + Sm::kQlf);      // [buf][plane][16][TS]
    uint32_t* scalew = reinterpret_cast<uint32_t*>(smem + Sm::kStage + Sm::kQlf + Sm::kTiles);   // [buf][plane][16]
    int* tile_ok = reinterpret_cast<int*>(scalew + 2 * 2 * kBlockSize);          // [buf]
    float* alpha = reinterpret_cast<float*>(smem + Sm::kStage + Sm::kQlf + Sm::kTiles + Sm::kScales);   // [128]
    float* sgn = alpha + kRows;                                                   // [D]
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
    // A fragments of the rows (natural dimension order): a0 = (row g, k 2t..2t+1), a1 = (g+8, ..),
    // a2 = (g, k 2t+8..2t+9), a3 = (g+8, ..) of each 16-deep k-step
    const int g = lane >> 2, t = lane & 3;
    const int Rg = warp * 16 + g, Rg8 = Rg + 8;
    uint32_t qa[KS][4];
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
        const int d0 = 16 * kk + 2 * t;
        qa[kk][0] = pack_h2(qh[Rg * D + d0], qh[Rg * D + d0 + 1]);
        qa[kk][1] = pack_h2(qh[Rg8 * D + d0], qh[Rg8 * D + d0 + 1]);
        qa[kk][2] = pack_h2(qh[Rg * D + d0 + 8], qh[Rg * D + d0 + 9]);
        qa[kk][3] = pack_h2(qh[Rg8 * D + d0 + 8], qh[Rg8 * D + d0 + 9]);
        // the low halves go to a fragment-ordered area read once per k-step in the main loop
        qlf[(warp * KS + kk) * 32 + lane] =
            make_uint4(pack_h2(ql[Rg * D + d0], ql[Rg * D + d0 + 1]), pack_h2(ql[Rg8 * D + d0], ql[Rg8 * D + d0 + 1]),
                       pack_h2(ql[Rg * D + d0 + 8], ql[Rg * D + d0 + 9]),
                       pack_h2(ql[Rg8 * D + d0 + 8], ql[Rg8 * D + d0 + 9]));
    }
    const uint4* my_qlf = qlf + warp * KS * 32 + lane;
    const float al_g = alpha[Rg], al_g8 = alpha[Rg8];
    const int qt_g = qt0 + Rg / G, qt_g8 = qt0 + Rg8 / G;
    const int lim_g = qt_g < qlen ? pos0 + qt_g : -1;     // last visible key of each row
    const int lim_g8 = qt_g8 < qlen ? pos0 + qt_g8 : -1;
    const int lim_w = max(lim_g, lim_g8);

    // keys this warp needs (up to the largest visible position among its rows) and the CTA
    const int last_qt = min(qlen - 1, qt0 + (warp * 16 + 15) / G);
    const int warp_lim = (qt0 + (warp * 16) / G < qlen) ? min(pos0 + last_qt, L - 1) : -1;
    const int nkb = warp_lim >= 0 ? warp_lim / kBlockSize + 1 : 0;
    const int cta_lim = min(pos0 + min(qlen - 1, qt0 + (kRows - 1) / G), L - 1);
    const int nkb_cta = cta_lim >= 0 ? cta_lim / kBlockSize + 1 : 0;

    // ---- cooperative dequantisation: codes of block kb in flight in registers, then into tiles
    const int32_t* table = p.block_tables + (int64_t)seq * p.max_blocks_per_seq;
    constexpr int kWordsPerThread = (2 * WPP + kPrefillThreads - 1) / kPrefillThreads;
    uint32_t cw[kWordsPerThread], sw[kWordsPerThread];
    int cur_ok = 0;
    auto fetch = [&](int kb) {   // this thread's code and scale words of block kb
        const int blk = __ldg(table + kb);
        cur_ok = blk >= 0 && (int64_t)blk < p.num_blocks;
#pragma unroll
        for (int u = 0; u < kWordsPerThread; ++u) {
            const int i = threadIdx.x + u * kPrefillThreads;
            cw[u] = 0u;
            sw[u] = 0u;
            if (i < 2 * WPP && cur_ok) {
                const int plane = i / WPP, tok = (i / Gm::KW) % kBlockSize, w = i % Gm::KW;
                const uint32_t* row = reinterpret_cast<const uint32_t*>(
                    p.cache + (((int64_t)blk * 2 + plane) * kBlockSize + tok) * H * Gm::RB + (int64_t)h * Gm::RB);
                cw[u] = __ldg(row + w);
                sw[u] = __ldg(row + Gm::KW);
            }
        }
    };
    auto dequant = [&](int buf) {   // the fetched words -> fp16 (code - zp) in natural order
#pragma unroll
        for (int u = 0; u < kWordsPerThread; ++u) {
            const int i = threadIdx.x + u * kPrefillThreads;
            if (i < 2 * WPP) {
                const int plane = i / WPP, tok = (i / Gm::KW) % kBlockSize, w = i % Gm::KW;
                const uint32_t zp = sw[u] & 15u;
                const uint32_t zl = zp_lo_half(zp) * 0x10001u, zh = zp_hi_half(zp) * 0x10001u;
                uint32_t o[4];
                unpack_word(cw[u], zl, zh, o);   // (e0,e4) (e1,e5) (e2,e6) (e3,e7)
                uint4 v;
                v.x = prmt(o[0], o[1], 0x5410u);   // (e0, e1)
                v.y = prmt(o[2], o[3], 0x5410u);   // (e2, e3)
                v.z = prmt(o[0], o[1], 0x7632u);   // (e4, e5)
                v.w = prmt(o[2], o[3], 0x7632u);   // (e6, e7)
                *reinterpret_cast<uint4*>(tiles + ((buf * 2 + plane) * kBlockSize + tok) * TS + 8 * w) = v;
                if (w == 0) scalew[(buf * 2 + plane) * kBlockSize + tok] = sw[u];
            }
        }
        if (threadIdx.x == 0) {
            tile_ok[buf] = cur_ok;
            if (!cur_ok) count_status(p.status, 1);
        }
    };

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_g = kNegBig, m_g8 = kNegBig, l_g = 0.0f, l_g8 = 0.0f;
    uint32_t eref = 0;

    __syncthreads();   // the q halves are consumed; the tiles area was never part of them
    if (nkb_cta > 0) {
        fetch(0);
        dequant(0);
        if (nkb_cta > 1) fetch(1);
    }
    __syncthreads();
    // ldmatrix row addresses: lane l serves row l % 8 of matrix l / 8
    const int lm = lane >> 3, lr = lane & 7;
    for (int kb = 0; kb < nkb_cta; ++kb) {
        const int buf = kb & 1;
        if (kb < nkb && tile_ok[buf]) {
            const __half* kt = tiles + (buf * 2 + 0) * kBlockSize * TS;
            const __half* vt = tiles + (buf * 2 + 1) * kBlockSize * TS;
            const uint32_t* kscale = scalew + (buf * 2 + 0) * kBlockSize;
            const uint32_t* vscale = scalew + (buf * 2 + 1) * kBlockSize;
            // ---- S = Q' (K - zp)^T over 16 keys (two 8-key tiles); matrices: keys 0-7 / 8-15 x
            // dims +0 / +8 of the k-step
            // (high and low halves accumulate separately: four independent mma chains)
            float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float sl[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const __half* krow = kt + ((lm >> 1) * 8 + lr) * TS + (lm & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t b[4];
                ldmatrix_x4(b, krow + 16 * kk);
                const uint4 al = my_qlf[kk * 32];
                mma_f16_16816(s[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b[0], b[1]);
                mma_f16_16816(s[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b[2], b[3]);
                mma_f16_16816(sl[0], al.x, al.y, al.z, al.w, b[0], b[1]);
                mma_f16_16816(sl[1], al.x, al.y, al.z, al.w, b[2], b[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] += sl[nt][e];
            }
            // ---- logits, causal mask, online softmax over rows g and g+8; s[nt][e] is key
            // 8 nt + 2t + (e & 1) of row g (e < 2) or g + 8
            const int kbase = kb * kBlockSize;
            float x[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int kt_ = 8 * nt + 2 * t + e;
                    const int key = kbase + kt_;
                    const float sk = __uint_as_float(kscale[kt_] & 0xFFFFFFF0u);
                    x[nt][e] = key <= lim_g ? s[nt][e] * sk * al_g : -INFINITY;
                    x[nt][2 + e] = key <= lim_g8 ? s[nt][2 + e] * sk * al_g8 : -INFINITY;
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
            // ---- V scale exponent reference over this lane's keys a row of the warp can see
            // (keys no row can see may sit in never-written slots: keep their words out)
            uint32_t svw[4];
            uint32_t emax = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int kt_ = 2 * t + (c & 1) + 8 * (c >> 1);   // keys 2t, 2t+1, 2t+8, 2t+9
                svw[c] = kbase + kt_ <= lim_w ? vscale[kt_] : 0u;
                emax = max(emax, (svw[c] >> 23) & 0xFFu);
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
            float sv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) sv[c] = __uint_as_float(svw[c] & 0xFFFFFFF0u) * wsc;
            // P_w as the A operand (C layout of two 8-key tiles == A layout of one 16-key tile),
            // high and low fp16 halves as for the queries
            uint32_t pa0, pa1, pa2, pa3, pl0, pl1, pl2, pl3;
            split_f16x2(pr[0][0] * sv[0], pr[0][1] * sv[1], pa0, pl0);   // row g, keys 2t, 2t+1
            split_f16x2(pr[0][2] * sv[0], pr[0][3] * sv[1], pa1, pl1);   // row g+8
            split_f16x2(pr[1][0] * sv[2], pr[1][1] * sv[3], pa2, pl2);   // row g, keys 2t+8, 2t+9
            split_f16x2(pr[1][2] * sv[2], pr[1][3] * sv[3], pa3, pl3);   // row g+8
            // ---- O += P_w (V - zp); matrices: keys 0-7 / 8-15 x dims +0 / +8, transposed
            const __half* vrow = vt + ((lm & 1) * 8 + lr) * TS + (lm >> 1) * 8;
#pragma unroll
            for (int nd = 0; nd < KS; ++nd) {
                uint32_t b[4];
                ldmatrix_x4_trans(b, vrow + 16 * nd);
                mma_f16_16816(o[2 * nd], pa0, pa1, pa2, pa3, b[0], b[1]);
                mma_f16_16816(o[2 * nd + 1], pa0, pa1, pa2, pa3, b[2], b[3]);
                mma_f16_16816(o[2 * nd], pl0, pl1, pl2, pl3, b[0], b[1]);
                mma_f16_16816(o[2 * nd + 1], pl0, pl1, pl2, pl3, b[2], b[3]);
            }
        }
        // the next block's tiles, then the codes of the block after it
        if (kb + 1 < nkb_cta) dequant(buf ^ 1);
        if (kb + 2 < nkb_cta) fetch(kb + 2);
        __syncthreads();
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
        const int d0 = 8 * nt + 2 * t;
        ostage[Rg * D + d0] = o[nt][0] * sc_g;
        ostage[Rg * D + d0 + 1] = o[nt][1] * sc_g;
        ostage[Rg8 * D + d0] = o[nt][2] * sc_g8;
        ostage[Rg8 * D + d0 + 1] = o[nt][3] * sc_g8;
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
    const size_t smem = PrefillSmem<D>::kBytes;
    auto kern = prefill_kernel<D, QT, OT>;
    cudaError_t err = opt_in_smem<prefill_kernel<D, QT, OT>>(smem);
    if (err != cudaSuccess) return err;
    const int BQ = kRows / p.G;
    dim3 grid((unsigned)(((max_query_len + BQ - 1) / BQ) * p.H), 1, p.num_seqs);
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
