/*
 * CPU oracle for the INT4 per-(token, head) KV-cache write.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct statement of what the
 * write path computes.  Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (page titles and sections):
 *  - "[Feature] Triton INT4 / INT2 per-token-head KV cache quantization" (vLLM PR #40633),
 *    description: random Hadamard pre-rotation, asymmetric 4-bit quantisation, 4-bit zero-point
 *    kept in the low 4 bits of the fp32 scale's mantissa; review note: quantise with the
 *    truncated scale so that write and read agree.
 *  - "tests/quantization/test_per_token_kv_cache.py", the INT4 reference in
 *    test_triton_unified_attention_per_token_head_scale (scale = (max - min) / 15 clamped at 1e-6,
 *    zero-point = round(-min / scale) clamped to [0, 15], codes = round(x / scale + zp) clamped to
 *    [0, 15], two codes per byte with the even element in the low nibble, scale bits & -16 | zp).
 *  - "PR #40835 report", get_kv_cache_shape: rows of head_size / 2 data bytes followed by one fp32
 *    scale, cache shape (num_blocks, 2, block_size, num_kv_heads, head_size / 2 + 4).
 *
 * Readings fixed where the pages leave a step open (each is listed in the design notes):
 *  - the rotation is y = c * H_d * (D * x), D = diag(signs), H_d the natural-order (Sylvester)
 *    Hadamard matrix, c = fp32(1 / sqrt(d)); the butterflies run at strides 1, 2, 4, ... in fp32
 *    with round-to-nearest-even after every add, then each element is multiplied by c once;
 *  - the scale is truncated (low 4 mantissa bits cleared) before it is used for the zero-point
 *    and the codes;
 *  - zp = clamp(rint(fp32(-min / s')), 0, 15) with an IEEE division and ties to even;
 *  - code_i = clamp(N(y_i * r + zp), 0, 15) where r = fp32(1 / s') and N(.) is the nearest
 *    integer, ties to even, of the EXACT real value y_i * r + zp (one rounding).  The pages'
 *    reference divides instead; oracle_codes_division_form() computes that form so that the tests
 *    can measure how often the two differ.
 *  - the scale word is stored little-endian at byte offset d/2 of the row.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_MAX_D 1024

static uint32_t bits_of(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float float_of(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static int is_pow2(int d) { return d >= 2 && d <= ORACLE_MAX_D && (d & (d - 1)) == 0; }

/* y = c * H_d * (D x): sign flip (exact), butterflies at strides 1, 2, ..., d/2, then scale by c. */
int oracle_rotate_f32(const float* x, const float* signs, int d, float* y) {
    if (!is_pow2(d)) return -1;
    float u[ORACLE_MAX_D];
    for (int i = 0; i < d; ++i) u[i] = x[i] * signs[i];
    for (int h = 1; h < d; h *= 2) {
        for (int i = 0; i < d; ++i) {
            if (i & h) continue;
            float a = u[i];
            float b = u[i + h];
            u[i] = a + b;
            u[i + h] = a - b;
        }
    }
    const float c = (float)(1.0 / sqrt((double)d));
    for (int i = 0; i < d; ++i) y[i] = u[i] * c;
    return 0;
}

/* Nearest integer (ties to even) of the exact real value p + zp, where p = y * r is formed
 * exactly in double (two 24-bit significands give at most 48 bits). */
static double nearest_of_shifted_product(float y, float r, int zp) {
    double p = (double)y * (double)r;
    double n0 = floor(p);
    double half = n0 + 0.5;
    double n;
    if (p < half) {
        n = n0;
    } else if (p > half) {
        n = n0 + 1.0;
    } else {
        /* exact tie: of the two neighbours of p + zp take the even one */
        n = (fmod(n0 + (double)zp, 2.0) == 0.0) ? n0 : n0 + 1.0;
    }
    return n + (double)zp;
}

static uint8_t clamp_code(double v) {
    if (v < 0.0) return 0;
    if (v > 15.0) return 15;
    return (uint8_t)v;
}

/* Quantise an already-rotated vector y: codes[d] in 0..15 and the stored 32-bit scale word
 * (truncated scale bits | zero-point). */
int oracle_quantize_rotated(const float* y, int d, uint8_t* codes, uint32_t* word) {
    if (d < 1 || d > ORACLE_MAX_D) return -1;
    float mn = y[0];
    float mx = y[0];
    for (int i = 1; i < d; ++i) {
        if (y[i] < mn) mn = y[i];
        if (y[i] > mx) mx = y[i];
    }
    float range = mx - mn;
    float s = range / 15.0f;
    if (!(s >= 1e-6f)) s = 1e-6f;
    uint32_t sb = bits_of(s) & 0xFFFFFFF0u;
    float sp = float_of(sb);
    float zq = -mn / sp;
    float zr = rintf(zq);
    int zp = zr < 0.0f ? 0 : (zr > 15.0f ? 15 : (int)zr);
    float r = 1.0f / sp;
    for (int i = 0; i < d; ++i) codes[i] = clamp_code(nearest_of_shifted_product(y[i], r, zp));
    *word = sb | (uint32_t)zp;
    return 0;
}

/* The codes as the pages' test reference forms them: t = fp32(y / s'), t = fp32(t + zp),
 * code = clamp(rint(t), 0, 15).  Used only to count how often this form differs. */
int oracle_codes_division_form(const float* y, int d, uint8_t* codes) {
    uint32_t word;
    uint8_t tmp[ORACLE_MAX_D];
    if (oracle_quantize_rotated(y, d, tmp, &word) != 0) return -1;
    float sp = float_of(word & 0xFFFFFFF0u);
    float zp = (float)(word & 0xFu);
    for (int i = 0; i < d; ++i) {
        float t = y[i] / sp;
        t = t + zp;
        codes[i] = clamp_code((double)rintf(t));
    }
    return 0;
}

/* Row bytes: byte j = code[2j] | code[2j+1] << 4 for j < d/2, then the scale word little-endian. */
static void pack_row(const uint8_t* codes, uint32_t word, int d, uint8_t* row) {
    for (int j = 0; j < d / 2; ++j) row[j] = (uint8_t)((codes[2 * j] & 0xF) | ((codes[2 * j + 1] & 0xF) << 4));
    row[d / 2 + 0] = (uint8_t)(word & 0xFF);
    row[d / 2 + 1] = (uint8_t)((word >> 8) & 0xFF);
    row[d / 2 + 2] = (uint8_t)((word >> 16) & 0xFF);
    row[d / 2 + 3] = (uint8_t)((word >> 24) & 0xFF);
}

/* One head vector (fp32, the exact upcast of the fp16/bf16 input) -> one cache row of d/2+4 bytes. */
int oracle_encode_row(const float* x, const float* signs, int d, uint8_t* row) {
    float y[ORACLE_MAX_D];
    uint8_t codes[ORACLE_MAX_D];
    uint32_t word;
    if (oracle_rotate_f32(x, signs, d, y) != 0) return -1;
    oracle_quantize_rotated(y, d, codes, &word);
    pack_row(codes, word, d, row);
    return 0;
}

/* The cache write.  k, v: [T, H, d] fp32; slots: [T]; cache: (num_blocks, 2, bs, H, d/2+4) bytes.
 * A slot < 0 is a padding token and is skipped; a slot >= num_blocks * bs is skipped and counted.
 * Returns the number of out-of-range slots, or -1 for an invalid head size. */
int64_t oracle_kv_int4_write(const float* k, const float* v, int64_t num_tokens, int num_kv_heads,
                             int d, const int64_t* slots, const float* signs, uint8_t* cache,
                             int64_t num_blocks, int block_size) {
    if (!is_pow2(d)) return -1;
    const int64_t row_bytes = d / 2 + 4;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) {
            ++bad;
            continue;
        }
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int p = 0; p < 2; ++p) {
            const float* src = (p == 0 ? k : v) + t * (int64_t)num_kv_heads * d;
            for (int h = 0; h < num_kv_heads; ++h) {
                uint8_t* row = cache + (((blk * 2 + p) * block_size + off) * num_kv_heads + h) * row_bytes;
                oracle_encode_row(src + (int64_t)h * d, signs, d, row);
            }
        }
    }
    return bad;
}
