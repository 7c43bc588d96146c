/*
 * kvq_oracle.c -- plain, slow CPU oracle for dynamic KV-cache quantization
 * and fused-dequantization paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product (the CUDA
 * library under dynamically_quantized_paged_gb300/) never links, imports or
 * calls it, and this file includes nothing from the product.
 *
 * What it computes, and where each step comes from:
 *
 *   [P1] "Dynamic KV Cache Quantization for Fast LLM Inference"
 *        - section "Understanding Dynamic Quantization Techniques for KV
 *          Caches (e.g., INT8, INT4)": the scale is the row's largest absolute
 *          value divided by 2^(bits-1)-1, the code is the rounded quotient
 *          x / scale, the scale is computed on the fly per head / per token;
 *          an all-zero tensor gets zero codes and scale 1.0; the INT8 range
 *          is [-127, 127]; dequantization multiplies the code by the scale.
 *          The same paragraph names a zero-point, which is what the
 *          asymmetric INT4 scheme below stores.
 *        - section "Recap of KV Caching ...": a new token's K/V are appended
 *          and the query attends to every cached token.
 *        - section "Integrating Dynamic Quantization with PagedAttention ...":
 *          fixed-size blocks, logical-to-physical block mapping.
 *   [P2] "What is KV Cache Optimization? Definition, Quantization & Memory
 *        Management in Enterprise AI?", section "Technical Architecture":
 *        capture K/V, quantize to FP8/INT8/INT4, store in non-contiguous
 *        pages, dequantize inside the attention kernel; bytes per token.
 *   [P3] "KV Cache Optimization: Strategies for Faster LLM Inference",
 *        section "How vLLM Implements KV Cache Optimization": blocks are
 *        allocated on demand, 16 tokens per block by default.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): rounding is round-half-to-even (the worked example's torch.round);
 * the INT8 scale is an IEEE fp32 division and the code an IEEE fp32 division
 * by the scale; FP8-E4M3 uses qmax = 448 (largest finite E4M3) and
 * round-to-nearest-even with saturation; INT4 is asymmetric over groups of 32
 * channels with an fp16 zero-point rounded down from the group minimum and an
 * fp16 scale rounded up from (max - zero) / 15; symmetric INT4 uses groups
 * of 32, an fp32 scale max|x| / 7 and two's-complement nibbles; attention is
 * exact fp64 over
 * the dequantized cache with softmax scale 1/sqrt(head_dim) and query head g
 * reading KV head g / (Hq / Hkv).
 *
 * Per-channel K ([P3] "KV Cache Optimization: Strategies for Faster LLM
 * Inference", section "KV Cache Quantization: When and How to Compress":
 * per-channel quantization keeps more than per-tensor).  Reading taken: the
 * K scale of a channel is taken over the tokens of one page (one scale per
 * page, KV head and channel); while a page is still filling its tokens are
 * stored with the INT8 token rule and their bf16 K rows are kept in a
 * residual slot; once full, the page is sealed: its K is re-quantized per
 * channel from those bf16 rows (the INT8 rule along the token axis, in the
 * normalized form described at orc_quant_kchan_page).  V keeps the token
 * rule throughout.  Dequantized K = code * channel factor * token scale,
 * where an open page has channel factors 1 and a sealed page has its
 * largest channel scale as every token's scale.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -fPIC -shared.
 * Floating-point: every fp32 step is a single IEEE operation in the order
 * written; no contraction, no reassociation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- scheme ids (the oracle's own copy of the numbering) ----------------- */
enum { ORC_INT8 = 1, ORC_FP8 = 2, ORC_INT4 = 3, ORC_INT4SYM = 4, ORC_INT8KC = 5 };

/* ---- number formats, from their definitions ------------------------------ */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
float orc_bf16_to_float(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_fp16_value(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int m = bits & 0x3ff;
    double v;
    if (e == 0x1f) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);          /* subnormal: m * 2^-24 */
    else v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -v : v;
}

/* Encode a binary16 value known to be exactly representable. */
static uint16_t fp16_bits_of_exact(double v) {
    uint16_t sign = 0;
    if (signbit(v)) { sign = 0x8000; v = -v; }
    if (isinf(v)) return sign | 0x7c00;
    if (v == 0.0) return sign;
    int e;
    frexp(v, &e);                       /* v = f * 2^e, f in [0.5, 1) */
    int unb = e - 1;                    /* v = 1.x * 2^unb */
    if (unb < -14) {                    /* subnormal */
        return sign | (uint16_t)(v / ldexp(1.0, -24));
    }
    double frac = v / ldexp(1.0, unb) - 1.0;
    return sign | (uint16_t)((unb + 15) << 10) | (uint16_t)(frac * 1024.0);
}

/* Directed rounding of a finite fp32 value to binary16.  The spacing of
 * binary16 numbers near x is 2^(E-10) for |x| in [2^E, 2^(E+1)), E >= -14,
 * and 2^-24 below 2^-14; x / spacing is exact in double, so floor/ceil give
 * the neighbours exactly.  Beyond the largest finite value 65504 the result
 * is 65504 or infinity depending on the direction. */
static double fp16_directed(float xf, int up) {
    double x = (double)xf;
    if (x == 0.0) return x;
    double ax = fabs(x);
    int e;
    frexp(ax, &e);
    int E = e - 1;
    if (E < -14) E = -14;
    double spacing = ldexp(1.0, E - 10);
    double k = x / spacing;
    double r = (up ? ceil(k) : floor(k)) * spacing;
    if (r > 65504.0) r = up ? INFINITY : 65504.0;
    if (r < -65504.0) r = up ? -65504.0 : -INFINITY;
    if (r == 0.0 && signbit(x)) r = -0.0;
    return r;
}

uint16_t orc_fp16_round_down(float x) { return fp16_bits_of_exact(fp16_directed(x, 0)); }
uint16_t orc_fp16_round_up(float x) { return fp16_bits_of_exact(fp16_directed(x, 1)); }

/* OCP 8-bit floating point, E4M3 ("fn" flavour): 1 sign, 4 exponent bits
 * (bias 7), 3 fraction bits; no infinities; S.1111.111 is NaN; the largest
 * finite magnitude is 1.75 * 2^8 = 448; subnormals are m/8 * 2^-6. */
double orc_e4m3_value(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xf;
    int m = code & 0x7;
    double v;
    if (e == 0xf && m == 0x7) v = NAN;
    else if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* The 127 finite non-negative E4M3 magnitudes, in code order (code c has
 * magnitude e4m3_mag[c]; they increase strictly with c), filled once when the
 * library is loaded from the definition above. */
static double e4m3_mag[0x7f];

__attribute__((constructor)) static void orc_init_e4m3_table(void) {
    for (int c = 0; c < 0x7f; ++c) e4m3_mag[c] = orc_e4m3_value((uint8_t)c);
}

/* Round-to-nearest-even into E4M3 with saturation to +-448: the nearest of
 * the 127 finite non-negative magnitudes to |y|, a tie going to the even code
 * (the even significand).  The sign of the result is the sign of y, zero
 * included.  The two magnitudes that bracket |y| are found by bisection over
 * the increasing table; the nearest of the two is taken. */
uint8_t orc_e4m3_encode(float yf) {
    double y = (double)yf;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs(y);
    if (a >= 448.0) return sign | 0x7e;
    int lo = 0, hi = 0x7e; /* invariant: e4m3_mag[lo] <= a < e4m3_mag[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (e4m3_mag[mid] <= a) lo = mid;
        else hi = mid;
    }
    double dlo = a - e4m3_mag[lo], dhi = e4m3_mag[hi] - a;
    int best;
    if (dlo < dhi) best = lo;
    else if (dhi < dlo) best = hi;
    else best = (lo % 2 == 0) ? lo : hi;
    return sign | (uint8_t)best;
}

/* ---- per-row quantizers ---------------------------------------------------- */

/* Symmetric INT8 of one (token, KV head) row, following the worked INT8
 * function of [P1] "Understanding Dynamic Quantization Techniques": the
 * largest magnitude; zero row -> zero codes and scale 1.0; scale =
 * absmax / 127 (fp32 division); code = round-half-even(x / scale) (fp32
 * division), kept inside [-127, 127]. */
void orc_quant_int8_row(const uint16_t* x, int n, int8_t* codes, float* scale_out) {
    float absmax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(orc_bf16_to_float(x[i]));
        if (a > absmax) absmax = a;
    }
    if (absmax == 0.0f) {
        for (int i = 0; i < n; ++i) codes[i] = 0;
        *scale_out = 1.0f;
        return;
    }
    float scale = absmax / 127.0f;
    for (int i = 0; i < n; ++i) {
        float r = rintf(orc_bf16_to_float(x[i]) / scale);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        codes[i] = (int8_t)r;
    }
    *scale_out = scale;
}

/* FP8-E4M3 of one (token, KV head) row: the same absmax rule with qmax = 448
 * (the largest finite E4M3); code = E4M3 round-to-nearest-even of x / scale,
 * saturating.  A zero row gets zero codes and scale 1.0. */
void orc_quant_fp8_row(const uint16_t* x, int n, uint8_t* codes, float* scale_out) {
    float absmax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(orc_bf16_to_float(x[i]));
        if (a > absmax) absmax = a;
    }
    if (absmax == 0.0f) {
        for (int i = 0; i < n; ++i) codes[i] = 0;
        *scale_out = 1.0f;
        return;
    }
    float scale = absmax / 448.0f;
    for (int i = 0; i < n; ++i) codes[i] = orc_e4m3_encode(orc_bf16_to_float(x[i]) / scale);
    *scale_out = scale;
}

/* Asymmetric INT4 of one row, per group of `group` channels along head_dim.
 * For each group: minimum mn and maximum mx (fp32); zero-point z = binary16
 * rounded down from mn; scale s = binary16 rounded up from (mx - z) / 15
 * (fp32 subtraction, fp32 division); s == 0 (a constant group equal to z)
 * becomes 1.0, the zero-row rule of [P1].  code = round-half-even((x - z) / s)
 * inside [0, 15].  Two codes per byte: the even channel in the low nibble.
 * Dequantization: code * s + z. */
void orc_quant_int4_row(const uint16_t* x, int n, int group, uint8_t* packed,
                        uint16_t* scales, uint16_t* zeros) {
    int ngroups = n / group;
    uint8_t q[1024];
    for (int gi = 0; gi < ngroups; ++gi) {
        const uint16_t* xg = x + gi * group;
        float mn = INFINITY, mx = -INFINITY;
        for (int i = 0; i < group; ++i) {
            float v = orc_bf16_to_float(xg[i]);
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        uint16_t zb = orc_fp16_round_down(mn);
        float zf = (float)orc_fp16_value(zb);
        float span = mx - zf;
        float sdiv = span / 15.0f;
        uint16_t sb = orc_fp16_round_up(sdiv);
        if (orc_fp16_value(sb) == 0.0) sb = 0x3c00; /* 1.0 */
        float sf = (float)orc_fp16_value(sb);
        for (int i = 0; i < group; ++i) {
            float r = rintf((orc_bf16_to_float(xg[i]) - zf) / sf);
            if (r < 0.0f) r = 0.0f;
            if (r > 15.0f) r = 15.0f;
            q[gi * group + i] = (uint8_t)r;
        }
        scales[gi] = sb;
        zeros[gi] = zb;
    }
    for (int j = 0; j < n / 2; ++j) packed[j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
}

/* Symmetric INT4 of one row in groups of `group` channels: [P1]
 * "Understanding Dynamic Quantization Techniques ..." with bits = 4, so the
 * scale is the group's largest magnitude over 2^(4-1)-1 = 7 (one IEEE fp32
 * division, kept in fp32), an all-zero group gets scale 1.0 and zero codes,
 * and the code is the half-to-even rounding of the IEEE fp32 quotient x /
 * scale, which lies in [-7, 7] by construction (clamped all the same).  Codes
 * are stored as 4-bit two's complement, two per byte, the even channel in
 * the low nibble.  Dequantization: code * scale. */
void orc_quant_int4sym_row(const uint16_t* x, int n, int group, uint8_t* packed, float* scales) {
    int ngroups = n / group;
    int8_t q[1024];
    for (int gi = 0; gi < ngroups; ++gi) {
        const uint16_t* xg = x + gi * group;
        float a = 0.0f;
        for (int i = 0; i < group; ++i) {
            float v = fabsf(orc_bf16_to_float(xg[i]));
            if (v > a) a = v;
        }
        float s = (a == 0.0f) ? 1.0f : a / 7.0f;
        for (int i = 0; i < group; ++i) {
            float r = (a == 0.0f) ? 0.0f : rintf(orc_bf16_to_float(xg[i]) / s);
            if (r < -7.0f) r = -7.0f;
            if (r > 7.0f) r = 7.0f;
            q[gi * group + i] = (int8_t)r;
        }
        scales[gi] = s;
    }
    for (int j = 0; j < n / 2; ++j)
        packed[j] = (uint8_t)(((uint8_t)q[2 * j] & 0xF) | (((uint8_t)q[2 * j + 1] & 0xF) << 4));
}

/* Per-channel INT8 of one (page, KV head) K block x[P][D] (bf16 bits): the
 * absmax rule of [P1] "Understanding Dynamic Quantization Techniques" taken
 * down each channel instead of along each token ([P3] "KV Cache
 * Quantization: When and How to Compress": per-channel), in a normalized
 * form that keeps every stored factor small:
 *   s_j   = (max over t of |x[t][j]|) / 127                   (fp32 division)
 *   S     = max over j of s_j                                  (the block's largest)
 *   r_j   = fp16 round-up of s_j / S  (fp32 division), a channel factor in
 *           [0, 1]; rounding up makes the effective scale e_j >= s_j up to
 *           the fp32 roundings, so no quotient passes 127 by more than a
 *           rounding step
 *   e_j   = r_j * S                                            (fp32 product)
 *   code  = round-half-even(x / e_j) (fp32 division), kept in [-127, 127];
 *           0 for a channel with e_j = 0 (an all-zero channel)
 *   tok_t = S for every token of the block.
 * An all-zero block stores codes 0, factors 1.0 and token scales 1.0 (the
 * zero-row convention of the INT8 rule).  Dequantized: code * r_j * tok_t. */
void orc_quant_kchan_page(const uint16_t* x, int P, int D, int8_t* codes, uint16_t* chan, float* tok) {
    float s[1024];
    float S = 0.0f;
    for (int j = 0; j < D; ++j) {
        float absmax = 0.0f;
        for (int t = 0; t < P; ++t) {
            float a = fabsf(orc_bf16_to_float(x[(int64_t)t * D + j]));
            if (a > absmax) absmax = a;
        }
        s[j] = absmax / 127.0f;
        if (s[j] > S) S = s[j];
    }
    if (S == 0.0f) {
        for (int64_t i = 0; i < (int64_t)P * D; ++i) codes[i] = 0;
        for (int j = 0; j < D; ++j) chan[j] = 0x3C00; /* 1.0 */
        for (int t = 0; t < P; ++t) tok[t] = 1.0f;
        return;
    }
    for (int j = 0; j < D; ++j) {
        float ratio = s[j] / S;
        chan[j] = orc_fp16_round_up(ratio);
        float e = (float)orc_fp16_value(chan[j]) * S;
        for (int t = 0; t < P; ++t) {
            int8_t q = 0;
            if (e != 0.0f) {
                float r = rintf(orc_bf16_to_float(x[(int64_t)t * D + j]) / e);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                q = (int8_t)r;
            }
            codes[(int64_t)t * D + j] = q;
        }
    }
    for (int t = 0; t < P; ++t) tok[t] = S;
}

/* ---- the paged cache image ------------------------------------------------- */

/* One layer's cache.  Layout (this library's design, restated here on its
 * own):
 *   8-bit schemes:  codes  [page][kv_head][page_size][head_dim]   1 B each
 *                   scales [page][kv_head][page_size]             fp32
 *   INT4:           codes  [page][kv_head][page_size][head_dim/2] 2 codes/B
 *                   scales, zeros [page][kv_head][page_size][head_dim/group]
 *                                                                 fp16 bits
 *   symmetric INT4: codes as INT4 (two's-complement nibbles)
 *                   scales [page][kv_head][page_size][head_dim/group] fp32
 *   per-channel K:  codes and scales as INT8 (K scales are the token
 *                   scales tok_t), plus
 *                   k_chan  [page][kv_head][head_dim]             fp16 bits
 *                   k_resid [resid_slots][kv_head][page_size][head_dim] bf16
 * A token at physical slot `slot` lives in page slot / page_size at offset
 * slot % page_size. */
typedef struct {
    int32_t scheme, num_pages, page_size, num_kv_heads, head_dim, group;
    void *k_codes, *v_codes, *k_scales, *v_scales, *k_zeros, *v_zeros;
    void *k_chan, *k_resid;
    int32_t resid_slots;
} orc_cache;

static int64_t row_code_bytes(const orc_cache* c) {
    return (c->scheme == ORC_INT4 || c->scheme == ORC_INT4SYM) ? c->head_dim / 2 : c->head_dim;
}

/* Quantize-append: token t's K and V rows ([T][Hkv][D] bf16) are quantized
 * per KV head and stored at slot_mapping[t]; a negative slot skips the token.
 * Per-channel K: both rows take the INT8 token rule (the page is open); a
 * token at offset 0 opens its page, setting that head's channel factors to
 * 1.0; with resid_slot given and resid_slot[t] >= 0, the token's bf16 K row
 * is also kept at offset slot % page_size of residual slot resid_slot[t].
 * Returns 0, or -1 if a slot or residual slot is outside its pool (nothing
 * written for it). */
int orc_append_kc(const orc_cache* c, const int64_t* slot_mapping, const int32_t* resid_slot,
                  const uint16_t* k, const uint16_t* v, int32_t T) {
    const int H = c->num_kv_heads, D = c->head_dim, P = c->page_size;
    const int64_t nslots = (int64_t)c->num_pages * P;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int32_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= nslots) { bad = 1; continue; }
        int64_t page = slot / P, off = slot % P;
        int32_t rs = resid_slot ? resid_slot[t] : -1;
        if (c->scheme == ORC_INT8KC && rs >= c->resid_slots) { bad = 1; continue; }
        for (int h = 0; h < H; ++h) {
            int64_t row = (page * H + h) * P + off; /* row index inside the pool */
            if (c->scheme == ORC_INT8KC) {
                const uint16_t* x = k + ((int64_t)t * H + h) * D;
                if (off == 0)
                    for (int j = 0; j < D; ++j) ((uint16_t*)c->k_chan)[(page * H + h) * D + j] = 0x3C00;
                if (rs >= 0)
                    memcpy((uint16_t*)c->k_resid + (((int64_t)rs * H + h) * P + off) * D, x,
                           sizeof(uint16_t) * (size_t)D);
            }
            for (int kv = 0; kv < 2; ++kv) {
                const uint16_t* x = (kv == 0 ? k : v) + ((int64_t)t * H + h) * D;
                uint8_t* codes = (uint8_t*)(kv == 0 ? c->k_codes : c->v_codes) + row * row_code_bytes(c);
                if (c->scheme == ORC_INT8 || c->scheme == ORC_INT8KC) {
                    float* sc = (float*)(kv == 0 ? c->k_scales : c->v_scales) + row;
                    orc_quant_int8_row(x, D, (int8_t*)codes, sc);
                } else if (c->scheme == ORC_FP8) {
                    float* sc = (float*)(kv == 0 ? c->k_scales : c->v_scales) + row;
                    orc_quant_fp8_row(x, D, codes, sc);
                } else if (c->scheme == ORC_INT4SYM) {
                    int ng = D / c->group;
                    float* sc = (float*)(kv == 0 ? c->k_scales : c->v_scales) + row * ng;
                    orc_quant_int4sym_row(x, D, c->group, codes, sc);
                } else {
                    int ng = D / c->group;
                    uint16_t* sc = (uint16_t*)(kv == 0 ? c->k_scales : c->v_scales) + row * ng;
                    uint16_t* zp = (uint16_t*)(kv == 0 ? c->k_zeros : c->v_zeros) + row * ng;
                    orc_quant_int4_row(x, D, c->group, codes, sc, zp);
                }
            }
        }
    }
    return bad ? -1 : 0;
}

int orc_append(const orc_cache* c, const int64_t* slot_mapping, const uint16_t* k,
               const uint16_t* v, int32_t T) {
    return orc_append_kc(c, slot_mapping, NULL, k, v, T);
}

/* Seal pages of the per-channel K scheme: for each i, page pages[i] (every KV
 * head) takes the per-channel rule (orc_quant_kchan_page) of the page_size
 * bf16 K rows kept in residual slot resid_slots[i]: its K codes, channel
 * factors and token scales are replaced; V is left as it is.  Returns 0, or
 * -1 if a page or slot id is outside its pool (that pair is skipped). */
int orc_seal_pages(const orc_cache* c, const int32_t* pages, const int32_t* resid_slots, int32_t n) {
    const int H = c->num_kv_heads, D = c->head_dim, P = c->page_size;
    int bad = 0;
    if (c->scheme != ORC_INT8KC) return -1;
    for (int32_t i = 0; i < n; ++i) {
        int32_t page = pages[i], rs = resid_slots[i];
        if (page < 0 || page >= c->num_pages || rs < 0 || rs >= c->resid_slots) { bad = 1; continue; }
        for (int h = 0; h < H; ++h) {
            const uint16_t* x = (const uint16_t*)c->k_resid + ((int64_t)rs * H + h) * P * D;
            int64_t row0 = ((int64_t)page * H + h) * P;
            orc_quant_kchan_page(x, P, D, (int8_t*)c->k_codes + row0 * D,
                                 (uint16_t*)c->k_chan + ((int64_t)page * H + h) * D, (float*)c->k_scales + row0);
        }
    }
    return bad ? -1 : 0;
}

/* Dequantize the row stored at pool row index `row` into fp64 (exact:
 * code * scale (+ zero) with every operand exactly representable). */
static void dequant_row(const orc_cache* c, int kv, int64_t row, double* out) {
    const int D = c->head_dim;
    const uint8_t* codes = (const uint8_t*)(kv == 0 ? c->k_codes : c->v_codes) + row * row_code_bytes(c);
    if (c->scheme == ORC_INT8 || (c->scheme == ORC_INT8KC && kv == 1)) {
        double s = ((const float*)(kv == 0 ? c->k_scales : c->v_scales))[row];
        for (int j = 0; j < D; ++j) out[j] = (double)(int8_t)codes[j] * s;
    } else if (c->scheme == ORC_INT8KC) {
        /* code * channel factor * token scale: 8 + 11 + 24 significant bits,
         * exact in fp64 */
        double s = ((const float*)c->k_scales)[row];
        const uint16_t* r = (const uint16_t*)c->k_chan + (row / c->page_size) * D;
        for (int j = 0; j < D; ++j) out[j] = (double)(int8_t)codes[j] * orc_fp16_value(r[j]) * s;
    } else if (c->scheme == ORC_FP8) {
        double s = ((const float*)(kv == 0 ? c->k_scales : c->v_scales))[row];
        for (int j = 0; j < D; ++j) out[j] = orc_e4m3_value(codes[j]) * s;
    } else if (c->scheme == ORC_INT4SYM) {
        int ng = D / c->group;
        const float* sc = (const float*)(kv == 0 ? c->k_scales : c->v_scales) + row * ng;
        for (int j = 0; j < D; ++j) {
            int nib = (j & 1) ? (codes[j / 2] >> 4) : (codes[j / 2] & 0xf);
            int code = nib >= 8 ? nib - 16 : nib; /* 4-bit two's complement */
            out[j] = (double)code * (double)sc[j / c->group];
        }
    } else {
        int ng = D / c->group;
        const uint16_t* sc = (const uint16_t*)(kv == 0 ? c->k_scales : c->v_scales) + row * ng;
        const uint16_t* zp = (const uint16_t*)(kv == 0 ? c->k_zeros : c->v_zeros) + row * ng;
        for (int j = 0; j < D; ++j) {
            int code = (j & 1) ? (codes[j / 2] >> 4) : (codes[j / 2] & 0xf);
            int gi = j / c->group;
            out[j] = (double)code * orc_fp16_value(sc[gi]) + orc_fp16_value(zp[gi]);
        }
    }
}

/* Decode attention, fp64.  For sequence b and query head g (KV head
 * g / (Hq/Hkv)): scores over every cached token t < seq_lens[b] (the token
 * just appended included), found through block_table[b][t / page_size];
 * softmax by max subtraction; output = sum_t p_t * V_t.  seq_len 0 gives a
 * zero output.  softmax_scale <= 0 means 1/sqrt(head_dim).
 * out is [B][Hq][D] fp64.  Returns 0, or -1 on an out-of-range page id. */
int orc_decode_attn(const orc_cache* c, const uint16_t* q, const int32_t* block_table,
                    const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t max_pages_per_seq,
                    double softmax_scale, double* out) {
    const int H = c->num_kv_heads, D = c->head_dim, P = c->page_size;
    const int G = Hq / H;
    if (softmax_scale <= 0.0) softmax_scale = 1.0 / sqrt((double)D);
    int bad = 0;
#pragma omp parallel for schedule(dynamic) collapse(2) reduction(| : bad)
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t hq = 0; hq < Hq; ++hq) {
            const int h = hq / G;
            const int32_t L = seq_lens[b];
            double* o = out + ((int64_t)b * Hq + hq) * D;
            for (int j = 0; j < D; ++j) o[j] = 0.0;
            if (L <= 0) continue;
            double qd[1024], kr[1024], vr[1024];
            for (int j = 0; j < D; ++j) qd[j] = orc_bf16_to_float(q[((int64_t)b * Hq + hq) * D + j]);
            double* s = (double*)malloc(sizeof(double) * (size_t)L);
            double m = -INFINITY;
            int ok = 1;
            for (int32_t t = 0; t < L; ++t) {
                int32_t page = block_table[(int64_t)b * max_pages_per_seq + t / P];
                if (page < 0 || page >= c->num_pages) { ok = 0; break; }
                dequant_row(c, 0, ((int64_t)page * H + h) * P + t % P, kr);
                double dot = 0.0;
                for (int j = 0; j < D; ++j) dot += qd[j] * kr[j];
                s[t] = dot * softmax_scale;
                if (s[t] > m) m = s[t];
            }
            if (!ok) { bad = 1; free(s); continue; }
            double l = 0.0;
            for (int32_t t = 0; t < L; ++t) {
                double p = exp(s[t] - m);
                l += p;
                int32_t page = block_table[(int64_t)b * max_pages_per_seq + t / P];
                dequant_row(c, 1, ((int64_t)page * H + h) * P + t % P, vr);
                for (int j = 0; j < D; ++j) o[j] += p * vr[j];
            }
            for (int j = 0; j < D; ++j) o[j] /= l;
            free(s);
        }
    }
    return bad ? -1 : 0;
}

/* ---- page allocation --------------------------------------------------------- */

/* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; the 64-bit finalizer constants as published by
 * Vigna): advance the state by the golden-ratio increment, then mix. */
static uint64_t splitmix64_next(uint64_t* state) {
    uint64_t z = (*state += 0x9e3779b97f4a7c15ULL);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

uint64_t orc_splitmix64(uint64_t* state) { return splitmix64_next(state); }

/* The initial free list of a pool of num_pages pages ([P3] "How vLLM
 * Implements KV Cache Optimization": blocks are handed out on demand from a
 * pool, scattered in memory).  Page ids 0..N-1 are shuffled by Fisher-Yates
 * (Durstenfeld's form: i from N-1 down to 1, j = next() mod (i+1), swap a[i]
 * and a[j]) driven by SplitMix64 seeded with `seed`.  The allocator hands
 * pages out from the END of this array (a stack), one at a time. */
void orc_free_list(int32_t num_pages, uint64_t seed, int32_t* out) {
    uint64_t st = seed;
    for (int32_t i = 0; i < num_pages; ++i) out[i] = i;
    for (int32_t i = num_pages - 1; i >= 1; --i) {
        uint64_t j = splitmix64_next(&st) % (uint64_t)(i + 1);
        int32_t tmp = out[i];
        out[i] = out[j];
        out[j] = tmp;
    }
}

/* ---- misc ---------------------------------------------------------------------- */

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
