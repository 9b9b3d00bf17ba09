/*
 * Plain CPU oracle for paged attention over a q8 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with the
 * CUDA library: no header, no helper, no table.
 *
 * Sources (pages, cited by title and section):
 *  - "shared/attention_kit.py" (WanGP attention kit): the q8 format
 *    (`quantize_q8`, `dequantize_q8_into`: int8 data, one FP16 scale per
 *    32 channels, scale = max|x|/127 clamped at 1e-8) and the two-set
 *    log-sum-exp merge `_merge_lse_`.
 *  - "shared/kernels/qk_quant_triton.py" (`_norm_rope_quant`, `_rows`):
 *    rounding half away from zero before the int8 cast; the weighted RMSNorm
 *    (fp32 statistics, output rounded to the activation dtype) and the fp32
 *    rotation of channel pairs that the fused store applies to keys.
 *  - "attention_impl.py" (fastkernels-b200, `_store_kvcache_nhd`,
 *    `StoreKVCache`): scatter by slot, slot < 0 skipped,
 *    block = slot // block_size, offset = slot % block_size; the torch SDPA
 *    reference paths `_cache_seq`, `_sdpa_one`, `_prefill_torch_from_cache`:
 *    paged gather, GQA by repeat_interleave, causal mask k_pos <= q_pos with
 *    key_offset = k_len - q_len.
 *  - "triton_turboquant_unified_attention.py" (vLLM unified kernel): the
 *    K and V load sites of its alternative formats (FP8 keys read as e4m3
 *    values; 4-bit values dequantized as idx * scale + zero with one fp16
 *    scale and zero per token); the seq_lens / query_start_loc meaning, the
 *    causal limit
 *    seq_offset <= context_len + query_pos, the 3D split-KV segments and the
 *    (max, expsum, acc) partial triples merged by the online-softmax rule.
 *
 * Precision: quantization takes its decisions in fp32, as the q8 pages do
 * (`x.float()`, then fp32 divide, round, clamp, FP16 store).  Attention is
 * fp64 over the exactly dequantized values code * (double)scale.
 *
 * Readings where the pages are silent or disagree (each is listed in the
 * design notes):
 *  - rounding is exact round-half-away-from-zero of the fp32 quotient
 *    (C `roundf`), not "+0.5*sign then truncate";
 *  - the divisor is the fp32 scale before its FP16 rounding;
 *  - the scale floor is 1e-8 (fp32), and FP16 conversion is round to nearest
 *    even;
 *  - the LSE is the natural log of sum_j exp(scale * q.k_j);
 *  - caches are HND: K codes [num_blocks, Hk, block_size, D] int8, K scales
 *    [num_blocks, Hk, block_size, D/32] fp16; V pages channel-major, codes
 *    [num_blocks, Hk, D, block_size], scales [num_blocks, Hk, D/32, block_size].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_GROUP 32

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern -> value.  bf16 is the upper half of an IEEE binary32. */
static float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary16 bit pattern -> value (exact; every binary16 is a binary32). */
float or_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t exp = (uint32_t)(h >> 10) & 0x1fu;
    uint32_t man = (uint32_t)h & 0x3ffu;
    float mag;
    if (exp == 0) {
        mag = ldexpf((float)man, -24);            /* zero or subnormal: man * 2^-24 */
    } else if (exp == 31) {
        mag = man ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(man | 0x400u), (int)exp - 25); /* 1.man * 2^(exp-15) */
    }
    return sign ? -mag : mag;
}

/*
 * binary32 -> binary16, round to nearest, ties to even (IEEE 754 default).
 * Written from the definition: find the two neighbouring binary16 values and
 * pick the nearer, the even one on a tie.  Overflow past the largest finite
 * binary16 (65504) rounds to infinity exactly when the value is at or above
 * 65520, the midpoint between 65504 and 2^16.
 */
uint16_t or_f32_to_f16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    float a = fabsf(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7c00u);   /* rounds to inf */
    /* binary16 step (ulp) at a: 2^(e-10) for normal a in [2^e, 2^(e+1)),
     * 2^-24 for subnormal a < 2^-14. */
    int e;
    if (a < ldexpf(1.0f, -14)) {
        e = -14;
    } else {
        (void)frexpf(a, &e);   /* a = m * 2^e, m in [0.5, 1) */
        e -= 1;                /* a in [2^e, 2^(e+1)) */
    }
    double ulp = ldexp(1.0, e - 10);
    double q = (double)a / ulp;          /* exact: a has 24 bits, ulp a power of two */
    double lo = floor(q);
    double rem = q - lo;
    double n;
    if (rem > 0.5) n = lo + 1.0;
    else if (rem < 0.5) n = lo;
    else n = (fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0;
    double r = n * ulp;                  /* the rounded magnitude, exact */
    /* encode r */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -14)) {
        uint16_t man = (uint16_t)(r / ldexp(1.0, -24));
        return (uint16_t)(sign | man);
    }
    int re;
    double m = frexp(r, &re);            /* r = m * 2^re, m in [0.5, 1) */
    int exp16 = re - 1 + 15;             /* r = 1.f * 2^(re-1) */
    if (exp16 >= 31) return (uint16_t)(sign | 0x7c00u);
    uint16_t man = (uint16_t)((m * 2.0 - 1.0) * 1024.0);
    return (uint16_t)(sign | ((uint16_t)exp16 << 10) | man);
}

/*
 * binary32 -> bfloat16 bits, round to nearest, ties to even.  bfloat16 keeps
 * the top 16 bits of a binary32 (same exponent range): the result is the
 * nearer of the two bfloat16 values that bracket x -- the truncation and the
 * next value up in magnitude -- the even one on a tie.  NaN stays NaN.
 */
uint16_t or_f32_to_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if (isnan(x)) return (uint16_t)((u >> 16) | 0x40u);   /* quiet NaN, sign kept */
    uint32_t lower = u >> 16;                 /* truncation toward zero */
    uint32_t rest = u & 0xffffu;              /* the dropped bits */
    if (rest > 0x8000u || (rest == 0x8000u && (lower & 1u))) lower += 1u;  /* carries into the exponent */
    return (uint16_t)lower;
}

/*
 * binary32 -> fp8 e4m3 ("e4m3fn": 1 sign, 4 exponent bits of bias 7, 3
 * mantissa bits, no infinities, NaN = S.1111.111), round to nearest even,
 * saturating: magnitudes past the largest finite value 448 give 448 (the
 * midpoint rule would send 464 and up to the NaN pattern).  Written from the
 * definition: the two fp8 values bracketing |x| are found from its exponent
 * and the nearer (the even one on a tie) is taken.  NaN gives 0x7f.
 */
uint8_t or_f32_to_e4m3(float x)
{
    uint8_t sign = (uint8_t)(signbit(x) ? 0x80u : 0u);
    float a = fabsf(x);
    if (isnan(x)) return 0x7fu;
    if (a >= 448.0f) return (uint8_t)(sign | 0x7eu);          /* 448 = 1.75 * 2^8 */
    /* spacing of e4m3 values at a: 2^(e - 3) for a in [2^e, 2^(e+1)),
     * e >= -6; 2^-9 below 2^-6 (subnormals) */
    int e;
    if (a < ldexpf(1.0f, -6)) {
        e = -6;
    } else {
        (void)frexpf(a, &e);   /* a = m * 2^e, m in [0.5, 1) */
        e -= 1;
    }
    double step = ldexp(1.0, e - 3);
    double q = (double)a / step;           /* exact */
    double lo = floor(q), rem = q - lo, n;
    if (rem > 0.5) n = lo + 1.0;
    else if (rem < 0.5) n = lo;
    else n = (fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0;
    double r = n * step;                   /* rounded magnitude, exact */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    int re;
    double m = frexp(r, &re);              /* r = m * 2^re, m in [0.5, 1) */
    int exp8 = re - 1 + 7;
    uint8_t man = (uint8_t)((m * 2.0 - 1.0) * 8.0);
    return (uint8_t)(sign | (uint8_t)(exp8 << 3) | man);
}

/* fp8 e4m3 bits -> value (exact). */
float or_e4m3_to_f32(uint8_t b)
{
    int sign = b >> 7, exp = (b >> 3) & 0xf, man = b & 7;
    float mag;
    if (exp == 15 && man == 7) mag = NAN;
    else if (exp == 0) mag = ldexpf((float)man, -9);            /* subnormal: man * 2^-9 */
    else mag = ldexpf((float)(man | 8), exp - 10);             /* 1.man * 2^(exp - 7) */
    return sign ? -mag : mag;
}

/*
 * 4-bit asymmetric quantization of one value row x [d] (bf16 bits), the
 * value format whose load site the TurboQuant page shows (V = idx * scale +
 * zero, one fp16 scale and zero per token):
 *   lo = min x, hi = max x                       (fp32)
 *   s32 = max((hi - lo) / 15, 1e-8)              (fp32)
 *   idx = clamp(round_half_away((x - lo) / s32), 0, 15)   (fp32 subtract, divide)
 *   scale = fp16(s32), zero = fp16(lo)           (round to nearest even)
 * idx of channel c goes to nibble c of `nib` (byte c / 2, low nibble for even c).
 */
void or_v4_quantize_row(const uint16_t *x_bf16, int32_t d, uint8_t *nib, uint16_t *scale_bits,
                        uint16_t *zero_bits)
{
    float lo = INFINITY, hi = -INFINITY;
    for (int32_t c = 0; c < d; ++c) {
        float v = or_bf16_to_f32(x_bf16[c]);
        if (v < lo) lo = v;
        if (v > hi) hi = v;
    }
    float s32 = (hi - lo) / 15.0f;
    if (s32 < 1e-8f) s32 = 1e-8f;
    for (int32_t c = 0; c < d; c += 2) nib[c / 2] = 0;
    for (int32_t c = 0; c < d; ++c) {
        float r = roundf((or_bf16_to_f32(x_bf16[c]) - lo) / s32);
        if (r > 15.0f) r = 15.0f;
        if (r < 0.0f) r = 0.0f;
        uint8_t i = (uint8_t)r;
        nib[c / 2] = (uint8_t)(nib[c / 2] | (c & 1 ? (uint8_t)(i << 4) : i));
    }
    *scale_bits = or_f32_to_f16_rne(s32);
    *zero_bits = or_f32_to_f16_rne(lo);
}

/* ------------------------------------------------------------------------ */
/* q8 quantization of one group of 32 channels                               */
/* ------------------------------------------------------------------------ */

/*
 * q8 format ("shared/attention_kit.py", `quantize_q8`):
 *   amax  = max |x| over the group                        (fp32)
 *   s32   = max(amax / 127, 1e-8)                         (fp32 divide, clamp_min)
 *   code  = clamp(round_half_away(x / s32), -127, 127)    (fp32 divide)
 *   scale = fp16(s32), round to nearest even
 * Rounding half away from zero follows "shared/kernels/qk_quant_triton.py"
 * (`_norm_rope_quant`), taken exactly (C roundf).
 */
void or_q8_quantize_group(const float *x, int8_t *codes, uint16_t *scale_bits)
{
    float amax = 0.0f;
    for (int i = 0; i < OR_GROUP; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s32 = amax / 127.0f;
    if (s32 < 1e-8f) s32 = 1e-8f;
    for (int i = 0; i < OR_GROUP; ++i) {
        float r = roundf(x[i] / s32);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        codes[i] = (int8_t)r;
    }
    *scale_bits = or_f32_to_f16_rne(s32);
}

/* Quantize rows of bf16 values: x [n_rows, d] -> codes [n_rows, d],
 * scales [n_rows, d/32]. */
void or_q8_quantize_rows(const uint16_t *x_bf16, int64_t n_rows, int32_t d,
                         int8_t *codes, uint16_t *scales)
{
    float buf[OR_GROUP];
    int32_t groups = d / OR_GROUP;
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int32_t g = 0; g < groups; ++g) {
            const uint16_t *src = x_bf16 + r * d + (int64_t)g * OR_GROUP;
            for (int i = 0; i < OR_GROUP; ++i) buf[i] = or_bf16_to_f32(src[i]);
            or_q8_quantize_group(buf, codes + r * d + (int64_t)g * OR_GROUP,
                                 scales + r * groups + g);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* kv_store: quantize and scatter by slot                                    */
/* ------------------------------------------------------------------------ */

/*
 * key, value: [n_tokens, hk, d] bf16 bits, contiguous.
 * K cache (HND): codes [num_blocks, hk, bs, d] int8, scales
 * [num_blocks, hk, bs, d/32] fp16 bits.  V cache: the same pages stored
 * channel-major, codes [num_blocks, hk, d, bs], scales
 * [num_blocks, hk, d/32, bs] (a layout reading; the values are the same).
 * Scatter ("attention_impl.py", `_store_kvcache_nhd`): slot < 0 is skipped;
 * block = slot / bs, offset = slot % bs.  A slot at or beyond
 * num_blocks * bs is skipped and counted in the return value.
 * Tokens are independent (two tokens with one slot are undefined), so the
 * token range is shared out over n_threads threads (<= 0: every core).
 */
typedef struct {
    const uint16_t *key, *value;
    const int64_t *slot_mapping;
    int64_t n0, n1;
    int32_t hk, d;
    int8_t *k_cache, *v_cache;
    uint16_t *k_scale, *v_scale;
    int64_t num_blocks;
    int32_t bs;
    int64_t bad;
} or_store_job;

static void *or_store_worker(void *arg)
{
    or_store_job *j = (or_store_job *)arg;
    int32_t groups = j->d / OR_GROUP;
    for (int64_t n = j->n0; n < j->n1; ++n) {
        int64_t slot = j->slot_mapping[n];
        if (slot < 0) continue;
        if (slot >= j->num_blocks * j->bs) { ++j->bad; continue; }
        int64_t block = slot / j->bs;
        int64_t offset = slot % j->bs;
        for (int32_t h = 0; h < j->hk; ++h) {
            int64_t row = (block * j->hk + h) * j->bs + offset;     /* HND row */
            const uint16_t *ks = j->key + (n * j->hk + h) * (int64_t)j->d;
            const uint16_t *vs = j->value + (n * j->hk + h) * (int64_t)j->d;
            or_q8_quantize_rows(ks, 1, j->d, j->k_cache + row * j->d, j->k_scale + row * groups);
            /* V: quantize the row, then place channel c at page row c */
            int8_t vcodes[1024];
            uint16_t vscales[32];
            or_q8_quantize_rows(vs, 1, j->d, vcodes, vscales);
            int64_t page = block * j->hk + h;
            for (int32_t c = 0; c < j->d; ++c)
                j->v_cache[(page * j->d + c) * j->bs + offset] = vcodes[c];
            for (int32_t g = 0; g < groups; ++g)
                j->v_scale[(page * groups + g) * j->bs + offset] = vscales[g];
        }
    }
    return NULL;
}

int64_t or_kv_store(const uint16_t *key, const uint16_t *value,
                    const int64_t *slot_mapping, int64_t n_tokens, int32_t hk,
                    int32_t d, int8_t *k_cache, uint16_t *k_scale,
                    int8_t *v_cache, uint16_t *v_scale, int64_t num_blocks,
                    int32_t bs, int32_t n_threads)
{
    if (n_threads <= 0) n_threads = (int32_t)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    if (n_tokens < (int64_t)n_threads * 64) n_threads = 1;
    or_store_job jobs[512];
    pthread_t tids[512];
    for (int32_t i = 0; i < n_threads; ++i) {
        or_store_job j = {key, value, slot_mapping, n_tokens * i / n_threads,
                          n_tokens * (i + 1) / n_threads, hk, d, k_cache, v_cache,
                          k_scale, v_scale, num_blocks, bs, 0};
        jobs[i] = j;
    }
    for (int32_t i = 0; i < n_threads; ++i) pthread_create(&tids[i], NULL, or_store_worker, &jobs[i]);
    int64_t bad = 0;
    for (int32_t i = 0; i < n_threads; ++i) {
        pthread_join(tids[i], NULL);
        bad += jobs[i].bad;
    }
    return bad;
}

/*
 * kv_store in the alternative format: keys as fp8 e4m3 (or_f32_to_e4m3 of
 * each bf16 value, no scale), values as 4-bit codes with a per-(token, head)
 * fp16 scale and zero (or_v4_quantize_row).  Caches (head-major pages):
 *   k_cache  uint8 [num_blocks][hk][bs][d]        e4m3 bits, token-major
 *   v_cache  uint8 [num_blocks][hk][d][bs / 2]    channel-major, keys 2j and
 *                                                  2j + 1 in the low and high
 *                                                  nibble of byte j
 *   v_scale, v_zero fp16 [num_blocks][hk][bs]
 * Scatter as or_kv_store (slot < 0 skipped, slots past the cache counted).
 */
int64_t or_kv_store_f8v4(const uint16_t *key, const uint16_t *value,
                         const int64_t *slot_mapping, int64_t n_tokens, int32_t hk, int32_t d,
                         uint8_t *k_cache, uint8_t *v_cache, uint16_t *v_scale,
                         uint16_t *v_zero, int64_t num_blocks, int32_t bs)
{
    int64_t bad = 0;
    uint8_t nib[512];
    for (int64_t n = 0; n < n_tokens; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        if (slot >= num_blocks * bs) { ++bad; continue; }
        int64_t block = slot / bs, offset = slot % bs;
        for (int32_t h = 0; h < hk; ++h) {
            int64_t page = block * hk + h;
            const uint16_t *ks = key + (n * hk + h) * (int64_t)d;
            const uint16_t *vs = value + (n * hk + h) * (int64_t)d;
            for (int32_t c = 0; c < d; ++c)
                k_cache[(page * bs + offset) * d + c] = or_f32_to_e4m3(or_bf16_to_f32(ks[c]));
            uint16_t sb, zb;
            or_v4_quantize_row(vs, d, nib, &sb, &zb);
            for (int32_t c = 0; c < d; ++c) {
                uint8_t idx = (uint8_t)((nib[c / 2] >> (4 * (c & 1))) & 0xfu);
                uint8_t *byte = v_cache + (page * d + c) * (bs / 2) + offset / 2;
                if (offset & 1) *byte = (uint8_t)((*byte & 0x0fu) | (idx << 4));
                else *byte = (uint8_t)((*byte & 0xf0u) | idx);
            }
            v_scale[page * bs + offset] = sb;
            v_zero[page * bs + offset] = zb;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Fused store: RMSNorm and rotation of the key rows, then q8                */
/* ------------------------------------------------------------------------ */

/*
 * One key row x [d] (bf16 bits) -> the fp32 values the fused store quantizes
 * ("shared/kernels/qk_quant_triton.py", `_rows`, with the readings noted):
 *  1. weighted RMSNorm when w != NULL (bf16 bits [d]):
 *       lane sums: lane l (0..31) takes channels l, l + 32, l + 64, ... in
 *       order, the first squared, each next one added by a fused
 *       multiply-add (the page's lane sums for d = 128); the 32 lane sums are
 *       then added pairwise, lane l with lane l ^ o for o = 16, 8, 4, 2, 1
 *       (the page sums the lanes by a tree whose order it does not fix);
 *       inv = 1 / sqrt(total / d + eps), the square root and the division
 *       each rounded once in fp32 (the page uses an approximate hardware
 *       rsqrt);
 *       y_c = bf16((x_c * inv) * w_c), each product rounded to fp32, the
 *       result rounded to the activation dtype;
 *     otherwise y = x;
 *  2. rotation when rope != NULL (fp32 [rot / 2][2]: cos, sin of pair p at
 *     this token's position), for the rot / 2 pairs (lead, trail) =
 *     (p, p + rot / 2), or (2p, 2p + 1) when interleaved:
 *       out_lead  = fma(cos, y_lead, (-sin) * y_trail)
 *       out_trail = fma(sin, y_lead, cos * y_trail)
 *     in fp32, the plain product rounded first (the page's tl.fma with fp
 *     fusion off); channels at and past rot keep y.  The rotated values stay
 *     fp32: they are quantized without a rounding to bf16.
 */
void or_norm_rope_row(const uint16_t *x, int32_t d, const uint16_t *w, float eps,
                      const float *rope, int32_t rot, int32_t interleaved, float *out)
{
    float y[1024];
    for (int32_t c = 0; c < d; ++c) y[c] = or_bf16_to_f32(x[c]);
    if (w) {
        float lanes[32], next[32];
        for (int32_t l = 0; l < 32; ++l) {
            float acc = y[l] * y[l];
            for (int32_t j = 1; j < d / 32; ++j) acc = fmaf(y[l + 32 * j], y[l + 32 * j], acc);
            lanes[l] = acc;
        }
        for (int32_t o = 16; o > 0; o >>= 1) {
            for (int32_t l = 0; l < 32; ++l) next[l] = lanes[l] + lanes[l ^ o];
            for (int32_t l = 0; l < 32; ++l) lanes[l] = next[l];
        }
        float inv = 1.0f / sqrtf(lanes[0] / (float)d + eps);
        for (int32_t c = 0; c < d; ++c) {
            float t = y[c] * inv;
            t = t * or_bf16_to_f32(w[c]);
            y[c] = or_bf16_to_f32(or_f32_to_bf16_rne(t));
        }
    }
    for (int32_t c = 0; c < d; ++c) out[c] = y[c];
    if (rope) {
        int32_t pairs = rot / 2;
        for (int32_t p = 0; p < pairs; ++p) {
            int32_t lead = interleaved ? 2 * p : p;
            int32_t trail = interleaved ? 2 * p + 1 : p + pairs;
            float cs = rope[2 * p], sn = rope[2 * p + 1];
            float prod_lead = (-sn) * y[trail];
            float prod_trail = cs * y[trail];
            out[lead] = fmaf(cs, y[lead], prod_lead);
            out[trail] = fmaf(sn, y[lead], prod_trail);
        }
    }
}

typedef struct {
    const uint16_t *key, *value;
    const int64_t *slot_mapping, *positions;
    int64_t n0, n1;
    int32_t hk, d;
    const uint16_t *w;
    float eps;
    const float *rope;
    int64_t max_pos;
    int32_t rot, interleaved;
    int8_t *k_cache, *v_cache;
    uint16_t *k_scale, *v_scale;
    int64_t num_blocks;
    int32_t bs;
    int64_t bad;
} or_fused_job;

static void *or_fused_worker(void *arg)
{
    or_fused_job *j = (or_fused_job *)arg;
    int32_t groups = j->d / OR_GROUP;
    float vals[1024];
    for (int64_t n = j->n0; n < j->n1; ++n) {
        int64_t slot = j->slot_mapping[n];
        if (slot < 0) continue;
        int64_t pos = j->rope ? j->positions[n] : 0;
        if (slot >= j->num_blocks * j->bs || (j->rope && (pos < 0 || pos >= j->max_pos))) {
            ++j->bad;
            continue;
        }
        int64_t block = slot / j->bs, offset = slot % j->bs;
        for (int32_t h = 0; h < j->hk; ++h) {
            int64_t row = (block * j->hk + h) * j->bs + offset;
            const uint16_t *ks = j->key + (n * j->hk + h) * (int64_t)j->d;
            const uint16_t *vs = j->value + (n * j->hk + h) * (int64_t)j->d;
            or_norm_rope_row(ks, j->d, j->w, j->eps,
                             j->rope ? j->rope + pos * (int64_t)j->rot : NULL, j->rot,
                             j->interleaved, vals);
            for (int32_t g = 0; g < groups; ++g)
                or_q8_quantize_group(vals + g * OR_GROUP, j->k_cache + row * j->d + g * OR_GROUP,
                                     j->k_scale + row * groups + g);
            int8_t vcodes[1024];
            uint16_t vscales[32];
            or_q8_quantize_rows(vs, 1, j->d, vcodes, vscales);
            int64_t page = block * j->hk + h;
            for (int32_t c = 0; c < j->d; ++c)
                j->v_cache[(page * j->d + c) * j->bs + offset] = vcodes[c];
            for (int32_t g = 0; g < groups; ++g)
                j->v_scale[(page * groups + g) * j->bs + offset] = vscales[g];
        }
    }
    return NULL;
}

/*
 * kv_store with the key rows normalized and rotated first (or_norm_rope_row;
 * norm_weight NULL skips the norm, rope NULL the rotation), then stored as
 * or_kv_store stores them; values are stored unchanged.  positions [n_tokens]
 * picks each token's row of rope (fp32 [max_pos][rot / 2][2]).  Tokens with a
 * slot beyond the cache or a position outside [0, max_pos) are skipped and
 * counted in the return value.
 */
int64_t or_kv_store_norm_rope(const uint16_t *key, const uint16_t *value,
                              const int64_t *slot_mapping, const int64_t *positions,
                              int64_t n_tokens, int32_t hk, int32_t d,
                              const uint16_t *norm_weight, float eps, const float *rope,
                              int64_t max_pos, int32_t rot, int32_t interleaved,
                              int8_t *k_cache, uint16_t *k_scale, int8_t *v_cache,
                              uint16_t *v_scale, int64_t num_blocks, int32_t bs,
                              int32_t n_threads)
{
    if (n_threads <= 0) n_threads = (int32_t)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    if (n_tokens < (int64_t)n_threads * 64) n_threads = 1;
    or_fused_job jobs[512];
    pthread_t tids[512];
    for (int32_t i = 0; i < n_threads; ++i) {
        or_fused_job j = {key, value, slot_mapping, positions, n_tokens * i / n_threads,
                          n_tokens * (i + 1) / n_threads, hk, d, norm_weight, eps, rope,
                          max_pos, rot, interleaved, k_cache, v_cache, k_scale, v_scale,
                          num_blocks, bs, 0};
        jobs[i] = j;
    }
    for (int32_t i = 0; i < n_threads; ++i)
        pthread_create(&tids[i], NULL, or_fused_worker, &jobs[i]);
    int64_t bad = 0;
    for (int32_t i = 0; i < n_threads; ++i) {
        pthread_join(tids[i], NULL);
        bad += jobs[i].bad;
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Paged attention in fp64                                                   */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;          /* [T, hq, d] bf16 bits */
    int32_t T, hq, hk, d;
    const int8_t *k_cache;
    const uint16_t *k_scale;
    const int8_t *v_cache;
    const uint16_t *v_scale;
    int64_t num_blocks;
    int32_t bs;
    const int32_t *cu_seqlens_q;    /* [S+1] */
    const int32_t *seq_lens;        /* [S] */
    int32_t S;
    const int32_t *block_table;     /* [S, bt_stride] */
    int32_t bt_stride;
    double softmax_scale;
    /* Options (defaults: NULL, 0, 1 -- plain causal attention):
     * sinks   [hq] per-q-head sink logit, in the units of the scaled scores,
     *         added to the softmax denominator only ("triton_turboquant_
     *         unified_attention.py", USE_SINKS: out = sum_i exp(s_i) v_i /
     *         (exp(sink) + sum_i exp(s_i))); NULL = none.
     * window  sliding window W > 0: the query at absolute position p sees
     *         keys p - (W - 1) .. p ("attention_impl.py", window_size =
     *         (sliding_window - 1, 0)); 0 = none.  Causal attention only.
     * causal  1: query i of a sequence sees keys 0 .. seq_len - q_len + i;
     *         0: every query sees keys 0 .. seq_len - 1 (a cached prefix
     *         attended in a pass of its own), seq_len may be below q_len. */
    const float *sinks;
    int32_t window;
    int32_t causal;
    /* Cache format: 0 = q8 (the caches above); 1 = fp8 keys and 4-bit values
     * (or_kv_store_f8v4: k_cache holds e4m3 bits, v_cache nibbles, v_scale
     * and v_zero one fp16 per key; k_scale unused). */
    int32_t fmt;
    const uint16_t *v_zero;
} or_problem;

/* HND row of key j of kv head h of sequence s, through the block table
 * ("attention_impl.py", `_cache_seq`: page j / bs, offset j % bs), or -1
 * when the table entry is missing or out of range. */
static int64_t or_kv_row(const or_problem *p, int32_t s, int32_t h, int64_t j)
{
    int64_t page = j / p->bs;
    int64_t off = j % p->bs;
    if (page >= p->bt_stride) return -1;
    int64_t blk = p->block_table[(int64_t)s * p->bt_stride + page];
    if (blk < 0 || blk >= p->num_blocks) return -1;
    return (blk * p->hk + h) * p->bs + off;
}

/* Dequantized channel c of the K row `row`: code * scale, exact in fp64
 * ("shared/attention_kit.py", `dequantize_q8_into`). */
static double or_dequant_k(const or_problem *p, int64_t row, int32_t c)
{
    if (p->fmt == 1)  /* fp8 key: the e4m3 value itself */
        return (double)or_e4m3_to_f32((uint8_t)p->k_cache[row * p->d + c]);
    int32_t groups = p->d / OR_GROUP;
    double code = (double)p->k_cache[row * p->d + c];
    double sc = (double)or_f16_to_f32(p->k_scale[row * groups + c / OR_GROUP]);
    return code * sc;
}

/* The same for V, whose pages are channel-major: page = row / bs, offset =
 * row % bs. */
static double or_dequant_v(const or_problem *p, int64_t row, int32_t c)
{
    if (p->fmt == 1) {  /* 4-bit value: idx * scale + zero, exact in fp64 */
        int64_t page = row / p->bs, off = row % p->bs;
        uint8_t byte = (uint8_t)p->v_cache[(page * p->d + c) * (p->bs / 2) + off / 2];
        double idx = (double)((byte >> (4 * (off & 1))) & 0xf);
        return idx * (double)or_f16_to_f32(p->v_scale[page * p->bs + off]) +
               (double)or_f16_to_f32(p->v_zero[page * p->bs + off]);
    }
    int32_t groups = p->d / OR_GROUP;
    int64_t page = row / p->bs, off = row % p->bs;
    double code = (double)p->v_cache[(page * p->d + c) * p->bs + off];
    double sc = (double)or_f16_to_f32(p->v_scale[(page * groups + c / OR_GROUP) * p->bs + off]);
    return code * sc;
}

/* Sequence of token t: the s with cu[s] <= t < cu[s+1] (linear scan). */
static int32_t or_seq_of_token(const or_problem *p, int32_t t)
{
    for (int32_t s = 0; s < p->S; ++s)
        if (p->cu_seqlens_q[s] <= t && t < p->cu_seqlens_q[s + 1]) return s;
    return -1;
}

/*
 * Attention of one (token t, q head h) over the visible keys j in [lo, hi):
 * visible means j <= context_len + i, context_len = seq_len - q_len,
 * i = t - cu[s] ("triton_turboquant_unified_attention.py", causal mask;
 * "attention_impl.py", `_sdpa_one` with key_offset = k_len - q_len).
 * GQA: q head h reads kv head h / (hq / hk).
 * Returns the partial triple (m, l, acc): m = max score, l = sum exp(s - m),
 * acc = sum exp(s - m) * v.  An empty range gives m = -inf, l = 0, acc = 0.
 * scores: scratch of at least hi - lo doubles.
 */
static int or_partial(const or_problem *p, int32_t t, int32_t h, int64_t lo,
                      int64_t hi, double *scores, double *m_out, double *l_out,
                      double *acc)
{
    int err = 0;
    int32_t s = or_seq_of_token(p, t);
    if (s < 0) return 1;
    int32_t q_len = p->cu_seqlens_q[s + 1] - p->cu_seqlens_q[s];
    int64_t ctx = (int64_t)p->seq_lens[s] - q_len;
    int64_t i = t - p->cu_seqlens_q[s];
    int64_t last = ctx + i;                     /* last visible key */
    if (!p->causal) {
        last = (int64_t)p->seq_lens[s] - 1;
    } else {
        if (ctx < 0) return 1;
        if (p->window > 0 && lo < last - (p->window - 1)) lo = last - (p->window - 1);
    }
    if (hi > last + 1) hi = last + 1;
    int32_t kvh = h / (p->hq / p->hk);
    const uint16_t *qrow = p->q + ((int64_t)t * p->hq + h) * p->d;
    for (int32_t c = 0; c < p->d; ++c) acc[c] = 0.0;
    if (hi <= lo) { *m_out = -INFINITY; *l_out = 0.0; return 0; }
    double m = -INFINITY;
    for (int64_t j = lo; j < hi; ++j) {
        int64_t row = or_kv_row(p, s, kvh, j);
        double dot = 0.0;
        if (row < 0) err = 1;
        else
            for (int32_t c = 0; c < p->d; ++c)
                dot += (double)or_bf16_to_f32(qrow[c]) *
                       or_dequant_k(p, row, c);
        scores[j - lo] = p->softmax_scale * dot;
        if (scores[j - lo] > m) m = scores[j - lo];
    }
    double l = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        int64_t row = or_kv_row(p, s, kvh, j);
        double w = exp(scores[j - lo] - m);
        l += w;
        if (row >= 0)
            for (int32_t c = 0; c < p->d; ++c)
                acc[c] += w * or_dequant_v(p, row, c);
    }
    *m_out = m;
    *l_out = l;
    return err;
}

/*
 * Merge of partial triples over disjoint key sets (the online-softmax rule of
 * the split-KV segments, and "shared/attention_kit.py" `_merge_lse_` in
 * natural-log form):
 *   M = max_k m_k;  w_k = exp(m_k - M)  (0 for an empty part);
 *   out = sum_k w_k acc_k / sum_k w_k l_k;  lse = M + ln sum_k w_k l_k.
 */
void or_merge_partials(int32_t n, const double *m, const double *l,
                       const double *acc, int32_t d, double *out, double *lse)
{
    double M = -INFINITY;
    for (int32_t k = 0; k < n; ++k) if (m[k] > M) M = m[k];
    double L = 0.0;
    for (int32_t c = 0; c < d; ++c) out[c] = 0.0;
    for (int32_t k = 0; k < n; ++k) {
        if (m[k] == -INFINITY) continue;
        double w = exp(m[k] - M);
        L += w * l[k];
        for (int32_t c = 0; c < d; ++c) out[c] += w * acc[(int64_t)k * d + c];
    }
    for (int32_t c = 0; c < d; ++c) out[c] /= L;
    *lse = M + log(L);
}

/*
 * Merge of two normalized attention results over disjoint key sets, row by
 * row ("shared/attention_kit.py" `_merge_lse_(out, lse, other, other_lse)`,
 * natural-log LSE):
 *   M = max(lse_a, lse_b);  e_x = exp(lse_x - M);
 *   out = (e_a out_a + e_b out_b) / (e_a + e_b);  lse = M + ln(e_a + e_b).
 * Rows with both LSEs -inf (no key on either side) get out = 0, lse = -inf.
 * out_a, out_b, out [rows, d]; lse_a, lse_b, lse [rows]; fp64 throughout.
 */
void or_merge_states(int64_t rows, int32_t d, const double *out_a, const double *lse_a,
                     const double *out_b, const double *lse_b, double *out, double *lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double a = lse_a[r], b = lse_b[r];
        const double M = a > b ? a : b;
        double *o = out + r * d;
        if (M == -INFINITY) {
            for (int32_t c = 0; c < d; ++c) o[c] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        const double ea = exp(a - M), eb = exp(b - M);
        const double sum = ea + eb;
        for (int32_t c = 0; c < d; ++c)
            o[c] = (ea * out_a[r * d + c] + eb * out_b[r * d + c]) / sum;
        lse[r] = M + log(sum);
    }
}

typedef struct {
    const or_problem *p;
    const int64_t *rows;     /* row r = token * hq + head */
    int64_t n_rows;
    int64_t next;            /* shared work counter */
    pthread_mutex_t lock;
    double *out, *lse;
    int64_t max_keys;
    int errors;
} or_job;

static void *or_worker(void *arg)
{
    or_job *job = (or_job *)arg;
    const or_problem *p = job->p;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(job->max_keys + 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)p->d);
    int errors = 0;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t k = job->next++;
        pthread_mutex_unlock(&job->lock);
        if (k >= job->n_rows) break;
        int64_t r = job->rows ? job->rows[k] : k;
        int32_t t = (int32_t)(r / p->hq), h = (int32_t)(r % p->hq);
        double m, l;
        errors |= or_partial(p, t, h, 0, job->max_keys, scores, &m, &l, acc);
        if (p->sinks) {
            /* the sink logit joins the denominator with no value */
            double sink = (double)p->sinks[h];
            if (sink > m) {
                double r = exp(m - sink);  /* 0 when the row has no key */
                l *= r;
                for (int32_t c = 0; c < p->d; ++c) acc[c] *= r;
                m = sink;
            }
            if (m > -INFINITY) l += exp(sink - m);
        }
        if (l == 0.0) {
            /* no key and no sink: out = 0, lse = -inf */
            for (int32_t c = 0; c < p->d; ++c) job->out[k * p->d + c] = 0.0;
            job->lse[k] = -INFINITY;
            continue;
        }
        /* one part: out = acc / l, lse = m + ln l */
        or_merge_partials(1, &m, &l, acc, p->d, job->out + k * p->d, job->lse + k);
    }
    pthread_mutex_lock(&job->lock);
    job->errors |= errors;
    pthread_mutex_unlock(&job->lock);
    free(scores);
    free(acc);
    return NULL;
}

static int or_run_rows(const or_problem *pp, const int64_t *rows, int64_t n_rows,
                       double *out, double *lse, int32_t n_threads);

/*
 * Full attention for the listed rows (row = token * hq + q head; rows == NULL
 * means all T * hq rows in order).  out [n_rows, d] and lse [n_rows] fp64.
 * n_threads <= 0 uses every online core.  Returns 0, or 1 when a row's
 * metadata was invalid (its result is then meaningless).
 */
int or_paged_attention(const uint16_t *q, int32_t T, int32_t hq, int32_t hk,
                       int32_t d, const int8_t *k_cache, const uint16_t *k_scale,
                       const int8_t *v_cache, const uint16_t *v_scale,
                       int64_t num_blocks, int32_t bs, const int32_t *cu_seqlens_q,
                       const int32_t *seq_lens, int32_t S,
                       const int32_t *block_table, int32_t bt_stride,
                       float softmax_scale, const int64_t *rows, int64_t n_rows,
                       double *out, double *lse, int32_t n_threads)
{
    or_problem p = {q, T, hq, hk, d, k_cache, k_scale, v_cache, v_scale,
                    num_blocks, bs, cu_seqlens_q, seq_lens, S, block_table,
                    bt_stride, (double)softmax_scale, NULL, 0, 1, 0, NULL};
    return or_run_rows(&p, rows, n_rows, out, lse, n_threads);
}

/*
 * or_paged_attention with the options of or_problem: per-q-head sinks (or
 * NULL), a sliding window (0 = none; causal only), causal (1) or
 * full-prefix (0) visibility, and the cache format (fmt, v_zero).  A row that sees no key and has no sink gets
 * out = 0 and lse = -inf; with a sink, lse = ln(exp(sink) + sum exp(s_i)).
 * Returns 0, 1 on invalid metadata, 2 on an invalid option.
 */
int or_paged_attention_ex(const uint16_t *q, int32_t T, int32_t hq, int32_t hk,
                          int32_t d, const int8_t *k_cache, const uint16_t *k_scale,
                          const int8_t *v_cache, const uint16_t *v_scale,
                          int64_t num_blocks, int32_t bs, const int32_t *cu_seqlens_q,
                          const int32_t *seq_lens, int32_t S,
                          const int32_t *block_table, int32_t bt_stride,
                          float softmax_scale, const float *sinks, int32_t window,
                          int32_t causal, int32_t fmt, const uint16_t *v_zero,
                          const int64_t *rows, int64_t n_rows,
                          double *out, double *lse, int32_t n_threads)
{
    if (window < 0 || (window > 0 && !causal) || fmt < 0 || fmt > 1 || (fmt == 1 && !v_zero))
        return 2;
    or_problem p = {q, T, hq, hk, d, k_cache, k_scale, v_cache, v_scale,
                    num_blocks, bs, cu_seqlens_q, seq_lens, S, block_table,
                    bt_stride, (double)softmax_scale, sinks, window, causal ? 1 : 0,
                    fmt, v_zero};
    return or_run_rows(&p, rows, n_rows, out, lse, n_threads);
}

static int or_run_rows(const or_problem *pp, const int64_t *rows, int64_t n_rows,
                       double *out, double *lse, int32_t n_threads)
{
    or_problem p = *pp;
    int32_t T = p.T, hq = p.hq, S = p.S;
    const int32_t *seq_lens = p.seq_lens;
    if (!rows) n_rows = (int64_t)T * hq;
    int64_t max_keys = 1;
    for (int32_t s = 0; s < S; ++s) if (seq_lens[s] > max_keys) max_keys = seq_lens[s];
    or_job job;
    job.p = &p; job.rows = rows; job.n_rows = n_rows; job.next = 0;
    job.out = out; job.lse = lse; job.max_keys = max_keys; job.errors = 0;
    pthread_mutex_init(&job.lock, NULL);
    if (n_threads <= 0) n_threads = (int32_t)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    pthread_t tids[512];
    for (int32_t i = 0; i < n_threads; ++i) pthread_create(&tids[i], NULL, or_worker, &job);
    for (int32_t i = 0; i < n_threads; ++i) pthread_join(tids[i], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.errors;
}

/*
 * Partial triple of one row over keys [lo, hi) (split-KV segment), for the
 * merge identities.  acc [d].
 */
int or_attention_partial(const uint16_t *q, int32_t T, int32_t hq, int32_t hk,
                         int32_t d, const int8_t *k_cache, const uint16_t *k_scale,
                         const int8_t *v_cache, const uint16_t *v_scale,
                         int64_t num_blocks, int32_t bs,
                         const int32_t *cu_seqlens_q, const int32_t *seq_lens,
                         int32_t S, const int32_t *block_table, int32_t bt_stride,
                         float softmax_scale, int32_t token, int32_t head,
                         int64_t lo, int64_t hi, double *m, double *l, double *acc)
{
    or_problem p = {q, T, hq, hk, d, k_cache, k_scale, v_cache, v_scale,
                    num_blocks, bs, cu_seqlens_q, seq_lens, S, block_table,
                    bt_stride, (double)softmax_scale, NULL, 0, 1, 0, NULL};
    int64_t n = hi > lo ? hi - lo : 1;
    double *scores = (double *)malloc(sizeof(double) * (size_t)n);
    int err = or_partial(&p, token, head, lo, hi, scores, m, l, acc);
    free(scores);
    return err;
}
