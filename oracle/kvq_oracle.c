/*
 * kvq_oracle.c -- plain CPU oracle for the block-quantized KV cache and the
 * single-token decode attention that reads it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only through seeded synthetic inputs.
 *
 * What it follows (the pages are three scraped articles on DeepSeek-R1
 * inference tuning):
 *   - "DeepSeek-R1 inference latency ... hardware-aware scheduling"
 *     (jsqmd.com/news/887038), section 2.1 "KV Cache block compression on the
 *     A100 bandwidth bottleneck", the function quantize_block: per block of
 *     64 rows, scale = max|x| / 7.5, codes = round(x / scale) clamped to
 *     [-8, 7] and stored as 8-bit integers.
 *   - "DeepSeek R1 performance overview" (aicoding.csdn.net), section 2.2
 *     "KV Cache dynamic compression": symmetric per-chunk INT8 quantization
 *     with a scale taken from a prior per-chunk extrema pass, and section 3.1,
 *     where decode reads an INT8 KV cache.
 *   - "DeepSeek R1 performance tips" (ddd.cn), section 4: KV pages addressed
 *     through a block table (vLLM PagedAttention); section 1: an FP8 KV cache
 *     as the default on Blackwell.
 *   - "hardware-aware scheduling" (jsqmd.com/news/887038), section 2.2: FP8
 *     E4M3 with dynamic range scaling driven by max|x|, and its error bound
 *     (half a unit in the last place of the 3-bit fraction).
 *
 * Readings taken where the pages are silent or inconsistent (each is listed in
 * the design notes):
 *   - a block is (sequence, head, 64 consecutive tokens); the tail block of a
 *     sequence uses only its valid rows;
 *   - arithmetic is IEEE binary32: the fp16 input is widened exactly, the
 *     scale is a / 7.5f (int4) or a / 127.0f (int8) rounded to nearest, the
 *     quotient x / scale is rounded to nearest, and rounding to an integer is
 *     half-to-even (nearbyintf under FE_TONEAREST);
 *   - clamp range [-8, 7] for int4 (the code, not the comment), [-127, 127]
 *     for int8; no zero-point;
 *   - an all-zero block has scale 0 and all codes 0;
 *   - int4 codes are packed two to a byte, the even element of the head
 *     dimension in the low nibble, as 4-bit two's complement; int8 codes are
 *     one two's-complement byte each;
 *   - FP8: the same block, scale = a / 448.0f (448 = the largest finite E4M3
 *     value, so max|x| maps to the top of the format), code = E4M3 of the
 *     binary32 quotient x / scale rounded to nearest, ties to the even
 *     fraction, saturating at +-448, sign kept (a quotient that rounds to
 *     zero keeps its sign); an all-zero block has scale 0 and codes 0x00;
 *   - decode attention is exact softmax attention of one query per
 *     (sequence, head) over the dequantized keys and values k^ = code * scale,
 *     evaluated here in binary64; an empty sequence yields a zero output.
 *
 * Build flags matter: -O2 -fno-fast-math -ffp-contract=off (see oracle/build.py).
 */
#include <float.h>
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs binary32 expressions evaluated in binary32 (FLT_EVAL_METHOD == 0)"
#endif

#define ORC_INT4 0
#define ORC_INT8 1
#define ORC_FP8 2
#define ORC_BLOCK 64

/* ---------------------------------------------------------------------------
 * binary16 -> binary32, written out from the IEEE 754 binary16 layout
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).  Exact for
 * every finite value, subnormals and signed zeros included.
 * ------------------------------------------------------------------------- */
float orc_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float v;
    if (e == 0) {
        v = ldexpf((float)m, -24);                 /* subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexpf((float)(m | 0x400), e - 25);    /* (1024 + m) * 2^(e-15-10) */
    }
    return sign ? -v : v;
}

/* ---------------------------------------------------------------------------
 * FP8 E4M3 (the OCP 8-bit format NVIDIA's E4M3 follows): 1 sign bit, 4
 * exponent bits with bias 7, 3 fraction bits; exponent field 0 holds the
 * subnormals f/8 * 2^-6; exponent field 15 with fraction 7 is NaN; there are no
 * infinities, so the largest finite value is 1.75 * 2^8 = 448 (0x7e).
 * ------------------------------------------------------------------------- */
double orc_e4m3_to_double(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 0xf;
    int f = c & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) v = ldexp((double)f, -9);          /* f/8 * 2^-6 */
    else v = ldexp((double)(8 + f), e - 10);       /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

/*
 * binary32 -> E4M3, round to nearest with ties to the even fraction,
 * saturating: the code whose value is nearest to |y| among the 127 finite
 * non-negative codes 0x00..0x7e (their values increase with the code), the
 * even one of two equally near, then y's sign bit.  Found by bisection over
 * that ordered table; |y| above 448 gets 0x7e.
 */
#define TAB(c) orc_e4m3_to_double((uint8_t)(c))
uint8_t orc_float_to_e4m3(float y)
{
    double ay = fabs((double)y);
    int lo = 0, hi = 126;
    if (ay >= TAB(126)) {
        lo = 126;
    } else {
        while (hi - lo > 1) {                  /* TAB(lo) <= ay < TAB(hi) */
            int mid = (lo + hi) / 2;
            if (TAB(mid) <= ay) lo = mid; else hi = mid;
        }
    }
    int c = lo;                                /* the nearer of lo and lo + 1; a tie goes to the even code */
    if (lo < 126) {
        double dlo = ay - TAB(lo), dhi = TAB(lo + 1) - ay;
        if (dhi < dlo || (dhi == dlo && ((lo + 1) & 1) == 0)) c = lo + 1;
    }
    return (uint8_t)(c | (signbit(y) ? 0x80 : 0));
}
#undef TAB

/* ---------------------------------------------------------------------------
 * One block of quantize_block.
 *   x      : pointer to row 0, element 0 of the block (fp16 bits)
 *   rows   : number of valid rows (1..64); rows beyond it get code 0
 *   row_stride : elements between consecutive rows
 *   D      : head dimension (elements per row)
 *   out    : codes of the block, 64 rows of D/2 (int4) or D (int8) bytes
 * returns the scale
 * ------------------------------------------------------------------------- */
static float quantize_one_block(int fmt, const uint16_t *x, int rows, int64_t row_stride,
                                int D, uint8_t *out)
{
    /* step 1: a = max |x| over the valid rows */
    float a = 0.0f;
    for (int r = 0; r < rows; r++)
        for (int d = 0; d < D; d++) {
            float v = fabsf(orc_half_to_float(x[r * row_stride + d]));
            if (v > a) a = v;
        }
    /* step 2: the scale */
    float scale = (fmt == ORC_INT4) ? a / 7.5f : (fmt == ORC_INT8) ? a / 127.0f : a / 448.0f;
    int lo = (fmt == ORC_INT4) ? -8 : -127;
    int hi = (fmt == ORC_INT4) ? 7 : 127;
    int row_bytes = (fmt == ORC_INT4) ? D / 2 : D;
    memset(out, 0, (size_t)ORC_BLOCK * row_bytes);
    if (scale == 0.0f) return scale;               /* all-zero block: every code 0 */
    if (fmt == ORC_FP8) {                          /* step 3 in E4M3: round the quotient to the format */
        for (int r = 0; r < rows; r++)
            for (int d = 0; d < D; d++) {
                float y = orc_half_to_float(x[r * row_stride + d]) / scale;
                out[r * row_bytes + d] = orc_float_to_e4m3(y);
            }
        return scale;
    }
    /* step 3: codes = clamp(round_half_even(x / scale)) and step 4: store */
    for (int r = 0; r < rows; r++) {
        for (int d = 0; d < D; d++) {
            float xv = orc_half_to_float(x[r * row_stride + d]);
            float y = xv / scale;
            float rq = nearbyintf(y);
            int q = (int)rq;
            if (q < lo) q = lo;
            if (q > hi) q = hi;
            if (fmt == ORC_INT4) {
                uint8_t nib = (uint8_t)(q & 0xf);
                uint8_t *byte = &out[r * row_bytes + d / 2];
                if (d % 2 == 0) *byte = (uint8_t)((*byte & 0xf0) | nib);
                else            *byte = (uint8_t)((*byte & 0x0f) | (nib << 4));
            } else {
                out[r * row_bytes + d] = (uint8_t)(int8_t)q;
            }
        }
    }
    return scale;
}

/*
 * Quantize a contiguous tensor x[T][H][D] (fp16 bits) block by block.
 *   codes  : [ceil(T/64)][H][64][D/2 or D]
 *   scales : [ceil(T/64)][H]
 * returns 0, or -1 on bad arguments.
 */
int orc_quantize(int fmt, const uint16_t *x, int64_t T, int32_t H, int32_t D,
                 uint8_t *codes, float *scales)
{
    if ((fmt != ORC_INT4 && fmt != ORC_INT8 && fmt != ORC_FP8) || T < 0 || H <= 0 || D <= 0 || (D % 2))
        return -1;
    fesetround(FE_TONEAREST);
    int row_bytes = (fmt == ORC_INT4) ? D / 2 : D;
    int64_t nb = (T + ORC_BLOCK - 1) / ORC_BLOCK;
    for (int64_t j = 0; j < nb; j++) {
        int rows = (int)((T - j * ORC_BLOCK) < ORC_BLOCK ? (T - j * ORC_BLOCK) : ORC_BLOCK);
        for (int h = 0; h < H; h++) {
            const uint16_t *src = x + (j * ORC_BLOCK * H + h) * (int64_t)D;
            uint8_t *dst = codes + ((j * H + h) * (int64_t)ORC_BLOCK) * row_bytes;
            scales[j * H + h] = quantize_one_block(fmt, src, rows, (int64_t)H * D, D, dst);
        }
    }
    return 0;
}

/* the value of the code of element (row, d) of one (page, head) code block
 * (a signed integer for int4 / int8, an E4M3 value for FP8), exact in binary64 */
static double code_at(int fmt, const uint8_t *blk, int D, int row, int d)
{
    if (fmt == ORC_INT4) {
        uint8_t byte = blk[row * (D / 2) + d / 2];
        int nib = (d % 2 == 0) ? (byte & 0xf) : (byte >> 4);
        return nib >= 8 ? nib - 16 : nib;
    }
    if (fmt == ORC_FP8) return orc_e4m3_to_double(blk[row * D + d]);
    return (int)(int8_t)blk[row * D + d];
}

/*
 * Dequantize the keys and values of one (sequence, head) from the paged cache
 * into binary64 arrays kh[L][D], vh[L][D]: element = code * scale.
 */
static void gather_dequant(int fmt, int32_t H, int32_t D, const uint8_t *k_codes,
                           const uint8_t *v_codes, const float *k_scales, const float *v_scales,
                           const int32_t *bt_row, int32_t L, int32_t h, double *kh, double *vh)
{
    int row_bytes = (fmt == ORC_INT4) ? D / 2 : D;
    size_t blk_bytes = (size_t)ORC_BLOCK * row_bytes;
    for (int32_t t = 0; t < L; t++) {
        int32_t page = bt_row[t / ORC_BLOCK];
        int row = t % ORC_BLOCK;
        const uint8_t *kb = k_codes + ((size_t)page * H + h) * blk_bytes;
        const uint8_t *vb = v_codes + ((size_t)page * H + h) * blk_bytes;
        double sk = (double)k_scales[(size_t)page * H + h];
        double sv = (double)v_scales[(size_t)page * H + h];
        for (int d = 0; d < D; d++) {
            kh[(size_t)t * D + d] = code_at(fmt, kb, D, row, d) * sk;
            vh[(size_t)t * D + d] = code_at(fmt, vb, D, row, d) * sv;
        }
    }
}

/* the attention of one query over token range [t0, t1): running max m,
 * denominator l and unnormalised numerator acc[D] (binary64) */
static void attend_range(const double *qv, const double *kh, const double *vh, int D,
                         int32_t t0, int32_t t1, double softmax_scale,
                         double *m_out, double *l_out, double *acc)
{
    double m = -INFINITY;
    for (int32_t t = t0; t < t1; t++) {
        double s = 0.0;
        for (int d = 0; d < D; d++) s += qv[d] * kh[(size_t)t * D + d];
        s *= softmax_scale;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int d = 0; d < D; d++) acc[d] = 0.0;
    for (int32_t t = t0; t < t1; t++) {
        double s = 0.0;
        for (int d = 0; d < D; d++) s += qv[d] * kh[(size_t)t * D + d];
        s *= softmax_scale;
        double p = exp(s - m);
        l += p;
        for (int d = 0; d < D; d++) acc[d] += p * vh[(size_t)t * D + d];
    }
    *m_out = m;
    *l_out = l;
}

/*
 * Decode attention over the paged cache, binary64 throughout:
 *   s_t = softmax_scale * sum_d q_d * k^_{t,d};  p = softmax(s);  o_d = sum_t p_t v^_{t,d}
 *
 * Grouped query heads: the cache holds Hkv heads and q holds Hq = g * Hkv
 * heads; query head i reads cache head i / g (consecutive query heads share a
 * cache head, the grouping of grouped-query / multi-query attention).  g = 1
 * is plain multi-head attention.
 *
 * num_splits <= 1 evaluates the definition directly.  num_splits > 1 cuts the
 * tokens of every (sequence, head) into that many contiguous ranges, evaluates
 * (m_i, l_i, acc_i) per range and merges them:
 *   m = max m_i,  l = sum l_i e^(m_i - m),  o = sum acc_i e^(m_i - m) / l
 * which equals the direct result up to rounding; tests use it to pin the merge
 * step of split decoding.
 *
 *   codes   : [num_pages][Hkv][64][D/2 or D];  scales : [num_pages][Hkv]
 *   block_table : [B][max_blocks]  page of block j of sequence b
 *   seq_lens    : [B]
 *   q           : fp16 bits [B][Hq][D]
 *   out         : binary64 [B][Hq][D]
 * returns 0, or -1 on bad arguments (Hq not a multiple of Hkv, a block-table
 * entry outside [0, num_pages) or a length beyond max_blocks * 64).
 */
int orc_decode_attention_gqa(int fmt, int32_t Hkv, int32_t Hq, int32_t D, int32_t num_pages,
                             const uint8_t *k_codes, const uint8_t *v_codes,
                             const float *k_scales, const float *v_scales,
                             const int32_t *block_table, int32_t max_blocks,
                             const int32_t *seq_lens, int32_t B, const uint16_t *q,
                             double softmax_scale, int32_t num_splits, double *out)
{
    if ((fmt != ORC_INT4 && fmt != ORC_INT8 && fmt != ORC_FP8) || Hkv <= 0 || Hq <= 0 || (Hq % Hkv) || D <= 0 || (D % 2) || B < 0)
        return -1;
    const int32_t g = Hq / Hkv;
    for (int32_t b = 0; b < B; b++) {
        int32_t L = seq_lens[b];
        if (L < 0 || L > max_blocks * ORC_BLOCK) return -1;
        for (int32_t j = 0; j < (L + ORC_BLOCK - 1) / ORC_BLOCK; j++) {
            int32_t pg = block_table[(size_t)b * max_blocks + j];
            if (pg < 0 || pg >= num_pages) return -1;
        }
    }
    double *qv = (double *)malloc(sizeof(double) * D);
    double *o = (double *)malloc(sizeof(double) * D);
    for (int32_t b = 0; b < B; b++) {
        int32_t L = seq_lens[b];
        double *kh = (double *)malloc(sizeof(double) * ((size_t)L * D + 1));
        double *vh = (double *)malloc(sizeof(double) * ((size_t)L * D + 1));
        for (int32_t hq = 0; hq < Hq; hq++) {
            const int32_t h = hq / g;  /* the cache head this query head reads */
            double *dst = out + ((size_t)b * Hq + hq) * D;
            if (L == 0) {
                for (int d = 0; d < D; d++) dst[d] = 0.0;
                continue;
            }
            gather_dequant(fmt, Hkv, D, k_codes, v_codes, k_scales, v_scales,
                           block_table + (size_t)b * max_blocks, L, h, kh, vh);
            for (int d = 0; d < D; d++)
                qv[d] = (double)orc_half_to_float(q[((size_t)b * Hq + hq) * D + d]);
            int32_t S = num_splits < 1 ? 1 : num_splits;
            if (S > L) S = L;
            double m_all = -INFINITY, l_all = 0.0;
            double *ms = (double *)malloc(sizeof(double) * S);
            double *ls = (double *)malloc(sizeof(double) * S);
            double *accs = (double *)malloc(sizeof(double) * S * D);
            for (int32_t i = 0; i < S; i++) {
                int32_t t0 = (int32_t)((int64_t)L * i / S);
                int32_t t1 = (int32_t)((int64_t)L * (i + 1) / S);
                attend_range(qv, kh, vh, D, t0, t1, softmax_scale, &ms[i], &ls[i], accs + (size_t)i * D);
                if (ms[i] > m_all) m_all = ms[i];
            }
            for (int d = 0; d < D; d++) o[d] = 0.0;
            for (int32_t i = 0; i < S; i++) {
                double w = exp(ms[i] - m_all);
                l_all += ls[i] * w;
                for (int d = 0; d < D; d++) o[d] += accs[(size_t)i * D + d] * w;
            }
            for (int d = 0; d < D; d++) dst[d] = o[d] / l_all;
            free(ms);
            free(ls);
            free(accs);
        }
        free(kh);
        free(vh);
    }
    free(qv);
    free(o);
    return 0;
}

/* multi-head attention: every query head has its own cache head (g = 1) */
int orc_decode_attention(int fmt, int32_t H, int32_t D, int32_t num_pages,
                         const uint8_t *k_codes, const uint8_t *v_codes,
                         const float *k_scales, const float *v_scales,
                         const int32_t *block_table, int32_t max_blocks,
                         const int32_t *seq_lens, int32_t B, const uint16_t *q,
                         double softmax_scale, int32_t num_splits, double *out)
{
    return orc_decode_attention_gqa(fmt, H, H, D, num_pages, k_codes, v_codes, k_scales, v_scales, block_table,
                                    max_blocks, seq_lens, B, q, softmax_scale, num_splits, out);
}

/*
 * max over (t, d) of |v^_{t,d}| for every (sequence, head): the normaliser of
 * the attention error measure.  out: binary64 [B][H]
 */
int orc_value_absmax(int fmt, int32_t H, int32_t D, const uint8_t *v_codes, const float *v_scales,
                     const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                     int32_t B, double *out)
{
    int row_bytes = (fmt == ORC_INT4) ? D / 2 : D;
    size_t blk_bytes = (size_t)ORC_BLOCK * row_bytes;
    for (int32_t b = 0; b < B; b++)
        for (int32_t h = 0; h < H; h++) {
            double mx = 0.0;
            for (int32_t t = 0; t < seq_lens[b]; t++) {
                int32_t page = block_table[(size_t)b * max_blocks + t / ORC_BLOCK];
                const uint8_t *vb = v_codes + ((size_t)page * H + h) * blk_bytes;
                double sv = (double)v_scales[(size_t)page * H + h];
                for (int d = 0; d < D; d++) {
                    double v = fabs(code_at(fmt, vb, D, t % ORC_BLOCK, d) * sv);
                    if (v > mx) mx = v;
                }
            }
            out[(size_t)b * H + h] = mx;
        }
    return 0;
}
