/*
 * kvq_oracle.c -- plain, slow, single-threaded CPU oracle for low-bit KV-cache
 * decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant generator with the CUDA path in
 * bit_kv_cache_07_gb300/csrc; both are written independently from the same
 * description of the method.
 *
 * Everything here works on ONE stream: one (batch row, KV head) pair, with
 * its T tokens of K and V (fp16, [T][d]) and the g query heads that share
 * that KV head.  The Python wrapper (oracle/kvq_oracle.py) loops streams.
 *
 * Sources (page title, section):
 *  - "KVTuner" review, observation 2: K per-channel asymmetric quantization;
 *    "Intra-Layer KV Cache Quantization Precision Pair Pruning": the pairs
 *    KV8, K8V4, KV4, K4V2, KV2.
 *  - KVQuant (arXiv 2401.18079) abstract + "technical approach": per-channel
 *    K, pre-RoPE K, non-uniform (NUQ) datatypes, per-vector dense-and-sparse
 *    outliers (~1 %).
 *  - InnerQ (arXiv 2602.23200), "Methodology" 1-4: per-token groups along the
 *    hidden dimension (64 channels), min/max per group with a shared scale,
 *    fp16 windows of recent and sink tokens.
 *  - "Hadamard rotation-based 2-bit quantization for KV cache compression":
 *    rotate V with a Hadamard matrix, quantize uniformly to 2 bits, apply the
 *    inverse after the attention sum.
 * The uniform quantizer (min/max per group, one shared scale) computes
 * scale=(max-min)/(2^b-1) and code=clamp(rint((x-min)/scale),0,2^b-1) in
 * fp32, correctly rounded step by step; attention is computed in fp64.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math.
 * -ffp-contract=off matters: the fp32 quantizer must not fuse into FMA.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 <-> binary32, written from the format definition.      */
/* ------------------------------------------------------------------------ */

/* Decode a binary16 bit pattern: sign, 5-bit exponent (bias 15), 10-bit
 * fraction.  exp==0 is subnormal (fraction * 2^-24), exp==31 is Inf/NaN. */
float orc_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexpf((float)(f + 1024), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a binary32 value to the nearest binary16, ties to even. */
uint16_t orc_float_to_half(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (isnan(x))
        return 0x7e00;
    if (a == 0.0)
        return sign;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-24, m in [0, 1024] */
        double m = rint(a * ldexp(1.0, 24)); /* exact product, RN-even */
        return (uint16_t)(sign | (uint16_t)m); /* m==1024 encodes 2^-14 */
    }
    int ex;
    frexp(a, &ex);            /* a = fr * 2^ex, fr in [0.5, 1) */
    int E = ex - 1;           /* a in [2^E, 2^(E+1)) */
    double m = rint(ldexp(a, 10 - E)); /* 11-bit significand, RN-even */
    if (m == 2048.0) {        /* rounded up to the next binade */
        m = 1024.0;
        E += 1;
    }
    if (E + 15 >= 31)
        return (uint16_t)(sign | 0x7c00); /* overflow -> Inf */
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(m - 1024.0));
}

/* ------------------------------------------------------------------------ */
/* Uniform asymmetric quantizer (min / scale), one group.                  */
/* ------------------------------------------------------------------------ */

/* Quantize n fp16 values x[i*stride] with b bits.
 *   mn, mx   : min and max of the fp32-widened inputs
 *   scale32  : (mx - mn) / (2^b - 1)                  (fp32, IEEE RN)
 *   code     : clamp(rint((x - mn) / scale32), 0, 2^b - 1)   (fp32, RN-even)
 *   stored   : min_h = fp16(mn) (exact: mn is an input), scale_h = fp16_RN(scale32)
 * A constant group (mx == mn) stores scale 0 and all-zero codes. */
void orc_quantize_uniform(const uint16_t *x, int n, int stride, int bits,
                          uint8_t *code, int code_stride,
                          uint16_t *min_h, uint16_t *scale_h)
{
    float mn = orc_half_to_float(x[0]);
    float mx = mn;
    for (int i = 1; i < n; i++) {
        float v = orc_half_to_float(x[(long)i * stride]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    float qmax = (float)((1 << bits) - 1);
    float scale = (mx - mn) / qmax;
    for (int i = 0; i < n; i++) {
        float v = orc_half_to_float(x[(long)i * stride]);
        int c = 0;
        if (scale != 0.0f) {
            float r = rintf((v - mn) / scale);
            if (r < 0.0f) r = 0.0f;
            if (r > qmax) r = qmax;
            c = (int)r;
        }
        code[(long)i * code_stride] = (uint8_t)c;
    }
    *min_h = orc_float_to_half(mn);
    *scale_h = orc_float_to_half(scale);
}

/* The InnerQ per-group quantizer on fp32 inputs x[i*stride] (i < n), b bits.
 *   mn, mx   : min / max
 *   mean     : (sum of x) / n in fp64 (exact: see below)
 *   symmetric when `hybrid`, mx > mn and |mean| * 2^(b+1) <= mx - mn (the
 *   mean lies within half an asymmetric step of zero: the group is centred):
 *     a       = max(|mn|, |mx|), qs = 2^(b-1) - 1
 *     scale32 = a / qs                                   (fp32 RN)
 *     code    = clamp(rint(x / scale32), -qs, qs) + 2^(b-1)   (fp32, RN-even)
 *     stored  : scale_h = fp16_RN(scale32), min_h = fp16(-2^(b-1) * scale_h),
 *               so that min_h + code * scale_h = (code - 2^(b-1)) * scale_h
 *     (if 2^(b-1) * scale_h overflows fp16 the group falls back to asymmetric)
 *   otherwise asymmetric, as orc_quantize_uniform: scale32 = (mx - mn) / (2^b - 1),
 *     code = clamp(rint((x - mn) / scale32), 0, 2^b - 1), min_h = fp16_RN(mn),
 *     scale_h = fp16_RN(scale32); a constant group stores scale 0, codes 0.
 * The inputs are fp16 values, or fp16 values divided by powers of two up to
 * 2^16 (the key normalisation), so each is an integer multiple of 2^-40 below
 * 2^16 in magnitude and the fp64 sum of n <= 128 of them is exact. */
void orc_quantize_group(const float *x, int n, int stride, int bits, int hybrid,
                        uint8_t *code, int code_stride, uint16_t *min_h, uint16_t *scale_h)
{
    float mn = x[0], mx = x[0];
    double sum = 0.0;
    for (int i = 0; i < n; i++) {
        float v = x[(long)i * stride];
        if (v < mn) mn = v;
        if (v > mx) mx = v;
        sum += (double)v;
    }
    double mean = sum / (double)n;
    if (hybrid && mx > mn && fabs(mean) * (double)(1 << (bits + 1)) <= (double)mx - (double)mn) {
        float a = fabsf(mn) > fabsf(mx) ? fabsf(mn) : fabsf(mx);
        float qs = (float)((1 << (bits - 1)) - 1);
        float scale = a / qs;
        uint16_t sh = orc_float_to_half(scale);
        float mf = -(float)(1 << (bits - 1)) * orc_half_to_float(sh);
        uint16_t mh = orc_float_to_half(mf);
        if (isfinite(orc_half_to_float(mh))) {
            for (int i = 0; i < n; i++) {
                float r = rintf(x[(long)i * stride] / scale);
                if (r < -qs) r = -qs;
                if (r > qs) r = qs;
                code[(long)i * code_stride] = (uint8_t)((int)r + (1 << (bits - 1)));
            }
            *min_h = mh;
            *scale_h = sh;
            return;
        }
    }
    float qmax = (float)((1 << bits) - 1);
    float scale = (mx - mn) / qmax;
    for (int i = 0; i < n; i++) {
        int c = 0;
        if (scale != 0.0f) {
            float r = rintf((x[(long)i * stride] - mn) / scale);
            if (r < 0.0f) r = 0.0f;
            if (r > qmax) r = qmax;
            c = (int)r;
        }
        code[(long)i * code_stride] = (uint8_t)c;
    }
    *min_h = orc_float_to_half(mn);
    *scale_h = orc_float_to_half(scale);
}

/* InnerQ per-channel key normalisation: for each channel c, n_c = 2^e with e
 * the smallest integer such that max_t |K_tc| <= 2^e over the given tokens
 * (1 for an all-zero channel).  A power of two, so K / n_c and q * n_c are
 * exact; |K / n_c| <= 1 on those tokens. */
void orc_key_norm(const uint16_t *K, int T, int d, float *norm)
{
    for (int c = 0; c < d; c++) {
        float m = 0.0f;
        for (int t = 0; t < T; t++) {
            float a = fabsf(orc_half_to_float(K[(size_t)t * d + c]));
            if (a > m) m = a;
        }
        float n = 1.0f;
        if (m > 0.0f) {
            int e;
            frexpf(m, &e);            /* m = f * 2^e, f in [0.5, 1) */
            n = ldexpf(1.0f, e);      /* 2^e >= m */
            if (ldexpf(1.0f, e - 1) >= m) n = ldexpf(1.0f, e - 1);  /* m a power of two */
        }
        norm[c] = n;
    }
}

/* ------------------------------------------------------------------------ */
/* Bit packing: code i of a row occupies bits [b*i, b*i + b) of the row's    */
/* little-endian bitstream (bit 0 = least significant bit of byte 0).       */
/* ------------------------------------------------------------------------ */

void orc_pack_bits(const uint8_t *codes, int n, int bits, uint8_t *out)
{
    int nbytes = (n * bits + 7) / 8;
    memset(out, 0, (size_t)nbytes);
    for (int i = 0; i < n; i++)
        for (int j = 0; j < bits; j++) {
            int bit = (codes[i] >> j) & 1;
            int pos = i * bits + j;
            out[pos / 8] |= (uint8_t)(bit << (pos % 8));
        }
}

void orc_unpack_bits(const uint8_t *in, int n, int bits, uint8_t *codes)
{
    for (int i = 0; i < n; i++) {
        int c = 0;
        for (int j = 0; j < bits; j++) {
            int pos = i * bits + j;
            c |= ((in[pos / 8] >> (pos % 8)) & 1) << j;
        }
        codes[i] = (uint8_t)c;
    }
}

/* ------------------------------------------------------------------------ */
/* Hadamard rotation of one V vector (n a power of two).                     */
/* ------------------------------------------------------------------------ */

/* v' = fp16_RN( c * (H v) ), H the Sylvester Hadamard matrix
 * H[i][j] = (-1)^popcount(i & j), c = fp32(1/sqrt(n)).  H v is evaluated by
 * the fast Walsh-Hadamard butterflies in fp32, stage widths h = 1, 2, 4, ...,
 * n/2; each butterfly maps (a, b) -> (a + b, a - b), every operation RN. */
void orc_hadamard_rotate(const uint16_t *v, int n, uint16_t *out)
{
    float y[1024];
    for (int i = 0; i < n; i++)
        y[i] = orc_half_to_float(v[i]);
    for (int h = 1; h < n; h *= 2)
        for (int i = 0; i < n; i += 2 * h)
            for (int j = i; j < i + h; j++) {
                float a = y[j], b = y[j + h];
                y[j] = a + b;
                y[j + h] = a - b;
            }
    float c = (float)(1.0 / sqrt((double)n));
    for (int i = 0; i < n; i++)
        out[i] = orc_float_to_half(y[i] * c);
}

/* Apply the normalised Hadamard matrix Hn = H / sqrt(n) to an fp64 vector,
 * written as the dense sum over the popcount definition of H.  Hn is
 * symmetric and Hn * Hn = I, so this is also the inverse rotation. */
void orc_hadamard_apply_f64(const double *x, int n, double *out)
{
    double inv = 1.0 / sqrt((double)n);
    for (int i = 0; i < n; i++) {
        double acc = 0.0;
        for (int j = 0; j < n; j++) {
            int neg = __builtin_popcount((unsigned)(i & j)) & 1;
            acc += neg ? -x[j] : x[j];
        }
        out[i] = acc * inv;
    }
}

/* ------------------------------------------------------------------------ */
/* Non-uniform (LUT) 3-bit quantizer with per-vector dense-and-sparse        */
/* outliers, one token vector of n channels.                                 */
/* ------------------------------------------------------------------------ */

/* Outliers: the k entries of largest |x| (ties -> lower channel index),
 * kept as fp16 values with their channel indices in ascending order; their
 * dense code is 0.  Dense part (the other n - k entries):
 *   mn, mx  : min / max (fp32)
 *   s32     : (mx - mn) / (L7 - L0)                     (fp32 RN)
 *   u       : (x - mn) / s32                            (fp32 RN)
 *   tau_i   : (L_i + L_{i+1}) * 0.5 - L0, i = 0..6     (fp32 RN)
 *   code    : #{ i : u > tau_i }   (the nearest LUT level; exact ties go down)
 *   stored  : min_h = fp16(mn), s_h = fp16_RN(s32)
 * A constant dense part (mx == mn) gives s 0 and all-zero codes. */
void orc_nuq_encode(const uint16_t *x, int n, int k, const float *lut,
                    uint8_t *code, uint16_t *min_h, uint16_t *s_h,
                    uint8_t *cols, uint16_t *vals)
{
    unsigned char is_out[1024];
    memset(is_out, 0, sizeof is_out);
    for (int j = 0; j < k; j++) {
        int best = -1;
        float bv = -1.0f;
        for (int i = 0; i < n; i++) {
            if (is_out[i]) continue;
            float a = fabsf(orc_half_to_float(x[i]));
            if (a > bv) { bv = a; best = i; }
        }
        is_out[best] = 1;
    }
    int m = 0;
    for (int i = 0; i < n; i++)
        if (is_out[i]) {
            cols[m] = (uint8_t)i;
            vals[m] = x[i];
            m++;
        }
    float mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < n; i++) {
        if (is_out[i]) continue;
        float v = orc_half_to_float(x[i]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    float span = lut[7] - lut[0];
    float s = (mx - mn) / span;
    float tau[7];
    for (int i = 0; i < 7; i++)
        tau[i] = (lut[i] + lut[i + 1]) * 0.5f - lut[0];
    for (int i = 0; i < n; i++) {
        int c = 0;
        if (!is_out[i] && s != 0.0f) {
            float u = (orc_half_to_float(x[i]) - mn) / s;
            for (int t = 0; t < 7; t++)
                if (u > tau[t]) c++;
        }
        code[i] = (uint8_t)c;
    }
    *min_h = orc_float_to_half(mn);
    *s_h = orc_float_to_half(s);
}

/* Reconstruct one NUQ vector in fp64: x^ = min_h + s_h * (L_code - L0) on the
 * dense part, the stored fp16 value on the outlier channels. */
void orc_nuq_decode(const uint8_t *code, int n, uint16_t min_h, uint16_t s_h,
                    const float *lut, int k, const uint8_t *cols,
                    const uint16_t *vals, double *out)
{
    double mn = orc_half_to_float(min_h), s = orc_half_to_float(s_h);
    for (int i = 0; i < n; i++)
        out[i] = mn + s * ((double)lut[code[i]] - (double)lut[0]);
    for (int j = 0; j < k; j++)
        out[cols[j]] = orc_half_to_float(vals[j]);
}

/* ------------------------------------------------------------------------ */
/* RoPE (rotate-half convention), fp64.                                      */
/* ------------------------------------------------------------------------ */

/* theta_i = base^(-2i/d) for i < d/2; channel pairs (i, i + d/2):
 *   x'_i       = x_i cos(t theta_i) - x_{i+d/2} sin(t theta_i)
 *   x'_{i+d/2} = x_{i+d/2} cos(t theta_i) + x_i sin(t theta_i)          */
void orc_rope_apply(double *x, int d, double pos, double base)
{
    int half = d / 2;
    for (int i = 0; i < half; i++) {
        double th = pow(base, -2.0 * (double)i / (double)d);
        double c = cos(pos * th), s = sin(pos * th);
        double a = x[i], b = x[i + half];
        x[i] = a * c - b * s;
        x[i + half] = b * c + a * s;
    }
}

/* ------------------------------------------------------------------------ */
/* Cache layout rule (which tokens are fp16, which are quantized).           */
/* ------------------------------------------------------------------------ */

typedef struct orc_cfg {
    int32_t d;            /* head dim */
    int32_t k_bits;       /* 2,4,8 uniform; 3 NUQ; 16 fp16 (then v_bits 16) */
    int32_t v_bits;
    int32_t gk;           /* K group: tokens per group (per-channel K) */
    int32_t gv;           /* V group: channels per group (per-token V) */
    int32_t n_sink;       /* S */
    int32_t n_recent;     /* R */
    int32_t v_hadamard;   /* rotate V before quantizing */
    int32_t k_pre_rope;   /* K stored before RoPE; rotate after dequant */
    int32_t outliers;     /* NUQ outliers per vector */
    double rope_theta;
    double sm_scale;      /* softmax scale (1/sqrt(d) when 0) */
    float k_lut[8];
    float v_lut[8];
    int32_t pos_offset;   /* absolute position of the stream's first token (a
                             context shard that starts later); RoPE angles use
                             pos_offset + t */
    int32_t gkc;          /* InnerQ K layout: per token, groups of gkc channels
                             along the hidden dimension (0: per channel over gk
                             tokens) */
    int32_t hybrid;       /* InnerQ: every uniform group picks a symmetric or an
                             asymmetric grid from its own statistics */
    int32_t k_norm;       /* InnerQ: per-channel key normalisation (InnerQ K
                             layout only) */
    int32_t norm_tokens;  /* the first norm_tokens tokens (the prefill) fix the
                             normalisation (<= 0: all T tokens) */
} orc_cfg;

/* Sinks are positions [0, S).  The quantized tokens are the
 * Nq = gk * floor((T - S - R) / gk) positions [S, S + Nq) (0 if T - S - R <= 0).
 * The rest, [S + Nq, T), is the fp16 recent window of W in [R, R + gk)
 * tokens.  In fp16 mode (16 bits) nothing is quantized and every token is
 * a window token. */
void orc_layout_counts(const orc_cfg *c, int T, int *S_eff, int *Nq, int *W)
{
    if (c->k_bits == 16) {
        *S_eff = 0;
        *Nq = 0;
        *W = T;
        return;
    }
    int s = T < c->n_sink ? T : c->n_sink;
    int rest = T - c->n_sink - c->n_recent;
    int nq = rest > 0 ? c->gk * (rest / c->gk) : 0;
    *S_eff = s;
    *Nq = nq;
    *W = T - s - nq;
}

static int row_bytes(int bits, int d) { return d * bits / 8; }

/* ------------------------------------------------------------------------ */
/* Build the stored representation of one stream from its T fp16 tokens.    */
/* ------------------------------------------------------------------------ */

/* Output arrays (caller allocated, sizes from Nq / W / S_eff):
 *  kc    [Nq][d*kb/8]            packed K codes, one row per token
 *  ks    uniform K: [Nq/gk][d][2] (min, scale) per channel per group
 *        NUQ K:     [Nq][2]       (min, s) per token
 *  vc    [Nq][d*vb/8]            packed V codes
 *  vs    uniform V: [Nq][d/gv][2] (min, scale) per token per channel group
 *        NUQ V:     [Nq][2]
 *  ksink, vsink [S_eff][d]       fp16 copies of the sink tokens
 *  kwin,  vwin  [W][d]           fp16 copies of the window tokens (position order)
 *  k_rowptr [Nq+1], k_cols [Nq*k], k_vals [Nq*k]  (NUQ K outliers, CSR)
 *  v_rowptr, v_cols, v_vals                        (NUQ V outliers, CSR)
 *  kn    [d]                     InnerQ key normalisation n_c (fp32 powers of two)
 *  With the InnerQ K layout (gkc > 0), ks is [Nq][d/gkc][2] (min, scale) per
 *  token per channel group, of the keys divided by n_c when k_norm is set.
 * V window tokens are stored unrotated even when V is Hadamard-rotated. */
void orc_build_stream(const orc_cfg *c, int T, const uint16_t *K, const uint16_t *V,
                      uint8_t *kc, uint16_t *ks, uint8_t *vc, uint16_t *vs,
                      uint16_t *ksink, uint16_t *vsink, uint16_t *kwin, uint16_t *vwin,
                      int32_t *k_rowptr, uint8_t *k_cols, uint16_t *k_vals,
                      int32_t *v_rowptr, uint8_t *v_cols, uint16_t *v_vals, float *kn)
{
    int d = c->d, S, Nq, W;
    orc_layout_counts(c, T, &S, &Nq, &W);
    uint8_t codes[1024];
    uint16_t rot[1024];

    for (int t = 0; t < S; t++) {
        memcpy(ksink + (size_t)t * d, K + (size_t)t * d, (size_t)d * 2);
        memcpy(vsink + (size_t)t * d, V + (size_t)t * d, (size_t)d * 2);
    }
    for (int w = 0; w < W; w++) {
        int t = S + Nq + w;
        memcpy(kwin + (size_t)w * d, K + (size_t)t * d, (size_t)d * 2);
        memcpy(vwin + (size_t)w * d, V + (size_t)t * d, (size_t)d * 2);
    }
    /* InnerQ key normalisation: fixed by the first norm_tokens tokens (the
     * prefill), whether or not any of them is quantized yet */
    if (c->k_norm) {
        int P = (c->norm_tokens > 0 && c->norm_tokens < T) ? c->norm_tokens : T;
        orc_key_norm(K, P, d, kn);
    }
    if (Nq == 0) {
        if (c->k_bits == 3) k_rowptr[0] = 0;
        if (c->v_bits == 3) v_rowptr[0] = 0;
        return;
    }

    /* K */
    int krow = row_bytes(c->k_bits, d);
    if (c->gkc > 0) {
        /* InnerQ: per token, groups of gkc channels along the hidden dimension,
         * on the normalised keys K / n_c */
        float xn[1024];
        int ng = d / c->gkc;
        for (int i = 0; i < Nq; i++) {
            const uint16_t *x = K + (size_t)(S + i) * d;
            for (int ch = 0; ch < d; ch++)
                xn[ch] = orc_half_to_float(x[ch]) / (c->k_norm ? kn[ch] : 1.0f);
            for (int j = 0; j < ng; j++) {
                uint16_t *e = ks + ((size_t)i * ng + j) * 2;
                orc_quantize_group(xn + j * c->gkc, c->gkc, 1, c->k_bits, c->hybrid,
                                   codes + j * c->gkc, 1, &e[0], &e[1]);
            }
            orc_pack_bits(codes, d, c->k_bits, kc + (size_t)i * krow);
        }
    } else if (c->k_bits == 3) {
        k_rowptr[0] = 0;
        for (int i = 0; i < Nq; i++) {
            const uint16_t *x = K + (size_t)(S + i) * d;
            orc_nuq_encode(x, d, c->outliers, c->k_lut, codes, &ks[2 * i], &ks[2 * i + 1],
                           k_cols + (size_t)i * c->outliers, k_vals + (size_t)i * c->outliers);
            orc_pack_bits(codes, d, 3, kc + (size_t)i * krow);
            k_rowptr[i + 1] = k_rowptr[i] + c->outliers;
        }
    } else {
        /* per channel, over groups of gk consecutive quantized tokens */
        uint8_t *gcodes = malloc((size_t)c->gk * d);
        float *gx = malloc(sizeof(float) * (size_t)c->gk * d);
        int ngrp = Nq / c->gk;
        for (int g = 0; g < ngrp; g++) {
            const uint16_t *base = K + (size_t)(S + g * c->gk) * d;
            for (size_t e = 0; e < (size_t)c->gk * d; e++) gx[e] = orc_half_to_float(base[e]);
            for (int ch = 0; ch < d; ch++) {
                uint16_t *e = ks + ((size_t)g * d + ch) * 2;
                if (c->hybrid)
                    orc_quantize_group(gx + ch, c->gk, d, c->k_bits, 1, gcodes + ch, d, &e[0], &e[1]);
                else
                    orc_quantize_uniform(base + ch, c->gk, d, c->k_bits,
                                         gcodes + ch, d, &e[0], &e[1]);
            }
            for (int r = 0; r < c->gk; r++)
                orc_pack_bits(gcodes + (size_t)r * d, d, c->k_bits,
                              kc + (size_t)(g * c->gk + r) * krow);
        }
        free(gcodes);
        free(gx);
    }

    /* V */
    int vrow = row_bytes(c->v_bits, d);
    for (int i = 0; i < Nq; i++) {
        const uint16_t *x = V + (size_t)(S + i) * d;
        if (c->v_hadamard) {
            orc_hadamard_rotate(x, d, rot);
            x = rot;
        }
        if (c->v_bits == 3) {
            if (i == 0) v_rowptr[0] = 0;
            orc_nuq_encode(x, d, c->outliers, c->v_lut, codes, &vs[2 * i], &vs[2 * i + 1],
                           v_cols + (size_t)i * c->outliers, v_vals + (size_t)i * c->outliers);
            v_rowptr[i + 1] = v_rowptr[i] + c->outliers;
        } else {
            int ng = d / c->gv;
            float xf[1024];
            for (int ch = 0; ch < d; ch++) xf[ch] = orc_half_to_float(x[ch]);
            for (int j = 0; j < ng; j++) {
                uint16_t *e = vs + ((size_t)i * ng + j) * 2;
                if (c->hybrid)
                    orc_quantize_group(xf + j * c->gv, c->gv, 1, c->v_bits, 1,
                                       codes + j * c->gv, 1, &e[0], &e[1]);
                else
                    orc_quantize_uniform(x + j * c->gv, c->gv, 1, c->v_bits,
                                         codes + j * c->gv, 1, &e[0], &e[1]);
            }
        }
        orc_pack_bits(codes, d, c->v_bits, vc + (size_t)i * vrow);
    }
}

/* ------------------------------------------------------------------------ */
/* Decode attention of one stream, fp64.                                     */
/* ------------------------------------------------------------------------ */

typedef struct orc_store {
    const uint8_t *kc; const uint16_t *ks; const uint8_t *vc; const uint16_t *vs;
    const uint16_t *ksink, *vsink, *kwin, *vwin;
    const int32_t *k_rowptr; const uint8_t *k_cols; const uint16_t *k_vals;
    const int32_t *v_rowptr; const uint8_t *v_cols; const uint16_t *v_vals;
    const float *kn;
} orc_store;

/* K of token t as stored, reconstructed in fp64 (dequantized, or the fp16
 * sink / window copy), then RoPE'd at position t in pre-RoPE mode. */
static void token_k(const orc_cfg *c, const orc_store *st, int S, int Nq, int t, double *kr)
{
    int d = c->d;
    uint8_t codes[1024];
    if (t < S) {
        for (int ch = 0; ch < d; ch++) kr[ch] = orc_half_to_float(st->ksink[(size_t)t * d + ch]);
    } else if (t >= S + Nq) {
        int w = t - S - Nq;
        for (int ch = 0; ch < d; ch++) kr[ch] = orc_half_to_float(st->kwin[(size_t)w * d + ch]);
    } else {
        int i = t - S;
        orc_unpack_bits(st->kc + (size_t)i * row_bytes(c->k_bits, d), d, c->k_bits, codes);
        if (c->gkc > 0) {
            int ng = d / c->gkc;
            for (int ch = 0; ch < d; ch++) {
                const uint16_t *e = st->ks + ((size_t)i * ng + ch / c->gkc) * 2;
                double v = (double)orc_half_to_float(e[0]) +
                           (double)codes[ch] * (double)orc_half_to_float(e[1]);
                kr[ch] = c->k_norm ? v * (double)st->kn[ch] : v;
            }
        } else if (c->k_bits == 3) {
            orc_nuq_decode(codes, d, st->ks[2 * i], st->ks[2 * i + 1], c->k_lut,
                           st->k_rowptr[i + 1] - st->k_rowptr[i], st->k_cols + st->k_rowptr[i],
                           st->k_vals + st->k_rowptr[i], kr);
        } else {
            int grp = i / c->gk;
            for (int ch = 0; ch < d; ch++) {
                const uint16_t *e = st->ks + ((size_t)grp * d + ch) * 2;
                kr[ch] = (double)orc_half_to_float(e[0]) +
                         (double)codes[ch] * (double)orc_half_to_float(e[1]);
            }
        }
    }
    if (c->k_pre_rope)
        orc_rope_apply(kr, d, (double)c->pos_offset + (double)t, c->rope_theta);
}

/* V of token t as stored, in fp64: dequantized (still in the rotated domain
 * when V is Hadamard-rotated), or the fp16 sink / window copy. */
static void token_v(const orc_cfg *c, const orc_store *st, int S, int Nq, int t, double *vr)
{
    int d = c->d;
    uint8_t codes[1024];
    if (t < S) {
        for (int ch = 0; ch < d; ch++) vr[ch] = orc_half_to_float(st->vsink[(size_t)t * d + ch]);
    } else if (t >= S + Nq) {
        int w = t - S - Nq;
        for (int ch = 0; ch < d; ch++) vr[ch] = orc_half_to_float(st->vwin[(size_t)w * d + ch]);
    } else {
        int i = t - S;
        orc_unpack_bits(st->vc + (size_t)i * row_bytes(c->v_bits, d), d, c->v_bits, codes);
        if (c->v_bits == 3) {
            orc_nuq_decode(codes, d, st->vs[2 * i], st->vs[2 * i + 1], c->v_lut,
                           st->v_rowptr[i + 1] - st->v_rowptr[i], st->v_cols + st->v_rowptr[i],
                           st->v_vals + st->v_rowptr[i], vr);
        } else {
            int ng = d / c->gv;
            for (int ch = 0; ch < d; ch++) {
                const uint16_t *e = st->vs + ((size_t)i * ng + ch / c->gv) * 2;
                vr[ch] = (double)orc_half_to_float(e[0]) +
                         (double)codes[ch] * (double)orc_half_to_float(e[1]);
            }
        }
    }
}

/* For each of the g query heads (q is [g][d] fp16, already RoPE'd):
 *   logit_t = sm_scale * q . k~_t over all T tokens (sinks, quantized, window)
 *   p_t     = exp(logit_t - max_t logit_t)
 *   o       = ( Hn * sum_{t quantized} p_t v^'_t  +  sum_{t fp16} p_t v_t ) / sum_t p_t
 *             in Hadamard mode (inverse rotation after the attention sum);
 *             otherwise sum_t p_t v~_t / sum_t p_t
 *   lse     = max + log(sum_t p_t)
 * out is [g][d], lse is [g], both fp64. */
void orc_decode_stream(const orc_cfg *c, int T, int g, const uint16_t *q,
                       const uint8_t *kc, const uint16_t *ks,
                       const uint8_t *vc, const uint16_t *vs,
                       const uint16_t *ksink, const uint16_t *vsink,
                       const uint16_t *kwin, const uint16_t *vwin,
                       const int32_t *k_rowptr, const uint8_t *k_cols, const uint16_t *k_vals,
                       const int32_t *v_rowptr, const uint8_t *v_cols, const uint16_t *v_vals,
                       const float *kn, double *out, double *lse)
{
    int d = c->d, S, Nq, W;
    orc_layout_counts(c, T, &S, &Nq, &W);
    orc_store st = { kc, ks, vc, vs, ksink, vsink, kwin, vwin,
                     k_rowptr, k_cols, k_vals, v_rowptr, v_cols, v_vals, kn };
    double sm = c->sm_scale != 0.0 ? c->sm_scale : 1.0 / sqrt((double)d);

    double *qv = malloc(sizeof(double) * (size_t)g * d);
    double *logit = malloc(sizeof(double) * (size_t)g * (T > 0 ? T : 1));
    double *mx = malloc(sizeof(double) * g), *L = malloc(sizeof(double) * g);
    double *oq = calloc((size_t)g * d, sizeof(double)), *ow = calloc((size_t)g * d, sizeof(double));
    double kr[1024], vr[1024], rot[1024];

    for (int i = 0; i < g * d; i++) qv[i] = orc_half_to_float(q[i]);
    for (int h = 0; h < g; h++) { mx[h] = -INFINITY; L[h] = 0.0; }

    for (int t = 0; t < T; t++) {
        token_k(c, &st, S, Nq, t, kr);
        for (int h = 0; h < g; h++) {
            double acc = 0.0;
            for (int ch = 0; ch < d; ch++) acc += qv[(size_t)h * d + ch] * kr[ch];
            double z = sm * acc;
            logit[(size_t)h * T + t] = z;
            if (z > mx[h]) mx[h] = z;
        }
    }
    for (int t = 0; t < T; t++) {
        token_v(c, &st, S, Nq, t, vr);
        int quant = (t >= S && t < S + Nq);
        for (int h = 0; h < g; h++) {
            double p = exp(logit[(size_t)h * T + t] - mx[h]);
            L[h] += p;
            double *dst = (quant ? oq : ow) + (size_t)h * d;
            for (int ch = 0; ch < d; ch++) dst[ch] += p * vr[ch];
        }
    }
    for (int h = 0; h < g; h++) {
        double *o = oq + (size_t)h * d;
        if (c->v_hadamard) {
            orc_hadamard_apply_f64(o, d, rot);
            memcpy(o, rot, sizeof(double) * d);
        }
        for (int ch = 0; ch < d; ch++)
            out[(size_t)h * d + ch] = (o[ch] + ow[(size_t)h * d + ch]) / L[h];
        lse[h] = mx[h] + log(L[h]);
    }
    free(qv); free(logit); free(mx); free(L); free(oq); free(ow);
}

/* ------------------------------------------------------------------------ */
/* Merge of attention results over disjoint parts of one context.           */
/* ------------------------------------------------------------------------ */

/* n parts of the same query rows (rows of d channels each): part r has the
 * normalised output o_r = sum_{t in r} p_t v_t / sum_{t in r} p_t and
 * lse_r = log sum_{t in r} exp(logit_t) (-inf for an empty part).  The
 * attention over the union is
 *   lse = log sum_r exp(lse_r),   o = sum_r exp(lse_r - lse) o_r.
 * outs [n][rows][d], lses [n][rows]; out [rows][d], lse [rows]; fp64.  The
 * largest lse_r is subtracted before exponentiating (an exact identity). */
void orc_merge_parts(int n, int rows, int d, const double *outs, const double *lses,
                     double *out, double *lse)
{
    for (int i = 0; i < rows; i++) {
        double m = -INFINITY;
        for (int r = 0; r < n; r++)
            if (lses[(size_t)r * rows + i] > m) m = lses[(size_t)r * rows + i];
        double L = 0.0;
        for (int ch = 0; ch < d; ch++) out[(size_t)i * d + ch] = 0.0;
        if (m == -INFINITY) {   /* every part empty */
            lse[i] = -INFINITY;
            continue;
        }
        for (int r = 0; r < n; r++) {
            double lr = lses[(size_t)r * rows + i];
            if (lr == -INFINITY) continue;
            double w = exp(lr - m);
            L += w;
            for (int ch = 0; ch < d; ch++)
                out[(size_t)i * d + ch] += w * outs[((size_t)r * rows + i) * d + ch];
        }
        for (int ch = 0; ch < d; ch++) out[(size_t)i * d + ch] /= L;
        lse[i] = m + log(L);
    }
}

/* ------------------------------------------------------------------------ */
/* Fitting a non-uniform level table (unweighted per-layer Lloyd).          */
/* ------------------------------------------------------------------------ */

/* The position of every dense value of a vector inside its dense range, on
 * the grid of 2^-16: outliers removed as orc_nuq_encode removes them (the k
 * largest |x|, ties to the lower channel), mn / mx the dense min / max
 * (fp32), u = (x - mn) / (mx - mn) (fp32, RN), position = rint(u * 2^16),
 * an integer in [0, 2^16].  The encoder maps mn to L0 and mx to L7 by the
 * same affine map, so a table fitted on these positions (scaled to [0, 1])
 * is one the encoder can use directly.  A vector whose dense part is
 * constant (mx == mn) gives no positions (the encoder codes it all 0).  With
 * `hadamard`, the vector is first rotated as orc_hadamard_rotate does.
 * Writes the positions of vector x (n channels) to pos and returns how many. */
static int nuq_fit_positions(const uint16_t *xin, int n, int k, int hadamard, int32_t *pos)
{
    uint16_t rot[1024];
    const uint16_t *x = xin;
    if (hadamard) {
        orc_hadamard_rotate(xin, n, rot);
        x = rot;
    }
    unsigned char is_out[1024];
    memset(is_out, 0, sizeof is_out);
    for (int j = 0; j < k; j++) {
        int best = -1;
        float bv = -1.0f;
        for (int i = 0; i < n; i++) {
            if (is_out[i]) continue;
            float a = fabsf(orc_half_to_float(x[i]));
            if (a > bv) { bv = a; best = i; }
        }
        is_out[best] = 1;
    }
    float mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < n; i++) {
        if (is_out[i]) continue;
        float v = orc_half_to_float(x[i]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    if (!(mx > mn)) return 0;
    float span = mx - mn;
    int m = 0;
    for (int i = 0; i < n; i++) {
        if (is_out[i]) continue;
        float u = (orc_half_to_float(x[i]) - mn) / span;
        pos[m++] = (int32_t)rintf(u * 65536.0f);
    }
    return m;
}

/* Lloyd's algorithm for 8 levels on the positions of all dense values of
 * nvec vectors x [nvec][n] (fp16), with the two end levels held at 0 and
 * 2^16 (every vector's dense min and max sit there):
 *   start        l_i = i * 2^16 / 7                              (fp64)
 *   assignment   a position p belongs to level #{i < 7 : p > (l_i + l_{i+1}) / 2}
 *                (the encoder's rule: an exact tie goes down)
 *   update       l_i = (sum of its positions) / (their count) for i = 1..6
 *                (exact integer sums, one fp64 division; an empty level
 *                keeps its value)
 * repeated until an update changes no level or max_iters updates were made.
 * lut[i] = fp16_RN(l_i / 2^16) as fp32; levels (if not NULL) gets the l_i
 * (fp64, positions).  Returns the number of updates made, or -1 if the
 * rounded levels are not strictly increasing. */
int orc_nuq_fit_lut(const uint16_t *x, long nvec, int n, int k, int hadamard, int max_iters, float *lut,
                    double *levels)
{
    int32_t *pos = malloc(sizeof(int32_t) * (size_t)nvec * (size_t)n);
    long np = 0;
    for (long v = 0; v < nvec; v++)
        np += nuq_fit_positions(x + (size_t)v * n, n, k, hadamard, pos + np);
    double l[8];
    for (int i = 0; i < 8; i++) l[i] = (double)i * 65536.0 / 7.0;
    int it = 0;
    while (it < max_iters) {
        double t[7];
        for (int i = 0; i < 7; i++) t[i] = (l[i] + l[i + 1]) / 2.0;
        long long cnt[8] = {0}, sum[8] = {0};
        for (long j = 0; j < np; j++) {
            int c = 0;
            for (int i = 0; i < 7; i++)
                if ((double)pos[j] > t[i]) c++;
            cnt[c] += 1;
            sum[c] += pos[j];
        }
        it++;
        int changed = 0;
        for (int i = 1; i < 7; i++) {
            if (cnt[i] == 0) continue;
            double nl = (double)sum[i] / (double)cnt[i];
            if (nl != l[i]) changed = 1;
            l[i] = nl;
        }
        if (!changed) break;
    }
    free(pos);
    if (levels)
        for (int i = 0; i < 8; i++) levels[i] = l[i];
    for (int i = 0; i < 8; i++) lut[i] = orc_half_to_float(orc_float_to_half((float)(l[i] / 65536.0)));
    for (int i = 1; i < 8; i++)
        if (!(lut[i] > lut[i - 1])) return -1;
    return it;
}

/* The positions of nvec vectors (as orc_nuq_fit_lut sees them), for tests:
 * writes at most cap positions, returns how many there are. */
long orc_nuq_fit_positions(const uint16_t *x, long nvec, int n, int k, int hadamard, int32_t *pos, long cap)
{
    int32_t tmp[1024];
    long np = 0;
    for (long v = 0; v < nvec; v++) {
        int m = nuq_fit_positions(x + (size_t)v * n, n, k, hadamard, tmp);
        for (int i = 0; i < m; i++) {
            if (np < cap) pos[np] = tmp[i];
            np++;
        }
    }
    return np;
}

/* ------------------------------------------------------------------------ */
/* Per-head bit allocation (RateQuant): distortion-rate fit and allocation.  */
/* ------------------------------------------------------------------------ */

/* Mean squared error of the cache's uniform quantizers on one stream's T
 * calibration tokens (fp16 K, V [T][d]) at `bits`: K per channel over the
 * floor(T / gk) whole groups of gk tokens (or, with the InnerQ layout, per
 * token over gkc-channel groups of the normalised keys), V per token over
 * gv-channel groups (rotated first when v_hadamard; the error is measured
 * where the quantizer works).  x^ = min_h + code * scale_h in fp64; hybrid
 * groups as configured.  dk, dv: sum of squared errors / number of values. */
void orc_quant_distortion(const orc_cfg *c, int T, const uint16_t *K, const uint16_t *V, int bits,
                          double *dk, double *dv)
{
    int d = c->d;
    uint8_t codes[1024];
    float xf[1024];
    uint16_t rot[1024];
    double sk = 0.0, sv = 0.0;
    long nk = 0, nv = 0;
    if (c->gkc > 0) {
        float kn[1024];
        if (c->k_norm) orc_key_norm(K, T, d, kn);
        for (int t = 0; t < T; t++) {
            for (int ch = 0; ch < d; ch++)
                xf[ch] = orc_half_to_float(K[(size_t)t * d + ch]) / (c->k_norm ? kn[ch] : 1.0f);
            for (int j = 0; j < d / c->gkc; j++) {
                uint16_t mh, sh;
                orc_quantize_group(xf + j * c->gkc, c->gkc, 1, bits, c->hybrid, codes, 1, &mh, &sh);
                for (int i = 0; i < c->gkc; i++) {
                    double xh = (double)orc_half_to_float(mh) + (double)codes[i] * (double)orc_half_to_float(sh);
                    double e = ((double)xf[j * c->gkc + i] - xh) * (c->k_norm ? (double)kn[j * c->gkc + i] : 1.0);
                    sk += e * e;
                    nk++;
                }
            }
        }
    } else {
        int ng = T / c->gk;
        float *gx = malloc(sizeof(float) * (size_t)c->gk);
        for (int g = 0; g < ng; g++)
            for (int ch = 0; ch < d; ch++) {
                uint16_t mh, sh;
                for (int i = 0; i < c->gk; i++)
                    gx[i] = orc_half_to_float(K[(size_t)(g * c->gk + i) * d + ch]);
                orc_quantize_group(gx, c->gk, 1, bits, c->hybrid, codes, 1, &mh, &sh);
                for (int i = 0; i < c->gk; i++) {
                    double e = (double)gx[i] -
                               ((double)orc_half_to_float(mh) + (double)codes[i] * (double)orc_half_to_float(sh));
                    sk += e * e;
                    nk++;
                }
            }
        free(gx);
    }
    for (int t = 0; t < T; t++) {
        const uint16_t *x = V + (size_t)t * d;
        if (c->v_hadamard) {
            orc_hadamard_rotate(x, d, rot);
            x = rot;
        }
        for (int ch = 0; ch < d; ch++) xf[ch] = orc_half_to_float(x[ch]);
        for (int j = 0; j < d / c->gv; j++) {
            uint16_t mh, sh;
            orc_quantize_group(xf + j * c->gv, c->gv, 1, bits, c->hybrid, codes, 1, &mh, &sh);
            for (int i = 0; i < c->gv; i++) {
                double e = (double)xf[j * c->gv + i] -
                           ((double)orc_half_to_float(mh) + (double)codes[i] * (double)orc_half_to_float(sh));
                sv += e * e;
                nv++;
            }
        }
    }
    *dk = nk ? sk / (double)nk : 0.0;
    *dv = nv ? sv / (double)nv : 0.0;
}

/* Fit D(b) = alpha * beta^-b to n points (b_i, D_i > 0): least squares of
 * ln D = ln alpha - b ln beta (RateQuant, "Methodology" 1 and the
 * distortion calibration of 3). */
void orc_fit_rd(int n, const double *b, const double *D, double *alpha, double *beta)
{
    double sb = 0, sy = 0, sbb = 0, sby = 0;
    for (int i = 0; i < n; i++) {
        double y = log(D[i]);
        sb += b[i];
        sy += y;
        sbb += b[i] * b[i];
        sby += b[i] * y;
    }
    double slope = (n * sby - sb * sy) / (n * sbb - sb * sb);  /* = -ln beta */
    double icpt = (sy - slope * sb) / n;                        /* = ln alpha */
    *alpha = exp(icpt);
    *beta = exp(-slope);
}

/* Reverse water-filling (RateQuant "Methodology" 1, per-component beta):
 * minimise sum_i w_i alpha_i beta_i^-b_i subject to sum_i b_i = B over real
 * b_i.  Stationarity: w_i alpha_i ln(beta_i) beta_i^-b_i = lambda, i.e.
 * b_i = (ln(w_i alpha_i ln beta_i) - ln lambda) / ln beta_i; ln lambda is
 * found by bisection so that the b_i sum to B.  (With a common beta this is
 * b_i = B/n + (ln w_i - ln wbar) / ln beta, wbar the geometric mean of
 * w_i alpha_i.)  Components need beta_i > 1. */
void orc_rate_waterfill(int n, const double *alpha, const double *beta, const double *w, double B, double *b)
{
    double lo = -1e3, hi = 1e3;
    for (int it = 0; it < 400; it++) {
        double mid = 0.5 * (lo + hi), sum = 0;
        for (int i = 0; i < n; i++) {
            double wi = w ? w[i] : 1.0;
            sum += (log(wi * alpha[i] * log(beta[i])) - mid) / log(beta[i]);
        }
        if (sum > B) lo = mid; else hi = mid;
    }
    double ll = 0.5 * (lo + hi);
    for (int i = 0; i < n; i++) {
        double wi = w ? w[i] : 1.0;
        b[i] = (log(wi * alpha[i] * log(beta[i])) - ll) / log(beta[i]);
    }
}

/* Greedy marginal-gain allocation (RateQuant "Methodology" 3, Alg. 1) on the
 * bit widths the cache supports, the ladder 2 -> 4 -> 8: every component
 * starts at 2 bits; while some next step fits the remaining budget
 * (total - sum of bits), take the step with the largest weighted distortion
 * reduction per added bit, w_i (D_i(b) - D_i(b')) / (b' - b) with the fitted
 * D_i; ties go to the lower component index.  bits_out[i] in {2, 4, 8}.
 * Returns the bits used (-1 if the budget is below 2 bits per component). */
int orc_rate_greedy(int n, const double *alpha, const double *beta, const double *w, int total, int *bits_out)
{
    int used = 2 * n;
    if (total < used) return -1;
    for (int i = 0; i < n; i++) bits_out[i] = 2;
    for (;;) {
        int best = -1;
        double bg = 0.0;
        for (int i = 0; i < n; i++) {
            int b0 = bits_out[i];
            if (b0 >= 8) continue;
            int b1 = b0 == 2 ? 4 : 8;
            if (used + (b1 - b0) > total) continue;
            double wi = w ? w[i] : 1.0;
            double gain = wi * (alpha[i] * pow(beta[i], -b0) - alpha[i] * pow(beta[i], -b1)) / (double)(b1 - b0);
            if (best < 0 || gain > bg) {
                best = i;
                bg = gain;
            }
        }
        if (best < 0) break;
        int b0 = bits_out[best];
        int b1 = b0 == 2 ? 4 : 8;
        used += b1 - b0;
        bits_out[best] = b1;
    }
    return used;
}
