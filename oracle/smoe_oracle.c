/*
 * smoe_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar CPU oracle for the SMOE group-quantised routed-expert
 * MoE layer.  Only the tests, the package smoke check and the benchmark's CPU
 * baseline may call it; the product path never links or executes it.  It
 * shares no code, header, table or constant generator with the CUDA library.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fPIC -shared -pthread
 * With contraction off every float operation below is rounded to fp32 on its
 * own, which is what makes the quantiser's codes reproducible bit for bit.
 *
 * Sources (page title, section):
 *   "SMOE Quantisation"  -- Quantisation Levels; L2-MSE Scale Optimiser;
 *                           Bit Packing; Decoding: Metal Kernel.
 *   ".smoe Binary Format" -- Expert Blob Architecture (codes then fp16 scales,
 *                           gate -> up -> down; byte counts per sub-tensor).
 *   "CMF v2 -- Format Specification" -- 2.2 MoE, execution semantics
 *                           (softmax over all logits, top-k with ties to the
 *                           lower index, selection-only expert_bias,
 *                           optional renormalisation, shared expert weighted
 *                           by sigmoid(shared_expert_gate . x) or 1).
 *   "Model Agnosticism"  -- SmoeModelConfig (router has max_experts_per_layer
 *                           rows; norm_topk_prob; moe_top_k <= 16; SiLU).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   G1  an all-zero group gets scale 0 and the code that rounds 0 (Q4: 8,
 *       Q2: 2); it decodes to exactly 0.
 *   G2  round() is round-half-to-even (rintf in the default rounding mode).
 *   G3  linspace(0.1, 1.0, 64) is evaluated in double the way numpy does
 *       (j*step + 0.1, last point exactly 1.0), then rounded to fp32; the
 *       candidate scale is that fp32 value times the fp32 absmax, rounded.
 *   G4  codes and the MSE use the fp32 candidate scale; the stored scale is
 *       that scale rounded to fp16 (nearest, ties to even).
 *   G5  encode is ((w / s) * L) + L with each step rounded to fp32, then
 *       rint and clamp to [0, 2L]; decode is ((c - L) / L) * s in fp32.
 *   MSE is accumulated in double; the first (smallest) candidate wins ties.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_GROUP 64
#define ORACLE_NCAND 64

/* ---------------------------------------------------------------- scalars */

/* bf16 -> fp32: the bf16 pattern is the top half of the fp32 pattern. */
static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE 754 binary16 -> fp32, written from the format definition. */
static float f16_bits_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return (float)(sign ? -v : v);
}

/* fp32 -> IEEE 754 binary16, round to nearest, ties to even, written from
 * the format definition with exact double arithmetic (frexp/ldexp/rint). */
static uint16_t f32_to_f16_bits(float f)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (isnan(f))
        return sign | 0x7e00;
    if (a >= 65520.0) /* 65504 + half an ulp rounds up to infinity */
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-24, m in [0, 1024] */
        double m = rint(a * ldexp(1.0, 24));
        return sign | (uint16_t)m; /* m == 1024 is the smallest normal */
    }
    int ex;
    (void)frexp(a, &ex); /* a = fr * 2^ex with fr in [0.5, 1) */
    int E = ex - 1;      /* a = (1 + t) * 2^E */
    double m = rint((ldexp(a, -E) - 1.0) * 1024.0);
    if (m == 1024.0) {
        m = 0.0;
        E += 1;
    }
    if (E + 15 >= 31)
        return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | (int)m);
}

/* ------------------------------------------------------ quantiser (a9) */

/* The 64 grid fractions linspace(0.1, 1.0, 64), reading G3. */
static void grid_fractions(float t[ORACLE_NCAND])
{
    double start = 0.1, stop = 1.0;
    double step = (stop - start) / (double)(ORACLE_NCAND - 1);
    for (int j = 0; j < ORACLE_NCAND; ++j) {
        double v = (double)j * step + start;
        if (j == ORACLE_NCAND - 1)
            v = stop;
        t[j] = (float)v;
    }
}

static float half_range(int bits) { return bits == 4 ? 7.5f : 1.5f; }

/* "SMOE Quantisation", L2-MSE Scale Optimiser: code = clamp(round(n*L + L)),
 * n = w / s; reading G5 fixes the fp32 order of operations. */
static uint8_t encode_one(float w, float s, float L, float cmax)
{
    float n = w / s;
    float q = n * L;
    q = q + L;
    float r = rintf(q);
    if (r < 0.0f)
        r = 0.0f;
    if (r > cmax)
        r = cmax;
    return (uint8_t)r;
}

/* "SMOE Quantisation", Decoding: weight = ((float)code - L) / L * scale. */
static float decode_one(uint8_t c, float s, float L)
{
    float lv = ((float)c - L) / L;
    return lv * s;
}

/* Quantise one group of n weights.  Outputs the codes, the chosen fp32 scale,
 * the chosen grid index (-1 for an all-zero group) and, if mse != NULL, the
 * reconstruction MSE of every candidate. */
static void quantize_group(const float *w, int n, int bits, const float t[ORACLE_NCAND],
                           uint8_t *codes, float *s_best, int *j_best, double *mse)
{
    const float L = half_range(bits);
    const float cmax = 2.0f * L;
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        float m = fabsf(w[i]);
        if (m > a)
            a = m;
    }
    if (a == 0.0f) { /* reading G1 */
        uint8_t zc = (uint8_t)rintf(L);
        for (int i = 0; i < n; ++i)
            codes[i] = zc;
        *s_best = 0.0f;
        *j_best = -1;
        if (mse)
            for (int j = 0; j < ORACLE_NCAND; ++j)
                mse[j] = 0.0;
        return;
    }
    int best = 0;
    double best_mse = INFINITY;
    for (int j = 0; j < ORACLE_NCAND; ++j) {
        float s = t[j] * a;
        double acc = 0.0;
        for (int i = 0; i < n; ++i) {
            uint8_t c = encode_one(w[i], s, L, cmax);
            double e = (double)w[i] - (double)decode_one(c, s, L);
            acc += e * e;
        }
        acc /= (double)n;
        if (mse)
            mse[j] = acc;
        if (acc < best_mse) { /* strict: first minimum wins */
            best_mse = acc;
            best = j;
        }
    }
    float s = t[best] * a;
    for (int i = 0; i < n; ++i)
        codes[i] = encode_one(w[i], s, L, cmax);
    *s_best = s;
    *j_best = best;
}

/* "SMOE Quantisation", Bit Packing: LSB-first, 8/bits codes per byte; element
 * idx goes to byte idx*bits/8 at bit (idx mod 8/bits)*bits. */
void oracle_pack(const uint8_t *codes, int64_t n, int bits, uint8_t *out)
{
    int64_t nbytes = (n * bits + 7) / 8;
    int per = 8 / bits;
    memset(out, 0, (size_t)nbytes);
    for (int64_t i = 0; i < n; ++i)
        out[i / per] |= (uint8_t)((codes[i] & ((1 << bits) - 1)) << ((i % per) * bits));
}

void oracle_unpack(const uint8_t *packed, int64_t n, int bits, uint8_t *codes)
{
    int per = 8 / bits;
    for (int64_t i = 0; i < n; ++i)
        codes[i] = (uint8_t)((packed[i / per] >> ((i % per) * bits)) & ((1 << bits) - 1));
}

/* Byte counts of one quantised sub-tensor (".smoe Binary Format", Expert Blob
 * Architecture): ceil(rows*cols*bits/8) code bytes, ceil(rows*cols/G)*2 scale
 * bytes. */
int64_t oracle_stream_bytes(int64_t rows, int64_t cols, int bits)
{
    return (rows * cols * bits + 7) / 8;
}

int64_t oracle_scales_bytes(int64_t rows, int64_t cols, int group)
{
    return ((rows * cols + group - 1) / group) * 2;
}

/* Bytes of one expert blob without padding: gate [f,d], up [f,d], down [d,f]. */
int64_t oracle_blob_bytes(int64_t d, int64_t f, int bits)
{
    int64_t one = oracle_stream_bytes(f, d, bits) + oracle_scales_bytes(f, d, ORACLE_GROUP);
    return 3 * one;
}

/* Quantise a row-major bf16 tensor of rows*cols elements (cols % 64 == 0) in
 * groups of 64 along the flattened order.  Writes the LSB-first code stream
 * and the fp16 scales.  Optional outputs: the per-group fp32 scale, the chosen
 * grid index, and all 64 candidate MSEs per group.  Returns 0, or -1 on bad
 * arguments. */
int oracle_quantize(const uint16_t *w_bf16, int64_t rows, int64_t cols, int bits,
                    uint8_t *codes_lsb, uint16_t *scales_f16, float *scale_f32,
                    int32_t *j_best, double *mse_all)
{
    if ((bits != 2 && bits != 4) || rows < 0 || cols <= 0 || cols % ORACLE_GROUP)
        return -1;
    float t[ORACLE_NCAND];
    grid_fractions(t);
    int64_t n = rows * cols, ngroups = n / ORACLE_GROUP;
    uint8_t *codes = (uint8_t *)malloc((size_t)(n > 0 ? n : 1));
    if (!codes)
        return -1;
    float w[ORACLE_GROUP];
    for (int64_t g = 0; g < ngroups; ++g) {
        for (int i = 0; i < ORACLE_GROUP; ++i)
            w[i] = bf16_bits_to_f32(w_bf16[g * ORACLE_GROUP + i]);
        float s;
        int jb;
        quantize_group(w, ORACLE_GROUP, bits, t, codes + g * ORACLE_GROUP, &s, &jb,
                       mse_all ? mse_all + g * ORACLE_NCAND : NULL);
        scales_f16[g] = f32_to_f16_bits(s);
        if (scale_f32)
            scale_f32[g] = s;
        if (j_best)
            j_best[g] = jb;
    }
    oracle_pack(codes, n, bits, codes_lsb);
    free(codes);
    return 0;
}

/* Dequantise an LSB-first stream + fp16 scales to a dense fp32 matrix. */
int oracle_dequantize(const uint8_t *codes_lsb, const uint16_t *scales_f16, int64_t rows,
                      int64_t cols, int bits, float *w_out)
{
    if ((bits != 2 && bits != 4) || cols % ORACLE_GROUP)
        return -1;
    const float L = half_range(bits);
    int per = 8 / bits;
    int64_t n = rows * cols;
    for (int64_t i = 0; i < n; ++i) {
        uint8_t c = (uint8_t)((codes_lsb[i / per] >> ((i % per) * bits)) & ((1 << bits) - 1));
        float s = f16_bits_to_f32(scales_f16[i / ORACLE_GROUP]);
        w_out[i] = decode_one(c, s, L);
    }
    return 0;
}

/* Expose the scalar helpers so that the tests can pin them. */
float oracle_f16_to_f32(uint16_t h) { return f16_bits_to_f32(h); }
uint16_t oracle_f32_to_f16(float f) { return f32_to_f16_bits(f); }
void oracle_grid(float *t) { grid_fractions(t); }
uint8_t oracle_encode(float w, float s, int bits)
{
    float L = half_range(bits);
    return encode_one(w, s, L, 2.0f * L);
}
float oracle_decode(uint8_t c, float s, int bits) { return decode_one(c, s, half_range(bits)); }

/* ------------------------------------------------------- router (a1-a3) */

/* logits[t,e] = sum_i Wr[e,i] x[t,i], accumulated in double, rounded to fp32
 * ("Model Agnosticism": the gate has max_experts_per_layer rows). */
void oracle_router_logits(const uint16_t *wr_bf16, const float *x, int64_t T, int32_t E,
                          int32_t d, float *logits)
{
    for (int64_t t = 0; t < T; ++t)
        for (int32_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int32_t i = 0; i < d; ++i)
                acc += (double)bf16_bits_to_f32(wr_bf16[(int64_t)e * d + i]) *
                       (double)x[t * d + i];
            logits[t * E + e] = (float)acc;
        }
}

/* "CMF v2", 2.2 MoE: scores are the softmax over all E logits, or with
 * router_sigmoid each expert's sigmoid(logit) on its own (double, the
 * selection key rounded to fp32); top-k chosen by the key, larger first,
 * ties to the lower expert index.  Key: the logit when no bias is given
 * (selecting on it selects on either score, both being increasing in the
 * logit); with an expert_bias, logit + bias for softmax scores, fl32(score) +
 * bias for sigmoid scores, each addition in fp32.  The bias never enters the
 * weights.  The selected scores are divided by their sum with norm_topk_prob,
 * then multiplied by routed_scaling_factor.  A routing mask ("CMF v2", 5:
 * expert bitfield, LSB-first, bit e set = expert e routable; nullable) limits
 * the selection to the routable experts and the softmax to them (its
 * normalisation runs over the routable set); its tail bits must be zero and
 * at least k experts routable.  Slots are written in rank order.  Returns 0,
 * or -1 on bad arguments. */
static int routable(const uint8_t *mask, int32_t e)
{
    return !mask || ((mask[e >> 3] >> (e & 7)) & 1);
}

int oracle_route_ex2(const float *logits, int64_t T, int32_t E, int32_t k, int32_t norm,
                     const float *bias, int32_t router_sigmoid, float routed_scaling_factor,
                     const uint8_t *mask, int32_t *ids, float *weights)
{
    if (E <= 0 || k < 1 || k > 16 || k > E || !(routed_scaling_factor > 0.0f) ||
        routed_scaling_factor > 3.0e38f)
        return -1;
    if (mask) {
        int32_t n = 0;
        for (int32_t e = 0; e < E; ++e)
            n += routable(mask, e);
        for (int32_t e = E; e < (E + 7) / 8 * 8; ++e)
            if ((mask[e >> 3] >> (e & 7)) & 1)
                return -1; /* tail bits beyond E must be zero */
        if (n < k)
            return -1;
    }
    float *key = (float *)malloc(sizeof(float) * (size_t)E);
    uint8_t *taken = (uint8_t *)malloc((size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    if (!key || !taken || !p) {
        free(key);
        free(taken);
        free(p);
        return -1;
    }
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        if (router_sigmoid) {
            for (int32_t e = 0; e < E; ++e)
                p[e] = 1.0 / (1.0 + exp(-(double)l[e]));
        } else {
            double m = -INFINITY;
            for (int32_t e = 0; e < E; ++e)
                if (routable(mask, e) && (double)l[e] > m)
                    m = (double)l[e];
            double z = 0.0;
            for (int32_t e = 0; e < E; ++e) {
                p[e] = routable(mask, e) ? exp((double)l[e] - m) : 0.0;
                z += p[e];
            }
            for (int32_t e = 0; e < E; ++e)
                p[e] /= z;
        }
        for (int32_t e = 0; e < E; ++e) {
            if (!bias)
                key[e] = l[e];
            else if (router_sigmoid)
                key[e] = (float)p[e] + bias[e];
            else
                key[e] = l[e] + bias[e];
            taken[e] = 0;
        }
        double sel = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e] || !routable(mask, e))
                    continue;
                if (best < 0 || key[e] > key[best]) /* strict: lower index on ties */
                    best = e;
            }
            taken[best] = 1;
            ids[t * k + j] = best;
            sel += p[best];
        }
        for (int32_t j = 0; j < k; ++j) {
            double pj = p[ids[t * k + j]];
            weights[t * k + j] = (float)((norm ? pj / sel : pj) * (double)routed_scaling_factor);
        }
    }
    free(key);
    free(taken);
    free(p);
    return 0;
}

int oracle_route_ex(const float *logits, int64_t T, int32_t E, int32_t k, int32_t norm,
                    const float *bias, int32_t router_sigmoid, float routed_scaling_factor,
                    int32_t *ids, float *weights)
{
    return oracle_route_ex2(logits, T, E, k, norm, bias, router_sigmoid, routed_scaling_factor,
                            NULL, ids, weights);
}

int oracle_route(const float *logits, int64_t T, int32_t E, int32_t k, int32_t norm,
                 const float *bias, int32_t *ids, float *weights)
{
    return oracle_route_ex2(logits, T, E, k, norm, bias, 0, 1.0f, NULL, ids, weights);
}

/* --------------------------------------------------- expert FFN (a5-a6) */

/* One expert's SwiGLU FFN on one token, from its blob (".smoe Binary Format",
 * Expert Blob Architecture: [gate codes][gate scales][up codes][up scales]
 * [down codes][down scales], no padding).  g and u are accumulated in double
 * and rounded to fp32; h = silu(g) * u (SiLU per the SARC activation field)
 * in double, rounded to fp32; out = W_down h in double, rounded to fp32.
 * If h_out != NULL the f values of h are written there. */
int oracle_expert_ffn(const uint8_t *blob, int32_t d, int32_t f, int bits, const float *x,
                      float *out, float *h_out)
{
    if ((bits != 2 && bits != 4) || d % ORACLE_GROUP || f % ORACLE_GROUP)
        return -1;
    int64_t cb = oracle_stream_bytes(f, d, bits), sb = oracle_scales_bytes(f, d, ORACLE_GROUP);
    const uint8_t *gate_c = blob;
    const uint16_t *gate_s = (const uint16_t *)(blob + cb);
    const uint8_t *up_c = blob + cb + sb;
    const uint16_t *up_s = (const uint16_t *)(blob + 2 * cb + sb);
    const uint8_t *down_c = blob + 2 * (cb + sb);
    const uint16_t *down_s = (const uint16_t *)(blob + 3 * cb + 2 * sb);

    float *wg = (float *)malloc(sizeof(float) * (size_t)f * d);
    float *wu = (float *)malloc(sizeof(float) * (size_t)f * d);
    float *wd = (float *)malloc(sizeof(float) * (size_t)f * d);
    float *h = (float *)malloc(sizeof(float) * (size_t)f);
    if (!wg || !wu || !wd || !h) {
        free(wg);
        free(wu);
        free(wd);
        free(h);
        return -1;
    }
    oracle_dequantize(gate_c, gate_s, f, d, bits, wg);
    oracle_dequantize(up_c, up_s, f, d, bits, wu);
    oracle_dequantize(down_c, down_s, d, f, bits, wd);
    for (int32_t r = 0; r < f; ++r) {
        double ga = 0.0, ua = 0.0;
        for (int32_t i = 0; i < d; ++i) {
            ga += (double)wg[(int64_t)r * d + i] * (double)x[i];
            ua += (double)wu[(int64_t)r * d + i] * (double)x[i];
        }
        float g = (float)ga, u = (float)ua;
        double hv = (double)g / (1.0 + exp(-(double)g)) * (double)u;
        h[r] = (float)hv;
    }
    for (int32_t i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int32_t r = 0; r < f; ++r)
            acc += (double)wd[(int64_t)i * f + r] * (double)h[r];
        out[i] = (float)acc;
    }
    if (h_out)
        memcpy(h_out, h, sizeof(float) * (size_t)f);
    free(wg);
    free(wu);
    free(wd);
    free(h);
    return 0;
}

/* ------------------------------------------------- MoE layer (a1-a7) */

/* Apply a given routing: y[t] = sum_j w[t,j] * FFN_{ids[t,j]}(x_t) in rank
 * order (double, rounded once), plus the shared expert's weighted output
 * ("CMF v2", 2.2 MoE: the shared expert is always added, with weight
 * sigmoid(shared_expert_gate . x) when that tensor is present, else 1).
 *   blobs[e]      expert e's blob (NULL allowed for an expert no token picks)
 *   shared_blob   nullable; shared expert of intermediate size fs
 *   shared_gate   nullable bf16 [d]
 * Returns 0, -1 on bad arguments, -2 if a selected expert's blob is NULL. */
/* expert_bits (nullable, [E]): each routed expert's own depth, 2 or 4
 * (mixed bit depth per expert, "CMF v2" 2.2: each expert its own dtype);
 * NULL = every expert at `bits`.  The shared expert is at `bits`. */
int oracle_moe_apply_mixed(int32_t d, int32_t f, int32_t E, int32_t k, int bits,
                           const int32_t *expert_bits, const uint8_t *const *blobs,
                           const uint8_t *shared_blob, int32_t fs, const uint16_t *shared_gate,
                           const float *x, int64_t T, const int32_t *ids, const float *wts,
                           float *y)
{
    if (d <= 0 || f <= 0 || E <= 0 || k < 1 || (bits != 2 && bits != 4))
        return -1;
    if (expert_bits)
        for (int32_t e = 0; e < E; ++e)
            if (expert_bits[e] != 2 && expert_bits[e] != 4)
                return -1;
    float *o = (float *)malloc(sizeof(float) * (size_t)d);
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = 0;
    if (!o || !acc) {
        rc = -1;
        goto done;
    }
    for (int64_t t = 0; t < T; ++t) {
        const float *xt = x + t * d;
        for (int32_t i = 0; i < d; ++i)
            acc[i] = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = ids[t * k + j];
            if (e < 0 || e >= E) {
                rc = -1;
                goto done;
            }
            const uint8_t *b = blobs[e];
            if (!b) {
                rc = -2;
                goto done;
            }
            if (oracle_expert_ffn(b, d, f, expert_bits ? expert_bits[e] : bits, xt, o, NULL)) {
                rc = -1;
                goto done;
            }
            for (int32_t i = 0; i < d; ++i)
                acc[i] += (double)wts[t * k + j] * (double)o[i];
        }
        if (shared_blob && fs > 0) {
            double sw = 1.0;
            if (shared_gate) {
                double z = 0.0;
                for (int32_t i = 0; i < d; ++i)
                    z += (double)bf16_bits_to_f32(shared_gate[i]) * (double)xt[i];
                sw = 1.0 / (1.0 + exp(-z));
            }
            if (oracle_expert_ffn(shared_blob, d, fs, bits, xt, o, NULL)) {
                rc = -1;
                goto done;
            }
            for (int32_t i = 0; i < d; ++i)
                acc[i] += sw * (double)o[i];
        }
        for (int32_t i = 0; i < d; ++i)
            y[t * d + i] = (float)acc[i];
    }
done:
    free(o);
    free(acc);
    return rc;
}

/* The same result as oracle_moe_apply_mixed, bit for bit, with the expert
 * FFNs of all (token, slot) items spread over nthreads POSIX threads: each
 * item runs the unchanged scalar oracle_expert_ffn on its own output row;
 * the combine then runs on the calling thread in exactly the serial order
 * (rank order in double, then the shared expert).  Only the benchmark's CPU
 * baseline uses it, to time the oracle on every host core. */
struct ffn_item {
    const uint8_t *blob;
    int32_t f, bits;
    const float *x;
    float *out;
};
struct ffn_pool {
    const struct ffn_item *items;
    int64_t n;
    int32_t d;
    int64_t next;
    int failed;
    pthread_mutex_t mu;
};

static void *ffn_worker(void *arg)
{
    struct ffn_pool *p = (struct ffn_pool *)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        const int64_t i = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (i >= p->n)
            return NULL;
        const struct ffn_item *it = &p->items[i];
        if (oracle_expert_ffn(it->blob, p->d, it->f, it->bits, it->x, it->out, NULL)) {
            pthread_mutex_lock(&p->mu);
            p->failed = 1;
            pthread_mutex_unlock(&p->mu);
        }
    }
}

int oracle_moe_apply_threads(int32_t d, int32_t f, int32_t E, int32_t k, int bits,
                             const int32_t *expert_bits, const uint8_t *const *blobs,
                             const uint8_t *shared_blob, int32_t fs, const uint16_t *shared_gate,
                             const float *x, int64_t T, const int32_t *ids, const float *wts,
                             float *y, int nthreads)
{
    if (d <= 0 || f <= 0 || E <= 0 || k < 1 || (bits != 2 && bits != 4) || nthreads < 1)
        return -1;
    if (expert_bits)
        for (int32_t e = 0; e < E; ++e)
            if (expert_bits[e] != 2 && expert_bits[e] != 4)
                return -1;
    const int has_sh = shared_blob && fs > 0;
    const int64_t per_t = k + (has_sh ? 1 : 0);
    struct ffn_item *items = (struct ffn_item *)malloc(sizeof(struct ffn_item) * (size_t)(T * per_t + 1));
    float *o = (float *)malloc(sizeof(float) * (size_t)(T * per_t * d + 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int rc = 0, started = 0;
    struct ffn_pool pool;
    if (!items || !o || !acc || !th) {
        rc = -1;
        goto done;
    }
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            const int32_t e = ids[t * k + j];
            if (e < 0 || e >= E) {
                rc = -1;
                goto done;
            }
            if (!blobs[e]) {
                rc = -2;
                goto done;
            }
            struct ffn_item *it = &items[t * per_t + j];
            it->blob = blobs[e];
            it->f = f;
            it->bits = expert_bits ? expert_bits[e] : bits;
            it->x = x + t * d;
            it->out = o + (t * per_t + j) * d;
        }
        if (has_sh) {
            struct ffn_item *it = &items[t * per_t + k];
            it->blob = shared_blob;
            it->f = fs;
            it->bits = bits;
            it->x = x + t * d;
            it->out = o + (t * per_t + k) * d;
        }
    }
    pool.items = items;
    pool.n = T * per_t;
    pool.d = d;
    pool.next = 0;
    pool.failed = 0;
    pthread_mutex_init(&pool.mu, NULL);
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, ffn_worker, &pool) != 0)
            break;
        ++started;
    }
    if (started == 0)
        ffn_worker(&pool);
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
    pthread_mutex_destroy(&pool.mu);
    if (pool.failed) {
        rc = -1;
        goto done;
    }
    for (int64_t t = 0; t < T; ++t) {
        const float *xt = x + t * d;
        for (int32_t i = 0; i < d; ++i)
            acc[i] = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            const float *oj = o + (t * per_t + j) * d;
            for (int32_t i = 0; i < d; ++i)
                acc[i] += (double)wts[t * k + j] * (double)oj[i];
        }
        if (has_sh) {
            double sw = 1.0;
            if (shared_gate) {
                double z = 0.0;
                for (int32_t i = 0; i < d; ++i)
                    z += (double)bf16_bits_to_f32(shared_gate[i]) * (double)xt[i];
                sw = 1.0 / (1.0 + exp(-z));
            }
            const float *os = o + (t * per_t + k) * d;
            for (int32_t i = 0; i < d; ++i)
                acc[i] += sw * (double)os[i];
        }
        for (int32_t i = 0; i < d; ++i)
            y[t * d + i] = (float)acc[i];
    }
done:
    free(items);
    free(o);
    free(acc);
    free(th);
    return rc;
}

int oracle_moe_apply(int32_t d, int32_t f, int32_t E, int32_t k, int bits,
                     const uint8_t *const *blobs, const uint8_t *shared_blob, int32_t fs,
                     const uint16_t *shared_gate, const float *x, int64_t T,
                     const int32_t *ids, const float *wts, float *y)
{
    return oracle_moe_apply_mixed(d, f, E, k, bits, NULL, blobs, shared_blob, fs, shared_gate, x,
                                  T, ids, wts, y);
}

/* Full layer forward for T tokens, each independent: router logits, route,
 * then oracle_moe_apply.  x is [T, d] fp32 (bf16 activations are widened
 * exactly by the caller); router_w is bf16 [E, d].  Optionally writes the
 * routing (ids/weights [T, k]) and the logits [T, E]. */
int oracle_moe_forward_ex(int32_t d, int32_t f, int32_t E, int32_t k, int32_t norm, int bits,
                          const int32_t *expert_bits, const uint16_t *router_w,
                          const float *expert_bias, int32_t router_sigmoid,
                          float routed_scaling_factor, const uint8_t *mask,
                          const uint8_t *const *blobs, const uint8_t *shared_blob, int32_t fs,
                          const uint16_t *shared_gate, const float *x, int64_t T, float *y,
                          int32_t *ids_out, float *w_out, float *logits_out)
{
    if (d <= 0 || f <= 0 || E <= 0 || k < 1 || k > 16 || k > E || (bits != 2 && bits != 4))
        return -1;
    float *logits = (float *)malloc(sizeof(float) * (size_t)(T * E + 1));
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T * k + 1));
    float *wts = (float *)malloc(sizeof(float) * (size_t)(T * k + 1));
    int rc = 0;
    if (!logits || !ids || !wts) {
        rc = -1;
        goto done;
    }
    oracle_router_logits(router_w, x, T, E, d, logits);
    if (oracle_route_ex2(logits, T, E, k, norm, expert_bias, router_sigmoid, routed_scaling_factor,
                         mask, ids, wts)) {
        rc = -1;
        goto done;
    }
    rc = oracle_moe_apply_mixed(d, f, E, k, bits, expert_bits, blobs, shared_blob, fs, shared_gate,
                                x, T, ids, wts, y);
    if (rc)
        goto done;
    if (ids_out)
        memcpy(ids_out, ids, sizeof(int32_t) * (size_t)(T * k));
    if (w_out)
        memcpy(w_out, wts, sizeof(float) * (size_t)(T * k));
    if (logits_out)
        memcpy(logits_out, logits, sizeof(float) * (size_t)(T * E));
done:
    free(logits);
    free(ids);
    free(wts);
    return rc;
}

int oracle_moe_forward(int32_t d, int32_t f, int32_t E, int32_t k, int32_t norm, int bits,
                       const uint16_t *router_w, const float *expert_bias,
                       const uint8_t *const *blobs, const uint8_t *shared_blob, int32_t fs,
                       const uint16_t *shared_gate, const float *x, int64_t T, float *y,
                       int32_t *ids_out, float *w_out, float *logits_out)
{
    return oracle_moe_forward_ex(d, f, E, k, norm, bits, NULL, router_w, expert_bias, 0, 1.0f,
                                 NULL, blobs, shared_blob, fs, shared_gate, x, T, y, ids_out,
                                 w_out, logits_out);
}
