/*
 * oracle.c -- plain, slow, single-threaded fp64 CPU oracle for the W4A16 NVFP4
 * mixture-of-experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  It shares no code, header,
 * table or constant with the CUDA library; it reads the same input bytes and
 * nothing else.
 *
 * What it computes, and where that is stated:
 *  - Atlas article "告别Python堆栈：Atlas用纯Rust重写LLM推理，在GB10上跑赢vLLM"
 *    (f.mffb.com.cn/a/497905.html), section "编译时内核选择和W4A16 Grouped GEMM":
 *    an MoE layer with two per-expert projections, gate_up and down, whose
 *    weights are packed 4-bit NVFP4 codes dequantised to BF16 and multiplied
 *    against BF16 activations by a BF16 MMA.
 *  - same article, section "KV Cache量化、MTP推测解码和调试工具链": the MoE layer
 *    takes gate logits, picks expert IDs, and the routed output is the layer
 *    output (the article debugs it against a higher-precision oracle, which
 *    is what this file is).
 *  - ATOM article "AMD ATOM推理引擎：如何用分页KV缓存和分段编译实现大模型推理性能翻倍"
 *    (itsolotime.com/archives/33112), section "8.1 MoE 路径：路由、专家并行与
 *    MORI 通信": MoE = token routing, top-k selection, expert compute and a
 *    final combine of the expert outputs per token.
 *  - "Rust 实现深度学习推理引擎：从计算图到异构硬件加速"
 *    (ybb.press/ai-applications/14151.html), section "三、计算图：节点、边与拓扑排序":
 *    the SiLU / SwiGLU activation of LLaMA-style FFNs.
 *
 * The NVFP4 format itself is not spelled out on those pages (they only name
 * "nvfp4" and "E2M1"); the decoders below follow the public OCP FP8 / MX
 * closed forms: E2M1 = 1 sign, 2 exponent (bias 1), 1 mantissa bit;
 * E4M3 = 1 sign, 4 exponent (bias 7), 3 mantissa bits, no infinities,
 * S.1111.111 = NaN.  A weight is code * block_scale * global_scale, with one
 * E4M3 block scale per 16 consecutive elements along K and one fp32 global
 * scale per expert matrix.
 *
 * Readings where the pages are silent:
 *  - packed codes: element 2i in the low nibble, 2i+1 in the high nibble;
 *  - gate_up rows 0..I-1 are the gate projection, rows I..2I-1 the up
 *    projection, and SwiGLU = silu(gate) * up;
 *  - routing selects on the fp32 logits, ties to the lower expert index,
 *    NaN treated as -infinity; the k gate weights are the softmax over the k
 *    selected logits (the same as a softmax over all E renormalised over the
 *    selected k);
 *  - the intermediate activation h (input of the down projection's BF16 MMA)
 *    is rounded to bf16, round-to-nearest-even; everything else is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- decoders */

/* E2M1 code (low 4 bits of `code`) -> value.  sign = bit 3, exponent = bits
 * 2..1 (bias 1), mantissa = bit 0.  exponent 0 is subnormal: 0.5 * m. */
double oracle_dec_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* E4M3 ("fn" variant) code -> value.  sign = bit 7, exponent = bits 6..3
 * (bias 7), mantissa = bits 2..0.  exponent 0 is subnormal: (m/8) * 2^-6.
 * exponent 15 with mantissa 7 is NaN; there are no infinities. */
double oracle_dec_e4m3(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* bf16 bit pattern -> value (exact). */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp64 -> bf16 bit pattern, round to nearest, ties to even, computed on the
 * value (not on bits): find the two neighbouring bf16 values and pick. */
uint16_t oracle_bf16_rne(double v)
{
    if (isnan(v)) return 0x7FC0u;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    /* bf16: 8 significant bits, exponent range of fp32 (normal >= 2^-126,
     * subnormal quantum 2^-133), max finite (2 - 2^-7) * 2^127. */
    int ex;
    frexp(a, &ex);              /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;             /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;     /* subnormal range keeps the quantum fixed */
    double q = ldexp(1.0, e - 7);
    double lo = floor(a / q) * q;
    double hi = lo + q;
    double r;
    if (a - lo < hi - a) r = lo;
    else if (a - lo > hi - a) r = hi;
    else r = (fmod(lo / q, 2.0) == 0.0) ? lo : hi;
    if (r > ldexp(2.0 - ldexp(1.0, -7), 127)) return (uint16_t)(sign | 0x7F80u); /* overflow -> inf */
    float f = (float)r;     /* exact: r has <= 8 significant bits in fp32 range */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

static double g_e2m1[16];
static double g_e4m3[256];
static int g_tables_ready = 0;

static void tables_init(void)
{
    if (g_tables_ready) return;
    for (unsigned c = 0; c < 16; ++c) g_e2m1[c] = oracle_dec_e2m1(c);
    for (unsigned c = 0; c < 256; ++c) g_e4m3[c] = oracle_dec_e4m3(c);
    g_tables_ready = 1;
}

/* One weight element W[e][n][kk] of a projection with N rows and K columns:
 * codes [E][N][K/2] (low nibble = even kk), scales [E][N][K/16], gs [E]. */
double oracle_weight(const uint8_t *codes, const uint8_t *scales, const float *gs,
                     int N, int K, int e, int n, int kk)
{
    tables_init();
    size_t row = (size_t)e * (size_t)N + (size_t)n;
    uint8_t byte = codes[row * (size_t)(K / 2) + (size_t)(kk / 2)];
    unsigned nib = (kk & 1) ? (byte >> 4) : (byte & 15u);
    uint8_t sc = scales[row * (size_t)(K / 16) + (size_t)(kk / 16)];
    return g_e2m1[nib] * g_e4m3[sc] * (double)gs[e];
}

/* Decode a whole weight row into `out[K]` (same formula, one row at a time so
 * that no full matrix is ever materialised). */
void oracle_decode_row(const uint8_t *codes, const uint8_t *scales, const float *gs,
                       int N, int K, int e, int n, double *out)
{
    tables_init();
    size_t row = (size_t)e * (size_t)N + (size_t)n;
    const uint8_t *c = codes + row * (size_t)(K / 2);
    const uint8_t *s = scales + row * (size_t)(K / 16);
    double g = (double)gs[e];
    for (int kk = 0; kk < K; ++kk) {
        unsigned nib = (kk & 1) ? (c[kk / 2] >> 4) : (c[kk / 2] & 15u);
        out[kk] = g_e2m1[nib] * g_e4m3[s[kk / 16]] * g;
    }
}

/* ------------------------------------------------------------ router logits */

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* The gate logits of the Atlas article's MoE layer (section "KV Cache量化、MTP
 * 推测解码和调试工具链": gate input -> gate logits -> expert IDs), exactly:
 * logits[t][e] = sum_h x[t][h] * Wr[e][h] (+ bias[e]) in fp64, rounded once to
 * fp32.  x bf16 [T][H], Wr bf16 [E][H], bias fp32 [E] or NULL. */
void oracle_router_logits_exact(const uint16_t *x, const uint16_t *wr, const float *bias, int T, int H, int E,
                                double *logits)
{
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += (double)bf16_to_float(x[(size_t)t * H + h]) * (double)bf16_to_float(wr[(size_t)e * H + h]);
            if (bias != NULL) acc += (double)bias[e];
            logits[(size_t)t * E + e] = acc;
        }
}

/* The same logits in fp32 with the library's fixed reduction order, so that
 * routing on them is reproducible bit for bit:
 *  - the hidden dimension is cut into 8-element chunks; part l (l = 0..31)
 *    takes chunks l, l+32, l+64, ... and accumulates x*w over its elements in
 *    ascending h with a fused multiply-add, starting from 0;
 *  - the 32 parts are combined in five rounds; in round r (strides 16, 8, 4,
 *    2, 1) every part l becomes part l + part (l XOR stride); the result is
 *    part 0 (an fp32 add is commutative, so every part ends equal);
 *  - the bias, if any, is added last. */
void oracle_router_logits(const uint16_t *x, const uint16_t *wr, const float *bias, int T, int H, int E,
                          float *logits)
{
    float part[32], next[32];
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            const uint16_t *xr = x + (size_t)t * H, *wrow = wr + (size_t)e * H;
            for (int l = 0; l < 32; ++l) {
                float acc = 0.0f;
                for (int chunk = l; chunk * 8 < H; chunk += 32)
                    for (int c = 0; c < 8; ++c) {
                        int h = chunk * 8 + c;
                        acc = fmaf(bf16_to_float(xr[h]), bf16_to_float(wrow[h]), acc);
                    }
                part[l] = acc;
            }
            for (int stride = 16; stride >= 1; stride /= 2) {
                for (int l = 0; l < 32; ++l) next[l] = part[l] + part[l ^ stride];
                memcpy(part, next, sizeof part);
            }
            float v = part[0];
            if (bias != NULL) v = v + bias[e];
            logits[(size_t)t * E + e] = v;
        }
}

/* ------------------------------------------------------------------ routing */

static double route_key(float v)
{
    return isnan(v) ? -INFINITY : (double)v;
}

/* Top-k routing of every token.  logits fp32 [T][E].  Writes ids [T][k]
 * (slot order: descending logit, ties to the lower expert index) and the
 * gate weights w [T][k] in fp64: softmax over the k selected logits.  If the
 * best selected logit is -infinity (all NaN / -inf), the weights are 1/k. */
void oracle_route(const float *logits, int T, int E, int k, int32_t *ids, double *w)
{
    char *taken = (char *)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * (size_t)E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            double bv = 0.0;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                double v = route_key(l[e]);
                if (best < 0 || v > bv) { best = e; bv = v; }  /* strict: keeps lower index on ties */
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        double lmax = route_key(l[ids[(size_t)t * k]]);
        if (lmax == -INFINITY) {
            for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = 1.0 / (double)k;
            continue;
        }
        double sum = 0.0;
        for (int j = 0; j < k; ++j) {
            double z = exp(route_key(l[ids[(size_t)t * k + j]]) - lmax);
            w[(size_t)t * k + j] = z;
            sum += z;
        }
        for (int j = 0; j < k; ++j) w[(size_t)t * k + j] /= sum;
    }
    free(taken);
}

/* -------------------------------------------------------------- permutation */

/* Group the T*k (token, slot) pairs by expert.  counts[e] = number of pairs
 * routed to e; offsets = exclusive scan of counts (E+1 entries); the sorted
 * order lists pairs by (expert, token) -- a token meets an expert at most once
 * -- so sorted_token[p] is the token of sorted row p and inv_perm[t*k+j] is
 * the sorted row of pair (t, j). */
void oracle_permute(const int32_t *ids, int T, int E, int k, int32_t *counts,
                    int32_t *offsets, int32_t *sorted_token, int32_t *inv_perm)
{
    int n = T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int i = 0; i < n; ++i) counts[ids[i]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int i = 0; i < n; ++i) {           /* ascending i = ascending (token, slot) */
        int e = ids[i];
        int p = fill[e]++;
        sorted_token[p] = i / k;
        inv_perm[i] = p;
    }
    free(fill);
}

/* ------------------------------------------------------------ expert FFN */

/* gate_up + SwiGLU for one activation row.  x: bf16 bits [H].  gate_up
 * weights have N = 2I rows, K = H.  h_exact [I] (fp64, may be NULL) and
 * h_bf16 [I] (bf16 bits of h_exact, RNE, may be NULL). */
void oracle_gate_up_swiglu_row(const uint16_t *x, int H, int I,
                               const uint8_t *codes, const uint8_t *scales, const float *gs,
                               int e, double *h_exact, uint16_t *h_bf16)
{
    double *xv = (double *)malloc(sizeof(double) * (size_t)H);
    double *wr = (double *)malloc(sizeof(double) * (size_t)H);
    for (int i = 0; i < H; ++i) xv[i] = oracle_bf16_to_double(x[i]);
    for (int f = 0; f < I; ++f) {
        double g = 0.0, u = 0.0;
        oracle_decode_row(codes, scales, gs, 2 * I, H, e, f, wr);
        for (int i = 0; i < H; ++i) g += xv[i] * wr[i];
        oracle_decode_row(codes, scales, gs, 2 * I, H, e, I + f, wr);
        for (int i = 0; i < H; ++i) u += xv[i] * wr[i];
        double h = g / (1.0 + exp(-g)) * u;
        if (h_exact) h_exact[f] = h;
        if (h_bf16) h_bf16[f] = oracle_bf16_rne(h);
    }
    free(xv);
    free(wr);
}

/* down projection for one row.  h: bf16 bits [I].  down weights have N = H
 * rows, K = I.  y [H] fp64. */
void oracle_down_row(const uint16_t *h, int H, int I,
                     const uint8_t *codes, const uint8_t *scales, const float *gs,
                     int e, double *y)
{
    double *hv = (double *)malloc(sizeof(double) * (size_t)I);
    double *wr = (double *)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; ++i) hv[i] = oracle_bf16_to_double(h[i]);
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        oracle_decode_row(codes, scales, gs, H, I, e, n, wr);
        for (int i = 0; i < I; ++i) acc += hv[i] * wr[i];
        y[n] = acc;
    }
    free(hv);
    free(wr);
}

/* Weighted combine back to token order for rows given in sorted order:
 * out[t][n] = sum_j w[t][j] * y[inv_perm[t*k+j]][n]  (fp64, ascending j). */
void oracle_combine(const double *y, const int32_t *inv_perm, const double *w, int T, int H, int k,
                    double *out)
{
    for (int t = 0; t < T; ++t) {
        double *o = out + (size_t)t * (size_t)H;
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            const double *yr = y + (size_t)inv_perm[(size_t)t * k + j] * (size_t)H;
            double wj = w[(size_t)t * k + j];
            for (int n = 0; n < H; ++n) o[n] += wj * yr[n];
        }
    }
}

/* ------------------------------------------------------------------ layer */

/* Layer output for the tokens listed in rows[0..nrows): out [nrows][H] fp64.
 * out[r] = sum_j w[t,j] * down_e(bf16(swiglu(gate_up_e(x[t])))), e = id[t,j].
 * ids / w must come from oracle_route (ids [T][k], w [T][k]). */
void oracle_layer_rows(const uint16_t *x, const int32_t *ids, const double *w,
                       const uint8_t *gu_codes, const uint8_t *gu_scales, const float *gu_gs,
                       const uint8_t *dn_codes, const uint8_t *dn_scales, const float *dn_gs,
                       int H, int I, int k, const int32_t *rows, int nrows, double *out)
{
    uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)I);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    for (int r = 0; r < nrows; ++r) {
        int t = rows[r];
        double *o = out + (size_t)r * (size_t)H;
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            double wj = w[(size_t)t * k + j];
            oracle_gate_up_swiglu_row(x + (size_t)t * (size_t)H, H, I, gu_codes, gu_scales, gu_gs,
                                      e, NULL, h);
            oracle_down_row(h, H, I, dn_codes, dn_scales, dn_gs, e, y);
            for (int n = 0; n < H; ++n) o[n] += wj * y[n];
        }
    }
    free(h);
    free(y);
}

/* Whole layer: route, then every token.  out [T][H] fp64; ids [T][k] and
 * w [T][k] are written too. */
void oracle_layer(const uint16_t *x, const float *logits,
                  const uint8_t *gu_codes, const uint8_t *gu_scales, const float *gu_gs,
                  const uint8_t *dn_codes, const uint8_t *dn_scales, const float *dn_gs,
                  int T, int H, int I, int E, int k, int32_t *ids, double *w, double *out)
{
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    oracle_route(logits, T, E, k, ids, w);
    for (int t = 0; t < T; ++t) rows[t] = t;
    oracle_layer_rows(x, ids, w, gu_codes, gu_scales, gu_gs, dn_codes, dn_scales, dn_gs,
                      H, I, k, rows, T, out);
    free(rows);
}

/* ====================================================== W4A4 (NVFP4 activations)
 *
 * The block-scaled FP4 variant of the layer: weights as above, and the
 * activations entering each projection (x for gate_up, h for down) quantized
 * to NVFP4 too, then multiplied in fp64.  The pages give no activation
 * quantizer (the ATOM article's section 8.2 lists a 4-bit-activation format
 * as an execution contract of its own; the Atlas article notes GB10 lacks the
 * native FP4 MMA that GB300 has); the reading taken here is the weights'
 * NVFP4 format without a global scale: per 16 consecutive elements one E4M3
 * scale s = RNE_e4m3(min(amax16 / 6, 448)) and codes RNE_e2m1(v / e4m3(s)),
 * ties to the even mantissa, saturating at +-6 (all codes 0 when e4m3(s) is
 * 0); the scale from amax16 / 6 computed in fp32, the codes by rounding
 * the exact quotient v / e4m3(s) (each code is the grid value c with c *
 * e4m3(s) nearest to v).  h is quantized from its value rounded to fp32. */

/* fp32 -> E4M3 code, round to nearest even, for 0 <= v <= 448 (finite). */
unsigned oracle_e4m3_rne(float v)
{
    /* candidates: every non-negative finite code, nearest by |value - v|;
     * on a tie the code with the even mantissa (even code) wins */
    unsigned best = 0;
    double bd = INFINITY;
    for (unsigned c = 0; c < 0x7F; ++c) {
        double d = fabs(oracle_dec_e4m3(c) - (double)v);
        if (d < bd || (d == bd && (c & 1u) == 0u && (best & 1u) == 1u)) {
            bd = d;
            best = c;
        }
    }
    return best;
}

/* fp32 -> E2M1 code: nearest of the 15 values, ties to the even mantissa,
 * saturating at +-6; -0 and values rounding to 0 give code 0. */
unsigned oracle_e2m1_rne(float v)
{
    double a = fabs((double)v);
    unsigned best = 0;
    double bd = INFINITY;
    for (unsigned c = 0; c < 8; ++c) {
        double d = fabs(oracle_dec_e2m1(c) - a);
        if (d < bd || (d == bd && (c & 1u) == 0u && (best & 1u) == 1u)) {
            bd = d;
            best = c;
        }
    }
    if (a > 6.0) best = 7;
    return (best != 0 && v < 0.0f) ? (best | 8u) : best;
}

/* E2M1 code of the exact quotient v / d (d > 0): the grid magnitude g whose
 * g * d is nearest to |v|, ties to the even mantissa, saturating at 6. */
static unsigned e2m1_of_quotient(float v, float d)
{
    double a = fabs((double)v);
    unsigned best = 0;
    double bd = INFINITY;
    for (unsigned c = 0; c < 8; ++c) {
        double dist = fabs(oracle_dec_e2m1(c) * (double)d - a);
        if (dist < bd || (dist == bd && (c & 1u) == 0u && (best & 1u) == 1u)) {
            bd = dist;
            best = c;
        }
    }
    return (best != 0 && v < 0.0f) ? (best | 8u) : best;
}

/* Quantize n fp32 values (n a multiple of 16) to NVFP4: codes [n/2] (element
 * 2i in the low nibble), E4M3 scales [n/16]. */
void oracle_quant_nvfp4(const float *v, int n, uint8_t *codes, uint8_t *scales)
{
    for (int b = 0; b < n / 16; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(v[16 * b + i]);
            if (a > amax) amax = a;
        }
        float q = amax / 6.0f;
        if (q > 448.0f) q = 448.0f;
        unsigned s = oracle_e4m3_rne(q);
        float d = (float)oracle_dec_e4m3(s);
        scales[b] = (uint8_t)s;
        for (int i = 0; i < 16; i += 2) {
            unsigned c0 = 0, c1 = 0;
            if (d != 0.0f) {
                c0 = e2m1_of_quotient(v[16 * b + i], d);
                c1 = e2m1_of_quotient(v[16 * b + i + 1], d);
            }
            codes[8 * b + i / 2] = (uint8_t)(c0 | (c1 << 4));
        }
    }
}

/* NVFP4 values (codes [n/2], scales [n/16], no global scale) -> fp64 [n]. */
static void dequant_nvfp4(const uint8_t *codes, const uint8_t *scales, int n, double *out)
{
    for (int i = 0; i < n; ++i) {
        unsigned c = (codes[i / 2] >> (4 * (i & 1))) & 15u;
        out[i] = oracle_dec_e2m1(c) * oracle_dec_e4m3(scales[i / 16]);
    }
}

/* The W4A4 layer for the tokens rows[0..nrows): x bf16 bits [T][H] quantized
 * per token, gate_up + SwiGLU in fp64 on the dequantized values, h rounded to
 * fp32 and quantized, down in fp64, the weighted sum over the k slots in
 * fp64.  out [nrows][H]. */
void oracle_w4a4_layer_rows(const uint16_t *x, const int32_t *ids, const double *w,
                            const uint8_t *gu_codes, const uint8_t *gu_scales, const float *gu_gs,
                            const uint8_t *dn_codes, const uint8_t *dn_scales, const float *dn_gs,
                            int H, int I, int k, const int32_t *rows, int nrows, double *out)
{
    float *xf = (float *)malloc(sizeof(float) * (size_t)H);
    uint8_t *xc = (uint8_t *)malloc((size_t)H / 2), *xs = (uint8_t *)malloc((size_t)H / 16);
    double *xq = (double *)malloc(sizeof(double) * (size_t)H);
    double *wr = (double *)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    float *hf = (float *)malloc(sizeof(float) * (size_t)I);
    uint8_t *hc = (uint8_t *)malloc((size_t)I / 2), *hs = (uint8_t *)malloc((size_t)I / 16);
    double *hq = (double *)malloc(sizeof(double) * (size_t)I);
    for (int r = 0; r < nrows; ++r) {
        int t = rows[r];
        double *o = out + (size_t)r * (size_t)H;
        for (int i = 0; i < H; ++i) xf[i] = bf16_to_float(x[(size_t)t * H + i]);
        oracle_quant_nvfp4(xf, H, xc, xs);
        dequant_nvfp4(xc, xs, H, xq);
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            for (int f = 0; f < I; ++f) {
                double g = 0.0, u = 0.0;
                oracle_decode_row(gu_codes, gu_scales, gu_gs, 2 * I, H, e, f, wr);
                for (int i = 0; i < H; ++i) g += xq[i] * wr[i];
                oracle_decode_row(gu_codes, gu_scales, gu_gs, 2 * I, H, e, I + f, wr);
                for (int i = 0; i < H; ++i) u += xq[i] * wr[i];
                hf[f] = (float)(g / (1.0 + exp(-g)) * u);
            }
            oracle_quant_nvfp4(hf, I, hc, hs);
            dequant_nvfp4(hc, hs, I, hq);
            for (int n = 0; n < H; ++n) {
                double acc = 0.0;
                oracle_decode_row(dn_codes, dn_scales, dn_gs, H, I, e, n, wr);
                for (int i = 0; i < I; ++i) acc += hq[i] * wr[i];
                o[n] += w[(size_t)t * k + j] * acc;
            }
        }
    }
    free(xf); free(xc); free(xs); free(xq); free(wr); free(hf); free(hc); free(hs); free(hq);
}
