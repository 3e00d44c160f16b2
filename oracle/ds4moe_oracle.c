/*
 * ds4moe CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 restatement of the routed-MoE expert layer of the
 * DwarfStar (ds4) engine, used to check the CUDA library.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load this
 * code; the product never does.  It shares no code, header or table with the
 * CUDA path.
 *
 * What the layer is (pages: "DwarfStar実地分析: DeepSeek V4 Flashをローカルで
 * 動かす狭域推論エンジン", §GGUFの対応範囲は意図的に狭い; "DS4 分布式Shell客户端",
 * §模型下载 and §设计动机): a routed mixture-of-experts feed-forward layer
 * whose routed experts are stored in 4-bit block-scaled MXFP4 (gate, up and
 * down projections) or, in the asymmetric 2-bit scheme, with a Q2_K down
 * projection.  The pages name the formats and the layer but give no formula;
 * the readings below are the plain ones and are listed in the design notes.
 *
 *   route   : per token, the k largest logits sorted by (value desc, index
 *             asc); w = softmax over those k logits only.
 *   group   : counts per expert, exclusive offsets, and the (token, slot)
 *             pairs stably sorted by (expert, token).
 *   expert  : g = Wg.x, u = Wu.x, h = silu(g)*u = g/(1+exp(-g))*u, y = Wd.h.
 *   combine : out[t] = sum_j w[t,j] * y[t,j].
 *   with a router and a shared expert (original precision, bf16 weights):
 *             logits = Wr.x before the routing, and out[t] += the shared
 *             expert's SwiGLU FFN of x (its h rounded to bf16).
 *
 * Formats (OCP Microscaling Formats v1.0): E2M1 magnitudes
 * {0,0.5,1,1.5,2,3,4,6} with bit 3 the sign; E8M0 byte b -> 2^(b-127)
 * (0xFF = NaN); 32-element blocks along the contraction axis; the element
 * 2i sits in the low nibble of byte i.  E4M3: bias 7, 3 mantissa bits,
 * subnormals m*2^-9, largest finite 448, S.1111.111 = NaN.
 *
 * Activation-precision modes (the GPU path's precisions are part of the
 * layer as built, so the oracle follows them):
 *   ACT_EXACT  (few-token decode path): x used exactly as its bf16 value,
 *              h kept in fp64.
 *   ACT_MXFP8  (prefill path): x -> MXFP8 along d; h is rounded to fp32
 *              (the precision the kernel takes its quantisation decision
 *              in) and then -> MXFP8 along f.
 *   ACT_MXFP8_X_ONLY (prefill path with the Q2_K down projection): x ->
 *              MXFP8, h kept in fp64.
 *   ACT_MXFP4  (all-FP4 prefill, both MMA operands E2M1): x -> MXFP4 along
 *              d; h rounded to fp32, then -> MXFP4 along f.
 * MXFP8 block rule (OCP v1.0 conversion): s = floor(log2(amax)) - 8 (E4M3
 * emax = 8), clamped to [-127, 127]; s = 0 when amax = 0; element code =
 * E4M3 round-to-nearest-even of v / 2^s, saturating to +-448.
 * MXFP4 activation block rule (the same conversion for E2M1): s =
 * floor(log2(amax)) - 2 (E2M1 emax = 2), clamped, s = 0 for amax = 0; code =
 * E2M1 round-to-nearest-even of v / 2^s (ties to the even code), saturating
 * to +-6; a negative value that rounds to zero keeps its sign (code 8).
 *
 * Q2_K-style super-block (256 weights = 16 sub-blocks of 16, 84 bytes):
 * bytes 0..15 scale byte j (low nibble sc_j, high nibble m_j); bytes 16..79
 * 2-bit q, weight i at byte 16 + i/4, bits 2*(i%4); bytes 80..81 fp16 d,
 * 82..83 fp16 dmin (little endian).  w_i = d*sc_j*q_i - dmin*m_j, j = i/16.
 *
 * NaN or infinite logits/activations are outside the layer's domain.
 * Parity pins live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ACT_EXACT = 0, ACT_MXFP8 = 1, ACT_MXFP8_X_ONLY = 2, ACT_MXFP4 = 3 };
enum { DOWN_MXFP4 = 0, DOWN_Q2K = 1 };

/* ------------------------------------------------------------------ */
/* number formats                                                      */
/* ------------------------------------------------------------------ */

/* E2M1 code (4 bits) -> value. */
double ds4o_e2m1(unsigned code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[code & 7u];
    return (code & 8u) ? -v : v;
}

/* E8M0 byte -> 2^(b-127); 0xFF is NaN. */
double ds4o_e8m0(unsigned b)
{
    if ((b & 0xFFu) == 0xFFu) return NAN;
    return ldexp(1.0, (int)(b & 0xFFu) - 127);
}

/* IEEE binary16 bits -> value. */
double ds4o_half(uint16_t h)
{
    int sign = h >> 15, ex = (h >> 10) & 31, man = h & 1023;
    double v;
    if (ex == 0) v = ldexp((double)man, -24);
    else if (ex == 31) v = man ? NAN : INFINITY;
    else v = ldexp((double)(1024 + man), ex - 25);
    return sign ? -v : v;
}

/* bfloat16 bits -> value (exact). */
double ds4o_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* E4M3 byte -> value. */
double ds4o_e4m3_decode(uint8_t b)
{
    int sign = b >> 7, ex = (b >> 3) & 15, man = b & 7;
    double v;
    if (ex == 15 && man == 7) return NAN;
    if (ex == 0) v = ldexp((double)man, -9);
    else v = ldexp((double)(8 + man), ex - 10);
    return sign ? -v : v;
}

/* value -> E4M3 byte, round to nearest even, saturating to +-448. */
uint8_t ds4o_e4m3_encode(double v)
{
    uint8_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                 /* subnormal range: multiples of 2^-9 */
        double q = nearbyint(ldexp(a, 9));    /* 0..8; 8 is the smallest normal */
        if (q >= 8.0) return sign | 0x08;
        return sign | (uint8_t)q;
    }
    int e;
    frexp(a, &e);                             /* a = m*2^e, m in [0.5,1) */
    e -= 1;                                   /* a = 1.f * 2^e, e in [-6, 8] */
    double m = nearbyint((ldexp(a, -e) - 1.0) * 8.0);   /* 0..8 */
    if (m >= 8.0) { m = 0.0; e += 1; }
    if (e > 8 || (e == 8 && m > 6.0)) return sign | 0x7E;
    return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

/* MXFP8 along one 32-element block: returns the E8M0 byte, writes codes. */
uint8_t ds4o_mxfp8_block(const double *v, uint8_t *codes)
{
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) if (fabs(v[i]) > amax) amax = fabs(v[i]);
    int s = 0;
    if (amax > 0.0) {
        int e;
        frexp(amax, &e);          /* floor(log2(amax)) = e - 1 */
        s = (e - 1) - 8;
        if (s < -127) s = -127;
        if (s > 127) s = 127;
    }
    for (int i = 0; i < 32; ++i) codes[i] = ds4o_e4m3_encode(ldexp(v[i], -s));
    return (uint8_t)(s + 127);
}

/* In-place: replace v[0..n) (n % 32 == 0) by its MXFP8 dequantised value. */
static void mxfp8_roundtrip(double *v, int n)
{
    uint8_t codes[32];
    for (int b = 0; b < n; b += 32) {
        uint8_t sb = ds4o_mxfp8_block(v + b, codes);
        double sc = ldexp(1.0, (int)sb - 127);
        for (int i = 0; i < 32; ++i) v[b + i] = ds4o_e4m3_decode(codes[i]) * sc;
    }
}

/* value -> E2M1 code (bit 3 sign), round to nearest even code, saturating to +-6. */
uint8_t ds4o_e2m1_encode(double v)
{
    uint8_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x8 : 0x0;
    double a = fabs(v);
    if (a >= 6.0) return sign | 7;
    if (a < 1.0) {                            /* subnormal step 0.5: codes 0, 1 and 2 (= 1.0) */
        return sign | (uint8_t)nearbyint(a * 2.0);
    }
    int e;
    frexp(a, &e);
    e -= 1;                                   /* a = 1.m * 2^e, e in {0, 1, 2} */
    double m = nearbyint((ldexp(a, -e) - 1.0) * 2.0);   /* 0, 1 or 2 */
    if (m >= 2.0) { m = 0.0; e += 1; }
    if (e > 2) return sign | 7;
    return sign | (uint8_t)(((e + 1) << 1) | (int)m);
}

/* MXFP4 of one 32-element activation block: returns the E8M0 byte, writes
 * one E2M1 code (0..15) per element. */
uint8_t ds4o_mxfp4_act_block(const double *v, uint8_t *codes)
{
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) if (fabs(v[i]) > amax) amax = fabs(v[i]);
    int s = 0;
    if (amax > 0.0) {
        int e;
        frexp(amax, &e);          /* floor(log2(amax)) = e - 1 */
        s = (e - 1) - 2;
        if (s < -127) s = -127;
        if (s > 127) s = 127;
    }
    for (int i = 0; i < 32; ++i) codes[i] = ds4o_e2m1_encode(ldexp(v[i], -s));
    return (uint8_t)(s + 127);
}

/* In-place: replace v[0..n) (n % 32 == 0) by its MXFP4 dequantised value. */
static void mxfp4_roundtrip(double *v, int n)
{
    uint8_t codes[32];
    for (int b = 0; b < n; b += 32) {
        uint8_t sb = ds4o_mxfp4_act_block(v + b, codes);
        double sc = ldexp(1.0, (int)sb - 127);
        for (int i = 0; i < 32; ++i) v[b + i] = ds4o_e2m1(codes[i]) * sc;
    }
}

/* One Q2_K-style weight: super-block pointer, index 0..255. */
double ds4o_q2k_weight(const uint8_t *sb, int i)
{
    uint16_t dbits = (uint16_t)(sb[80] | (sb[81] << 8));
    uint16_t mbits = (uint16_t)(sb[82] | (sb[83] << 8));
    double d = ds4o_half(dbits), dmin = ds4o_half(mbits);
    int j = i / 16;
    int sc = sb[j] & 15, mm = sb[j] >> 4;
    int q = (sb[16 + i / 4] >> (2 * (i % 4))) & 3;
    return d * sc * q - dmin * mm;
}

/* ------------------------------------------------------------------ */
/* weights                                                             */
/* ------------------------------------------------------------------ */
typedef struct {
    int d, E, f, k, down_fmt;
    const uint8_t *gate_codes, *gate_scales;  /* [E][f][d/2], [E][f][d/32] */
    const uint8_t *up_codes, *up_scales;
    const uint8_t *down_codes, *down_scales;  /* MXFP4 [E][d][f/2], [E][d][f/32] */
    const uint8_t *down_q2k;                  /* Q2_K  [E][d][f/256][84] */
} ds4o_layer;

/* Dot of one MXFP4 row (K elements) with v: sum_c e2m1(code_c)*2^(s-127)*v_c. */
static double mxfp4_row_dot(const uint8_t *codes, const uint8_t *scales, int K, const double *v)
{
    double acc = 0.0;
    for (int c = 0; c < K; ++c) {
        unsigned byte = codes[c / 2];
        unsigned code = (c & 1) ? (byte >> 4) : (byte & 15u);
        double w = ds4o_e2m1(code) * ds4o_e8m0(scales[c / 32]);
        acc += w * v[c];
    }
    return acc;
}

static double q2k_row_dot(const uint8_t *row, int K, const double *v)
{
    double acc = 0.0;
    for (int c = 0; c < K; ++c) acc += ds4o_q2k_weight(row + (size_t)(c / 256) * 84, c % 256) * v[c];
    return acc;
}

/* One expert's FFN on the activation vector xin[d]; writes y[d]. */
static void expert_ffn(const ds4o_layer *L, int e, const double *xin, int act_mode, double *y)
{
    const int d = L->d, f = L->f;
    double *h = (double *)malloc(sizeof(double) * (size_t)f);
    #pragma omp parallel for schedule(static)
    for (int i = 0; i < f; ++i) {
        size_t r = (size_t)e * f + i;
        double g = mxfp4_row_dot(L->gate_codes + r * (d / 2), L->gate_scales + r * (d / 32), d, xin);
        double u = mxfp4_row_dot(L->up_codes + r * (d / 2), L->up_scales + r * (d / 32), d, xin);
        h[i] = g / (1.0 + exp(-g)) * u;
    }
    if (act_mode == ACT_MXFP8 || act_mode == ACT_MXFP4) {
        for (int i = 0; i < f; ++i) h[i] = (double)(float)h[i];
        if (act_mode == ACT_MXFP8) mxfp8_roundtrip(h, f);
        else mxfp4_roundtrip(h, f);
    }
    #pragma omp parallel for schedule(static)
    for (int m = 0; m < d; ++m) {
        size_t r = (size_t)e * d + m;
        if (L->down_fmt == DOWN_Q2K)
            y[m] = q2k_row_dot(L->down_q2k + r * (size_t)(f / 256) * 84, f, h);
        else
            y[m] = mxfp4_row_dot(L->down_codes + r * (f / 2), L->down_scales + r * (f / 32), f, h);
    }
    free(h);
}

static void token_input(const ds4o_layer *L, const uint16_t *x_row, int act_mode, double *xin)
{
    for (int c = 0; c < L->d; ++c) xin[c] = ds4o_bf16(x_row[c]);
    if (act_mode == ACT_MXFP4) mxfp4_roundtrip(xin, L->d);
    else if (act_mode != ACT_EXACT) mxfp8_roundtrip(xin, L->d);
}

/* ------------------------------------------------------------------ */
/* routing and grouping                                                */
/* ------------------------------------------------------------------ */
typedef struct { double v; int i; } keyed;

static int cmp_keyed(const void *a, const void *b)
{
    const keyed *x = (const keyed *)a, *y = (const keyed *)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

/* Top-k by (value desc, index asc) and softmax over the selected k. */
void ds4o_route(const float *logits, int T, int E, int k, int32_t *idx, double *w)
{
    keyed *buf = (keyed *)malloc(sizeof(keyed) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double v = logits[(size_t)t * E + e];
            buf[e].v = isnan(v) ? -INFINITY : v;
            buf[e].i = e;
        }
        qsort(buf, (size_t)E, sizeof(keyed), cmp_keyed);
        double z = 0.0;
        for (int j = 0; j < k; ++j) z += exp(buf[j].v - buf[0].v);
        for (int j = 0; j < k; ++j) {
            idx[(size_t)t * k + j] = buf[j].i;
            w[(size_t)t * k + j] = exp(buf[j].v - buf[0].v) / z;
        }
    }
    free(buf);
}

/* counts[E], offsets[E+1], pairs sorted by (expert, token): perm_tok/perm_slot
 * [T*k], inv[T*k] = position of pair (t, j) in that order. */
void ds4o_group(const int32_t *idx, int T, int E, int k, int32_t *counts, int32_t *offsets,
                int32_t *perm_tok, int32_t *perm_slot, int32_t *inv)
{
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int p = 0; p < T * k; ++p) counts[idx[p]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int pos = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (idx[(size_t)t * k + j] == e) {
                    perm_tok[pos] = t;
                    perm_slot[pos] = j;
                    inv[(size_t)t * k + j] = pos;
                    ++pos;
                }
}

/* ------------------------------------------------------------------ */
/* layer forward                                                       */
/* ------------------------------------------------------------------ */
static ds4o_layer make_layer(int d, int E, int f, int k, int down_fmt,
                             const uint8_t *gc, const uint8_t *gs, const uint8_t *uc, const uint8_t *us,
                             const uint8_t *dc, const uint8_t *ds, const uint8_t *dq)
{
    ds4o_layer L = {d, E, f, k, down_fmt, gc, gs, uc, us, dc, ds, dq};
    return L;
}

/* Routed forward for the tokens listed in tokens[0..n): out[n][d] (fp64).
 * idx/w are the routing of those tokens' rows (row t of the full batch). */
void ds4o_forward(int d, int E, int f, int k, int down_fmt, int act_mode,
                  const uint8_t *gc, const uint8_t *gs, const uint8_t *uc, const uint8_t *us,
                  const uint8_t *dc, const uint8_t *ds, const uint8_t *dq,
                  const uint16_t *x, const int32_t *idx, const double *w,
                  int n, const int32_t *tokens, double *out)
{
    ds4o_layer L = make_layer(d, E, f, k, down_fmt, gc, gs, uc, us, dc, ds, dq);
    double *xin = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int q = 0; q < n; ++q) {
        int t = tokens[q];
        double *o = out + (size_t)q * d;
        for (int m = 0; m < d; ++m) o[m] = 0.0;
        token_input(&L, x + (size_t)t * d, act_mode, xin);
        for (int j = 0; j < k; ++j) {
            expert_ffn(&L, idx[(size_t)t * k + j], xin, act_mode, y);
            double wj = w[(size_t)t * k + j];
            for (int m = 0; m < d; ++m) o[m] += wj * y[m];
        }
    }
    free(xin);
    free(y);
}

/* Brute force: every expert's FFN for every listed token, weighted by a mask
 * that is w[t,j] for the routed experts and 0 for all others. */
void ds4o_forward_dense(int d, int E, int f, int k, int down_fmt, int act_mode,
                        const uint8_t *gc, const uint8_t *gs, const uint8_t *uc, const uint8_t *us,
                        const uint8_t *dc, const uint8_t *ds, const uint8_t *dq,
                        const uint16_t *x, const int32_t *idx, const double *w,
                        int n, const int32_t *tokens, double *out)
{
    ds4o_layer L = make_layer(d, E, f, k, down_fmt, gc, gs, uc, us, dc, ds, dq);
    double *xin = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int q = 0; q < n; ++q) {
        int t = tokens[q];
        double *o = out + (size_t)q * d;
        for (int m = 0; m < d; ++m) o[m] = 0.0;
        token_input(&L, x + (size_t)t * d, act_mode, xin);
        for (int e = 0; e < E; ++e) {
            double mask = 0.0;
            for (int j = 0; j < k; ++j)
                if (idx[(size_t)t * k + j] == e) mask = w[(size_t)t * k + j];
            expert_ffn(&L, e, xin, act_mode, y);
            for (int m = 0; m < d; ++m) o[m] += mask * y[m];
        }
    }
    free(xin);
    free(y);
}

/* Decoded weight matrices of one expert (fp64), for library-routine checks:
 * wg[f][d], wu[f][d], wd[d][f]. */
void ds4o_dequant_expert(int d, int E, int f, int down_fmt, int e,
                         const uint8_t *gc, const uint8_t *gs, const uint8_t *uc, const uint8_t *us,
                         const uint8_t *dc, const uint8_t *ds, const uint8_t *dq,
                         double *wg, double *wu, double *wd)
{
    (void)E;
    for (int i = 0; i < f; ++i) {
        size_t r = (size_t)e * f + i;
        for (int c = 0; c < d; ++c) {
            unsigned bg = gc[r * (d / 2) + c / 2], bu = uc[r * (d / 2) + c / 2];
            unsigned cg = (c & 1) ? bg >> 4 : bg & 15u, cu = (c & 1) ? bu >> 4 : bu & 15u;
            wg[(size_t)i * d + c] = ds4o_e2m1(cg) * ds4o_e8m0(gs[r * (d / 32) + c / 32]);
            wu[(size_t)i * d + c] = ds4o_e2m1(cu) * ds4o_e8m0(us[r * (d / 32) + c / 32]);
        }
    }
    for (int m = 0; m < d; ++m) {
        size_t r = (size_t)e * d + m;
        for (int c = 0; c < f; ++c) {
            if (down_fmt == DOWN_Q2K) {
                wd[(size_t)m * f + c] = ds4o_q2k_weight(dq + (r * (size_t)(f / 256) + c / 256) * 84, c % 256);
            } else {
                unsigned b = dc[r * (f / 2) + c / 2];
                unsigned cd = (c & 1) ? b >> 4 : b & 15u;
                wd[(size_t)m * f + c] = ds4o_e2m1(cd) * ds4o_e8m0(ds[r * (f / 32) + c / 32]);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* router projection and shared expert (original precision, bf16)      */
/* ------------------------------------------------------------------ */
/* "DwarfStar実地分析", §GGUFの対応範囲は意図的に狭い: the shared expert, the
 * projections and the routing stay at original precision; only the routed
 * experts are quantised.  Weights and activations here are bf16.
 *
 * Router: logits[t][e] = sum_c Wr[e][c] * x[t][c], exact in fp64 (the caller
 * rounds to fp32, the precision the kernel takes the top-k decision in). */
void ds4o_router_logits(int d, int E, const uint16_t *wr, const uint16_t *x, int T, double *logits)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += ds4o_bf16(wr[(size_t)e * d + c]) * ds4o_bf16(x[(size_t)t * d + c]);
            logits[(size_t)t * E + e] = acc;
        }
}

/* bf16 round-to-nearest-even of an fp32 value, returned as its value. */
static double bf16_round(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;
    float r;
    memcpy(&r, &u, 4);
    return (double)r;
}

/* Shared expert for the listed tokens: y[q][m] = sum_i Wd[m][i] * h_i with
 * g = Wg.x, u = Wu.x (fp64), h = bf16(fp32(g/(1+exp(-g))*u)) -- h kept in
 * bf16 like the model's activations, the rounding decided on fp32 h as the
 * kernel does.  Wg, Wu [fs][d], Wd [d][fs] bf16. */
void ds4o_shared_ffn(int d, int fs, const uint16_t *wg, const uint16_t *wu, const uint16_t *wd,
                     const uint16_t *x, int n, const int32_t *tokens, double *y)
{
    double *xin = (double *)malloc(sizeof(double) * (size_t)d);
    double *h = (double *)malloc(sizeof(double) * (size_t)fs);
    for (int q = 0; q < n; ++q) {
        const int t = tokens[q];
        for (int c = 0; c < d; ++c) xin[c] = ds4o_bf16(x[(size_t)t * d + c]);
        #pragma omp parallel for schedule(static)
        for (int i = 0; i < fs; ++i) {
            double g = 0.0, u = 0.0;
            for (int c = 0; c < d; ++c) {
                g += ds4o_bf16(wg[(size_t)i * d + c]) * xin[c];
                u += ds4o_bf16(wu[(size_t)i * d + c]) * xin[c];
            }
            h[i] = bf16_round((float)(g / (1.0 + exp(-g)) * u));
        }
        #pragma omp parallel for schedule(static)
        for (int m = 0; m < d; ++m) {
            double acc = 0.0;
            for (int i = 0; i < fs; ++i) acc += ds4o_bf16(wd[(size_t)m * fs + i]) * h[i];
            y[(size_t)q * d + m] = acc;
        }
    }
    free(xin);
    free(h);
}

/* MXFP8 of n values (n % 32 == 0): codes[n], scales[n/32]. */
void ds4o_mxfp4_act(const double *v, int n, uint8_t *codes, uint8_t *scales)
{
    for (int b = 0; b < n / 32; ++b) scales[b] = ds4o_mxfp4_act_block(v + 32 * b, codes + 32 * b);
}

void ds4o_mxfp8(const double *v, int n, uint8_t *codes, uint8_t *scales)
{
    for (int b = 0; b < n / 32; ++b) scales[b] = ds4o_mxfp8_block(v + 32 * b, codes + 32 * b);
}

int ds4o_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
