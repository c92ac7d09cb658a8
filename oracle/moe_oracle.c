/*
 * moe_oracle.c -- plain, slow, CPU-only oracle of the fused FP8 Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the package smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or constant
 * generator with the CUDA library, and it never calls it.
 *
 * Source pages (cited by title and section):
 *   [WT1] "Mega-MoE 内核代码导读：从 Dispatch 到 WGMMA 的融合流水线" (mlqm.cn/news/378595)
 *   [WT2] Mega-MoE walkthrough, part 2: index table vs. pull, round-robin, L1 pool
 *         (kwkr.cn/news/1317662)
 *   [SYM] "DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析"
 *   [DC]  "Dispatch/Combine: 博客理论 ↔ DeepEP 源码 ↔ DeepGEMM Mega MoE 三方对比分析"
 *   [FUSED] "MOE融合算子" (mkbk-pku.cn/pages/6d132f)
 * FP8 E4M3 follows the OCP 8-bit floating point specification (bias 7, no infinities,
 * S.1111.111 is NaN, largest finite magnitude 448).
 *
 * Readings of points the pages leave open (each is also listed in the design notes):
 *   - quantisation scale of a group: sf = max(amax, 1e-4) / 448 in fp32, not rounded to
 *     a power of two; values are encoded round-to-nearest-even with saturation to +-448.
 *     The power-of-two variant (UE8M0-representable scales, for the hardware block-scaled
 *     path): sf = the smallest power of two >= max(amax, 1e-4) / 448 (fp32 quotient), so
 *     every |value / sf| <= 448;
 *   - SwiGLU: h = silu(gate) * up with silu(z) = z / (1 + exp(-z)), gate = rows 0..I-1 of
 *     the gate_up weight, up = rows I..2I-1; h is rounded to fp32 and re-quantised per
 *     1x128 group before the down projection;
 *   - the top-k gate weight is applied after the down projection (plain definition
 *     Output = sum_k w_k * Expert_k), sums in ascending k, result rounded to bf16;
 *   - expert id -1 means "skip"; any other id outside [0, E) is an error.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ FP8 E4M3 ---- */

/* Value of one E4M3 code, written out from the format definition. */
double orc_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int expo = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant / 8.0, 1 - 7);          /* subnormal: 0.m * 2^(1-bias) */
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7); /* normal: 1.m * 2^(e-bias) */
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------ MXFP4 -------- */

/* Value of one FP4 E2M1 code (the element format of OCP Microscaling MXFP4): bit 3 sign,
 * bits 2..1 exponent with bias 1, bit 0 mantissa; exponent 0 is subnormal (0.m * 2^0),
 * and there is no infinity or NaN. */
double orc_e2m1_decode(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int expo = (code >> 1) & 0x3;
    int mant = code & 0x1;
    double mag;
    if (expo == 0)
        mag = (double)mant / 2.0;                         /* subnormal: 0.m * 2^(1-bias) */
    else
        mag = ldexp(1.0 + (double)mant / 2.0, expo - 1);  /* normal: 1.m * 2^(e-bias) */
    return sign ? -mag : mag;
}

/* Value of one E8M0 (UE8M0) scale byte: 2^(b - 127); 0xFF is NaN (OCP MX scale format). */
double orc_e8m0_decode(uint8_t b)
{
    return b == 0xFF ? NAN : ldexp(1.0, (int)b - 127);
}

static double g_dec[256];
static double g_dec4[16];
static int g_dec_ready = 0;

void orc_init(void)
{
    for (int c = 0; c < 256; ++c)
        g_dec[c] = orc_e4m3_decode((uint8_t)c);
    for (int c = 0; c < 16; ++c)
        g_dec4[c] = orc_e2m1_decode((uint8_t)c);
    g_dec_ready = 1;
}

static inline double dec(uint8_t c) { return g_dec[c]; }

/* Nearest finite E4M3 code to v (ties to the even code), i.e. round-to-nearest-even with
 * saturation: the search runs over every finite non-negative code, so anything beyond
 * 448 lands on 448.  NaN maps to the NaN code 0x7F. */
uint8_t orc_e4m3_encode(float v)
{
    if (!g_dec_ready)
        orc_init();
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(g_dec[c] - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(sign | best);
}

void orc_e4m3_encode_array(int64_t n, const float *v, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(v[i]);
}

void orc_e4m3_decode_array(int64_t n, const uint8_t *c, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_decode(c[i]);
}

/* bf16 round-to-nearest-even of an fp32 value (upper 16 bits after rounding). */
uint16_t orc_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return 0x7FC0;
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

void orc_bf16_rne_array(int64_t n, const float *v, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_rne(v[i]);
}

/* ------------------------------------------------------------------ routing ----- */

/* Packed 64-bit slot claim ([WT1] §4.2, [SYM] §12.2): arrivals are taken in the order
 * given; each adds (1 << 32) | count to one shared word and gets the old low 32 bits as
 * its first slot.  Returns the final word (high = arrivals, low = total slots). */
uint64_t orc_packed_claim(int n, const uint32_t *counts, uint32_t *starts)
{
    uint64_t word = 0;
    for (int i = 0; i < n; ++i) {
        uint64_t old = word;
        word += (1ull << 32) | (uint64_t)counts[i];
        starts[i] = (uint32_t)old;
    }
    return word;
}

/* Round-robin source choice by min-peeling ([WT2] §2.5, [SYM] §7.5).  p is the position
 * of a row among the rows one expert receives; recv[r] is how many rows source r sends
 * it.  Each round, A = number of sources with rows left and L = the smallest such
 * remainder; the round holds A*L rows: position q of the round goes to the (q mod A)-th
 * active source in ascending id, at slot offset + q div A, where offset counts the slots
 * every still-active source used in earlier rounds.  Returns 0, or 1 if p >= sum(recv). */
int orc_round_robin_one(int R, const uint32_t *recv, uint32_t p, uint32_t *src, uint32_t *slot)
{
    uint32_t rem[256];
    uint32_t offset = 0;
    if (R > 256)
        return 1;
    for (int r = 0; r < R; ++r)
        rem[r] = recv[r];
    for (;;) {
        uint32_t A = 0, L = UINT32_MAX;
        for (int r = 0; r < R; ++r)
            if (rem[r] > 0) {
                ++A;
                if (rem[r] < L)
                    L = rem[r];
            }
        if (A == 0)
            return 1;
        if ((uint64_t)p < (uint64_t)A * L) {
            uint32_t which = p % A, nth = 0;
            for (int r = 0; r < R; ++r)
                if (rem[r] > 0) {
                    if (nth == which) {
                        *src = (uint32_t)r;
                        break;
                    }
                    ++nth;
                }
            *slot = offset + p / A;
            return 0;
        }
        p -= A * L;
        offset += L;
        for (int r = 0; r < R; ++r)
            rem[r] -= (rem[r] < L ? rem[r] : L);
    }
}

/* Whole sequence for one expert: positions 0..sum(recv)-1. */
int orc_round_robin(int R, const uint32_t *recv, uint32_t *src, uint32_t *slot)
{
    uint64_t n = 0;
    for (int r = 0; r < R; ++r)
        n += recv[r];
    for (uint64_t p = 0; p < n; ++p)
        if (orc_round_robin_one(R, recv, (uint32_t)p, src + p, slot + p))
            return 1;
    return 0;
}

/* Expert segments of the pool ([WT2] §2.4): expert e starts at M-block
 * sum_{e'<e} ceil(n_e' / BM).  off has E+1 entries. */
void orc_block_offsets(int E, const uint32_t *counts, int BM, int32_t *off)
{
    off[0] = 0;
    for (int e = 0; e < E; ++e)
        off[e + 1] = off[e] + (int32_t)((counts[e] + (uint32_t)BM - 1) / (uint32_t)BM);
}

/* Direct counting of routed rows per expert and per (expert, source); source r owns
 * tokens [r*T/R, (r+1)*T/R).  Returns 0, or 1 if an id other than -1 lies outside [0,E). */
int orc_route_counts(int T, int k, int E, int R, const int64_t *idx,
                     uint32_t *counts, uint32_t *recv)
{
    int bad = 0, Tsrc = T / R;
    memset(counts, 0, sizeof(uint32_t) * (size_t)E);
    memset(recv, 0, sizeof(uint32_t) * (size_t)E * (size_t)R);
    for (int t = 0; t < T; ++t)
        for (int kk = 0; kk < k; ++kk) {
            int64_t e = idx[(int64_t)t * k + kk];
            if (e == -1)
                continue;
            if (e < -1 || e >= E) {
                bad = 1;
                continue;
            }
            counts[e] += 1;
            recv[e * R + t / Tsrc] += 1;
        }
    return bad;
}

/* ------------------------------------------------------------------ expert FFN ---- */

/* Weight formats of the expert FFN.
 *   ORC_W_FP8:   [N][K] e4m3 codes, fp32 scales [N/128][K/128], one per 128x128 block;
 *   ORC_W_MXFP4: [N][K/2] bytes of packed E2M1 codes, element 2j in the low nibble of byte j
 *                and element 2j+1 in the high nibble, with E8M0 scales [N][K/32], one per 32
 *                consecutive elements of a row (the OCP Microscaling MXFP4 block: 32 elements
 *                sharing one power-of-two scale).  The pages name FP8 x FP4 weights for their
 *                SM100 kernel ("DeepGEMM Mega MoE 对称内存（Symmetric Memory）深度分析" §11
 *                file table) without fixing the FP4 format; MXFP4 is the reading taken. */
enum { ORC_W_FP8 = 0, ORC_W_MXFP4 = 1 };

/* Element (n, c) of a row-major weight of K columns: code value times its block scale. */
static inline double wval(int wfmt, const uint8_t *w, const void *s, int64_t n, int64_t c, int64_t K)
{
    if (wfmt == ORC_W_MXFP4) {
        const uint8_t byte = w[n * (K / 2) + c / 2];
        const uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
        return g_dec4[code] * orc_e8m0_decode(((const uint8_t *)s)[n * (K / 32) + c / 32]);
    }
    return dec(w[n * K + c]) * (double)((const float *)s)[(n / 128) * (K / 128) + c / 128];
}

/* One expert on one token ([WT1] §六: Linear1 gate_up, SwiGLU, Linear2 down).
 *   x [H] e4m3 with xsf [H/128];  w1 [2I][H] with s1;  w2 [H][I] with s2, in weight format
 *   wfmt (above).
 * Every operand is dequantised element by element (code value times its block scale),
 * products are summed in double.  Outputs: y [H] (double); optional hq [I] codes and
 * hsf [I/128] scales of the re-quantised SwiGLU output. */
/* Scale rule of the SwiGLU re-quantisation: 0 = max(amax, 1e-4) / 448, 1 = the smallest
 * power of two >= that quotient.  Set before calling the numerics (not thread-safe). */
static int g_scale_pow2 = 0;
void orc_set_scale_rule(int pow2) { g_scale_pow2 = pow2 != 0; }

/* Smallest power of two >= v for a positive normal fp32 v: with v = f * 2^e, f in
 * [0.5, 1), it is v itself when f == 0.5, else 2^e. */
float orc_pow2_ceil(float v)
{
    int e;
    const float f = frexpf(v, &e);
    return f == 0.5f ? v : ldexpf(1.0f, e);
}

void orc_expert_ffn_fmt(int wfmt, int H, int I, const uint8_t *x, const float *xsf,
                        const uint8_t *w1, const void *s1,
                        const uint8_t *w2, const void *s2,
                        double *y, uint8_t *hq, float *hsf)
{
    const int KB2 = I / 128;
    double *dx = (double *)malloc(sizeof(double) * (size_t)H);
    float *h = (float *)malloc(sizeof(float) * (size_t)I);
    double *hd = (double *)malloc(sizeof(double) * (size_t)I);
    if (!g_dec_ready)
        orc_init();

    for (int c = 0; c < H; ++c)
        dx[c] = dec(x[c]) * (double)xsf[c / 128];

    for (int n = 0; n < I; ++n) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            g += dx[c] * wval(wfmt, w1, s1, n, c, H);
            u += dx[c] * wval(wfmt, w1, s1, I + n, c, H);
        }
        double silu = g / (1.0 + exp(-g));
        h[n] = (float)(silu * u);
    }

    for (int j = 0; j < KB2; ++j) {
        float amax = 0.0f;
        for (int n = j * 128; n < j * 128 + 128; ++n)
            amax = fmaxf(amax, fabsf(h[n]));
        float sf = fmaxf(amax, 1e-4f) / 448.0f;
        if (g_scale_pow2)
            sf = orc_pow2_ceil(sf);
        for (int n = j * 128; n < j * 128 + 128; ++n) {
            uint8_t q = orc_e4m3_encode(h[n] / sf);
            hd[n] = dec(q) * (double)sf;
            if (hq)
                hq[n] = q;
        }
        if (hsf)
            hsf[j] = sf;
    }

    for (int c = 0; c < H; ++c) {
        double acc = 0.0;
        for (int n = 0; n < I; ++n)
            acc += hd[n] * wval(wfmt, w2, s2, c, n, I);
        y[c] = acc;
    }
    free(dx);
    free(h);
    free(hd);
}

/* The FP8-weight form of orc_expert_ffn_fmt. */
void orc_expert_ffn(int H, int I, const uint8_t *x, const float *xsf,
                    const uint8_t *w1, const float *s1,
                    const uint8_t *w2, const float *s2,
                    double *y, uint8_t *hq, float *hsf)
{
    orc_expert_ffn_fmt(ORC_W_FP8, H, I, x, xsf, w1, s1, w2, s2, y, hq, hsf);
}

/* ------------------------------------------------------------------ layer ---------- */

/* Diagnostic combine mode ([SYM] §8.2 keeps the per-slot combine planes in bf16): when set,
 * each slot's weighted expert output is rounded to fp32 and then to bf16 (one plane value),
 * and the planes are summed in fp32 in ascending k, as a bf16 combine buffer followed by an
 * fp32 reduce computes it.  Off (default): the sum of w_k * y_k is kept in double.  Set
 * before calling the numerics (not thread-safe). */
static int g_plane_bf16 = 0;
void orc_set_plane_bf16(int on) { g_plane_bf16 = on != 0; }

static inline float bf16_bits_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* The layer on a list of tokens: out[t] = bf16( sum over k ascending of w[t,k] *
 * Expert_{idx[t,k]}(x[t]) ), skipping idx == -1; a token with no valid slot gives 0
 * ([DC] §1: Output(T) = sum_k w_k * Expert_k(T)).  out_bf16 [ntok][H] receives the bf16
 * bits, out_f32 (optional) the fp32 value before the bf16 rounding.  Returns 1 if a
 * token names an expert outside [0, E) other than -1 (that slot is skipped). */
int orc_forward_tokens_fmt(int wfmt, int T, int H, int I, int E, int k,
                           const uint8_t *x, const float *xsf,
                           const int64_t *idx, const float *w,
                           const uint8_t *w1, const void *s1,
                           const uint8_t *w2, const void *s2,
                           int ntok, const int32_t *tokens,
                           uint16_t *out_bf16, float *out_f32)
{
    int bad = 0;
    (void)T;
    if (!g_dec_ready)
        orc_init();
    /* per-expert strides of the weights (bytes) and scales (elements of their type) */
    const int mx = wfmt == ORC_W_MXFP4;
    const int64_t w1e = mx ? (int64_t)2 * I * (H / 2) : (int64_t)2 * I * H;
    const int64_t w2e = mx ? (int64_t)H * (I / 2) : (int64_t)H * I;
    const int64_t s1e = mx ? (int64_t)2 * I * (H / 32) : (int64_t)(2 * I / 128) * (H / 128);
    const int64_t s2e = mx ? (int64_t)H * (I / 32) : (int64_t)(H / 128) * (I / 128);
    const size_t ssz = mx ? sizeof(uint8_t) : sizeof(float);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int i = 0; i < ntok; ++i) {
        const int t = tokens[i];
        double *acc = (double *)calloc((size_t)H, sizeof(double));
        float *accf = (float *)calloc((size_t)H, sizeof(float));
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
        for (int kk = 0; kk < k; ++kk) {
            int64_t e = idx[(int64_t)t * k + kk];
            if (e == -1)
                continue;
            if (e < -1 || e >= E) {
                bad |= 1;
                continue;
            }
            orc_expert_ffn_fmt(wfmt, H, I, x + (int64_t)t * H, xsf + (int64_t)t * (H / 128),
                               w1 + e * w1e, (const char *)s1 + e * s1e * ssz,
                               w2 + e * w2e, (const char *)s2 + e * s2e * ssz, y, NULL, NULL);
            const double wk = (double)w[(int64_t)t * k + kk];
            if (g_plane_bf16) {
                for (int c = 0; c < H; ++c)
                    accf[c] += bf16_bits_value(orc_bf16_rne((float)(wk * y[c])));
            } else {
                for (int c = 0; c < H; ++c)
                    acc[c] += wk * y[c];
            }
        }
        for (int c = 0; c < H; ++c) {
            float f = g_plane_bf16 ? accf[c] : (float)acc[c];
            out_bf16[(int64_t)i * H + c] = orc_bf16_rne(f);
            if (out_f32)
                out_f32[(int64_t)i * H + c] = f;
        }
        free(acc);
        free(accf);
        free(y);
    }
    return bad;
}

/* The FP8-weight form of orc_forward_tokens_fmt. */
int orc_forward_tokens(int T, int H, int I, int E, int k,
                       const uint8_t *x, const float *xsf,
                       const int64_t *idx, const float *w,
                       const uint8_t *w1, const float *s1,
                       const uint8_t *w2, const float *s2,
                       int ntok, const int32_t *tokens,
                       uint16_t *out_bf16, float *out_f32)
{
    return orc_forward_tokens_fmt(ORC_W_FP8, T, H, I, E, k, x, xsf, idx, w, w1, s1, w2, s2, ntok, tokens,
                                  out_bf16, out_f32);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
