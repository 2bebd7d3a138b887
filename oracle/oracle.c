/*
 * oracle.c -- plain, slow, scalar fp64 CPU oracle for the two fused ops
 *
 *   fused_add_rms_norm -> quant_fp8   (fuse_norm_quant)
 *   silu_and_mul       -> quant_fp8   (fuse_act_quant)
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or constant with the CUDA library; it has its own bf16
 * and e4m3 codecs and keeps every intermediate in fp64.
 *
 * Sources, cited by page title and section:
 *  [FUS]  "Fusion torch.compile passes" (data-sketchers.com wiki, vLLM
 *         design-fusions page): section "RMSNorm + Quantization
 *         (fuse_norm_quant)" -- the two norm variants, the in-place residual
 *         update, and the three FP8 scale modes (static per-tensor, dynamic
 *         per-token, dynamic per-token-group of 128/64 columns); section
 *         "SiLU+Mul + Quantization (fuse_act_quant)" -- SiLU(gate)*up then
 *         FP8 quant without materialising the activation; "Quick Reference"
 *         table rows fuse_norm_quant / fuse_act_quant.
 *         Section "MLA Dual RMSNorm (fuse_mla_dual_rms_norm)" -- the
 *         paired q_c / kv_c RMSNorms of MLA attention (each with its own
 *         weight and eps) in one call, and its per-token-quant variant where
 *         q goes to FP8 with a per-token scale and kv stays bf16.
 *         Section "RMSNorm + Padding (fuse_act_padding)" -- residual add +
 *         RMSNorm fused with the padding of the hidden dimension to the
 *         multiple the next GEMM needs (GPT-OSS, hidden 2880).
 *         Section "QK Norm + RoPE (enable_qk_norm_rope_fusion)" -- split
 *         QKV, per-head RMSNorm of Q and K, then rotary embedding, in one
 *         kernel (models that normalise Q and K per head before RoPE).
 *  [NVFP4] NVIDIA's NVFP4 format ([FUS] "Quick Reference" names FP4 for both
 *         fusions and the "Support Matrix" NVFP4 dynamic on sm100+, but the
 *         pages define neither): E2M1 elements (the OCP Microscaling spec's
 *         FP4: sign, 2 exponent bits with bias 1, 1 mantissa bit; values
 *         +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}), blocks of 16 consecutive
 *         elements, an E4M3 scale per block and an fp32 scale per tensor.
 *  [OFP8] OCP 8-bit Floating Point Specification (OFP8), E4M3 encoding:
 *         bias 7, no infinities, S.1111.111 is NaN, max normal 448
 *         (S.1111.110), min normal 2^-6, min subnormal 2^-9.
 *
 * The pages never write the RMSNorm, SiLU or quantisation formulas out.  The
 * readings taken here (each the plainest one the pages support):
 *  - RMSNorm: y_j = r_j / sqrt(mean_j(r_j^2) + eps) * w_j, eps inside the
 *    square root, the mean over the whole hidden dimension.
 *  - The fused-add variant normalises the bf16-rounded sum r = bf16(x + res),
 *    which is also the residual it writes back.
 *  - y is NOT rounded to bf16 before quantising: the fusion exists to avoid
 *    materialising that full-precision intermediate.
 *  - Scales are dequantisation scales: q = e4m3(y / s), so y ~= q * s.
 *    Dynamic scales are s = fp32(max(amax, A_MIN) / 448), the division uses
 *    the stored fp32 scale, and A_MIN is the fp32 number nearest 1e-10
 *    (it only keeps an all-zero row or group away from 0/0).
 *  - Per-group scales cover G contiguous columns; the scale tensor is
 *    [T, n/G] fp32, row-major.
 *  - The per-group options that the GEMM side on sm100 wants (the "Support
 *    Matrix" ties per-group FP8 there to DeepGEMM; the formats come from
 *    the OCP Microscaling spec, E8M0): UE8M0 scales are the smallest power
 *    of two >= max(amax, A_MIN) / 448 (an exponent with no mantissa), and
 *    the column-major layout stores scale (t, g) at [g, t] of a [n/G, T4]
 *    tensor, T4 = T rounded up to a multiple of 4 (16-byte rows); the
 *    padding columns are not written.
 *  - silu(g) = g / (1 + exp(-g)); the gate is columns [0, I) and the up
 *    projection columns [I, 2I) of one [T, 2I] row.
 *  - A norm whose output stays in the activation dtype (the MLA dual
 *    norm's bf16 rows) rounds y once, to nearest even bf16.
 *  - e4m3 conversion rounds to nearest, ties to even mantissa, saturates
 *    finite overflow (and infinity) to +-448, keeps the sign of zero, and
 *    maps NaN to 0x7F.
 *  - NaN and infinite inputs: every formula above is evaluated in IEEE
 *    arithmetic as written, and the amax of a row or group is the largest
 *    |y| among its non-NaN elements (a NaN never wins the comparison; 0 when
 *    there is none).  So a NaN in r makes inv and every y NaN; an infinity
 *    in r makes sum(r^2) infinite and inv = 0, so y = +-0 at finite r and
 *    inf * 0 = NaN at the infinite one; silu(-inf) = -inf / inf is NaN.
 *
 * Build: plain C11, -ffp-contract=off so that no multiply-add is fused and
 * the results are the same on every host architecture.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_STATIC = 0, ORC_PER_TOKEN = 1, ORC_PER_GROUP = 2 };
/* Per-group options, or-ed into the mode: power-of-two (UE8M0) scales and a
 * column-major scale layout. */
enum { ORC_UE8M0 = 0x100, ORC_COL_MAJOR = 0x200 };

#define ORC_E4M3_MAX 448.0

/* ------------------------------------------------------------------ codecs */

/* Round a finite v to the nearest number with `p` significant bits whose
 * exponent is at least `emin` (below it the spacing stays 2^(emin-p+1), i.e.
 * gradual underflow), ties to even.  Division and multiplication by the power
 * of two `quantum` are exact, and nearbyint rounds half to even under the
 * default rounding mode, so the only rounding is the one intended. */
static double round_to_precision(double v, int p, int emin)
{
    if (v == 0.0 || !isfinite(v))
        return v;
    int e = ilogb(v);
    if (e < emin)
        e = emin;
    double quantum = ldexp(1.0, e - (p - 1));
    double m = v / quantum;
    return nearbyint(m) * quantum;
}

/* bf16 is the upper half of an IEEE binary32, so decoding is exact. */
double orc_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* bf16: 8 significant bits, emin -126, overflow to infinity (IEEE RNE). */
uint16_t orc_bf16_encode(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    double r = round_to_precision(v, 8, -126);
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max)
        r = signbit(r) ? -INFINITY : INFINITY;
    float f = (float)r; /* exact: r is a bf16 value or an infinity */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

double orc_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 0x7;
    if (e == 15 && m == 7)
        return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9)           /* 0.m * 2^-6 */
                          : ldexp((double)(8 + m), e - 10); /* 1.m * 2^(e-7) */
    return s ? -mag : mag;
}

/* e4m3 (OCP E4M3FN): 4 significant bits, emin -6, satfinite at 448. */
uint8_t orc_e4m3_encode(double v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    double r = isinf(a) ? ORC_E4M3_MAX : round_to_precision(a, 4, -6);
    if (r > ORC_E4M3_MAX)
        r = ORC_E4M3_MAX;
    if (r == 0.0)
        return sign;
    int e = ilogb(r);
    if (e < -6) /* subnormal: r = k * 2^-9, k = 1..7 */
        return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    int mant = (int)((r / ldexp(1.0, e) - 1.0) * 8.0);
    return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | mant));
}

/* e2m1 ([NVFP4] elements): 2 significant bits, emin 0 (subnormal spacing
 * 0.5), no infinities or NaN; RNE with saturation at 6.  Code: sign bit 3,
 * exponent bits 2..1, mantissa bit 0. */
double orc_e2m1_decode(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

uint8_t orc_e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    double r = isinf(a) ? 6.0 : round_to_precision(a, 2, 0);
    if (r > 6.0)
        r = 6.0;
    if (r == 0.0) /* keeps the sign of zero */
        return sign;
    int e = ilogb(r);
    if (e < 0) /* subnormal: 0.5 */
        return (uint8_t)(sign | 0x1);
    int mant = (int)((r / ldexp(1.0, e) - 1.0) * 2.0);
    return (uint8_t)(sign | (uint8_t)(((e + 1) << 1) | mant));
}

void orc_e2m1_decode_n(double *out, const uint8_t *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e2m1_decode(in[i]);
}

void orc_e2m1_encode_n(uint8_t *out, const double *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e2m1_encode(in[i]);
}

void orc_bf16_decode_n(double *out, const uint16_t *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_decode(in[i]);
}

void orc_bf16_encode_n(uint16_t *out, const double *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_encode(in[i]);
}

void orc_e4m3_decode_n(double *out, const uint8_t *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_decode(in[i]);
}

void orc_e4m3_encode_n(uint8_t *out, const double *in, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(in[i]);
}

/* ------------------------------------------------------------ quantisation */

/* The fp32 number nearest 1e-10: floor on a dynamic amax. */
double orc_amax_floor(void) { return (double)1e-10f; }

static float dynamic_scale(double amax)
{
    double a = amax > orc_amax_floor() ? amax : orc_amax_floor();
    return (float)(a / ORC_E4M3_MAX);
}

/* UE8M0 scale: the smallest power of two s with s >= max(amax, A_MIN)/448,
 * decided by exact comparisons with 448 * 2^e. */
static double ue8m0_scale(double amax)
{
    const double a = fmax(amax, orc_amax_floor());
    int e;
    frexp(a / ORC_E4M3_MAX, &e);
    while (ldexp(ORC_E4M3_MAX, e) < a)
        ++e;
    while (ldexp(ORC_E4M3_MAX, e - 1) >= a)
        --e;
    return ldexp(1.0, e);
}

/* quant_fp8 of one row y[0..n) ([FUS] "RMSNorm + Quantization": static
 * per-tensor, dynamic per-token, dynamic per-token-group).
 *   STATIC    : s = scale[0] (input)
 *   PER_TOKEN : s = fp32(max(amax_j |y_j|, A_MIN) / 448), written to scale[t]
 *   PER_GROUP : same over columns [g*G, (g+1)*G), written to scale[t*n/G + g]
 *               (UE8M0: the power-of-two scale; COL_MAJOR: scale[g*T4 + t])
 * then v_j = y_j / s (fp64, with the stored fp32 s) and q_j = e4m3(v_j).
 * v (optional) receives v_j for the tolerance checker.  T: rows in all. */
static void quantize_row(uint8_t *q, double *v, float *scale, const double *y,
                         int64_t t, int64_t T, int64_t n, int mode, int64_t G)
{
    const int flags = mode & ~0xFF;
    mode &= 0xFF;
    if (mode == ORC_STATIC) {
        double s = (double)scale[0];
        for (int64_t j = 0; j < n; ++j) {
            double vj = y[j] / s;
            q[j] = orc_e4m3_encode(vj);
            if (v)
                v[j] = vj;
        }
        return;
    }
    int64_t width = (mode == ORC_PER_TOKEN) ? n : G;
    int64_t ngroups = n / width;
    for (int64_t g = 0; g < ngroups; ++g) {
        const double *yg = y + g * width;
        double amax = 0.0;
        for (int64_t j = 0; j < width; ++j)
            if (fabs(yg[j]) > amax)
                amax = fabs(yg[j]);
        float s32 = (flags & ORC_UE8M0) ? (float)ue8m0_scale(amax) : dynamic_scale(amax);
        if (flags & ORC_COL_MAJOR)
            scale[g * ((T + 3) / 4 * 4) + t] = s32;
        else
            scale[t * ngroups + g] = s32;
        double s = (double)s32;
        for (int64_t j = 0; j < width; ++j) {
            double vj = yg[j] / s;
            q[g * width + j] = orc_e4m3_encode(vj);
            if (v)
                v[g * width + j] = vj;
        }
    }
}

static int check_mode(int mode, int64_t n, int64_t G)
{
    const int flags = mode & ~0xFF;
    if (flags & ~(ORC_UE8M0 | ORC_COL_MAJOR))
        return -1;
    mode &= 0xFF;
    if ((mode == ORC_STATIC || mode == ORC_PER_TOKEN) && flags == 0)
        return 0;
    if (mode == ORC_PER_GROUP && G > 0 && n % G == 0)
        return 0;
    return -1;
}

/* NVFP4 quantisation of one row y[0..n), n % 16 == 0 ([NVFP4]):
 *   for each block b of 16 columns:
 *     sf_b = e4m3(gs * max_j |y_j| / 6)          (the stored E4M3 code)
 *     v_j  = y_j * gs / decode(sf_b), or 0 when decode(sf_b) == 0
 *     q_j  = e2m1(v_j)
 * q4 packs two codes a byte, column 2i in the low nibble of byte i; sf holds
 * the n/16 block codes; v (optional) receives v_j. */
static void nvfp4_row(uint8_t *q4, uint8_t *sf, double *v, const double *y, int64_t n, float gs)
{
    for (int64_t b = 0; b < n / 16; ++b) {
        const double *yb = y + b * 16;
        double amax = 0.0;
        for (int j = 0; j < 16; ++j)
            if (fabs(yb[j]) > amax)
                amax = fabs(yb[j]);
        uint8_t code = orc_e4m3_encode((double)gs * amax / 6.0);
        sf[b] = code;
        double s = orc_e4m3_decode(code);
        for (int j = 0; j < 16; ++j) {
            double vj = s > 0.0 ? yb[j] * (double)gs / s : 0.0;
            uint8_t e = orc_e2m1_encode(vj);
            int64_t col = b * 16 + j;
            if (col % 2 == 0)
                q4[col / 2] = e;
            else
                q4[col / 2] = (uint8_t)(q4[col / 2] | (e << 4));
            if (v)
                v[col] = vj;
        }
    }
}

/* ------------------------------------------------------------------ ops */

/* fused_add_rms_norm(x, residual) -> quant_fp8(y), rows t = 0..T-1, each
 * of H columns ([FUS] "RMSNorm + Quantization", fused-add variant; with
 * residual == NULL the plain rms_norm(x) -> quant_fp8(y) variant):
 *   r_j  = bf16(x_j + res_j)   (the fp64 sum is exact unless the exponents
 *                               are more than 45 apart, and then the smaller
 *                               addend is far below half a bf16 ulp, so the
 *                               RNE result is the same as for the exact sum)
 *   residual_out_j = r_j       (the residual is updated in place)
 *   inv  = 1 / sqrt((sum_j r_j^2) / H + eps)
 *   y_j  = r_j * inv * w_j     (fp64, never rounded to bf16)
 *   q    = quant_fp8(y)
 * Layouts: x, residual, residual_out, v: [T, H]; weight [H]; q [T, H];
 * scale as in quantize_row.  Returns 0, or -1 on a bad mode/shape. */
int orc_fused_add_rms_norm_fp8(uint8_t *q, uint16_t *residual_out, float *scale,
                               double *v, const uint16_t *x,
                               const uint16_t *residual, const uint16_t *weight,
                               int64_t T, int64_t H, float eps, int mode,
                               int64_t G)
{
    if (T < 0 || H <= 0 || check_mode(mode, H, G) != 0)
        return -1;
    double *r = (double *)malloc((size_t)H * sizeof(double));
    double *y = (double *)malloc((size_t)H * sizeof(double));
    if (!r || !y) {
        free(r);
        free(y);
        return -2;
    }
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *xt = x + t * H;
        for (int64_t j = 0; j < H; ++j) {
            if (residual) {
                double sum = orc_bf16_decode(xt[j]) + orc_bf16_decode(residual[t * H + j]);
                uint16_t rb = orc_bf16_encode(sum);
                residual_out[t * H + j] = rb;
                r[j] = orc_bf16_decode(rb);
            } else {
                r[j] = orc_bf16_decode(xt[j]);
            }
        }
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j)
            ss += r[j] * r[j];
        double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
        for (int64_t j = 0; j < H; ++j)
            y[j] = r[j] * inv * orc_bf16_decode(weight[j]);
        quantize_row(q + t * H, v ? v + t * H : NULL, scale, y, t, T, H, mode, G);
    }
    free(r);
    free(y);
    return 0;
}

/* rms_norm(x, weight, eps) with a bf16 output, rows t = 0..T-1 ([FUS] "MLA
 * Dual RMSNorm": q_c and kv_c each go through rms_norm with their own weight
 * and eps, and the normalised rows stay bf16):
 *   y_j   = x_j / sqrt(mean_j(x_j^2) + eps) * w_j     (fp64)
 *   out_j = bf16(y_j)                                 (one rounding)
 * Layouts: x and out [T, H] row-major, weight [H]; y (optional) [T, H]. */
int orc_rms_norm_bf16(uint16_t *out, double *y, const uint16_t *x,
                      const uint16_t *weight, int64_t T, int64_t H, float eps)
{
    if (T < 0 || H <= 0)
        return -1;
    double *r = (double *)malloc((size_t)H * sizeof(double));
    if (!r)
        return -2;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < H; ++j)
            r[j] = orc_bf16_decode(x[t * H + j]);
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j)
            ss += r[j] * r[j];
        double mean = ss / (double)H;
        double inv = 1.0 / sqrt(mean + (double)eps);
        for (int64_t j = 0; j < H; ++j) {
            double yj = r[j] * inv * orc_bf16_decode(weight[j]);
            out[t * H + j] = orc_bf16_encode(yj);
            if (y)
                y[t * H + j] = yj;
        }
    }
    free(r);
    return 0;
}

/* fused_add_rms_norm(x, residual) -> pad, rows t = 0..T-1 ([FUS] "RMSNorm +
 * Padding (fuse_act_padding)"): the normalised row stays bf16 and is written
 * into a row of Hp >= H columns whose tail is zero:
 *   r_j    = bf16(x_j + residual_j)   (-> residual_out; r = x without residual)
 *   y_j    = r_j / sqrt(mean_j(r_j^2) + eps) * w_j          (fp64)
 *   out_j  = bf16(y_j) for j < H, 0 for H <= j < Hp          (one rounding)
 * Layouts: x, residual, residual_out [T, H]; out [T, Hp]; y (optional) [T, H]. */
int orc_fused_add_rms_norm_pad(uint16_t *out, uint16_t *residual_out, double *y,
                               const uint16_t *x, const uint16_t *residual,
                               const uint16_t *weight, int64_t T, int64_t H,
                               int64_t Hp, float eps)
{
    if (T < 0 || H <= 0 || Hp < H)
        return -1;
    double *r = (double *)malloc((size_t)H * sizeof(double));
    if (!r)
        return -2;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *xrow = x + t * H;
        for (int64_t j = 0; j < H; ++j) {
            if (residual) {
                uint16_t rb = orc_bf16_encode(orc_bf16_decode(xrow[j]) +
                                              orc_bf16_decode(residual[t * H + j]));
                residual_out[t * H + j] = rb;
                r[j] = orc_bf16_decode(residual_out[t * H + j]);
            } else {
                r[j] = orc_bf16_decode(xrow[j]);
            }
        }
        double sq = 0.0;
        for (int64_t j = 0; j < H; ++j)
            sq += r[j] * r[j];
        double scale = 1.0 / sqrt(sq / (double)H + (double)eps);
        for (int64_t j = 0; j < Hp; ++j) {
            double yj = j < H ? r[j] * scale * orc_bf16_decode(weight[j]) : 0.0;
            out[t * Hp + j] = j < H ? orc_bf16_encode(yj) : 0;
            if (y && j < H)
                y[t * H + j] = yj;
        }
    }
    free(r);
    return 0;
}

/* fused_qk_norm_rope(qkv) ([FUS] "QK Norm + RoPE"): for every token t and
 * every Q head (weight q_weight) and K head (weight k_weight) of qkv
 * [T, (Hq + 2 Hkv) * D] (Q heads, then K heads, then V heads, each D
 * contiguous columns):
 *   y_j = x_j / sqrt(mean_j(x_j^2) + eps) * w_j                  (fp64)
 * then the rotary embedding with c_i = cache[pos_t, i] and
 * s_i = cache[pos_t, D/2 + i], i < D/2, on the pairs (a, b) = (i, i + D/2)
 * (neox) or (2i, 2i + 1) (gptj):
 *   o_a = y_a c_i - y_b s_i,   o_b = y_b c_i + y_a s_i           (fp64)
 * written back in place as bf16 (one rounding); V heads are not touched.
 * o (optional) receives the pre-rounding values [T, (Hq + Hkv) * D].
 * Returns -1 on bad sizes or a position outside [0, max_pos). */
int orc_qk_norm_rope(uint16_t *qkv, double *o, const uint16_t *q_weight,
                     const uint16_t *k_weight, const float *cos_sin_cache,
                     const int64_t *positions, int64_t T, int64_t Hq, int64_t Hkv,
                     int64_t D, int64_t max_pos, float eps, int is_neox)
{
    if (T < 0 || Hq < 0 || Hkv < 0 || D <= 0 || D % 2 != 0 || max_pos <= 0)
        return -1;
    for (int64_t t = 0; t < T; ++t)
        if (positions[t] < 0 || positions[t] >= max_pos)
            return -1;
    double *y = (double *)malloc((size_t)D * sizeof(double));
    double *rot = (double *)malloc((size_t)D * sizeof(double));
    if (!y || !rot) {
        free(y);
        free(rot);
        return -2;
    }
    const int64_t row = (Hq + 2 * Hkv) * D;
    for (int64_t t = 0; t < T; ++t) {
        const float *cs = cos_sin_cache + positions[t] * D;
        for (int64_t h = 0; h < Hq + Hkv; ++h) {
            uint16_t *head = qkv + t * row + h * D;
            const uint16_t *w = h < Hq ? q_weight : k_weight;
            double sq = 0.0;
            for (int64_t j = 0; j < D; ++j) {
                double xj = orc_bf16_decode(head[j]);
                sq += xj * xj;
            }
            double inv_rms = 1.0 / sqrt(sq / (double)D + (double)eps);
            for (int64_t j = 0; j < D; ++j)
                y[j] = orc_bf16_decode(head[j]) * inv_rms * orc_bf16_decode(w[j]);
            for (int64_t i = 0; i < D / 2; ++i) {
                int64_t a = is_neox ? i : 2 * i;
                int64_t b = is_neox ? i + D / 2 : 2 * i + 1;
                double c = (double)cs[i], sn = (double)cs[D / 2 + i];
                rot[a] = y[a] * c - y[b] * sn;
                rot[b] = y[b] * c + y[a] * sn;
            }
            for (int64_t j = 0; j < D; ++j) {
                head[j] = orc_bf16_encode(rot[j]);
                if (o)
                    o[(t * (Hq + Hkv) + h) * D + j] = rot[j];
            }
        }
    }
    free(y);
    free(rot);
    return 0;
}

/* fused_add_rms_norm(x, residual) -> NVFP4 ([FUS] "RMSNorm + Quantization",
 * the FP4 output of the "Quick Reference"; [NVFP4]): r, residual_out and y as
 * in orc_fused_add_rms_norm_fp8, then nvfp4_row(y) with the per-tensor scale
 * gs.  Layouts: q4 [T, H/2] bytes; sf [T, H/16] E4M3 codes; v [T, H]. */
int orc_fused_add_rms_norm_nvfp4(uint8_t *q4, uint8_t *sf, uint16_t *residual_out, double *v,
                                 const uint16_t *x, const uint16_t *residual,
                                 const uint16_t *weight, float gs, int64_t T, int64_t H,
                                 float eps)
{
    if (T < 0 || H <= 0 || H % 16 != 0)
        return -1;
    double *r = (double *)malloc((size_t)H * sizeof(double));
    double *y = (double *)malloc((size_t)H * sizeof(double));
    if (!r || !y) {
        free(r);
        free(y);
        return -2;
    }
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < H; ++j) {
            double xj = orc_bf16_decode(x[t * H + j]);
            if (residual) {
                uint16_t rb = orc_bf16_encode(xj + orc_bf16_decode(residual[t * H + j]));
                residual_out[t * H + j] = rb;
                const double stored = orc_bf16_decode(rb); /* the stored residual */
                r[j] = stored;
            } else {
                r[j] = xj;
            }
        }
        double sumsq = 0.0;
        for (int64_t j = 0; j < H; ++j)
            sumsq += r[j] * r[j];
        double rinv = 1.0 / sqrt(sumsq / (double)H + (double)eps);
        for (int64_t j = 0; j < H; ++j)
            y[j] = r[j] * rinv * orc_bf16_decode(weight[j]);
        nvfp4_row(q4 + t * (H / 2), sf + t * (H / 16), v ? v + t * H : NULL, y, H, gs);
    }
    free(r);
    free(y);
    return 0;
}

/* silu_and_mul(gate_up) -> NVFP4 ([FUS] "SiLU+Mul + Quantization", the FP4
 * output; [NVFP4]): a_j = silu(g_j) * u_j as in orc_silu_mul_fp8, then
 * nvfp4_row(a).  Layouts: q4 [T, I/2]; sf [T, I/16]; v [T, I]. */
int orc_silu_mul_nvfp4(uint8_t *q4, uint8_t *sf, double *v, const uint16_t *gate_up, float gs,
                       int64_t T, int64_t I)
{
    if (T < 0 || I <= 0 || I % 16 != 0)
        return -1;
    double *act = (double *)malloc((size_t)I * sizeof(double));
    if (!act)
        return -2;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *gu = gate_up + t * 2 * I;
        for (int64_t j = 0; j < I; ++j) {
            double g = orc_bf16_decode(gu[j]);
            act[j] = g / (1.0 + exp(-g)) * orc_bf16_decode(gu[I + j]);
        }
        nvfp4_row(q4 + t * (I / 2), sf + t * (I / 16), v ? v + t * I : NULL, act, I, gs);
    }
    free(act);
    return 0;
}

/* silu_and_mul(gate_up) -> quant_fp8(a), rows t = 0..T-1 ([FUS] "SiLU+Mul +
 * Quantization"):
 *   g_j = gate_up[t, j], u_j = gate_up[t, I + j]   (gate half, then up half)
 *   a_j = g_j / (1 + exp(-g_j)) * u_j              (fp64, never materialised)
 *   q   = quant_fp8(a)
 * Layouts: gate_up [T, 2I]; q and v [T, I]; scale as in quantize_row. */
int orc_silu_mul_fp8(uint8_t *q, float *scale, double *v,
                     const uint16_t *gate_up, int64_t T, int64_t I, int mode,
                     int64_t G)
{
    if (T < 0 || I <= 0 || check_mode(mode, I, G) != 0)
        return -1;
    double *a = (double *)malloc((size_t)I * sizeof(double));
    if (!a)
        return -2;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *row = gate_up + t * 2 * I;
        for (int64_t j = 0; j < I; ++j) {
            double g = orc_bf16_decode(row[j]);
            double u = orc_bf16_decode(row[I + j]);
            a[j] = g / (1.0 + exp(-g)) * u;
        }
        quantize_row(q + t * I, v ? v + t * I : NULL, scale, a, t, T, I, mode, G);
    }
    free(a);
    return 0;
}
