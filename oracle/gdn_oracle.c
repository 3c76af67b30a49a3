/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code with the CUDA path.
 *
 * Sources (cited by page title and section):
 *   [gdn.rs]  logicaffeine_compile/codegen_cuda/gdn.rs -- kernel `gdn_step`
 *             (the recurrence and its output scale, and the key-head pairing
 *             note) and kernel `gdn_gate_norm` (RMS norm, then the silu gate).
 *   [ssm]     metrale_model_layers/layers/ops/ssm_gdn_a.rs -- launchers
 *             `gdn_prefill_regresident` (token-sequential prefill),
 *             `ssm_h_state_f32_to_f16` / `ssm_h_state_f16_to_f32` (h-state
 *             converters, round-to-nearest-even).
 *
 * Everything is written as the plain definition, in loops, in fp64, with no
 * blocking, fusion or reordering:
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
 *   o_t = S_t q_t / sqrt(D)
 * for every value head h, whose key/query head is g = h mod NK.
 *
 * Layouts (all contiguous; the tests pack strided device buffers from these):
 *   S      [batch][nv][d][d] double, row a = value index, column b = key index
 *   q, k   [batch][nk*d] float      v, z  [batch][nv*d] float
 *   alpha, beta [batch][nv] float   o     [batch][nv*d] double
 * Prefill adds a token axis after batch: q,k [batch][T][nk*d], v [batch][T][nv*d],
 * alpha,beta [batch][T][nv], o [batch][T][nv*d].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* One gated delta-rule step of one value head ([gdn.rs] `gdn_step`), as the
 * matrix definition:
 *   Sk   = S k                          (matrix-vector product)
 *   r    = beta (v - alpha Sk)          (the delta-rule correction)
 *   S   <- alpha S + r k^T              (decay plus rank-1 write)
 *   o    = S q / sqrt(d)                (read-out with the new state, scaled by
 *                                        1/sqrt(D), which the page keeps ahead
 *                                        of the norm)
 * `work` holds d doubles. */
static void head_step(int d, double *S, const double *q, const double *k,
                      const double *v, double alpha, double beta, double *o,
                      double *work)
{
    for (int a = 0; a < d; ++a) {
        double acc = 0.0;
        for (int b = 0; b < d; ++b) acc += S[(int64_t)a * d + b] * k[b];
        work[a] = acc;
    }
    for (int a = 0; a < d; ++a) {
        double r = beta * (v[a] - alpha * work[a]);
        for (int b = 0; b < d; ++b)
            S[(int64_t)a * d + b] = alpha * S[(int64_t)a * d + b] + r * k[b];
    }
    double scale = 1.0 / sqrt((double)d);
    for (int a = 0; a < d; ++a) {
        double acc = 0.0;
        for (int b = 0; b < d; ++b) acc += S[(int64_t)a * d + b] * q[b];
        o[a] = acc * scale;
    }
}

static void widen(const float *src, double *dst, int n)
{
    for (int i = 0; i < n; ++i) dst[i] = (double)src[i];
}

/* One decode step for `batch` sequences ([gdn.rs] `gdn_step`; [ssm]
 * `gdn_decode`).  Value head h reads key/query head g = h mod nk: the page's
 * note says the heads are tiled, not repeat-interleaved. */
void orc_decode(int batch, int nk, int nv, int d, double *S,
                const float *q, const float *k, const float *v,
                const float *alpha, const float *beta, double *o)
{
    double *qd = malloc(sizeof(double) * d), *kd = malloc(sizeof(double) * d);
    double *vd = malloc(sizeof(double) * d), *work = malloc(sizeof(double) * d);
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < nv; ++h) {
            int g = h % nk;
            widen(q + ((int64_t)b * nk + g) * d, qd, d);
            widen(k + ((int64_t)b * nk + g) * d, kd, d);
            widen(v + ((int64_t)b * nv + h) * d, vd, d);
            head_step(d, S + ((int64_t)b * nv + h) * d * d, qd, kd, vd,
                      (double)alpha[(int64_t)b * nv + h], (double)beta[(int64_t)b * nv + h],
                      o + ((int64_t)b * nv + h) * d, work);
        }
    }
    free(qd); free(kd); free(vd); free(work);
}

/* Gated RMS norm of each head's output ([gdn.rs] `gdn_gate_norm`): normalise
 * by the root of the mean square over the head's D outputs plus eps, scale by
 * the shared weight gn, THEN multiply by silu(z) = z / (1 + e^-z). */
void orc_gated_rmsnorm(int64_t heads, int d, const double *o, const float *z,
                       const float *gn, double eps, double *out)
{
    for (int64_t h = 0; h < heads; ++h) {
        const double *oh = o + h * d;
        double ss = 0.0;
        for (int a = 0; a < d; ++a) ss += oh[a] * oh[a];
        double den = sqrt(ss / (double)d + eps);
        for (int a = 0; a < d; ++a) {
            double zz = (double)z[h * d + a];
            double silu = zz / (1.0 + exp(-zz));
            out[h * d + a] = (double)gn[a] * oh[a] / den * silu;
        }
    }
}

/* Token-sequential prefill ([ssm] `gdn_prefill_regresident`): the decode step
 * applied to tokens t = 0..T-1 in order, the state carried across tokens, and
 * the raw output o recorded for every token (no norm). */
void orc_prefill(int batch, int T, int nk, int nv, int d, double *S,
                 const float *q, const float *k, const float *v,
                 const float *alpha, const float *beta, double *o)
{
    for (int b = 0; b < batch; ++b) {
        for (int t = 0; t < T; ++t) {
            int64_t bt = (int64_t)b * T + t;
            orc_decode(1, nk, nv, d, S + (int64_t)b * nv * d * d,
                       q + bt * nk * d, k + bt * nk * d, v + bt * nv * d,
                       alpha + bt * nv, beta + bt * nv, o + bt * nv * d);
        }
    }
}

/* ---------------------------------------------------------------------------
 * h-state converters ([ssm] `ssm_h_state_f32_to_f16`, `ssm_h_state_f16_to_f32`).
 * Written from the IEEE 754 binary32/binary16 encodings and the
 * roundTiesToEven rule, in integer arithmetic.
 *   binary32: 1 sign, 8 exponent (bias 127), 23 fraction bits.
 *   binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits; subnormals are
 *             multiples of 2^-24; the largest finite value is 65504.
 * ------------------------------------------------------------------------- */

uint16_t orc_f32_to_f16_bits(uint32_t x)
{
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ex = (x >> 23) & 0xffu;
    uint32_t fr = x & 0x7fffffu;

    if (ex == 0xffu) {                          /* inf or NaN */
        if (fr == 0) return (uint16_t)(sign | 0x7c00u);
        /* NaN stays NaN: quiet bit set, top fraction bits kept */
        return (uint16_t)(sign | 0x7c00u | 0x0200u | (fr >> 13));
    }
    if (ex == 0) {
        /* zero or binary32 subnormal (< 2^-126): far below half of the
         * smallest binary16 subnormal 2^-24, so it rounds to a signed zero */
        return sign;
    }
    /* value = M * 2^(E-23), M = 1.fraction as a 24-bit integer */
    int32_t E = (int32_t)ex - 127;
    uint32_t M = fr | 0x800000u;
    /* Result quantum: 2^(E-10) in the normal range, 2^-24 below 2^-14.
     * Number of quanta = M * 2^(E-23-qe) = M >> s with s = 13 + max(0, -14-E). */
    int32_t s = 13 + (E < -14 ? (-14 - E) : 0);
    uint32_t n;
    if (s > 25) {
        n = 0;                                   /* below half a quantum */
    } else {
        n = M >> s;
        uint32_t rem = M & ((1u << s) - 1u);
        uint32_t half = 1u << (s - 1);
        if (rem > half || (rem == half && (n & 1u))) n += 1;   /* ties to even */
    }
    if (E < -14) {
        /* subnormal range: the encoding is the quantum count itself; a count of
         * 1024 carries into the smallest normal (exponent field 1). */
        return (uint16_t)(sign | n);
    }
    if (n == 2048u) { n = 1024u; E += 1; }       /* rounding carried a bit */
    if (E > 15) return (uint16_t)(sign | 0x7c00u);  /* overflow to infinity */
    return (uint16_t)(sign | (uint32_t)(E + 15) << 10 | (n - 1024u));
}

uint32_t orc_f16_to_f32_bits(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t ex = (h >> 10) & 0x1fu;
    uint32_t fr = h & 0x3ffu;
    if (ex == 0x1fu) return sign | 0x7f800000u | (fr << 13);  /* inf / NaN */
    if (ex == 0) {
        if (fr == 0) return sign;                             /* signed zero */
        /* subnormal: fr * 2^-24; normalise so the leading bit is 2^10 */
        int32_t E = -14;
        while ((fr & 0x400u) == 0) { fr <<= 1; E -= 1; }
        return sign | (uint32_t)(E + 127) << 23 | ((fr & 0x3ffu) << 13);
    }
    return sign | (ex - 15u + 127u) << 23 | (fr << 13);
}

void orc_f32_to_f16_array(const uint32_t *src, uint16_t *dst, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i) dst[i] = orc_f32_to_f16_bits(src[i]);
}

void orc_f16_to_f32_array(const uint16_t *src, uint32_t *dst, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i) dst[i] = orc_f16_to_f32_bits(src[i]);
}

/* ---------------------------------------------------------------------------
 * Producers upstream of the recurrence, for the fused decode from projections
 * (ssm_gdn_a.rs `gdn_decode_f32_conv_norm`; gdn.rs `gk_conv_silu_l2`,
 * `gk_gdn_gates`).
 * ------------------------------------------------------------------------- */

/* Depthwise causal conv over `channels` channels with a `taps`-deep ring
 * ([gdn.rs] `gk_conv_silu`): the ring is a shift register, ring[t][c] for
 * t = 0..taps-1, entry taps-1 the newest.  Shift every channel up by one,
 * append this token's x, reduce with the per-channel taps w[t][c], apply
 * silu(a) = a / (1 + e^-a).  The ring is updated in place. */
void orc_conv_silu(int taps, int channels, float *ring, const float *x,
                   const float *w, double *y)
{
    for (int c = 0; c < channels; ++c) {
        for (int t = 0; t + 1 < taps; ++t)
            ring[(int64_t)t * channels + c] = ring[(int64_t)(t + 1) * channels + c];
        ring[(int64_t)(taps - 1) * channels + c] = x[c];
        double acc = 0.0;
        for (int t = 0; t < taps; ++t)
            acc += (double)ring[(int64_t)t * channels + c] * (double)w[(int64_t)t * channels + c];
        y[c] = acc / (1.0 + exp(-acc));
    }
}

/* Per-head L2 normalisation ([gdn.rs] `gk_conv_silu_l2`, q and k heads):
 * y / sqrt(sum_head y^2 + eps), eps added to the sum (not the mean). */
void orc_l2norm_heads(int heads, int d, double *y, double eps)
{
    for (int h = 0; h < heads; ++h) {
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += y[(int64_t)h * d + i] * y[(int64_t)h * d + i];
        double den = sqrt(ss + eps);
        for (int i = 0; i < d; ++i) y[(int64_t)h * d + i] /= den;
    }
}

/* The two gates of a value head ([gdn.rs] `gk_gdn_gates`): write strength
 * beta = sigmoid(br) and decay alpha = (1 + e^(ar + dt))^rate, where `rate`
 * already holds the negative decay rate, so alpha = exp(rate * softplus(ar + dt)). */
void orc_gates(int n, const float *br, const float *ar, const float *dt,
               const float *rate, double *beta, double *alpha)
{
    for (int i = 0; i < n; ++i) {
        beta[i] = 1.0 / (1.0 + exp(-(double)br[i]));
        alpha[i] = pow(1.0 + exp((double)ar[i] + (double)dt[i]), (double)rate[i]);
    }
}

/* orc_decode with fp64 token inputs (for inputs the oracle itself computed,
 * e.g. by orc_conv_silu / orc_l2norm_heads / orc_gates), same layouts. */
void orc_decode_f64(int batch, int nk, int nv, int d, double *S,
                    const double *q, const double *k, const double *v,
                    const double *alpha, const double *beta, double *o)
{
    double *work = malloc(sizeof(double) * d);
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < nv; ++h) {
            int g = h % nk;
            head_step(d, S + ((int64_t)b * nv + h) * d * d,
                      q + ((int64_t)b * nk + g) * d, k + ((int64_t)b * nk + g) * d,
                      v + ((int64_t)b * nv + h) * d,
                      alpha[(int64_t)b * nv + h], beta[(int64_t)b * nv + h],
                      o + ((int64_t)b * nv + h) * d, work);
        }
    }
    free(work);
}

/* ---------------------------------------------------------------------------
 * Int8 activation groups of the normed output ([gdn.rs] `gdn_gate_norm_q`,
 * the gate norm with the activation quantisation fused in for the int8
 * o-projection that follows).  The output vector of a token is cut into
 * groups of 32 consecutive values (a head's D outputs hold D/32 groups).  A
 * group's scale is its largest magnitude divided by 127, or 1 when the group
 * is all zero; each value's code is value / scale rounded to the nearest
 * integer, ties to even.  The page takes these decisions in fp32 on the fp32
 * output, so this function does the same: fp32 division on the given fp32
 * values (IEEE, correctly rounded), then the rounding rule below, written
 * out in double (exact for fp32 operands).
 * ------------------------------------------------------------------------- */
static double round_half_even(double r)
{
    double f = floor(r);
    double frac = r - f;
    if (frac > 0.5 || (frac == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;
    return f;
}

/* n values (a multiple of 32) -> n codes and n/32 scales. */
void orc_quant_q8_groups(int64_t n, const float *y, int8_t *code, float *scale)
{
    for (int64_t g0 = 0; g0 < n; g0 += 32) {
        float am = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float m = fabsf(y[g0 + i]);
            if (m > am) am = m;
        }
        float sc = am > 0.0f ? am / 127.0f : 1.0f;
        scale[g0 / 32] = sc;
        for (int i = 0; i < 32; ++i) {
            float r = y[g0 + i] / sc;
            code[g0 + i] = (int8_t)round_half_even((double)r);
        }
    }
}
