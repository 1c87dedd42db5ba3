/*
 * CPU oracle for integer-only training (NITI dynamic-shift requantisation and
 * the DFP16 shared-exponent linear path).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path calls, links or loads
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline do. It shares no code, header, table or constant with the CUDA
 * library.
 *
 * Every function is the plain definition of one step, written as nested loops
 * with int64 accumulation. The loop nest order of a contraction is chosen for
 * memory access only: every sum is an exact integer sum, so the order of the
 * terms does not change the result. Results that must fit int32 are checked,
 * and a value outside int32 aborts the process (ora_fail).
 *
 * Sources (the web pages this follows):
 *   [ODT]   "Integer On-Device Training: Overview" (TI C2000 MCU AI user
 *           guide), section 3 "The NITI Algorithm", "The Solution: Dynamic
 *           Shifts", Steps 1-5, and the note on delta propagation with
 *           target_bits = 7; section 4 (compute_loss writes dy,
 *           INTODT_Backward reads it); section 7 "Supported Configurations"
 *           (Conv2D, Conv2D+ReLU, Linear, Linear+ReLU).
 *   [TGR]   TiGrIS "Compilation Pipeline", normalisation pass 3 "Matrix
 *           product relabel" (weight indexed W[oc*IC + ic]) and the emission
 *           stage's "Layout transpose" (NHWC activations, weights
 *           [OC][KH][KW][IC]).
 *   [DFP]   "Mixed Precision Training of Convolutional Neural Networks using
 *           Integer Operations", section 3 "The Dynamic Fixed Point Format"
 *           and 3.1 "DFP Tensor Primitives" (f = i * 2^Es, one signed 8-bit
 *           exponent per tensor, products carry exponent Ea + Eb, down-convert
 *           by a right shift Rs with a new exponent).
 *   [APT]   "Adaptive Precision Training for Resource Constrained Devices",
 *           section III (k-bit weights, minimum resolution epsilon, Gavg,
 *           Algorithm 1).
 *
 * Readings where the pages leave a step open are stated at each function.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static void ora_fail(const char *what)
{
    fprintf(stderr, "oracle: %s\n", what);
    abort();
}

static int32_t checked_i32(int64_t v)
{
    if (v < INT32_MIN || v > INT32_MAX)
        ora_fail("int32 overflow in a contraction result");
    return (int32_t)v;
}

/* ---------------------------------------------------------------- scalars */

/* [ODT] Step 2: bits_needed = ceil(log2(max_val + 1)). For an integer m >= 0
 * this is the number of binary digits of m (0 for m = 0), counted here one bit
 * at a time, with no floating-point logarithm. */
int32_t ora_bitlen(uint64_t m)
{
    int32_t n = 0;
    while (m != 0) {
        n += 1;
        m >>= 1;
    }
    return n;
}

/* [ODT] Step 2: shift = max(0, bits_needed - target_bits). */
int32_t ora_shift_from_max(uint64_t max_abs, int32_t target_bits)
{
    int32_t s = ora_bitlen(max_abs) - target_bits;
    return s > 0 ? s : 0;
}

/* floor(a / 2^s) for s in 0..62, by exact integer division. */
static int64_t floor_div_pow2(int64_t a, int32_t s)
{
    int64_t d = (int64_t)1 << s;
    int64_t q = a / d;            /* C division truncates toward zero */
    if ((a % d) != 0 && a < 0)
        q -= 1;                   /* step down to the floor for negatives */
    return q;
}

/* [ODT] Step 3: "round(G >> shift) // round-half-up". Reading: the value
 * G / 2^s rounded to the nearest integer with ties going up (toward +inf),
 * i.e. floor((G + 2^(s-1)) / 2^s); shift 0 is the identity.
 * Examples: s=1: 3 -> 2, -3 -> -1, -1 -> 0. For s >= 63 every value that an
 * int64 operand here can hold rounds to 0, which is what the formula gives. */
int64_t ora_rhu(int64_t x, int32_t s)
{
    if (s < 0)
        ora_fail("negative shift");
    if (s == 0)
        return x;
    if (s >= 63) {
        /* |x| < 2^62 for every caller; (x + 2^(s-1)) / 2^s is then in [0, 1). */
        if (x >= ((int64_t)1 << 62) || x < -((int64_t)1 << 62))
            ora_fail("rhu operand out of range");
        return 0;
    }
    /* x + 2^(s-1) cannot overflow for the |x| < 2^62 operands used here */
    return floor_div_pow2(x + ((int64_t)1 << (s - 1)), s);
}

/* [ODT] Step 5: sat_int8, the full int8 range [-128, 127]. */
int64_t ora_sat8(int64_t v)
{
    if (v < -128) return -128;
    if (v > 127) return 127;
    return v;
}

/* DFP16 mantissa saturation: symmetric [-32767, 32767] (one code, -32768,
 * is left unused so that negation never overflows). */
int64_t ora_sat16(int64_t v)
{
    if (v < -32767) return -32767;
    if (v > 32767) return 32767;
    return v;
}

/* [ODT] Step 1: max_val = max(|G|) over one whole tensor. |INT32_MIN| = 2^31
 * is returned exactly, in an unsigned 32-bit value. */
uint32_t ora_absmax32(const int32_t *v, int64_t n)
{
    uint64_t m = 0;
    for (int64_t i = 0; i < n; i++) {
        int64_t a = v[i];
        uint64_t u = (uint64_t)(a < 0 ? -a : a);
        if (u > m) m = u;
    }
    return (uint32_t)m;
}

uint64_t ora_absmax64(const int64_t *v, int64_t n)
{
    uint64_t m = 0;
    for (int64_t i = 0; i < n; i++) {
        int64_t a = v[i];
        if (a == INT64_MIN) ora_fail("INT64_MIN in absmax64");
        uint64_t u = (uint64_t)(a < 0 ? -a : a);
        if (u > m) m = u;
    }
    return m;
}

/* ---------------------------------------------------- requantisation (int8) */

/* Steps 1-3 applied to a forward or gradient contraction Y, then sat_int8 and
 * (for a ReLU layer) the ReLU: out = relu ? max(0, sat8(rhu(Y, s))) :
 * sat8(rhu(Y, s)). The shift comes from the max of the raw int32 tensor
 * (before ReLU). Returns the shift; *max_out receives max|Y|. */
int32_t ora_requant(const int32_t *Y, int64_t n, int32_t target_bits, int relu,
                    int8_t *out, uint32_t *max_out)
{
    uint32_t m = ora_absmax32(Y, n);
    int32_t s = ora_shift_from_max(m, target_bits);
    for (int64_t i = 0; i < n; i++) {
        int64_t q = ora_sat8(ora_rhu(Y[i], s));
        if (relu && q < 0) q = 0;
        out[i] = (int8_t)q;
    }
    if (max_out) *max_out = m;
    return s;
}

/* Delta propagation ([ODT] note under Step 5, target_bits = 7): the dgrad
 * contraction D is requantised like Y and then gated by the ReLU of the layer
 * below: out = (a_prev > 0) ? sat8(rhu(D, s)) : 0. a_prev == NULL means no
 * gate (the layer below has no ReLU). */
int32_t ora_requant_mask(const int32_t *D, const int8_t *a_prev, int64_t n,
                         int32_t target_bits, int8_t *out, uint32_t *max_out)
{
    uint32_t m = ora_absmax32(D, n);
    int32_t s = ora_shift_from_max(m, target_bits);
    for (int64_t i = 0; i < n; i++) {
        int64_t q = ora_sat8(ora_rhu(D[i], s));
        if (a_prev && a_prev[i] <= 0) q = 0;
        out[i] = (int8_t)q;
    }
    if (max_out) *max_out = m;
    return s;
}

/* Top error written by the user's compute_loss ([ODT] section 4): an MSE
 * error against an integer target of target_mag on the true class and 0
 * elsewhere, saturated to int8: delta = sat8(logit - target_mag*[j == label]). */
void ora_top_error(const int8_t *logits, const int32_t *labels, int B, int C,
                   int32_t target_mag, int8_t *delta)
{
    for (int b = 0; b < B; b++) {
        if (labels[b] < 0 || labels[b] >= C) ora_fail("label out of range");
        for (int j = 0; j < C; j++) {
            int64_t t = (j == labels[b]) ? target_mag : 0;
            delta[(int64_t)b * C + j] = (int8_t)ora_sat8((int64_t)logits[(int64_t)b * C + j] - t);
        }
    }
}

/* [ODT] Steps 1-5 on one weight tensor. Reading of Step 4: the operand of the
 * second shift is G_quantized, the tensor already shifted and saturated in
 * Step 3, exactly as the step is written:
 *   s  = max(0, bitlen(max|G|) - target_bits)
 *   Gq = sat8(rhu(G, s))
 *   ws = max(0, s - mu_weight)
 *   dW = rhu(Gq, ws)
 *   W  = sat8(W - dW)
 * Writes shift and weight_shift; returns the number of nonzero dW. */
int64_t ora_niti_update(int8_t *W, const int32_t *G, int64_t n, int32_t target_bits,
                        int32_t mu_weight, int32_t *shift_out, int32_t *wshift_out,
                        uint32_t *max_out)
{
    uint32_t m = ora_absmax32(G, n);
    int32_t s = ora_shift_from_max(m, target_bits);
    int32_t ws = s - mu_weight > 0 ? s - mu_weight : 0;
    int64_t nonzero = 0;
    for (int64_t i = 0; i < n; i++) {
        int64_t gq = ora_sat8(ora_rhu(G[i], s));
        int64_t dw = ora_rhu(gq, ws);
        if (dw != 0) nonzero++;
        W[i] = (int8_t)ora_sat8((int64_t)W[i] - dw);
    }
    if (shift_out) *shift_out = s;
    if (wshift_out) *wshift_out = ws;
    if (max_out) *max_out = m;
    return nonzero;
}

/* ------------------------------------------------- int8 Linear contractions */

/* Forward: Y[b, oc] = sum_ic X[b, ic] * W[oc, ic]; W indexed W[oc*IC + ic]
 * ([TGR] pass 3). */
void ora_linear_fwd(const int8_t *X, const int8_t *W, int B, int IC, int OC, int32_t *Y)
{
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; b++) {
        const int8_t *x = X + (int64_t)b * IC;
        for (int oc = 0; oc < OC; oc++) {
            const int8_t *w = W + (int64_t)oc * IC;
            int64_t acc = 0;
            for (int ic = 0; ic < IC; ic++)
                acc += (int64_t)x[ic] * (int64_t)w[ic];
            Y[(int64_t)b * OC + oc] = checked_i32(acc);
        }
    }
}

/* Delta propagation: D[b, ic] = sum_oc delta[b, oc] * W[oc, ic]. */
void ora_linear_dgrad(const int8_t *delta, const int8_t *W, int B, int IC, int OC, int32_t *D)
{
#pragma omp parallel
    {
        int64_t *acc = (int64_t *)malloc(sizeof(int64_t) * (size_t)(IC > 0 ? IC : 1));
        if (!acc) ora_fail("out of memory");
#pragma omp for schedule(static)
        for (int b = 0; b < B; b++) {
            for (int ic = 0; ic < IC; ic++) acc[ic] = 0;
            for (int oc = 0; oc < OC; oc++) {
                int64_t d = delta[(int64_t)b * OC + oc];
                const int8_t *w = W + (int64_t)oc * IC;
                for (int ic = 0; ic < IC; ic++)
                    acc[ic] += d * (int64_t)w[ic];
            }
            for (int ic = 0; ic < IC; ic++)
                D[(int64_t)b * IC + ic] = checked_i32(acc[ic]);
        }
        free(acc);
    }
}

/* Weight gradient, summed over the batch (no mean): G[oc, ic] = sum_b
 * delta[b, oc] * A[b, ic], where A is the layer's int8 input. */
void ora_linear_wgrad(const int8_t *delta, const int8_t *A, int B, int IC, int OC, int32_t *G)
{
#pragma omp parallel
    {
        int64_t *acc = (int64_t *)malloc(sizeof(int64_t) * (size_t)(IC > 0 ? IC : 1));
        if (!acc) ora_fail("out of memory");
#pragma omp for schedule(static)
        for (int oc = 0; oc < OC; oc++) {
            for (int ic = 0; ic < IC; ic++) acc[ic] = 0;
            for (int b = 0; b < B; b++) {
                int64_t d = delta[(int64_t)b * OC + oc];
                const int8_t *a = A + (int64_t)b * IC;
                for (int ic = 0; ic < IC; ic++)
                    acc[ic] += d * (int64_t)a[ic];
            }
            for (int ic = 0; ic < IC; ic++)
                G[(int64_t)oc * IC + ic] = checked_i32(acc[ic]);
        }
        free(acc);
    }
}

/* Static per-channel requantisation of the TI library's forward ([ODT]
 * section 4: each layer holds INT32 offsets and const k (shift) and mult
 * arrays; section 6, step 2: the exported OSS chain Add(offset) -> Mul ->
 * Mul -> Floor -> Clip). Reading: the two multiplies are the integer mult
 * and a right shift by k, i.e.
 *   out[b][c] = clip(floor((Y[b][c] + offset[c]) * mult[c] / 2^k[c]), lo, 127)
 * with lo = 0 for a ReLU layer (the clamp at the output zero point) and -128
 * otherwise; the product is formed in int64. */
void ora_requant_static(const int32_t *Y, int B, int C, const int32_t *offset, const int32_t *mult,
                        const int32_t *k, int relu, int8_t *out)
{
    for (int b = 0; b < B; b++)
        for (int c = 0; c < C; c++) {
            if (k[c] < 0 || k[c] > 62) ora_fail("static shift out of range");
            int64_t v = ((int64_t)Y[(int64_t)b * C + c] + offset[c]) * (int64_t)mult[c];
            int64_t q = floor_div_pow2(v, k[c]);
            int64_t lo = relu ? 0 : -128;
            if (q < lo) q = lo;
            if (q > 127) q = 127;
            out[(int64_t)b * C + c] = (int8_t)q;
        }
}

/* Gradient of the offsets: the offset is added to every row of Y, so its
 * gradient is the delta summed over the batch rows: g[c] = sum_b delta[b][c]. */
void ora_offset_grad(const int8_t *delta, int B, int C, int32_t *g)
{
    for (int c = 0; c < C; c++) {
        int64_t acc = 0;
        for (int b = 0; b < B; b++) acc += delta[(int64_t)b * C + c];
        g[c] = checked_i32(acc);
    }
}

/* Update of the INT32 offsets. Reading (the pages say only that offsets are
 * updated by the backward pass): the same NITI Steps 1-5 as for weights,
 * applied to the offset gradient, with the result saturated to int32:
 * s = max(0, bitlen(max|g|) - target_bits), Gq = sat8(rhu(g, s)),
 * dO = rhu(Gq, max(0, s - mu)), offset = sat32(offset - dO). */
int64_t ora_offset_update(int32_t *offset, const int32_t *g, int C, int32_t target_bits, int32_t mu_weight,
                          int32_t *shift_out, int32_t *wshift_out, uint32_t *max_out)
{
    uint32_t m = ora_absmax32(g, C);
    int32_t s = ora_shift_from_max(m, target_bits);
    int32_t ws = s - mu_weight > 0 ? s - mu_weight : 0;
    int64_t nonzero = 0;
    for (int c = 0; c < C; c++) {
        int64_t d = ora_rhu(ora_sat8(ora_rhu(g[c], s)), ws);
        if (d != 0) nonzero++;
        int64_t v = (int64_t)offset[c] - d;
        if (v < INT32_MIN) v = INT32_MIN;
        if (v > INT32_MAX) v = INT32_MAX;
        offset[c] = (int32_t)v;
    }
    if (shift_out) *shift_out = s;
    if (wshift_out) *wshift_out = ws;
    if (max_out) *max_out = m;
    return nonzero;
}

/* UINT8-input variants for the first trainable layer of a partial model
 * ([ODT] section 4: the frozen part ends in a ReLU layer, so the library
 * receives UINT8 activations in [0, 255]). */
void ora_linear_fwd_u8(const uint8_t *X, const int8_t *W, int B, int IC, int OC, int32_t *Y)
{
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; b++) {
        const uint8_t *x = X + (int64_t)b * IC;
        for (int oc = 0; oc < OC; oc++) {
            const int8_t *w = W + (int64_t)oc * IC;
            int64_t acc = 0;
            for (int ic = 0; ic < IC; ic++)
                acc += (int64_t)x[ic] * (int64_t)w[ic];
            Y[(int64_t)b * OC + oc] = checked_i32(acc);
        }
    }
}

void ora_linear_wgrad_u8(const int8_t *delta, const uint8_t *A, int B, int IC, int OC, int32_t *G)
{
#pragma omp parallel
    {
        int64_t *acc = (int64_t *)malloc(sizeof(int64_t) * (size_t)(IC > 0 ? IC : 1));
        if (!acc) ora_fail("out of memory");
#pragma omp for schedule(static)
        for (int oc = 0; oc < OC; oc++) {
            for (int ic = 0; ic < IC; ic++) acc[ic] = 0;
            for (int b = 0; b < B; b++) {
                int64_t d = delta[(int64_t)b * OC + oc];
                const uint8_t *a = A + (int64_t)b * IC;
                for (int ic = 0; ic < IC; ic++)
                    acc[ic] += d * (int64_t)a[ic];
            }
            for (int ic = 0; ic < IC; ic++)
                G[(int64_t)oc * IC + ic] = checked_i32(acc[ic]);
        }
        free(acc);
    }
}

/* ReLU mask bits ([ODT] section 8, "ReLU Mask Buffers": BATCH_SIZE *
 * ceil(out_size / 8) bytes per ReLU layer): bit j % 8 of byte j / 8 of row b
 * is 1 where A[b][j] > 0. */
void ora_pack_relu_mask(const int8_t *A, int B, int F, uint8_t *mask)
{
    int64_t bytes = (F + 7) / 8;
    for (int b = 0; b < B; b++)
        for (int64_t k = 0; k < bytes; k++) {
            unsigned v = 0;
            for (int j = 0; j < 8; j++) {
                int64_t f = k * 8 + j;
                if (f < F && A[(int64_t)b * F + f] > 0) v |= 1u << j;
            }
            mask[(int64_t)b * bytes + k] = (uint8_t)v;
        }
}

/* ------------------------------------------------------ int8 conv (NHWC) */

static int conv_out(int in, int k, int stride, int pad)
{
    return (in + 2 * pad - k) / stride + 1;
}

/* Conv2D ([ODT] section 7: dense, groups = 1, dilation = 1) written as the
 * direct 7-deep loop. X [B][H][W][IC] (NHWC), Wt [OC][KH][KW][IC],
 * Y [B][OH][OW][OC]. Taps that fall in the zero padding contribute 0. */
void ora_conv2d_fwd(const int8_t *X, const int8_t *Wt, int B, int H, int Wd, int IC,
                    int OC, int KH, int KW, int stride, int pad, int32_t *Y)
{
    int OH = conv_out(H, KH, stride, pad), OW = conv_out(Wd, KW, stride, pad);
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; b++)
        for (int oh = 0; oh < OH; oh++)
            for (int ow = 0; ow < OW; ow++)
                for (int oc = 0; oc < OC; oc++) {
                    int64_t acc = 0;
                    for (int kh = 0; kh < KH; kh++) {
                        int ih = oh * stride - pad + kh;
                        if (ih < 0 || ih >= H) continue;
                        for (int kw = 0; kw < KW; kw++) {
                            int iw = ow * stride - pad + kw;
                            if (iw < 0 || iw >= Wd) continue;
                            const int8_t *x = X + (((int64_t)b * H + ih) * Wd + iw) * IC;
                            const int8_t *w = Wt + (((int64_t)oc * KH + kh) * KW + kw) * IC;
                            for (int ic = 0; ic < IC; ic++)
                                acc += (int64_t)x[ic] * (int64_t)w[ic];
                        }
                    }
                    Y[(((int64_t)b * OH + oh) * OW + ow) * OC + oc] = checked_i32(acc);
                }
}

/* Conv2D delta propagation as a scatter: every output delta sends
 * delta[b,oh,ow,oc] * Wt[oc,kh,kw,ic] to the input position it was computed
 * from. D [B][H][W][IC]. */
void ora_conv2d_dgrad(const int8_t *delta, const int8_t *Wt, int B, int H, int Wd, int IC,
                      int OC, int KH, int KW, int stride, int pad, int32_t *D)
{
    int OH = conv_out(H, KH, stride, pad), OW = conv_out(Wd, KW, stride, pad);
    int64_t img = (int64_t)H * Wd * IC;
#pragma omp parallel
    {
        int64_t *acc = (int64_t *)malloc(sizeof(int64_t) * (size_t)(img > 0 ? img : 1));
        if (!acc) ora_fail("out of memory");
#pragma omp for schedule(static)
        for (int b = 0; b < B; b++) {
            memset(acc, 0, sizeof(int64_t) * (size_t)img);
            for (int oh = 0; oh < OH; oh++)
                for (int ow = 0; ow < OW; ow++)
                    for (int oc = 0; oc < OC; oc++) {
                        int64_t d = delta[(((int64_t)b * OH + oh) * OW + ow) * OC + oc];
                        if (d == 0) continue;
                        for (int kh = 0; kh < KH; kh++) {
                            int ih = oh * stride - pad + kh;
                            if (ih < 0 || ih >= H) continue;
                            for (int kw = 0; kw < KW; kw++) {
                                int iw = ow * stride - pad + kw;
                                if (iw < 0 || iw >= Wd) continue;
                                const int8_t *w = Wt + (((int64_t)oc * KH + kh) * KW + kw) * IC;
                                int64_t *a = acc + ((int64_t)ih * Wd + iw) * IC;
                                for (int ic = 0; ic < IC; ic++)
                                    a[ic] += d * (int64_t)w[ic];
                            }
                        }
                    }
            for (int64_t i = 0; i < img; i++)
                D[(int64_t)b * img + i] = checked_i32(acc[i]);
        }
        free(acc);
    }
}

/* Conv2D weight gradient: G[oc,kh,kw,ic] = sum over b, oh, ow of
 * delta[b,oh,ow,oc] * X[b, oh*stride-pad+kh, ow*stride-pad+kw, ic]
 * (padding taps contribute 0). */
void ora_conv2d_wgrad(const int8_t *delta, const int8_t *X, int B, int H, int Wd, int IC,
                      int OC, int KH, int KW, int stride, int pad, int32_t *G)
{
    int OH = conv_out(H, KH, stride, pad), OW = conv_out(Wd, KW, stride, pad);
    int64_t per_oc = (int64_t)KH * KW * IC;
#pragma omp parallel
    {
        int64_t *acc = (int64_t *)malloc(sizeof(int64_t) * (size_t)(per_oc > 0 ? per_oc : 1));
        if (!acc) ora_fail("out of memory");
#pragma omp for schedule(static)
        for (int oc = 0; oc < OC; oc++) {
            memset(acc, 0, sizeof(int64_t) * (size_t)per_oc);
            for (int b = 0; b < B; b++)
                for (int oh = 0; oh < OH; oh++)
                    for (int ow = 0; ow < OW; ow++) {
                        int64_t d = delta[(((int64_t)b * OH + oh) * OW + ow) * OC + oc];
                        if (d == 0) continue;
                        for (int kh = 0; kh < KH; kh++) {
                            int ih = oh * stride - pad + kh;
                            if (ih < 0 || ih >= H) continue;
                            for (int kw = 0; kw < KW; kw++) {
                                int iw = ow * stride - pad + kw;
                                if (iw < 0 || iw >= Wd) continue;
                                const int8_t *x = X + (((int64_t)b * H + ih) * Wd + iw) * IC;
                                int64_t *g = acc + ((int64_t)kh * KW + kw) * IC;
                                for (int ic = 0; ic < IC; ic++)
                                    g[ic] += d * (int64_t)x[ic];
                            }
                        }
                    }
            for (int64_t i = 0; i < per_oc; i++)
                G[(int64_t)oc * per_oc + i] = checked_i32(acc[i]);
        }
        free(acc);
    }
}

/* Global average pooling as an integer sum: P[b, c] = sum over the HW spatial
 * positions of A[b, pos, c]. The division by HW is left out; the NITI shift
 * that follows rescales the tensor. */
void ora_gap_fwd(const int8_t *A, int B, int HW, int C, int32_t *P)
{
    for (int b = 0; b < B; b++)
        for (int c = 0; c < C; c++) {
            int64_t acc = 0;
            for (int p = 0; p < HW; p++)
                acc += A[((int64_t)b * HW + p) * C + c];
            P[(int64_t)b * C + c] = checked_i32(acc);
        }
}

/* Backward of the integer sum pooling: every position receives the pooled
 * delta, gated by the ReLU of the layer below:
 * D[b, pos, c] = (A[b, pos, c] > 0) ? dP[b, c] : 0. */
void ora_gap_bwd(const int8_t *dP, const int8_t *A, int B, int HW, int C, int8_t *D)
{
    for (int b = 0; b < B; b++)
        for (int p = 0; p < HW; p++)
            for (int c = 0; c < C; c++) {
                int64_t i = ((int64_t)b * HW + p) * C + c;
                D[i] = A[i] > 0 ? dP[(int64_t)b * C + c] : 0;
            }
}

/* ------------------------------------------------------------- DFP16 path */

/* [DFP] 3.1: the product of two DFP tensors is an integer tensor whose
 * exponent is the sum of the operands' exponents; the FMA chain shares it.
 * The sum is kept exact in int64 here (no 32-bit wraparound).
 * P[b, oc] = sum_ic X[b, ic] * W[oc, ic]. */
void ora_dfp_linear_fwd(const int16_t *X, const int16_t *W, int B, int IC, int OC, int64_t *P)
{
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; b++) {
        const int16_t *x = X + (int64_t)b * IC;
        for (int oc = 0; oc < OC; oc++) {
            const int16_t *w = W + (int64_t)oc * IC;
            int64_t acc = 0;
            for (int ic = 0; ic < IC; ic++)
                acc += (int64_t)x[ic] * (int64_t)w[ic];
            P[(int64_t)b * OC + oc] = acc;
        }
    }
}

/* P[b, ic] = sum_oc delta[b, oc] * W[oc, ic]. */
void ora_dfp_linear_dgrad(const int16_t *delta, const int16_t *W, int B, int IC, int OC, int64_t *P)
{
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; b++) {
        int64_t *p = P + (int64_t)b * IC;
        for (int ic = 0; ic < IC; ic++) p[ic] = 0;
        for (int oc = 0; oc < OC; oc++) {
            int64_t d = delta[(int64_t)b * OC + oc];
            const int16_t *w = W + (int64_t)oc * IC;
            for (int ic = 0; ic < IC; ic++)
                p[ic] += d * (int64_t)w[ic];
        }
    }
}

/* P[oc, ic] = sum_b delta[b, oc] * A[b, ic]. */
void ora_dfp_linear_wgrad(const int16_t *delta, const int16_t *A, int B, int IC, int OC, int64_t *P)
{
#pragma omp parallel for schedule(static)
    for (int oc = 0; oc < OC; oc++) {
        int64_t *p = P + (int64_t)oc * IC;
        for (int ic = 0; ic < IC; ic++) p[ic] = 0;
        for (int b = 0; b < B; b++) {
            int64_t d = delta[(int64_t)b * OC + oc];
            const int16_t *a = A + (int64_t)b * IC;
            for (int ic = 0; ic < IC; ic++)
                p[ic] += d * (int64_t)a[ic];
        }
    }
}

/* [DFP] 3.1 down-conversion of a wide integer tensor to DFP-16: right shift
 * by Rs bits and add Rs to the shared exponent. Reading: Rs is the smallest
 * shift that brings max|P| within target_bits (15) bits, the same rule as the
 * NITI shift; the shift rounds half up and the result saturates to
 * [-32767, 32767]. Returns Rs; the caller adds it to the exponent. */
int32_t ora_dfp_down(const int64_t *P, int64_t n, int32_t target_bits, int16_t *out,
                     uint64_t *max_out)
{
    uint64_t m = ora_absmax64(P, n);
    int32_t rs = ora_shift_from_max(m, target_bits);
    for (int64_t i = 0; i < n; i++)
        out[i] = (int16_t)ora_sat16(ora_rhu(P[i], rs));
    if (max_out) *max_out = m;
    return rs;
}

/* [DFP] 3.1: converting a floating-point tensor to DFP-16 derives the shared
 * exponent from the exponent of its absolute maximum. Reading: with
 * max|f| = frac * 2^e (frac in [0.5, 1)), E = e - 15, so every mantissa
 * f * 2^-E is below 2^15 in magnitude; mantissas are rounded to nearest, ties
 * to even (the IEEE default), and saturated to [-32767, 32767]. An all-zero
 * tensor gets exponent 0. Inputs must be finite. Returns E (the caller checks
 * the int8 range). */
int32_t ora_dfp_from_float(const float *f, int64_t n, int16_t *out)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(f[i]);
        if (!(a <= 3.4028235e38f)) ora_fail("non-finite input");
        if (a > m) m = a;
    }
    int e = 0;
    if (m > 0.0f) frexpf(m, &e);
    int32_t E = m > 0.0f ? e - 15 : 0;
    for (int64_t i = 0; i < n; i++) {
        float v = ldexpf(f[i], -E);          /* exact: a power-of-two scaling below 2^15 */
        long q = lrintf(v);                  /* round to nearest, ties to even */
        if (q > 32767) q = 32767;
        if (q < -32767) q = -32767;
        out[i] = (int16_t)q;
    }
    return E;
}

/* DFP-16 to float: f = i * 2^E ([DFP] 3.1), one rounding at most (exact
 * whenever the result is a normal or exactly representable subnormal float). */
void ora_dfp_to_float(const int16_t *m, int64_t n, int32_t E, float *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = ldexpf((float)m[i], E);
}

/* [DFP] section 3: Blocked-DFP gains range through several fine-grained
 * exponents per tensor. The page gives no block shape; reading: each row of a
 * [rows][cols] tensor is cut into blocks of `block` consecutive elements (the
 * last one shorter when block does not divide cols), and every block is a
 * DFP-16 tensor of its own (ora_dfp_from_float on the block).
 * exps: [rows][ceil(cols / block)]. */
void ora_bdfp_from_float(const float *f, int64_t rows, int64_t cols, int32_t block, int16_t *out, int32_t *exps)
{
    const int64_t nb = (cols + block - 1) / block;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t j = 0; j < nb; j++) {
            const int64_t c0 = j * block;
            const int64_t len = cols - c0 < block ? cols - c0 : block;
            exps[r * nb + j] = ora_dfp_from_float(f + r * cols + c0, len, out + r * cols + c0);
        }
}

void ora_bdfp_to_float(const int16_t *m, const int32_t *exps, int64_t rows, int64_t cols, int32_t block, float *out)
{
    const int64_t nb = (cols + block - 1) / block;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t j = 0; j < nb; j++) {
            const int64_t c0 = j * block;
            const int64_t len = cols - c0 < block ? cols - c0 : block;
            ora_dfp_to_float(m + r * cols + c0, len, exps[r * nb + j], out + r * cols + c0);
        }
}

/* Linear forward with FP32 output over Blocked-DFP operands whose blocks run
 * along the contraction (x [B][IC] and W [OC][IC], both blocked along IC with
 * the same block length): each block's products sum exactly in int64 (P_j,
 * exponent Ex_j + Ew_j by [DFP] 3.1); the blocks are added in double, in
 * block order, P_j * 2^(Ex_j + Ew_j) (each term exact), and the sum is rounded
 * once to float ([DFP] section 4: the kernels produce FP32 outputs). */
void ora_bdfp_linear_fwd_f32(const int16_t *x, const int32_t *ex, const int16_t *W, const int32_t *ew, int B, int IC,
                             int OC, int block, float *y)
{
    const int nb = (IC + block - 1) / block;
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; b++)
        for (int oc = 0; oc < OC; oc++) {
            double acc = 0.0;
            for (int j = 0; j < nb; j++) {
                const int k1 = (j + 1) * block < IC ? (j + 1) * block : IC;
                int64_t p = 0;
                for (int k = j * block; k < k1; k++) p += (int64_t)x[(int64_t)b * IC + k] * W[(int64_t)oc * IC + k];
                acc += ldexp((double)p, ex[b * nb + j] + ew[oc * nb + j]);
            }
            y[(int64_t)b * OC + oc] = (float)acc;
        }
}

/* FP32 output of a DFP contraction ([DFP] section 4: the kernels produce FP32
 * outputs): the exact int64 sum P rounded to float (to nearest, ties to even),
 * then scaled by 2^(Ea + Eb). */
void ora_p64_to_float(const int64_t *P, int64_t n, int32_t E, float *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = ldexpf((float)P[i], E);
}

/* Linear forward with FP32 output by the page's partial-accumulation scheme
 * ([DFP] section 4, "Handling overflows": INT16 products overflow an INT32
 * accumulator after a few terms, so the kernels keep accumulation chains short,
 * shift the inputs by one bit, convert each chain's INT32 partial to FP32, scale
 * it by 2^(E_inp + E_wt) and accumulate it into the FP32 output). Steps, in the
 * page's order:
 *   1. with input_shift = 1 every input mantissa becomes rhu(x, 1) and the
 *      input exponent E_inp = ex + 1 (with 0, x and ex unchanged);
 *   2. the contraction over IC is cut into chains of `chain` consecutive terms
 *      (the last one shorter when chain does not divide IC);
 *   3. a chain's products sum in an INT32 accumulator that wraps modulo 2^32 as
 *      the hardware's two's-complement accumulator does (the page's point is
 *      that the shift and the chain length keep this from happening);
 *   4. the chain's INT32 value is converted to FP32 (to nearest, ties to even)
 *      and scaled by 2^(E_inp + ew), the product formed exactly in double and
 *      rounded once to FP32;
 *   5. the terms are added to the FP32 output, which starts at 0, in increasing
 *      chain order, each addition rounded to FP32.
 * Readings (the page fixes none of them): the chain length is a parameter, the
 * shift rounds half up as the down-conversion does, and the accumulator wraps. */
void ora_dfp_linear_fwd_f32_chained(const int16_t *x, int32_t ex, const int16_t *W, int32_t ew, int B, int IC,
                                    int OC, int chain, int input_shift, float *y)
{
    if (chain < 1) ora_fail("chain length must be >= 1");
    const int32_t e_inp = input_shift ? ex + 1 : ex;
    const double scale = ldexp(1.0, e_inp + ew);
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; b++)
        for (int oc = 0; oc < OC; oc++) {
            float out = 0.0f;
            for (int k0 = 0; k0 < IC; k0 += chain) {
                const int k1 = k0 + chain < IC ? k0 + chain : IC;
                uint32_t acc = 0;                     /* INT32 accumulator, two's complement */
                for (int k = k0; k < k1; k++) {
                    int64_t xv = x[(int64_t)b * IC + k];
                    if (input_shift) xv = ora_rhu(xv, 1);
                    const int64_t prod = xv * (int64_t)W[(int64_t)oc * IC + k];
                    acc += (uint32_t)(prod & 0xFFFFFFFF);
                }
                const int64_t p32 = acc >= 0x80000000u ? (int64_t)acc - ((int64_t)1 << 32) : (int64_t)acc;
                const float pf = (float)p32;
                const float term = (float)((double)pf * scale);
                out = out + term;
            }
            y[(int64_t)b * OC + oc] = out;
        }
}

/* Integer SGD on a DFP weight tensor of `bits`-bit mantissas (bits <= 16)
 * with exponent E_W, learning rate 2^-eta: W <- W - G * 2^(E_G - eta - E_W).
 * With k = E_W + eta - E_G the step is dW = rhu(Gm, k) for k >= 0 and
 * Gm * 2^-k for k < 0; then W is saturated to the symmetric bits-bit range
 * [-(2^(bits-1) - 1), 2^(bits-1) - 1] (bits = 16 is sat16). A left shift
 * beyond 17 bits already exceeds every representable difference, so it is
 * capped at 17 without changing the saturated result. Returns the number of
 * nonzero dW. */
int64_t ora_dfp_update(int16_t *W, const int16_t *Gm, int64_t n, int32_t k, int32_t bits)
{
    const int64_t lim = ((int64_t)1 << (bits - 1)) - 1;
    int64_t nonzero = 0;
    for (int64_t i = 0; i < n; i++) {
        int64_t dw;
        if (k >= 0)
            dw = ora_rhu(Gm[i], k);
        else
            dw = (int64_t)Gm[i] * ((int64_t)1 << (-k > 17 ? 17 : -k));
        if (dw != 0) nonzero++;
        int64_t v = (int64_t)W[i] - dw;
        if (v > lim) v = lim;
        if (v < -lim) v = -lim;
        W[i] = (int16_t)v;
    }
    return nonzero;
}

/* [APT] "Adaptive Precision Training for Resource Constrained Devices",
 * section III: a layer's weights are a k-bit quantised tensor; its precision k
 * is raised or lowered by Algorithm 1. Reading: the weights are k-bit
 * mantissas with one shared power-of-two exponent E (the DFP representation
 * of [DFP] section 3), so the minimum resolution epsilon is 2^E. Going from
 * bits_old to bits_new = bits_old + d:
 *   d >= 0: W <- W * 2^d, E <- E - d (every value kept exactly);
 *   d <  0: W <- clamp(rhu(W, -d), +-(2^(bits_new-1) - 1)), E <- E - d.
 * Returns the exponent change (-d). */
int32_t ora_dfp_set_bits(int16_t *W, int64_t n, int32_t bits_old, int32_t bits_new)
{
    const int32_t d = bits_new - bits_old;
    const int64_t lim = ((int64_t)1 << (bits_new - 1)) - 1;
    for (int64_t i = 0; i < n; i++) {
        int64_t v = d >= 0 ? (int64_t)W[i] * ((int64_t)1 << d) : ora_rhu(W[i], -d);
        if (v > lim) v = lim;
        if (v < -lim) v = -lim;
        W[i] = (int16_t)v;
    }
    return -d;
}

/* sum of |x| over an int16 tensor (the numerator of [APT] Equation 4's mean) */
int64_t ora_abs_sum16(const int16_t *x, int64_t n)
{
    int64_t s = 0;
    for (int64_t i = 0; i < n; i++) s += x[i] < 0 ? -(int64_t)x[i] : (int64_t)x[i];
    return s;
}

/* Threads of the OpenMP loops over output rows (the results do not depend on it: every
 * output element is computed by one thread, in the same order). */
void ora_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
int ora_max_threads(void) { return omp_get_max_threads(); }
