/*
 * fsa_oracle.c -- plain, slow FP64 CPU oracle of Fused-Softmax quantized
 * attention (forward pass).  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg may call it; the product path
 * never does.  It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (cited by title and section/paragraph; "para N" counts the body
 * paragraphs of the article from its first one, "Making AI calculations..."):
 *   [NEWS]  "Fused-Softmax shifts an AI attention bottleneck onto faster GPU
 *            hardware" (article on arXiv:2611.09225)
 *            para 5: frozen reference maximum, threshold-triggered recovery
 *            para 6: Schraudolph exponential folded into the score product,
 *                    two-stage integer -> BF16 -> low-precision P conversion,
 *                    row sum by a second product on the same quantized P
 *            para 7: error split (operand quantization vs. softmax redesign)
 *            para 8: formats; the MXFP4 variant keeps six-bit P
 *   [SUMM]  "Fused softmax makes quantized attention faster on AMD GPUs"
 *            (summary of the same preprint), "What the evidence shows",
 *            bullet "Move work, keep correction"
 *   [EFQ]   "EFQ-Softmax: Exp-Free Quantization for Softmax", sections
 *            "B. Block-Scaled E2M1 Probability Representation" (32-element
 *            blocks with a shared E8M0 power-of-two scale) and
 *            "D. Algorithmic Cost and Method Boundary" (masks are applied
 *            before the score shift)
 *   Schraudolph, "A Fast, Compact Approximation of the Exponential Function",
 *            Neural Computation 11(4), 1999 (the exponent-field trick and its
 *            RMS-optimal shift constant).
 *
 * The pages give no equations; every step below follows the plainest reading
 * of the prose, and each reading is listed in the design notes of the repo.
 * All arithmetic is in double precision.  Rounding to an integer uses
 * nearbyint() in the default round-to-nearest-even mode.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_ERR_ARG 1
#define ORA_ERR_NOMEM 2

/* ------------------------------------------------------------------------
 * Element formats of the MX (microscaling) operands.
 *   0: E4M3 (MXFP8 elements and MXFP8's P)
 *   1: E2M3 (MXFP6 elements; P of both MXFP6 and MXFP4 -- [NEWS] para 8)
 *   2: E2M1 (MXFP4 elements)
 * Each is sign + ebits exponent + mbits mantissa with the given bias,
 * subnormals when the exponent field is 0, and a largest finite value maxv
 * (E4M3 reserves its all-ones code for NaN; the two narrow types have no
 * Inf/NaN).
 * ---------------------------------------------------------------------- */
typedef struct {
    int ebits, mbits, bias;
    double maxv;
} ora_fmt;

static const ora_fmt ORA_FMTS[3] = {
    {4, 3, 7, 448.0}, /* E4M3: max 1.75 * 2^8 */
    {2, 3, 1, 7.5},   /* E2M3: max 1.875 * 2^2 */
    {2, 1, 1, 6.0},   /* E2M1: max 1.5 * 2^2 */
};

int ora_num_formats(void) { return 3; }

/* Value of an element code. */
double ora_decode_elem(int fmt, int code)
{
    const ora_fmt *f = &ORA_FMTS[fmt];
    int sign = (code >> (f->ebits + f->mbits)) & 1;
    int e = (code >> f->mbits) & ((1 << f->ebits) - 1);
    int m = code & ((1 << f->mbits) - 1);
    double v;
    if (fmt == 0 && e == 15 && m == 7) return NAN; /* E4M3 NaN code */
    if (e == 0)
        v = ldexp((double)m, 1 - f->bias - f->mbits);
    else
        v = ldexp(1.0 + ldexp((double)m, -f->mbits), e - f->bias);
    return sign ? -v : v;
}

/* Round |a| to the grid of a binary format with mbits stored mantissa bits
 * and smallest normal exponent emin, ties to even (no overflow handling). */
static double round_to_grid(double a, int mbits, int emin)
{
    int k;
    double fr, quantum;
    if (a == 0.0) return 0.0;
    fr = frexp(a, &k);   /* a = fr * 2^k, fr in [0.5, 1) */
    (void)fr;
    k -= 1;              /* a in [2^k, 2^(k+1)) */
    if (k < emin) k = emin;                 /* subnormal: fixed quantum */
    quantum = ldexp(1.0, k - mbits);
    return nearbyint(a / quantum) * quantum; /* exact scaling, RNE */
}

/* Code of the element nearest to v (ties to even), saturating at +-maxv.
 * The sign bit follows the sign of v, also when v rounds to zero. */
int ora_encode_elem(int fmt, double v)
{
    const ora_fmt *f = &ORA_FMTS[fmt];
    int sign = signbit(v) ? 1 : 0;
    int emin = 1 - f->bias;
    double a = fabs(v), q;
    int code;
    q = round_to_grid(a, f->mbits, emin);
    if (q > f->maxv) q = f->maxv;
    if (q < ldexp(1.0, emin)) {
        /* zero or subnormal: exponent field 0 */
        code = (int)(q / ldexp(1.0, emin - f->mbits));
    } else {
        int k;
        double fr = frexp(q, &k);
        int e = k - 1;
        int m = (int)((ldexp(fr, 1) - 1.0) * (double)(1 << f->mbits));
        code = ((e + f->bias) << f->mbits) | m;
    }
    return code | (sign << (f->ebits + f->mbits));
}

/* ------------------------------------------------------------------------
 * BF16 helpers.  A bf16 is the upper half of an IEEE binary32.
 * ---------------------------------------------------------------------- */
double ora_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to bf16 (8 significant bits, exponent range of binary32,
 * ties to even).  Values beyond the finite range become Inf. */
uint16_t ora_double_to_bf16(double v)
{
    int sign = signbit(v) ? 1 : 0;
    double a = fabs(v), q;
    uint32_t bits;
    float f;
    if (isnan(v)) return 0x7FC0;
    q = round_to_grid(a, 7, -126);
    if (q > ldexp(255.0 / 128.0, 127)) q = INFINITY; /* beyond 0x7F7F */
    f = (float)q;   /* exact: q has at most 8 significant bits */
    memcpy(&bits, &f, 4);
    return (uint16_t)((bits >> 16) | ((uint32_t)sign << 15));
}

/* ------------------------------------------------------------------------
 * MX block scale.  The pages do not print the scale rule; the reading used
 * here: the shared E8M0 scale 2^X of a block is the smallest power of two
 * for which the block's largest magnitude fits the element format without
 * saturating, i.e. the smallest integer X with amax <= maxv * 2^X, clamped
 * to the E8M0 range [-127, 127]; an all-zero block takes X = -127.
 * ---------------------------------------------------------------------- */
int ora_mx_scale_exp(int fmt, double amax)
{
    const ora_fmt *f = &ORA_FMTS[fmt];
    int X, k;
    if (!(amax > 0.0)) return -127;
    frexp(amax / f->maxv, &k);       /* amax/maxv in [2^(k-1), 2^k) */
    X = k;                           /* candidate; fix up exactly below */
    while (X > -200 && amax <= f->maxv * ldexp(1.0, X - 1)) X--;
    while (amax > f->maxv * ldexp(1.0, X)) X++;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X;
}

/* Quantize one block of n <= 32 values: writes element codes, returns X.
 * If deq != NULL it receives the block's dequantized values. */
static int mx_block(int fmt, const double *x, int n, uint8_t *codes, double *deq)
{
    double amax = 0.0;
    int i, X;
    for (i = 0; i < n; i++)
        if (fabs(x[i]) > amax) amax = fabs(x[i]);
    X = ora_mx_scale_exp(fmt, amax);
    for (i = 0; i < n; i++) {
        int c = ora_encode_elem(fmt, ldexp(x[i], -X)); /* exact scaling */
        if (codes) codes[i] = (uint8_t)c;
        if (deq) deq[i] = ldexp(ora_decode_elem(fmt, c), X);
    }
    return X;
}

/* Public MX quantizer on bf16 input x[batch][rows][cols].
 * block_axis = 1: blocks of 32 run along cols;
 *   codes[batch][rows][cols], scales[batch][rows][ceil(cols/32)].
 * block_axis = 0: blocks of 32 run along rows and the output is transposed;
 *   codes[batch][cols][rows], scales[batch][cols][ceil(rows/32)].
 * Scales are E8M0 bytes X + 127.  The last block of a line may be short. */
int ora_mx_quantize(const uint16_t *x, int64_t batch, int64_t rows, int64_t cols,
                    int block_axis, int fmt, uint8_t *codes, uint8_t *scales)
{
    int64_t b, line, nlines, len, nblk, j;
    double buf[32];
    uint8_t cbuf[32];
    if (!x || !codes || !scales || batch < 0 || rows < 0 || cols < 0 ||
        fmt < 0 || fmt > 2 || (block_axis != 0 && block_axis != 1))
        return ORA_ERR_ARG;
    nlines = block_axis ? rows : cols;
    len = block_axis ? cols : rows;
    nblk = (len + 31) / 32;
    for (b = 0; b < batch; b++) {
        const uint16_t *xb = x + b * rows * cols;
        for (line = 0; line < nlines; line++) {
            for (j = 0; j < nblk; j++) {
                int64_t i0 = j * 32, n = len - i0 < 32 ? len - i0 : 32, i;
                int X;
                for (i = 0; i < n; i++) {
                    int64_t r = block_axis ? line : i0 + i;
                    int64_t c = block_axis ? i0 + i : line;
                    buf[i] = ora_bf16_to_double(xb[r * cols + c]);
                }
                X = mx_block(fmt, buf, (int)n, cbuf, NULL);
                for (i = 0; i < n; i++)
                    codes[(b * nlines + line) * len + i0 + i] = cbuf[i];
                scales[(b * nlines + line) * nblk + j] = (uint8_t)(X + 127);
            }
        }
    }
    return ORA_OK;
}

/* ------------------------------------------------------------------------
 * Schraudolph exponential in BF16 units ([NEWS] para 6).
 * For a shifted score x = s - m (natural-log units) the affine map
 *     y = 2^7 * (x * log2(e) + 127) - c
 * puts x*log2(e) into the exponent field of a bf16 (7 mantissa bits, bias
 * 127); the integer round(y), clamped to [0, 0x7F7F] so it stays a
 * non-negative finite bf16 pattern, reinterpreted as a bf16 IS the
 * approximation of e^x.  c = 7 is Schraudolph's RMS-optimal shift 60801
 * (given in units of 2^-20 of an octave) rescaled to units of 2^-7 and
 * rounded: 60801 / 2^13 = 7.42.
 * ---------------------------------------------------------------------- */
#define ORA_SCHR_C 7.0

double ora_schraudolph_y(double x)
{
    return 128.0 * (x * M_LOG2E + 127.0) - ORA_SCHR_C;
}

int ora_schraudolph_code(double y)
{
    double r = nearbyint(y);
    if (r < 0.0) r = 0.0;
    if (r > 32639.0) r = 32639.0; /* 0x7F7F, largest finite bf16 */
    return (int)r;
}

/* ------------------------------------------------------------------------
 * Attention oracle.
 * ---------------------------------------------------------------------- */
typedef struct {
    int qkv_fmt;        /* -1: Q/K/V not quantized; else element format */
    int p_fmt;          /* -1: P not quantized; else element format of P */
    int exp_mode;       /* 0: exact exp;  1: Schraudolph bf16 code;
                           2: EFQ-Softmax E2M1 codes (P quantization built in) */
    int max_mode;       /* 0: frozen reference (tile 0) + rollback gate;
                           1: exact row max over all keys (conventional);
                           2: running row max, O and l rescaled when it grows
                              (online attention) */
    int l_from_unquantized; /* 1: l sums the unquantized P (conventional) */
    int tile;           /* keys per KV tile (the gate's granularity) */
    double threshold;   /* gate threshold theta; +Inf disables the gate */
    double sm_scale;    /* score scale; <= 0 means 1/sqrt(D) */
    int gate_mode;      /* 0: the FP32 gate, tile max - m > theta;
                           1: the shortcut on converted values: the tile's
                              largest P block scale (frozen reference) exceeds
                              the scale of a block whose largest weight is the
                              code of theta (needs p_fmt >= 0, exp_mode 1) */
    double efq_tau, efq_h;  /* EFQ affine rule: code = clip(floor((r - tau) / h), 0, 7) */
} ora_params;

typedef struct {
    /* inputs */
    const uint16_t *q, *k, *v;
    int64_t Sq, Sk;             /* query rows and keys per head */
    int D;
    const ora_params *p;
    const double *kd, *vd;      /* dequantized K[Sk][D] and V[Sk][D] of this head */
    int64_t bh;                 /* head index (b*H + h) */
    const int64_t *rows;        /* row indices within the head */
    const int64_t *out_idx;     /* output slot of each row */
    int64_t nrows;
    /* outputs */
    double *out_f64;            /* [n][D] or NULL */
    uint16_t *out_bf16;         /* [n][D] or NULL */
    uint8_t *bits;              /* [n][n_t] or NULL */
    double *margins;            /* [n][n_t] or NULL: tile max - m - theta */
    double *row_m, *row_l;      /* [n] or NULL */
    int64_t count;              /* rollbacks counted by this worker */
    int err;
} ora_job;

/* The gate shortcut on converted values ("Fused-Softmax shifts ...", para
 * 12: the fastest four-bit implementation's shortcut can miss a recovery
 * trigger): with the frozen reference, a tile whose largest score passes it
 * by d has largest weight code c(d); its largest P block scale is
 * X(bf16(c(d))).  The shortcut fires when that scale exceeds the scale of a
 * block whose largest weight is c(theta).  X is a step function, so the
 * shortcut misses triggers with d just above theta (within theta's scale
 * binade). */
static int gate_shortcut_fires(int p_fmt, double d, double theta)
{
    const int cd = ora_schraudolph_code(ora_schraudolph_y(d));
    const int ct = ora_schraudolph_code(ora_schraudolph_y(theta));
    return ora_mx_scale_exp(p_fmt, ora_bf16_to_double((uint16_t)cd)) >
           ora_mx_scale_exp(p_fmt, ora_bf16_to_double((uint16_t)ct));
}

/* EFQ-Softmax probability codes for one block of n <= 32 keys ("EFQ-Softmax:
 * Exp-Free Quantization for Softmax", sections "B. Block-Scaled E2M1
 * Probability Representation" and "C. EFQ-Softmax Probability Code
 * Generation"): from the shifted scores z_j = s_j - m (m the running row
 * maximum, masked keys excluded) take u_j = z_j log2(e); the block's
 * exponent-only scale is 2^X with X the smallest integer such that the block's
 * largest probability 2^(max u) <= 6 * 2^X (6 = the largest E2M1 value),
 * clamped to [-127, 127]; the residual r_j = u_j - X is mapped to an E2M1
 * code by uniformly spaced thresholds, code = clip(floor((r - tau) / h), 0,
 * 7); the quantized probability is that code's E2M1 value times 2^X. */
static void efq_block(const double *z, int n, double tau, double h, double *pq)
{
    double umax = -INFINITY, u[32];
    int j, X;
    for (j = 0; j < n; j++) {
        u[j] = z[j] * M_LOG2E;
        if (u[j] > umax) umax = u[j];
    }
    if (umax == -INFINITY) {            /* every key of the block masked */
        for (j = 0; j < n; j++) pq[j] = 0.0;
        return;
    }
    X = (int)ceil(umax - log2(6.0));
    while (exp2(umax) > ldexp(6.0, X)) X++;
    while (exp2(umax) <= ldexp(6.0, X - 1)) X--;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    for (j = 0; j < n; j++) {
        double k = floor((u[j] - X - tau) / h);
        int code = k < 0.0 ? 0 : (k > 7.0 ? 7 : (int)k);
        pq[j] = ldexp(ora_decode_elem(2, code), X);
    }
}

/* One query row: the KV-tile loop of the method, step by step. */
static int attention_row(ora_job *J, int64_t i, int64_t slot)
{
    const ora_params *P = J->p;
    const int64_t S = J->Sk;    /* keys */
    const int D = J->D;
    const int64_t n_t = (S + P->tile - 1) / P->tile;
    const double sm = P->sm_scale > 0.0 ? P->sm_scale : 1.0 / sqrt((double)D);
    double qd[256], O[256], l = 0.0, m = 0.0;
    double *s = NULL, *pv = NULL, *pq = NULL;
    int64_t t, j, d;
    int64_t fired_count = 0;

    s = (double *)malloc(sizeof(double) * (size_t)P->tile);
    pv = (double *)malloc(sizeof(double) * (size_t)P->tile);
    pq = (double *)malloc(sizeof(double) * (size_t)P->tile);
    if (!s || !pv || !pq) { free(s); free(pv); free(pq); return ORA_ERR_NOMEM; }

    /* Step 1: the query row, MX-quantized along D when quantization is on. */
    {
        const uint16_t *qr = J->q + (J->bh * J->Sq + i) * D;
        for (d = 0; d < D; d++) qd[d] = ora_bf16_to_double(qr[d]);
        if (P->qkv_fmt >= 0)
            for (d = 0; d < D; d += 32)
                mx_block(P->qkv_fmt, qd + d, D - d < 32 ? (int)(D - d) : 32, NULL, qd + d);
    }
    for (d = 0; d < D; d++) O[d] = 0.0;

    /* Exact row max for the conventional reading. */
    if (P->max_mode == 1) {
        m = -INFINITY;
        for (j = 0; j < S; j++) {
            double acc = 0.0;
            for (d = 0; d < D; d++) acc += qd[d] * J->kd[j * D + d];
            if (sm * acc > m) m = sm * acc;
        }
    }

    for (t = 0; t < n_t; t++) {
        int64_t j0 = t * P->tile;
        int64_t j1 = j0 + P->tile < S ? j0 + P->tile : S; /* keys >= S masked */
        int64_t n = j1 - j0;
        double tmax = -INFINITY;

        /* Step 2: scores of this tile. */
        for (j = 0; j < n; j++) {
            double acc = 0.0;
            for (d = 0; d < D; d++) acc += qd[d] * J->kd[(j0 + j) * D + d];
            s[j] = sm * acc;
            if (s[j] > tmax) tmax = s[j];
        }

        /* Step 3: reference maximum ([NEWS] para 5).  Tile 0 freezes it;
         * later tiles keep it unless a score passes it by more than the
         * threshold, in which case the reference moves to this tile's max
         * and the accumulated O and l are rescaled by e^(m_old - m_new). */
        if (P->max_mode == 0) {
            if (t == 0) {
                m = tmax;
            } else {
                double margin = (tmax - m) - P->threshold;
                int fire = tmax - m > P->threshold;
                if (P->gate_mode == 1 && P->p_fmt >= 0)
                    fire = gate_shortcut_fires(P->p_fmt, tmax - m, P->threshold);
                if (J->margins) J->margins[slot * n_t + t] = margin;
                if (fire) {
                    double r = exp(m - tmax);
                    for (d = 0; d < D; d++) O[d] *= r;
                    l *= r;
                    m = tmax;
                    fired_count++;
                    if (J->bits) J->bits[slot * n_t + t] = 1;
                }
            }
        } else if (P->max_mode == 2) {
            /* online attention: the running maximum, exact rescale on growth */
            if (t == 0) {
                m = tmax;
            } else if (tmax > m) {
                double r = exp(m - tmax);
                for (d = 0; d < D; d++) O[d] *= r;
                l *= r;
                m = tmax;
            }
        }

        /* Step 4: weights of this tile. */
        if (P->exp_mode == 2) {
            /* EFQ: the quantized probabilities come directly from the shifted
             * scores, block by block (blocks aligned to the absolute key) */
            int64_t b0;
            for (j = 0; j < n; j++) pv[j] = s[j] - m;
            for (b0 = 0; b0 < n; b0 += 32)
                efq_block(pv + b0, n - b0 < 32 ? (int)(n - b0) : 32, P->efq_tau, P->efq_h, pq + b0);
            for (j = 0; j < n; j++) pv[j] = pq[j];
        }
        for (j = 0; j < n && P->exp_mode != 2; j++) {
            if (P->exp_mode == 0) {
                pv[j] = exp(s[j] - m);
            } else {
                /* integer reinterpretation: the rounded y is a bf16 pattern */
                int code = ora_schraudolph_code(ora_schraudolph_y(s[j] - m));
                pv[j] = ora_bf16_to_double((uint16_t)code);
            }
        }

        /* Step 5: second stage -- the bf16 weights are MX-quantized along the
         * keys in blocks of 32 aligned to the absolute key index. */
        if (P->exp_mode != 2)
            for (j = 0; j < n; j++) pq[j] = pv[j];
        if (P->p_fmt >= 0 && P->exp_mode != 2) {
            int64_t b0;
            for (b0 = 0; b0 < n; b0 += 32)
                mx_block(P->p_fmt, pv + b0, n - b0 < 32 ? (int)(n - b0) : 32, NULL, pq + b0);
        }

        /* Step 6: O += P V and l += P 1 on the same quantized P ([NEWS]
         * para 6), or l from the unquantized P in the conventional reading. */
        for (j = 0; j < n; j++) {
            const double *vr = J->vd + (j0 + j) * D;
            for (d = 0; d < D; d++) O[d] += pq[j] * vr[d];
            l += P->l_from_unquantized ? pv[j] : pq[j];
        }
    }

    /* Step 7: normalisation and output rounding. */
    for (d = 0; d < D; d++) {
        double o = O[d] / l;
        if (J->out_f64) J->out_f64[slot * D + d] = o;
        if (J->out_bf16) J->out_bf16[slot * D + d] = ora_double_to_bf16(o);
    }
    if (J->row_m) J->row_m[slot] = m;
    if (J->row_l) J->row_l[slot] = l;
    free(s); free(pv); free(pq);
    J->count += fired_count;
    return ORA_OK;
}

static void *worker(void *arg)
{
    ora_job *J = (ora_job *)arg;
    int64_t r;
    for (r = 0; r < J->nrows && !J->err; r++)
        J->err = attention_row(J, J->rows[r], J->out_idx[r]);
    return NULL;
}

/* Dequantized K and V of one head.  K blocks run along D (the score
 * contraction axis); V blocks run along the keys (the P V contraction axis). */
static int prepare_head(const uint16_t *k, const uint16_t *v, int64_t bh, int64_t S,
                        int D, int fmt, double *kd, double *vd)
{
    int64_t j, d, i;
    const uint16_t *kb = k + bh * S * D, *vb = v + bh * S * D;
    double buf[32];
    for (j = 0; j < S * D; j++) {
        kd[j] = ora_bf16_to_double(kb[j]);
        vd[j] = ora_bf16_to_double(vb[j]);
    }
    if (fmt < 0) return ORA_OK;
    for (j = 0; j < S; j++)
        for (d = 0; d < D; d += 32)
            mx_block(fmt, kd + j * D + d, D - d < 32 ? (int)(D - d) : 32, NULL, kd + j * D + d);
    for (d = 0; d < D; d++)
        for (j = 0; j < S; j += 32) {
            int n = S - j < 32 ? (int)(S - j) : 32;
            for (i = 0; i < n; i++) buf[i] = vd[(j + i) * D + d];
            mx_block(fmt, buf, n, NULL, buf);
            for (i = 0; i < n; i++) vd[(j + i) * D + d] = buf[i];
        }
    return ORA_OK;
}

/* Attention of q [B*H][Sq][D] over k, v [B*H][Sk][D] (bf16 bit patterns).
 * rows: global query-row indices bh*Sq + i to compute (n_rows of them,
 * grouped by head in any order), or NULL for every row (n_rows ignored).
 * Output slot r holds the r-th requested row.  Outputs may be NULL.
 * bits/margins are [n][n_t] with n_t = ceil(Sk / tile); bits must be zeroed
 * by the caller.  Returns the rollback count through *rollback_count (may be
 * NULL). */
int ora_attention_qk(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t BH, int64_t Sq, int64_t Sk, int D, const ora_params *p,
                     const int64_t *rows, int64_t n_rows, int n_threads,
                     double *out_f64, uint16_t *out_bf16, uint8_t *bits,
                     double *margins, double *row_m, double *row_l,
                     int64_t *rollback_count)
{
    const int64_t S = Sk;
    int64_t bh, r, total = 0;
    int err = ORA_OK;
    int64_t *hrows = NULL, *hslot = NULL;
    double *kd = NULL, *vd = NULL;
    if (p && p->exp_mode == 2 && (!(p->efq_h > 0.0) || p->tile % 32 != 0)) return ORA_ERR_ARG;
    if (!q || !k || !v || !p || BH < 0 || Sq < 1 || Sk < 1 || D < 1 || D > 256 || p->tile < 1 ||
        (p->qkv_fmt < -1 || p->qkv_fmt > 2) || (p->p_fmt < -1 || p->p_fmt > 2))
        return ORA_ERR_ARG;
    if (n_threads < 1) n_threads = 1;
    if (!rows) n_rows = BH * Sq;
    hrows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_rows + 1));
    hslot = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_rows + 1));
    kd = (double *)malloc(sizeof(double) * (size_t)(S * D));
    vd = (double *)malloc(sizeof(double) * (size_t)(S * D));
    if (!hrows || !hslot || !kd || !vd) { err = ORA_ERR_NOMEM; goto done; }

    for (bh = 0; bh < BH && !err; bh++) {
        int64_t nh = 0, per, w;
        pthread_t th[256];
        ora_job jobs[256];
        int nt;
        for (r = 0; r < n_rows; r++) {
            int64_t g = rows ? rows[r] : r;
            if (g < 0 || g >= BH * Sq) { err = ORA_ERR_ARG; goto done; }
            if (g / Sq == bh) { hrows[nh] = g % Sq; hslot[nh] = r; nh++; }
        }
        if (nh == 0) continue;
        prepare_head(k, v, bh, S, D, p->qkv_fmt, kd, vd);
        nt = n_threads > 256 ? 256 : n_threads;
        if (nt > nh) nt = (int)nh;
        per = (nh + nt - 1) / nt;
        for (w = 0; w < nt; w++) {
            ora_job *J = &jobs[w];
            int64_t a = w * per, b = a + per < nh ? a + per : nh;
            memset(J, 0, sizeof(*J));
            J->q = q; J->k = k; J->v = v; J->Sq = Sq; J->Sk = Sk; J->D = D; J->p = p;
            J->kd = kd; J->vd = vd; J->bh = bh;
            J->rows = hrows + a; J->out_idx = hslot + a; J->nrows = b > a ? b - a : 0;
            J->out_f64 = out_f64; J->out_bf16 = out_bf16; J->bits = bits;
            J->margins = margins; J->row_m = row_m; J->row_l = row_l;
            if (nt == 1) worker(J);
            else pthread_create(&th[w], NULL, worker, J);
        }
        for (w = 0; w < nt; w++) {
            if (nt > 1) pthread_join(th[w], NULL);
            if (jobs[w].err) err = jobs[w].err;
            total += jobs[w].count;
        }
    }
done:
    if (rollback_count) *rollback_count = total;
    free(hrows); free(hslot); free(kd); free(vd);
    return err;
}

/* Self-attention: Sq = Sk = S. */
int ora_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  int64_t BH, int64_t S, int D, const ora_params *p,
                  const int64_t *rows, int64_t n_rows, int n_threads,
                  double *out_f64, uint16_t *out_bf16, uint8_t *bits,
                  double *margins, double *row_m, double *row_l,
                  int64_t *rollback_count)
{
    return ora_attention_qk(q, k, v, BH, S, S, D, p, rows, n_rows, n_threads, out_f64, out_bf16,
                            bits, margins, row_m, row_l, rollback_count);
}
