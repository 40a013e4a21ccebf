/*
 * CPU oracle for the widened contraction  --  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  The product path never calls it and shares no
 * code with it.
 *
 * What it computes:
 *
 *   head dtype h: binary16 ("Tensor Programs, Part 1", section "One
 *   Program and One Numerical Contract") or bfloat16 (the BF16 head of the
 *   ContractionEpilogue row of the OpKind table, "ML compiler internals",
 *   section "The OpKind vocabulary").
 *
 *   for every output row m and output feature n
 *       acc = +0.0 in binary32
 *       for k = 0 .. K-1 (ascending):  acc = RN32(acc + RN32(x[m,k] * W[n,k]))
 *       FP32 output (the DenseContraction row: f32 result, no head
 *       rounding):  y = acc, or RN32(acc + b[n]) with a bias
 *       head output:
 *           t = RN_h(acc)                           rounding before the bias
 *           t = RN_h(t + b[n])                      when a bias is given
 *           t = step(t) for each epilogue step      each step rounds to h
 *           y = t
 *
 *   The ContractionEpilogue row says the head's result keeps its dtype and
 *   every step of the pointwise chain rounds through it.  Activations are
 *   compositions of primitives ("ML compiler internals", section "SwiGLU and
 *   GeLU FFN"), so each primitive rounds:
 *       ADD r:      t = RN_h(t + r[m,n])
 *       MUL r:      t = RN_h(t * r[m,n])
 *       SILU:       x / (1 + exp(-x)) over Neg, Exp, Add, Div:
 *                   a = RN_h(-t), e = RN_h(exp(a)), d = RN_h(1 + e), t = RN_h(t / d)
 *       GELU_TANH:  the sigmoid form x / (1 + exp(-c2 (x + c1 x^3))) over
 *                   Mul, Add, Neg, Exp, Div with c1 = RN_h(0.044715),
 *                   c2 = RN_h(2 sqrt(2/pi)):
 *                   s = RN_h(t*t), c = RN_h(s*t), u = RN_h(c1*c), v = RN_h(t+u),
 *                   z = RN_h(c2*v), a = RN_h(-z), e = RN_h(exp(a)),
 *                   d = RN_h(1+e), t = RN_h(t/d)
 *       GELU_ERF:   0.5 x (1 + erf(x / sqrt 2)) over Mul, Erf, Add:
 *                   s = RN_h(c3*t) with c3 = RN_h(1/sqrt 2), e = RN_h(erf(s)),
 *                   d = RN_h(1 + e), p = RN_h(t*d), t = RN_h(0.5*p)
 *   (the pages name the primitives, not their order or constants; this is
 *   the plain reading).  Each primitive is evaluated in binary64 and rounded
 *   once to h.  For +, -, * and / of h values binary64 holds more than
 *   2p+2 significand bits, so that equals the correctly rounded h result;
 *   exp and erf come from the C library in binary64.
 *
 * Products of two bfloat16 numbers are exact in binary32 inside its normal
 * range (8 + 8 significand bits); outside it the oracle rounds the product
 * to binary32, which is its plain reading of "products accumulate in FP32".
 *
 * RN_h is written here from the IEEE 754 definitions: binary16 (p = 11,
 * emin = -14, emax = 15) and bfloat16 (the upper half of binary32: p = 8,
 * emin = -126, emax = 127), gradual underflow, overflow to infinity, ties
 * to even.
 *
 * Pins (tests/test_oracle_contraction.py): the binary64 roundings against
 * exact rational arithmetic and against the pinned binary32 -> binary16
 * conversion on every binary32 value, hand-worked chains under
 * tests/golden/, closed forms of SiLU and GELU at exact points, the f16
 * head with no steps against the base oracle, and brute force on tiny
 * shapes.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <pthread.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

/* from oracle_linear.c (pinned there) */
float oracle_f16_to_f32(uint16_t h);
uint16_t oracle_f32_to_f16_rn(float v);

enum { ORC_F16 = 0, ORC_BF16 = 1 };
enum { ORC_ADD = 1, ORC_MUL = 2, ORC_SILU = 3, ORC_GELU_TANH = 4, ORC_GELU_ERF = 5 };

/* ---- bfloat16 -> binary32 (exact: bfloat16 is the upper half of binary32) */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float out;
    memcpy(&out, &bits, 4);
    return out;
}

/*
 * Round a binary64 value to the binary format with p significand bits
 * (hidden bit included), minimum normal exponent emin and maximum
 * exponent emax; round to nearest, ties to even; returns the rounded value
 * (infinity on overflow).  The quantum at |v| is 2^(max(floor(log2|v|),
 * emin) - p + 1); dividing by it is an exact power-of-two scaling, and
 * rint() rounds half to even in the default rounding mode.
 */
static double round_to_format(double v, int p, int emin, int emax)
{
    if (v != v || v == 0.0 || isinf(v)) return v;
    int e2;
    frexp(v, &e2);                 /* |v| = f * 2^e2, f in [0.5, 1) */
    int lead = e2 - 1;             /* floor(log2 |v|) */
    int q = (lead < emin ? emin : lead) - (p - 1);
    double n = rint(ldexp(fabs(v), -q));
#if ORACLE_MUTATION == 11
    n = trunc(ldexp(fabs(v), -q));  /* planted mistake: rounding toward zero */
#endif
    double r = ldexp(n, q);
    /* largest finite value: (2 - 2^(1-p)) * 2^emax */
    double maxv = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (r > maxv) r = INFINITY;
    return v < 0 ? -r : r;
}

uint16_t oracle_f64_to_f16_rn(double v)
{
    if (v != v) return 0x7e00u;
    double r = round_to_format(v, 11, -14, 15);
    /* r is a binary16 value, so it is exact in binary32 */
    return oracle_f32_to_f16_rn((float)r);
}

uint16_t oracle_f64_to_bf16_rn(double v)
{
    if (v != v) return 0x7fc0u;
    double r = round_to_format(v, 8, -126, 127);
    float f = (float)r;            /* exact: a bfloat16 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static double hval(uint16_t bits, int dt)
{
    return dt == ORC_BF16 ? (double)oracle_bf16_to_f32(bits) : (double)oracle_f16_to_f32(bits);
}

static uint16_t hround(double v, int dt)
{
    return dt == ORC_BF16 ? oracle_f64_to_bf16_rn(v) : oracle_f64_to_f16_rn(v);
}

/* one primitive: evaluate in binary64, round once to h; returns h bits */
#define RH(expr) hround((expr), dt)
#define V(bits) hval((bits), dt)

/* SiLU as Neg, Exp, Add, Div, each rounded to h */
static uint16_t step_silu(uint16_t t, int dt)
{
    uint16_t a = RH(-V(t));
    uint16_t e = RH(exp(V(a)));
    uint16_t d = RH(1.0 + V(e));
#if ORACLE_MUTATION == 12
    /* planted mistake: the whole activation rounded once */
    return RH(V(t) / (1.0 + exp(-V(t))));
#endif
    return RH(V(t) / V(d));
}

/* GELU, tanh approximation in its sigmoid form */
static uint16_t step_gelu_tanh(uint16_t t, int dt)
{
    const uint16_t c1 = RH(0.044715);
    const uint16_t c2 = RH(2.0 * sqrt(2.0 / acos(-1.0)));
    uint16_t s = RH(V(t) * V(t));
    uint16_t c = RH(V(s) * V(t));
    uint16_t u = RH(V(c1) * V(c));
    uint16_t v = RH(V(t) + V(u));
    uint16_t z = RH(V(c2) * V(v));
    uint16_t a = RH(-V(z));
    uint16_t e = RH(exp(V(a)));
    uint16_t d = RH(1.0 + V(e));
    return RH(V(t) / V(d));
}

/* GELU, erf form */
static uint16_t step_gelu_erf(uint16_t t, int dt)
{
    const uint16_t c3 = RH(1.0 / sqrt(2.0));
    uint16_t s = RH(V(c3) * V(t));
    uint16_t e = RH(erf(V(s)));
    uint16_t d = RH(1.0 + V(e));
    uint16_t p = RH(V(t) * V(d));
#if ORACLE_MUTATION == 13
    /* planted mistake: the factor 0.5 left out */
    return p;
#endif
    return RH(0.5 * V(p));
}

typedef struct {
    int num_steps;
    const int* ops;
    const uint16_t* const* operands;  /* [M, ld] row-major, NULL for activations */
    const int64_t* lds;
} orc_steps;

/* bias and epilogue steps applied to one head value t at (m, n) */
static uint16_t epilogue_value(uint16_t t, const uint16_t* b, int dt, const orc_steps* st,
                               int64_t m, int64_t n)
{
    if (b) t = RH(V(t) + V(b[n]));
    for (int s = 0; s < st->num_steps; ++s) {
        switch (st->ops[s]) {
        case ORC_ADD: t = RH(V(t) + V(st->operands[s][m * st->lds[s] + n])); break;
#if ORACLE_MUTATION == 14
        /* planted mistake: the multiplier read transposed */
        case ORC_MUL: t = RH(V(t) * V(st->operands[s][n * st->lds[s] + m])); break;
#else
        case ORC_MUL: t = RH(V(t) * V(st->operands[s][m * st->lds[s] + n])); break;
#endif
        case ORC_SILU: t = step_silu(t, dt); break;
        case ORC_GELU_TANH: t = step_gelu_tanh(t, dt); break;
        case ORC_GELU_ERF: t = step_gelu_erf(t, dt); break;
        default: break;
        }
    }
    return t;
}

typedef struct {
    const uint16_t* x; const uint16_t* w; const uint16_t* b;
    const uint16_t* proj_in;   /* epilogue-only mode: head values given */
    int dt, out_f32;
    void* y; uint16_t* proj;
    int64_t M, N, K;
    orc_steps st;
    int64_t m_begin, m_end;
} orc_job;

static void orc_rows(const orc_job* j)
{
    const int dt = j->dt;
    for (int64_t m = j->m_begin; m < j->m_end; ++m) {
        for (int64_t n = 0; n < j->N; ++n) {
            uint16_t t;
            if (j->proj_in) {
                t = j->proj_in[m * j->N + n];
            } else {
                float acc = 0.0f;
                const uint16_t* xr = j->x + m * j->K;
                const uint16_t* wr = j->w + n * j->K;
                for (int64_t k = 0; k < j->K; ++k) {
                    float xv = dt == ORC_BF16 ? oracle_bf16_to_f32(xr[k]) : oracle_f16_to_f32(xr[k]);
                    float wv = dt == ORC_BF16 ? oracle_bf16_to_f32(wr[k]) : oracle_f16_to_f32(wr[k]);
                    float prod = xv * wv;          /* RN32; exact in the normal range */
                    acc = acc + prod;              /* one RN32 per term */
                }
                if (j->out_f32) {
                    float yv = j->b ? acc + (float)hval(j->b[n], dt) : acc;
                    ((float*)j->y)[m * j->N + n] = yv;
                    continue;
                }
#if ORACLE_MUTATION == 15
                /* planted mistake: bfloat16 head rounded as binary16 */
                t = oracle_f64_to_f16_rn((double)acc);
#else
                t = hround((double)acc, dt);
#endif
                if (j->proj) j->proj[m * j->N + n] = t;
            }
            ((uint16_t*)j->y)[m * j->N + n] = epilogue_value(t, j->b, dt, &j->st, m, n);
        }
    }
}

static void* orc_thread(void* arg)
{
    orc_rows((const orc_job*)arg);
    return 0;
}

static int orc_run(orc_job base, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > base.M) nthreads = (int)base.M;
    orc_job jobs[256];
    pthread_t tids[256];
    int64_t per = base.M / nthreads, extra = base.M % nthreads, start = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t cnt = per + (t < extra ? 1 : 0);
        jobs[t] = base;
        jobs[t].m_begin = start;
        jobs[t].m_end = start + cnt;
        start += cnt;
    }
    int launched = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], 0, orc_thread, &jobs[t]) != 0) break;
        launched = t;
    }
    orc_rows(&jobs[0]);
    for (int t = 1; t <= launched; ++t) pthread_join(tids[t], 0);
    for (int t = launched + 1; t < nthreads; ++t) orc_rows(&jobs[t]);
    return 0;
}

static int steps_ok(int num_steps, const int* ops, const uint16_t* const* operands, const int64_t* lds,
                    int64_t N)
{
    if (num_steps < 0 || num_steps > 8) return 0;
    for (int s = 0; s < num_steps; ++s) {
        if (ops[s] < ORC_ADD || ops[s] > ORC_GELU_ERF) return 0;
        if ((ops[s] == ORC_ADD || ops[s] == ORC_MUL) && (!operands[s] || lds[s] < N)) return 0;
    }
    return 1;
}

/*
 * x [M,K], w [N,K] (read in place), b [N] or NULL, all in the head dtype
 * (0 binary16, 1 bfloat16) as bit patterns; y [M,N] of binary32 values when
 * out_f32 (no steps then), else head-dtype bits.  proj (optional) receives
 * RN_h of the sum.  Step s: ops[s] with operand s ([M, lds[s]] row-major
 * head-dtype bits) for ADD and MUL.  Rows are split over nthreads; each
 * element is computed by one thread in a fixed order.  Returns 0, or -1 on
 * bad arguments.
 */
int oracle_contraction(const uint16_t* x, const uint16_t* w, const uint16_t* b, int dtype, int out_f32,
                       void* y, uint16_t* proj, int64_t M, int64_t N, int64_t K,
                       int num_steps, const int* ops, const uint16_t* const* operands, const int64_t* lds,
                       int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || (dtype != ORC_F16 && dtype != ORC_BF16)) return -1;
    if (M == 0 || N == 0) return 0;
    if (!y || (K > 0 && (!x || !w))) return -1;
    if (out_f32 && num_steps != 0) return -1;
    if (!steps_ok(num_steps, ops, operands, lds, N)) return -1;
    orc_job base = {x, w, b, 0, dtype, out_f32 ? 1 : 0, y, proj, M, N, K,
                    {num_steps, ops, operands, lds}, 0, 0};
    return orc_run(base, nthreads);
}

/*
 * The head part alone: y = steps(RN_h(t + b[n])) for given head values t
 * [M,N] (used to bound how a difference in the head value propagates).
 */
int oracle_epilogue(const uint16_t* t, const uint16_t* b, int dtype, uint16_t* y, int64_t M, int64_t N,
                    int num_steps, const int* ops, const uint16_t* const* operands, const int64_t* lds,
                    int nthreads)
{
    if (M < 0 || N < 0 || (dtype != ORC_F16 && dtype != ORC_BF16)) return -1;
    if (M == 0 || N == 0) return 0;
    if (!t || !y || !steps_ok(num_steps, ops, operands, lds, N)) return -1;
    orc_job base = {0, 0, b, t, dtype, 0, y, 0, M, N, 0, {num_steps, ops, operands, lds}, 0, 0};
    return orc_run(base, nthreads);
}

void oracle_f64_to_f16_rn_array(const double* in, uint16_t* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_f64_to_f16_rn(in[i]);
}

void oracle_f64_to_bf16_rn_array(const double* in, uint16_t* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_f64_to_bf16_rn(in[i]);
}

void oracle_bf16_to_f32_array(const uint16_t* in, float* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_bf16_to_f32(in[i]);
}
