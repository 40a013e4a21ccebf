/*
 * CPU oracle for y = FP16(x . W^T) + b  --  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  The product path (the CUDA library and its
 * Python binding) never calls it and shares no code with it.
 *
 * What it computes, and where it comes from ("Tensor Programs, Part 1",
 * section "One Program and One Numerical Contract", the proj formula, the
 * two-rule contract and the Figure 1.1 caption):
 *
 *   for every output row m and output feature n
 *       acc  = +0.0 in binary32
 *       for k = 0 .. K-1 (ascending):  acc = RN32(acc + x[m,k] * W[n,k])
 *       proj = RN16(acc)                     rounding BEFORE the bias
 *       y    = RN16(proj + b[n])             bias broadcast over rows
 *
 * The product of two binary16 numbers is exact in binary32 (11 + 11
 * significand bits, exponents from 2^-48 to 2^32), so one binary32 rounding
 * per addition is the only rounding inside the sum (rule 1: FP32
 * accumulation, no per-product FP16 rounding).  The pages allow any
 * summation order; this oracle fixes ascending k, which is one legal order.
 * The bias add is done in binary32 and rounded once to binary16; that is
 * the Inductor capture's widen-add-narrow sequence, and it equals a direct
 * binary16 add (the MAX capture) because binary32 has more than 2*11+2
 * significand bits, which makes the double rounding innocuous.
 *
 * RN16 is written here from the IEEE 754 definition of binary16
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits, gradual
 * underflow to 2^-24, overflow to infinity, round to nearest with ties to
 * even).  Nothing here depends on a compiler's half-precision type.
 *
 * Pins (tests/): exhaustive comparison of both conversions with independent
 * implementations, the worked examples under tests/golden/, brute force
 * against exact rational arithmetic on tiny shapes, the Higham error
 * interval on random data, and the identity / permutation / symmetry
 * invariants.  Every function below is pinned by at least one of those.
 *
 * Mutation switches (ORACLE_MUTATION, compiled in only by the test that
 * checks the pins have teeth) plant one plausible mistake each.
 */
#include <stdint.h>
#include <string.h>
#include <pthread.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

/* ---- binary16 -> binary32 (exact: every binary16 value is a binary32). */
float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t f = h & 0x3ffu;
    uint32_t bits;
    if (e == 0) {
        /* zero or subnormal: value = f * 2^-24.  Normalise f into a
           binary32 normal number (2^-24 .. 2^-15 are all binary32 normals). */
        if (f == 0) {
            bits = sign;
        } else {
            int shift = 0;
            while ((f & 0x400u) == 0) { f <<= 1; ++shift; }
            f &= 0x3ffu;
            /* value = 1.f * 2^(-14 - shift) */
            uint32_t e32 = (uint32_t)(127 - 14 - shift);
            bits = sign | (e32 << 23) | (f << 13);
        }
    } else if (e == 31) {
        /* infinity or NaN; the NaN payload moves to the top fraction bits */
        bits = sign | 0x7f800000u | (f << 13);
    } else {
        bits = sign | ((e - 15u + 127u) << 23) | (f << 13);
    }
    float out;
    memcpy(&out, &bits, 4);
    return out;
}

/* ---- binary32 -> binary16, round to nearest, ties to even. */
uint16_t oracle_f32_to_f16_rn(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t e = (u >> 23) & 0xffu;
    uint32_t m = u & 0x7fffffu;

    if (e == 255) {
        if (m == 0) return (uint16_t)(sign | 0x7c00u);          /* infinity */
        /* NaN: keep it a NaN (quiet bit set), keep the top payload bits */
        return (uint16_t)(sign | 0x7e00u | (m >> 13));
    }
    /* |v| = sig * 2^ex with an integer significand sig < 2^24 */
    uint64_t sig;
    int ex;
    if (e == 0) { sig = m; ex = -149; }
    else        { sig = m | 0x800000u; ex = (int)e - 150; }
    if (sig == 0) return sign;                                   /* +-0 */

    /* p = floor(log2|v|) */
    int bitlen = 0;
    for (uint64_t t = sig; t; t >>= 1) ++bitlen;
    int p = ex + bitlen - 1;

    /* quantum (weight of the last fraction bit) of binary16 at |v| */
    int q = (p < -14) ? -24 : p - 10;

    /* n = round_half_even(|v| / 2^q) */
    int shift = q - ex;
    uint64_t n;
    if (shift <= 0) {
        n = sig << (-shift);              /* exact, no rounding needed */
    } else if (shift >= 60) {
        n = 0;                            /* far below half a quantum */
    } else {
        n = sig >> shift;
        uint64_t rem = sig & ((1ull << shift) - 1ull);
        uint64_t half = 1ull << (shift - 1);
        if (rem > half || (rem == half && (n & 1ull))) ++n;
    }

    if (q == -24) {
        /* subnormal range: encoding is n itself; n == 1024 is exactly the
           smallest normal number 2^-14, whose encoding is also 0x400 */
        return (uint16_t)(sign | (uint16_t)n);
    }
    if (n == 2048) { n = 1024; ++q; }     /* rounding carried into the exponent */
    int biased = q + 10 + 15;
    if (biased >= 31) return (uint16_t)(sign | 0x7c00u);         /* overflow */
    return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)(n - 1024));
}

void oracle_f16_to_f32_array(const uint16_t* in, float* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_f16_to_f32(in[i]);
}

void oracle_f32_to_f16_rn_array(const float* in, uint16_t* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_f32_to_f16_rn(in[i]);
}

/* ---- the linear op ------------------------------------------------------ */

typedef struct {
    const uint16_t* x; const uint16_t* w; const uint16_t* b;
    uint16_t* y; uint16_t* proj;
    int64_t M, N, K;
    int64_t m_begin, m_end;
} oracle_job;

static void oracle_rows(const oracle_job* j)
{
    for (int64_t m = j->m_begin; m < j->m_end; ++m) {
        const uint16_t* xr = j->x + m * j->K;
        for (int64_t n = 0; n < j->N; ++n) {
#if ORACLE_MUTATION == 2
            /* planted mistake: W read as [K, N] (transposed operand) */
            const uint16_t* wr = j->w + n;
#else
            const uint16_t* wr = j->w + n * j->K;
#endif
            float acc = 0.0f;
#if ORACLE_MUTATION == 3
            /* planted mistake: the last term of the sum is dropped */
            int64_t kend = j->K > 0 ? j->K - 1 : 0;
#else
            int64_t kend = j->K;
#endif
            for (int64_t k = 0; k < kend; ++k) {
#if ORACLE_MUTATION == 2
                float wv = oracle_f16_to_f32(wr[k * j->N]);
#else
                float wv = oracle_f16_to_f32(wr[k]);
#endif
                float prod = oracle_f16_to_f32(xr[k]) * wv;     /* exact */
#if ORACLE_MUTATION == 4
                /* planted mistake: each product rounded to binary16 */
                prod = oracle_f16_to_f32(oracle_f32_to_f16_rn(prod));
#endif
                acc = acc + prod;                               /* one RN32 */
#if ORACLE_MUTATION == 5
                /* planted mistake: binary16 accumulator */
                acc = oracle_f16_to_f32(oracle_f32_to_f16_rn(acc));
#endif
            }
            uint16_t p = oracle_f32_to_f16_rn(acc);             /* rule 2 */
#if ORACLE_MUTATION == 1
            /* planted mistake: bias added before the projection rounding */
            uint16_t yv = oracle_f32_to_f16_rn(acc + oracle_f16_to_f32(j->b[n]));
#elif ORACLE_MUTATION == 6
            /* planted mistake: bias indexed by the row instead of the column */
            uint16_t yv = oracle_f32_to_f16_rn(oracle_f16_to_f32(p) +
                                               oracle_f16_to_f32(j->b[m % j->N]));
#elif ORACLE_MUTATION == 7
            /* planted mistake: bias subtracted */
            uint16_t yv = oracle_f32_to_f16_rn(oracle_f16_to_f32(p) -
                                               oracle_f16_to_f32(j->b[n]));
#else
            uint16_t yv = oracle_f32_to_f16_rn(oracle_f16_to_f32(p) +
                                               oracle_f16_to_f32(j->b[n]));
#endif
            j->y[m * j->N + n] = yv;
            if (j->proj) j->proj[m * j->N + n] = p;
        }
    }
}

static void* oracle_thread(void* arg)
{
    oracle_rows((const oracle_job*)arg);
    return 0;
}

/*
 * x [M,K], w [N,K] (out_features x in_features, read in place: the
 * transpose is never formed), b [N], y [M,N]; all row-major binary16 bit
 * patterns.  proj (optional, may be NULL) receives RN16 of the sum.
 * Rows are split over nthreads threads; each element is computed by one
 * thread in a fixed order, so the result does not depend on nthreads.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_linear_f16(const uint16_t* x, const uint16_t* w, const uint16_t* b,
                      uint16_t* y, uint16_t* proj,
                      int64_t M, int64_t N, int64_t K, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (!y || !b || (K > 0 && (!x || !w))) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > M) nthreads = (int)M;

    oracle_job jobs[256];
    pthread_t tids[256];
    int64_t per = M / nthreads, extra = M % nthreads, start = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t cnt = per + (t < extra ? 1 : 0);
        jobs[t] = (oracle_job){x, w, b, y, proj, M, N, K, start, start + cnt};
        start += cnt;
    }
    int launched = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], 0, oracle_thread, &jobs[t]) != 0) break;
        launched = t;
    }
    oracle_rows(&jobs[0]);
    for (int t = 1; t <= launched; ++t) pthread_join(tids[t], 0);
    /* rows of threads that could not be started are done here */
    for (int t = launched + 1; t < nthreads; ++t) oracle_rows(&jobs[t]);
    return 0;
}
