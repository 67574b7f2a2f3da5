/*
 * CPU oracle for the routed-token grouped GEMM and its routing-probability
 * gradient.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product library never does.
 * It shares no code, header or table with the CUDA path.
 *
 * What it computes, plainly and slowly, in binary64 with a fixed ascending
 * summation order (compiled with -ffp-contract=off, no BLAS):
 *
 *   Y[r,n]   = sum_{c=0..K-1} X[r,c] * W[e(r),n,c]           grouped GEMM
 *   Yb[r,n]  = bf16_rne(Y[r,n])                             stored output
 *   P[s,r]   = sum_{n in slot s} G[t(r),n] * Yb[r,n]        private slot partial
 *   D[r]     = sum_{n=0..N-1} G[t(r),n] * Yb[r,n]           dprob of row r
 *   dW[e,n,c] = sum_{r in expert e} dY[r,n] * X[r,c]        weight gradient
 *
 * where e(r) is the expert whose row range [off[e], off[e+1]) holds r, and
 * t(r) = row_src[r] / topk is the token the permuted row came from.
 *
 * Sources: "Trillion-Parameter Pretraining Goes Bitwise-Deterministic: NVIDIA
 * Cuts the Determinism Tax to About 2%", section "Interpretation" (the
 * grouped-GEMM epilogue writes dprob[token] from several N-tiles; each N-tile
 * gets a private slot, slots are combined in a fixed order); "NVIDIA fait
 * passer le déterminisme bit à bit de Megatron Core à 2432 GPU ...", section
 * "Optimisation pour le Nemotron à mille milliards de paramètres" (private
 * output slots for the grouped-GEMM writers, fixed reduction order).  dprob is
 * the derivative of sum_{t,j} prob[t,j] * <expert_out[t,j], grad_out[t]> with
 * respect to prob, i.e. the dot product of the stored expert output row with
 * the token's output gradient.
 *
 * Parallelism: OpenMP over independent requested rows only, so the thread
 * count cannot change a single bit of the result.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32 pattern. */
static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a binary64 value to bfloat16 (1 sign, 8 exponent, 7 fraction bits;
 * emin = -126, subnormal quantum 2^-133, largest finite (2 - 2^-7) * 2^127)
 * with round-to-nearest, ties-to-even, straight from the IEEE 754 rule: scale
 * the value by its quantum so that representable values become integers,
 * round that to the nearest integer (even on a tie), scale back.  Overflow
 * gives an infinity of the value's sign; NaN gives the quiet NaN 0x7FC0 with
 * the input's sign.  Returns the 16-bit pattern.
 */
uint16_t oracle_bf16_rne(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);              /* a in [2^(e-1), 2^e) */
    int qexp = e - 8;                /* 8 significant bits for normal values */
    if (e - 1 < -126)
        qexp = -133;                 /* subnormal range: fixed quantum */
    double n = ldexp(a, -qexp);      /* exact: scaling by a power of two */
    double fl = floor(n);
    double frac = n - fl;            /* exact */
    double r;
    if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = ldexp(r, qexp);
    const double maxfin = ldexp(255.0, 120);   /* (2 - 2^-7) * 2^127 */
    if (v > maxfin)
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;              /* exact: v is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFFu));
}

void oracle_bf16_rne_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_rne(x[i]);
}

/* Expert owning permuted row r: the e with off[e] <= r < off[e+1].  When
 * several experts are empty the first non-empty one that contains r wins,
 * which is the only one whose range is non-empty. */
static int expert_of_row(const int32_t* off, int E, int64_t r)
{
    for (int e = 0; e < E; ++e)
        if (off[e] <= r && r < off[e + 1])
            return e;
    return -1;
}

/*
 * For each requested permuted row rows[i] (i < nrows) compute
 *   Y[i, n]   (binary64, may be NULL)
 *   Yb[i, n]  (bf16 bits, may be NULL)
 *   P[i, s]   (binary64 slot partials over columns [s*slot_width, ...), may be NULL)
 *   D[i]      (binary64 full dot, may be NULL)
 * X: [R,K] bf16 bits, W: [E,N,K] bf16 bits, G: [T,N] bf16 bits,
 * off: [E+1], row_src: [R] flat routing index t*topk + j.
 * G / row_src may be NULL when P and D are NULL.
 * Returns 0, or -1 if a requested row is not covered by any expert.
 */
int oracle_expert_rows(const uint16_t* X, const uint16_t* W, const uint16_t* G,
                       const int32_t* off, const int32_t* row_src,
                       int64_t R, int E, int K, int N, int topk,
                       const int64_t* rows, int64_t nrows, int slot_width,
                       double* Y, uint16_t* Yb, double* P, double* D)
{
    int bad = 0;
    int S = (N + slot_width - 1) / slot_width;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        int e = (r >= 0 && r < R) ? expert_of_row(off, E, r) : -1;
        if (e < 0) {
            bad |= 1;
            continue;
        }
        const uint16_t* x = X + r * (int64_t)K;
        const uint16_t* w = W + (int64_t)e * N * K;
        const uint16_t* g = NULL;
        if (G)
            g = G + (int64_t)(row_src[r] / topk) * N;
        double dsum = 0.0;
        for (int s = 0; s < S; ++s) {
            double psum = 0.0;
            int n_end = (s + 1) * slot_width < N ? (s + 1) * slot_width : N;
            for (int n = s * slot_width; n < n_end; ++n) {
                const uint16_t* wn = w + (int64_t)n * K;
                double y = 0.0;
                for (int c = 0; c < K; ++c)
                    y += bf16_value(x[c]) * bf16_value(wn[c]);
                uint16_t yb = oracle_bf16_rne(y);
                if (Y)
                    Y[i * N + n] = y;
                if (Yb)
                    Yb[i * N + n] = yb;
                if (g) {
                    double term = bf16_value(g[n]) * bf16_value(yb);
                    psum += term;
                    dsum += term;   /* columns visited in ascending n */
                }
            }
            if (P)
                P[i * S + s] = psum;
        }
        if (D && g)
            D[i] = dsum;
    }
    return bad ? -1 : 0;
}

/*
 * dprob of already-stored bf16 expert outputs (the unfused epilogue's input):
 * for each requested row, P[i, s] and D[i] from Yb = expert_out[r, :] directly.
 */
void oracle_dprob_from_output(const uint16_t* G, const uint16_t* expert_out,
                              const int32_t* row_src, int64_t R, int N, int topk,
                              const int64_t* rows, int64_t nrows, int slot_width,
                              double* P, double* D)
{
    int S = (N + slot_width - 1) / slot_width;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows[i];
        const uint16_t* y = expert_out + r * (int64_t)N;
        const uint16_t* g = G + (int64_t)(row_src[r] / topk) * N;
        for (int s = 0; s < S; ++s) {
            double psum = 0.0;
            int n_end = (s + 1) * slot_width < N ? (s + 1) * slot_width : N;
            for (int n = s * slot_width; n < n_end; ++n)
                psum += bf16_value(g[n]) * bf16_value(y[n]);
            if (P)
                P[i * S + s] = psum;
        }
        if (D) {
            double d = 0.0;
            for (int n = 0; n < N; ++n)
                d += bf16_value(g[n]) * bf16_value(y[n]);
            D[i] = d;
        }
    }
}

/*
 * Weight gradient of the grouped GEMM (the FFN-out projection's wgrad): for
 * each requested entry (e, n, c) = ent[3i], ent[3i+1], ent[3i+2],
 *   dW[e, n, c] = sum_{r = off[e]} ^ {off[e+1]-1} dY[r, n] * X[r, c]
 * in binary64, rows ascending; an expert without rows gives 0.
 * X: [R,K] bf16 bits (the GEMM's input rows), dY: [R,N] bf16 bits (gradient
 * at expert_out), off: [E+1].
 */
void oracle_wgrad_entries(const uint16_t* X, const uint16_t* dY, const int32_t* off, int E, int K, int N,
                          const int64_t* ent, int64_t nent, double* out)
{
    (void)E;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < nent; ++i) {
        int64_t e = ent[3 * i], n = ent[3 * i + 1], c = ent[3 * i + 2];
        double acc = 0.0;
        for (int64_t r = off[e]; r < off[e + 1]; ++r)
            acc += bf16_value(dY[r * (int64_t)N + n]) * bf16_value(X[r * (int64_t)K + c]);
        out[i] = acc;
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
