/*
 * Oracle for the causal long convolution: plain, slow, double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this code.  The product
 * (the CUDA library and its Python binding) never calls it, and it shares no
 * code, header, table or constant with the product.
 *
 * What it computes (FlashFFTConv page, section 3.4 "The FFT Convolution and
 * Its Hardware Mismatch"):
 *   - the convolution  (u * k)[i] = sum_j u[j] k[i - j]  over the indices
 *     where both are defined, restricted to the causal outputs i = 0..N-1;
 *   - the same result through the convolution theorem
 *     u * k = F^-1(F u . F k), with u and k zero-padded to length 2N so the
 *     circular convolution equals the linear one on the kept outputs;
 *   - the DFT with element (j, k) = exp(-2 pi i j k / n) (section 3.4,
 *     "The Monarch FFT Decomposition", definition of F_N); the inverse uses
 *     exp(+2 pi i j k / n) and divides by n;
 *   - the gated form y = v . ((u . w) * k) (section 3.4, "Gating operation
 *     fusion"), here with v = w_out and w = w_in of the same shape as u.
 *
 * The FFT is the textbook iterative radix-2 Cooley-Tukey transform (bit
 * reversal, then log2(n) butterfly passes); twiddles come from cos/sin of the
 * exact angle at every use.  Nothing is blocked, fused or reordered beyond
 * that definition.
 *
 * Further functions, each with its definition at its head: the causal
 * correlation and the two gradients of the convolution (input and kernel),
 * the partial convolution (kernel cut to T taps), the circular convolution,
 * and the frequency-sparse forms (the masked convolution, its DFT-sum twin
 * and the masked correlation).
 *
 * Pins (tests that run without a GPU): brute-force DFT and direct
 * convolution on small sizes, the delta / shifted-delta kernels, u = delta,
 * constant u (prefix sums), linearity, commutativity, Parseval, single-tone
 * transforms, numpy's FFT as an independent library, and hand-worked
 * fixtures; adjoint identities for the correlations and gradients;
 * windowed and modular brute-force sums for the partial and circular forms;
 * single-bin closed forms and the all-ones weight for the masked forms; and
 * planted mistakes for every group.  No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_PI 3.14159265358979323846264338327950288

/* 1 if n is a power of two (n >= 1). */
static int is_pow2(int64_t n) { return n >= 1 && (n & (n - 1)) == 0; }

/*
 * In-place DFT of length n (a power of two) of the complex vector (re, im).
 * sign = -1: forward transform X[k] = sum_j x[j] exp(-2 pi i j k / n).
 * sign = +1: inverse transform x[j] = (1/n) sum_k X[k] exp(+2 pi i j k / n).
 * Returns 0 on success, -1 if n is not a power of two.
 */
int oracle_fft(double *re, double *im, int64_t n, int sign)
{
    if (!is_pow2(n) || (sign != 1 && sign != -1)) return -1;
    /* bit-reversal permutation */
    for (int64_t i = 1, j = 0; i < n; ++i) {
        int64_t bit = n >> 1;
        for (; j & bit; bit >>= 1) j ^= bit;
        j ^= bit;
        if (i < j) {
            double t = re[i]; re[i] = re[j]; re[j] = t;
            t = im[i]; im[i] = im[j]; im[j] = t;
        }
    }
    /* butterfly passes: combine pairs of length-len/2 transforms; the
     * twiddle exp(sign 2 pi i j / len) is evaluated once per (len, j) */
    for (int64_t len = 2; len <= n; len <<= 1) {
        int64_t half = len >> 1;
        for (int64_t j = 0; j < half; ++j) {
            double ang = sign * 2.0 * ORACLE_PI * (double)j / (double)len;
            double wr = cos(ang), wi = sin(ang);
            for (int64_t start = 0; start < n; start += len) {
                int64_t a = start + j, b = a + half;
                double tr = re[b] * wr - im[b] * wi;
                double ti = re[b] * wi + im[b] * wr;
                re[b] = re[a] - tr; im[b] = im[a] - ti;
                re[a] += tr;        im[a] += ti;
            }
        }
    }
    if (sign == 1) {
        for (int64_t i = 0; i < n; ++i) { re[i] /= (double)n; im[i] /= (double)n; }
    }
    return 0;
}

/*
 * Brute-force DFT, O(n^2), any n >= 1: the definition written out.  Used only
 * to pin oracle_fft on small sizes.
 */
int oracle_dft_direct(const double *re, const double *im, double *out_re,
                      double *out_im, int64_t n, int sign)
{
    if (n < 1 || (sign != 1 && sign != -1)) return -1;
    for (int64_t k = 0; k < n; ++k) {
        double sr = 0.0, si = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            /* reduce j*k mod n first so the angle stays exact for large n */
            int64_t m = (j * k) % n;
            double ang = sign * 2.0 * ORACLE_PI * (double)m / (double)n;
            double c = cos(ang), s = sin(ang);
            sr += re[j] * c - im[j] * s;
            si += re[j] * s + im[j] * c;
        }
        out_re[k] = sign == 1 ? sr / (double)n : sr;
        out_im[k] = sign == 1 ? si / (double)n : si;
    }
    return 0;
}

/*
 * Causal convolution of one row through the convolution theorem:
 * y[t] = sum_{j=0}^{t} u[j] k[t-j], t = 0..N-1, computed as the first N
 * outputs of IDFT_{2N}(DFT_{2N}(u0) . DFT_{2N}(k0)) where u0, k0 are u, k
 * zero-padded to 2N.  N must be a power of two.  Returns 0 or -1.
 */
int oracle_causal_conv(const double *u, const double *k, double *y, int64_t N)
{
    if (!is_pow2(N)) return -1;
    int64_t L = 2 * N;
    double *ur = calloc((size_t)L, sizeof(double)), *ui = calloc((size_t)L, sizeof(double));
    double *kr = calloc((size_t)L, sizeof(double)), *ki = calloc((size_t)L, sizeof(double));
    if (!ur || !ui || !kr || !ki) { free(ur); free(ui); free(kr); free(ki); return -1; }
    memcpy(ur, u, (size_t)N * sizeof(double));
    memcpy(kr, k, (size_t)N * sizeof(double));
    oracle_fft(ur, ui, L, -1);
    oracle_fft(kr, ki, L, -1);
    for (int64_t i = 0; i < L; ++i) {
        double pr = ur[i] * kr[i] - ui[i] * ki[i];
        double pi = ur[i] * ki[i] + ui[i] * kr[i];
        ur[i] = pr; ui[i] = pi;
    }
    oracle_fft(ur, ui, L, 1);
    memcpy(y, ur, (size_t)N * sizeof(double));
    free(ur); free(ui); free(kr); free(ki);
    return 0;
}

/* Gated row: y = w_out . conv(u . w_in, k), all products in double. */
int oracle_causal_conv_gated(const double *u, const double *w_in, const double *w_out,
                             const double *k, double *y, int64_t N)
{
    double *x = malloc((size_t)N * sizeof(double));
    if (!x) return -1;
    for (int64_t i = 0; i < N; ++i) x[i] = u[i] * w_in[i];
    int rc = oracle_causal_conv(x, k, y, N);
    if (rc == 0)
        for (int64_t i = 0; i < N; ++i) y[i] *= w_out[i];
    free(x);
    return rc;
}

/*
 * Batched rows: u, y are [rows][N] with row r = b*H + h using kernel row
 * k[h] = k + h*N (k is [H][N]).  w_in / w_out may be NULL (ungated).
 * Rows [row_begin, row_end) only, so callers can split the work.
 */
int oracle_causal_conv_rows(const double *u, const double *w_in, const double *w_out,
                            const double *k, double *y, int64_t H, int64_t N,
                            int64_t row_begin, int64_t row_end)
{
    for (int64_t r = row_begin; r < row_end; ++r) {
        int64_t h = r % H;
        int rc;
        if (w_in && w_out)
            rc = oracle_causal_conv_gated(u + r * N, w_in + r * N, w_out + r * N,
                                          k + h * N, y + r * N, N);
        else
            rc = oracle_causal_conv(u + r * N, k + h * N, y + r * N, N);
        if (rc) return rc;
    }
    return 0;
}

/*
 * Compensated (Neumaier) sum of u[j] k[t-j] for j = 0..t: one causal output
 * straight from the definition, O(t).  Any N (not only powers of two).
 */
double oracle_direct_causal_conv_at(const double *u, const double *k, int64_t N, int64_t t)
{
    if (t < 0 || t >= N) return NAN;
    double s = 0.0, c = 0.0;
    for (int64_t j = 0; j <= t; ++j) {
        double v = u[j] * k[t - j];
        double nt = s + v;
        if (fabs(s) >= fabs(v)) c += (s - nt) + v;
        else c += (v - nt) + s;
        s = nt;
    }
    return s + c;
}

/* Direct O(N^2) causal convolution of one row (all N outputs). */
int oracle_direct_causal_conv(const double *u, const double *k, double *y, int64_t N)
{
    if (N < 1) return -1;
    for (int64_t t = 0; t < N; ++t) y[t] = oracle_direct_causal_conv_at(u, k, N, t);
    return 0;
}

/*
 * Backward pass (FlashFFTConv page, section 3.4 "Kernel Fusion and
 * Recomputation Strategies", recomputation in the backward pass: gradients
 * of the convolution output with respect to the input u and the kernel k).
 * For y[t] = sum_{j<=t} u[j] k[t-j] and an output gradient dy:
 *   du[j] = sum_{t=j}^{N-1} dy[t] k[t-j]            (correlation of dy with k)
 *   dk[i] = sum_b sum_{t=i}^{N-1} dy_b[t] u_b[t-i]   (correlation of dy with u, summed over the batch)
 * Through the DFT: with zero padding to 2N, sum_t a[t] b[t-i] is the first
 * N outputs of IDFT_{2N}(DFT(a0) . conj(DFT(b0))), because the padded b is
 * zero at the indices t - i + 2N >= N that the circular form adds.
 */
int oracle_causal_corr(const double *a, const double *b, double *out, int64_t N)
{
    if (!is_pow2(N)) return -1;
    const int64_t L2 = 2 * N;
    double *ar = calloc((size_t)L2, sizeof(double)), *ai = calloc((size_t)L2, sizeof(double));
    double *br = calloc((size_t)L2, sizeof(double)), *bi = calloc((size_t)L2, sizeof(double));
    if (!ar || !ai || !br || !bi) { free(ar); free(ai); free(br); free(bi); return -1; }
    memcpy(ar, a, (size_t)N * sizeof(double));
    memcpy(br, b, (size_t)N * sizeof(double));
    oracle_fft(ar, ai, L2, -1);
    oracle_fft(br, bi, L2, -1);
    for (int64_t i = 0; i < L2; ++i) {  /* A . conj(B) */
        double pr = ar[i] * br[i] + ai[i] * bi[i];
        double pi = ai[i] * br[i] - ar[i] * bi[i];
        ar[i] = pr; ai[i] = pi;
    }
    oracle_fft(ar, ai, L2, 1);
    memcpy(out, ar, (size_t)N * sizeof(double));
    free(ar); free(ai); free(br); free(bi);
    return 0;
}

/* One correlation output sum_{t=i}^{N-1} a[t] b[t-i] by the definition (compensated sum). */
double oracle_direct_causal_corr_at(const double *a, const double *b, int64_t N, int64_t i)
{
    if (i < 0 || i >= N) return NAN;
    double s = 0.0, c = 0.0;
    for (int64_t t = i; t < N; ++t) {
        double v = a[t] * b[t - i];
        double nt = s + v;
        if (fabs(s) >= fabs(v)) c += (s - nt) + v;
        else c += (v - nt) + s;
        s = nt;
    }
    return s + c;
}

/*
 * Input gradient of rows [row_begin, row_end) of a [rows][N] batch (row r =
 * b*H + h uses k[h]).  Gated (y = w_out . conv(u . w_in, k)):
 * du = w_in . corr(w_out . dy, k); w_in / w_out NULL for the plain form.
 */
int oracle_input_grad_rows(const double *dy, const double *w_in, const double *w_out,
                           const double *k, double *du, int64_t H, int64_t N,
                           int64_t row_begin, int64_t row_end)
{
    double *g = malloc((size_t)N * sizeof(double));
    if (!g) return -1;
    for (int64_t r = row_begin; r < row_end; ++r) {
        int64_t h = r % H;
        for (int64_t t = 0; t < N; ++t) g[t] = w_out ? dy[r * N + t] * w_out[r * N + t] : dy[r * N + t];
        int rc = oracle_causal_corr(g, k + h * N, du + r * N, N);
        if (rc) { free(g); return rc; }
        if (w_in)
            for (int64_t t = 0; t < N; ++t) du[r * N + t] *= w_in[r * N + t];
    }
    free(g);
    return 0;
}

/*
 * Kernel gradient of channels [h_begin, h_end): dk[h] = sum_b corr(g_b, x_b)
 * with g = w_out . dy and x = u . w_in (plain form: g = dy, x = u).  u, dy,
 * w_in, w_out are [B][H][N]; dk is [H][N].
 */
int oracle_kernel_grad_channels(const double *u, const double *dy, const double *w_in,
                                const double *w_out, double *dk, int64_t B, int64_t H,
                                int64_t N, int64_t h_begin, int64_t h_end)
{
    double *g = malloc((size_t)N * sizeof(double)), *x = malloc((size_t)N * sizeof(double));
    double *c = malloc((size_t)N * sizeof(double));
    if (!g || !x || !c) { free(g); free(x); free(c); return -1; }
    for (int64_t h = h_begin; h < h_end; ++h) {
        for (int64_t i = 0; i < N; ++i) dk[h * N + i] = 0.0;
        for (int64_t b = 0; b < B; ++b) {
            int64_t r = b * H + h;
            for (int64_t t = 0; t < N; ++t) {
                g[t] = w_out ? dy[r * N + t] * w_out[r * N + t] : dy[r * N + t];
                x[t] = w_in ? u[r * N + t] * w_in[r * N + t] : u[r * N + t];
            }
            int rc = oracle_causal_corr(g, x, c, N);
            if (rc) { free(g); free(x); free(c); return rc; }
            for (int64_t i = 0; i < N; ++i) dk[h * N + i] += c[i];
        }
    }
    free(g); free(x); free(c);
    return 0;
}

/*
 * Partial convolution (FlashFFTConv page, "Architectural Extensions: Partial
 * and Frequency-Sparse Convolutions": the kernel is zero beyond its first T
 * taps, so each output only sees the last T inputs):
 *   y[t] = sum_{j = max(0, t-T+1)}^{t} u[j] k[t-j],  t = 0..N-1.
 * Computed as the causal convolution of u with k cut to its first T taps
 * (N a power of two).
 */
int oracle_partial_conv(const double *u, const double *k, double *y, int64_t N, int64_t T)
{
    if (T < 1 || T > N) return -1;
    double *kt = calloc((size_t)N, sizeof(double));
    if (!kt) return -1;
    memcpy(kt, k, (size_t)T * sizeof(double));
    int rc = oracle_causal_conv(u, kt, y, N);
    free(kt);
    return rc;
}

/* One partial-convolution output by the definition (compensated sum), any N. */
double oracle_direct_partial_conv_at(const double *u, const double *k, int64_t N, int64_t T, int64_t t)
{
    if (t < 0 || t >= N || T < 1) return NAN;
    double s = 0.0, c = 0.0;
    int64_t j0 = t - T + 1 > 0 ? t - T + 1 : 0;
    for (int64_t j = j0; j <= t; ++j) {
        double v = u[j] * k[t - j];
        double nt = s + v;
        if (fabs(s) >= fabs(v)) c += (s - nt) + v;
        else c += (v - nt) + s;
        s = nt;
    }
    return s + c;
}

/*
 * Circular (non-causal) convolution of length N (FlashFFTConv page, the
 * convolution theorem without zero padding; the pages' non-causal
 * workloads): y[t] = sum_{j=0}^{N-1} u[j] k[(t - j) mod N], through the
 * N-point DFT: y = IDFT_N(DFT_N(u) . DFT_N(k)).  N a power of two.
 */
int oracle_circular_conv(const double *u, const double *k, double *y, int64_t N)
{
    if (!is_pow2(N)) return -1;
    double *ur = malloc((size_t)N * sizeof(double)), *ui = calloc((size_t)N, sizeof(double));
    double *kr = malloc((size_t)N * sizeof(double)), *ki = calloc((size_t)N, sizeof(double));
    if (!ur || !ui || !kr || !ki) { free(ur); free(ui); free(kr); free(ki); return -1; }
    memcpy(ur, u, (size_t)N * sizeof(double));
    memcpy(kr, k, (size_t)N * sizeof(double));
    oracle_fft(ur, ui, N, -1);
    oracle_fft(kr, ki, N, -1);
    for (int64_t i = 0; i < N; ++i) {
        double cr = ur[i] * kr[i] - ui[i] * ki[i];
        double ci = ur[i] * ki[i] + ui[i] * kr[i];
        ur[i] = cr; ui[i] = ci;
    }
    oracle_fft(ur, ui, N, 1);
    memcpy(y, ur, (size_t)N * sizeof(double));
    free(ur); free(ui); free(kr); free(ki);
    return 0;
}

/*
 * Frequency-sparse causal convolution (FlashFFTConv page, "Architectural
 * Extensions: Partial and Frequency-Sparse Convolutions", the
 * frequency-sparse part): the kernel's spectrum is zeroed on some bins
 * before the product.  mask[f], f = 0..N, weighs bin f of the 2N-point
 * spectrum of the real kernel; bin 2N - f (f = 1..N-1) takes the same
 * weight, so the weighted spectrum keeps the conjugate symmetry of a real
 * signal and the result is real:
 *   y = first N outputs of IDFT_2N( DFT_2N(u0) . DFT_2N(k0) . m ),
 *   m[f] = mask[f] for f <= N, mask[2N - f] for f > N.
 * N a power of two.  Returns 0 or -1.
 */
int oracle_masked_causal_conv(const double *u, const double *k, const double *mask, double *y, int64_t N)
{
    if (!is_pow2(N)) return -1;
    int64_t L2 = 2 * N;
    double *ur = calloc((size_t)L2, sizeof(double)), *ui = calloc((size_t)L2, sizeof(double));
    double *kr = calloc((size_t)L2, sizeof(double)), *ki = calloc((size_t)L2, sizeof(double));
    if (!ur || !ui || !kr || !ki) { free(ur); free(ui); free(kr); free(ki); return -1; }
    memcpy(ur, u, (size_t)N * sizeof(double));
    memcpy(kr, k, (size_t)N * sizeof(double));
    oracle_fft(ur, ui, L2, -1);
    oracle_fft(kr, ki, L2, -1);
    for (int64_t f = 0; f < L2; ++f) {
        double w = f <= N ? mask[f] : mask[L2 - f];
        double pr = (ur[f] * kr[f] - ui[f] * ki[f]) * w;
        double pi = (ur[f] * ki[f] + ui[f] * kr[f]) * w;
        ur[f] = pr; ui[f] = pi;
    }
    oracle_fft(ur, ui, L2, 1);
    memcpy(y, ur, (size_t)N * sizeof(double));
    free(ur); free(ui); free(kr); free(ki);
    return 0;
}

/*
 * The same outputs from the definition of the DFT, with no FFT (brute
 * force, O(N^2), any N >= 1).  Only the bins f = 0..N are formed:
 *   U[f] = sum_n u[n] exp(-i pi f n / N), K[f] likewise, P[f] = mask[f] U[f] K[f];
 * the other half of the spectrum is the conjugate of this one, so the
 * inverse transform of length 2N reads
 *   y[t] = (1 / 2N) (P[0] + (-1)^t P[N] + 2 sum_{f=1}^{N-1} Re(P[f] exp(+i pi f t / N))).
 * Angles are reduced exactly (f n mod 2N) before cos / sin.
 */
int oracle_direct_masked_causal_conv(const double *u, const double *k, const double *mask, double *y, int64_t N)
{
    if (N < 1) return -1;
    int64_t L2 = 2 * N;
    double *pr = malloc((size_t)(N + 1) * sizeof(double)), *pi = malloc((size_t)(N + 1) * sizeof(double));
    if (!pr || !pi) { free(pr); free(pi); return -1; }
    for (int64_t f = 0; f <= N; ++f) {
        double Ur = 0.0, Ui = 0.0, Kr = 0.0, Ki = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double a = ORACLE_PI * (double)((f * n) % L2) / (double)N;
            double c = cos(a), s = sin(a);
            Ur += u[n] * c; Ui -= u[n] * s;
            Kr += k[n] * c; Ki -= k[n] * s;
        }
        pr[f] = (Ur * Kr - Ui * Ki) * mask[f];
        pi[f] = (Ur * Ki + Ui * Kr) * mask[f];
    }
    for (int64_t t = 0; t < N; ++t) {
        double s = pr[0] + ((t & 1) ? -pr[N] : pr[N]);
        for (int64_t f = 1; f < N; ++f) {
            double a = ORACLE_PI * (double)((f * t) % L2) / (double)N;
            s += 2.0 * (pr[f] * cos(a) - pi[f] * sin(a));
        }
        y[t] = s / (double)L2;
    }
    free(pr); free(pi);
    return 0;
}

/*
 * Adjoint in u of the frequency-sparse convolution: the masked causal
 * correlation
 *   out = first N outputs of IDFT_2N( DFT_2N(a0) . conj(DFT_2N(b0)) . m ),
 * m mirrored as in oracle_masked_causal_conv.  With a = dy and b = k it is
 * the input gradient of y = masked causal conv(u, k) (the adjoint of a
 * product with a real, conjugate-symmetric weight is the product with the
 * conjugate spectrum and the same weight).  N a power of two.
 */
int oracle_masked_causal_corr(const double *a, const double *b, const double *mask, double *out, int64_t N)
{
    if (!is_pow2(N)) return -1;
    int64_t L2 = 2 * N;
    double *ar = calloc((size_t)L2, sizeof(double)), *ai = calloc((size_t)L2, sizeof(double));
    double *br = calloc((size_t)L2, sizeof(double)), *bi = calloc((size_t)L2, sizeof(double));
    if (!ar || !ai || !br || !bi) { free(ar); free(ai); free(br); free(bi); return -1; }
    memcpy(ar, a, (size_t)N * sizeof(double));
    memcpy(br, b, (size_t)N * sizeof(double));
    oracle_fft(ar, ai, L2, -1);
    oracle_fft(br, bi, L2, -1);
    for (int64_t f = 0; f < L2; ++f) {
        double wgt = f <= N ? mask[f] : mask[L2 - f];
        double cr = (ar[f] * br[f] + ai[f] * bi[f]) * wgt;
        double ci = (ai[f] * br[f] - ar[f] * bi[f]) * wgt;
        ar[f] = cr; ai[f] = ci;
    }
    oracle_fft(ar, ai, L2, 1);
    memcpy(out, ar, (size_t)N * sizeof(double));
    free(ar); free(ai); free(br); free(bi);
    return 0;
}
