/*
 * oracle.c -- plain, slow, fp64 CPU reference for the three stencil ops.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or run this code.  The
 * CUDA library never links, calls or shares code with it.
 *
 * Every function is the textbook definition written out, with no blocking,
 * fusion or reordering:
 *
 *  - ora_convt_planes: transposed convolution in SCATTER form.  Each input
 *    element x[n,ci,i] adds x*w[ci,co,k] to the output at o = i*s - p + k*d,
 *    per spatial dim, and is dropped when o falls outside [0, L_out).  Bias is
 *    added last.  Kimi-K2.6__l2_p50 states this input-to-output mapping where it
 *    derives which outputs each input element reaches; Kimi-K2.6__l1_p74 states
 *    the same mapping with the dilation factor on k (an input at i reaches
 *    i, i+d, ..., i+(K-1)d) and checks it on small worked examples.
 *  - ora_avgpool_planes: average pool, zero padding, divisor = kD*kH*kW when
 *    count_include_pad (Kimi-K2.6__l1_p46 fixes the divisor at 27 for the
 *    k3/s2/p1 pool), else the number of in-range taps.
 *  - ora_ct3d_scale_pool_bias_planes: the l2_p50 model in its literal order:
 *    t = convT(x)+conv_bias; t *= scale1; t = AvgPool3d(pool_k) (stride pool_k,
 *    no padding, floor mode); t += bias[co]; t *= scale2.
 *
 * Output sizes: transposed conv (L-1)*s - 2p + d*(k-1) + op + 1; pooling
 * floor((L + 2p - k)/s) + 1 (ceil mode: ceil(...) + 1, minus one when the last
 * window would start beyond L + p).
 *
 * Inputs are the fp32 arrays the GPU path also receives; every product and sum
 * is formed in double.  Work is split over output planes (n, c) with OpenMP;
 * the arithmetic order inside a plane does not depend on the thread count.
 * Build with -ffp-contract=off so x86 and Arm hosts give identical results.
 *
 * Return value of every entry point: 0 on success, -1 on a bad argument.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int ora_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ora_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int64_t ora_convt_len(int64_t L, int k, int s, int p, int d, int op)
{
    return (L - 1) * s - 2 * (int64_t)p + (int64_t)d * (k - 1) + op + 1;
}

int64_t ora_pool_len(int64_t L, int k, int s, int p, int ceil_mode)
{
    int64_t span = L + 2 * (int64_t)p - k;
    if (span < 0) return 0;
    int64_t n;
    if (ceil_mode) {
        n = (span + s - 1) / s + 1;
        if ((n - 1) * s >= L + p) n -= 1;
    } else {
        n = span / s + 1;
    }
    return n;
}

/* One (n, co) plane of the transposed convolution, scatter form, into a
 * zero-initialised double buffer of O[0]*O[1]*O[2] elements. */
static void convt_plane(const float *x, const int64_t in[5], const float *w,
                        const float *b, int64_t cout, const int k[3],
                        const int s[3], const int p[3], const int d[3],
                        const int64_t O[3], int64_t n, int64_t co, double *t)
{
    const int64_t cin = in[1], L0 = in[2], L1 = in[3], L2 = in[4];
    const int64_t osz = O[0] * O[1] * O[2];
    memset(t, 0, (size_t)osz * sizeof(double));
    for (int64_t ci = 0; ci < cin; ++ci) {
        const float *xp = x + ((n * cin + ci) * L0) * L1 * L2;
        const float *wp = w + (ci * cout + co) * (int64_t)k[0] * k[1] * k[2];
        for (int64_t i0 = 0; i0 < L0; ++i0)
        for (int64_t i1 = 0; i1 < L1; ++i1)
        for (int64_t i2 = 0; i2 < L2; ++i2) {
            const double xv = (double)xp[(i0 * L1 + i1) * L2 + i2];
            for (int k0 = 0; k0 < k[0]; ++k0) {
                const int64_t o0 = i0 * s[0] - p[0] + (int64_t)k0 * d[0];
                if (o0 < 0 || o0 >= O[0]) continue;
                for (int k1 = 0; k1 < k[1]; ++k1) {
                    const int64_t o1 = i1 * s[1] - p[1] + (int64_t)k1 * d[1];
                    if (o1 < 0 || o1 >= O[1]) continue;
                    for (int k2 = 0; k2 < k[2]; ++k2) {
                        const int64_t o2 = i2 * s[2] - p[2] + (int64_t)k2 * d[2];
                        if (o2 < 0 || o2 >= O[2]) continue;
                        const double wv = (double)wp[(k0 * k[1] + k1) * k[2] + k2];
                        t[(o0 * O[1] + o1) * O[2] + o2] += xv * wv;
                    }
                }
            }
        }
    }
    if (b) {
        const double bv = (double)b[co];
        for (int64_t j = 0; j < osz; ++j) t[j] += bv;
    }
}

static int bad_conv_args(const int64_t in[5], int64_t cout, const int k[3],
                         const int s[3], const int p[3], const int d[3],
                         const int op[3])
{
    for (int i = 0; i < 5; ++i) if (in[i] < 0) return 1;
    if (cout <= 0) return 1;
    for (int i = 0; i < 3; ++i)
        if (k[i] < 1 || s[i] < 1 || p[i] < 0 || d[i] < 1 || op[i] < 0) return 1;
    return 0;
}

/* Transposed convolution over up to three spatial dims (pass 1 for unused
 * leading dims).  x: [N, Cin, L0, L1, L2]; w: [Cin, Cout, k0, k1, k2]; b: [Cout]
 * or NULL.  sel holds nsel (n, co) pairs; y receives those planes compactly,
 * [nsel][O0][O1][O2].  sel == NULL means every plane in (n, co) order. */
int ora_convt_planes(const float *x, const int64_t in[5], const float *w,
                     const float *b, int64_t cout, const int k[3], const int s[3],
                     const int p[3], const int d[3], const int op[3],
                     const int64_t *sel, int64_t nsel, double *y)
{
    if (!x || !w || !y || bad_conv_args(in, cout, k, s, p, d, op)) return -1;
    int64_t O[3];
    for (int i = 0; i < 3; ++i) {
        O[i] = ora_convt_len(in[2 + i], k[i], s[i], p[i], d[i], op[i]);
        if (O[i] <= 0) return -1;
    }
    const int64_t osz = O[0] * O[1] * O[2];
    const int64_t nplanes = sel ? nsel : in[0] * cout;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < nplanes; ++j) {
        const int64_t n = sel ? sel[2 * j] : j / cout;
        const int64_t co = sel ? sel[2 * j + 1] : j % cout;
        if (n < 0 || n >= in[0] || co < 0 || co >= cout) { err = 1; continue; }
        convt_plane(x, in, w, b, cout, k, s, p, d, O, n, co, y + j * osz);
    }
    return err ? -1 : 0;
}

/* Average pool of one plane t (dims T[3], double) into out (dims P[3]). */
static void avgpool_plane(const double *t, const int64_t T[3], const int k[3],
                          const int s[3], const int p[3], int count_include_pad,
                          const int64_t P[3], double *out)
{
    for (int64_t a = 0; a < P[0]; ++a)
    for (int64_t b = 0; b < P[1]; ++b)
    for (int64_t c = 0; c < P[2]; ++c) {
        const int64_t st[3] = {a * s[0] - p[0], b * s[1] - p[1], c * s[2] - p[2]};
        double sum = 0.0;
        int64_t inside = 0;
        int64_t padded = 1;
        for (int i = 0; i < 3; ++i) {
            int64_t end = st[i] + k[i];
            if (end > T[i] + p[i]) end = T[i] + p[i];
            padded *= end - st[i];
        }
        for (int64_t u = st[0]; u < st[0] + k[0]; ++u)
        for (int64_t v = st[1]; v < st[1] + k[1]; ++v)
        for (int64_t q = st[2]; q < st[2] + k[2]; ++q) {
            if (u < 0 || u >= T[0] || v < 0 || v >= T[1] || q < 0 || q >= T[2]) continue;
            sum += t[(u * T[1] + v) * T[2] + q];
            ++inside;
        }
        const int64_t div = count_include_pad ? padded : inside;
        out[(a * P[1] + b) * P[2] + c] = div > 0 ? sum / (double)div : 0.0;
    }
}

/* AvgPool3d on x [N, C, D, H, W].  sel: nsel (n, c) pairs or NULL for all. */
int ora_avgpool_planes(const float *x, const int64_t in[5], const int k[3],
                       const int s[3], const int p[3], int count_include_pad,
                       int ceil_mode, const int64_t *sel, int64_t nsel, double *y)
{
    if (!x || !y) return -1;
    for (int i = 0; i < 5; ++i) if (in[i] < 0) return -1;
    for (int i = 0; i < 3; ++i)
        if (k[i] < 1 || s[i] < 1 || p[i] < 0 || 2 * p[i] > k[i]) return -1;
    const int64_t T[3] = {in[2], in[3], in[4]};
    int64_t P[3];
    for (int i = 0; i < 3; ++i) {
        P[i] = ora_pool_len(T[i], k[i], s[i], p[i], ceil_mode);
        if (P[i] <= 0) return -1;
    }
    const int64_t isz = T[0] * T[1] * T[2], osz = P[0] * P[1] * P[2];
    const int64_t nplanes = sel ? nsel : in[0] * in[1];
    int err = 0;
#pragma omp parallel
    {
        double *t = (double *)malloc((size_t)(isz > 0 ? isz : 1) * sizeof(double));
        if (!t) err = 1;
#pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < nplanes; ++j) {
            if (!t) continue;
            const int64_t n = sel ? sel[2 * j] : j / in[1];
            const int64_t c = sel ? sel[2 * j + 1] : j % in[1];
            if (n < 0 || n >= in[0] || c < 0 || c >= in[1]) { err = 1; continue; }
            const float *xp = x + (n * in[1] + c) * isz;
            for (int64_t q = 0; q < isz; ++q) t[q] = (double)xp[q];
            avgpool_plane(t, T, k, s, p, count_include_pad, P, y + j * osz);
        }
        free(t);
    }
    return err ? -1 : 0;
}

/* The l2_p50 chain: convT(+conv_bias) -> *scale1 -> AvgPool3d(pool_k) -> +bias
 * -> *scale2, one (n, co) plane at a time.  conv_bias may be NULL. */
int ora_ct3d_scale_pool_bias_planes(const float *x, const int64_t in[5],
                                    const float *w, const float *conv_bias,
                                    const float *bias, int64_t cout,
                                    const int k[3], const int s[3], const int p[3],
                                    const int d[3], const int op[3], int pool_k,
                                    double scale1, double scale2,
                                    const int64_t *sel, int64_t nsel, double *y)
{
    if (!x || !w || !bias || !y || pool_k < 1 ||
        bad_conv_args(in, cout, k, s, p, d, op)) return -1;
    int64_t O[3], P[3];
    for (int i = 0; i < 3; ++i) {
        O[i] = ora_convt_len(in[2 + i], k[i], s[i], p[i], d[i], op[i]);
        if (O[i] <= 0) return -1;
        P[i] = ora_pool_len(O[i], pool_k, pool_k, 0, 0);
        if (P[i] <= 0) return -1;
    }
    const int pk[3] = {pool_k, pool_k, pool_k}, pz[3] = {0, 0, 0};
    const int64_t tsz = O[0] * O[1] * O[2], osz = P[0] * P[1] * P[2];
    const int64_t nplanes = sel ? nsel : in[0] * cout;
    int err = 0;
#pragma omp parallel
    {
        double *t = (double *)malloc((size_t)tsz * sizeof(double));
        if (!t) err = 1;
#pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < nplanes; ++j) {
            if (!t) continue;
            const int64_t n = sel ? sel[2 * j] : j / cout;
            const int64_t co = sel ? sel[2 * j + 1] : j % cout;
            if (n < 0 || n >= in[0] || co < 0 || co >= cout) { err = 1; continue; }
            convt_plane(x, in, w, conv_bias, cout, k, s, p, d, O, n, co, t);
            for (int64_t q = 0; q < tsz; ++q) t[q] *= scale1;
            double *out = y + j * osz;
            avgpool_plane(t, O, pk, pk, pz, 1, P, out);
            const double bv = (double)bias[co];
            for (int64_t q = 0; q < osz; ++q) out[q] = (out[q] + bv) * scale2;
        }
        free(t);
    }
    return err ? -1 : 0;
}
