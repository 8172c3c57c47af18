/*
 * CPU oracle for the forward 2-D convolution with unstructured-sparse weights.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plainly written reference
 * that the CUDA path is checked against.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load it; the library never does, and
 * the two share no code, headers, tables or helpers.
 *
 * Everything is computed in fp64 (inputs arrive as fp32 values widened
 * exactly to double).  Definitions followed:
 *
 *  - Tuteja et al., "Theoretical and Empirical Analysis of Sparse Convolution",
 *    Sec. 3 Eq.(1): C[h,w,oc] = sum_ic sum_kh sum_kw X[h+kh-P, w+kw-P, ic] *
 *    W[kh,kw,ic,oc], with the kernel range clipped so X is never indexed
 *    outside [0,H) x [0,W) (i.e. implicit zero padding); no kernel flip.
 *    Generalised to stride s: the input row is e*s + r - pad (Escoin,
 *    "Direct sparse convolution", Algorithm 2 reads in[f(0, y*stride, x*stride)
 *    + offset]).
 *  - Same page, Eq.(2): output extent E = floor((H + 2P - K) / s) + 1.
 *  - Same page, Eq.(3): the sparse form, a sum over the nonzeros of output
 *    channel oc whose shifted input position lies inside the image.
 *  - Escoin (arXiv 1802.10280), "CONV layer" Algorithm 1: the seven-loop
 *    nest over (n, m, e, f, c, r, s) -> oracle_dense7.
 *  - Escoin, "Sparse weights" (CSR: value / colidx / rowptr) and Algorithm 2
 *    (for each image, each output channel, each nonzero of that row, every
 *    output position) -> oracle_csr.  The column index of the M x CRS lowered
 *    filter matrix is read as colidx = (c*R + r)*S + s.
 *
 * Every output also gets abs_sum = sum |w * x| over the same terms, which
 * scales the parity tolerance.
 *
 * Pins (tests/test_oracle_pins.py): lowering identity O = W * I by brute-force
 * im2col, torch CPU conv2d in float64, CSR == dense at every density,
 * linearity, identity / shifted delta filters, single-nonzero enumeration.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

int oracle_out_dim(int in, int k, int stride, int pad)
{
    if (stride < 1 || k < 1 || pad < 0) return -1;
    int num = in + 2 * pad - k;
    if (num < 0) return 0;
    return num / stride + 1;
}

int oracle_num_cpus(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int check_dims(int N, int C, int H, int W, int M, int R, int S, int stride, int pad)
{
    if (N < 0 || C < 1 || H < 1 || W < 1 || M < 1 || R < 1 || S < 1 || stride < 1 || pad < 0)
        return -1;
    return 0;
}

/* Escoin Algorithm 1: seven nested loops over a dense M x C x R x S filter. */
int oracle_dense7(int N, int C, int H, int W, int M, int R, int S, int stride, int pad,
                  const double *x, const double *w, double *y, double *abs_sum)
{
    if (check_dims(N, C, H, W, M, R, S, stride, pad)) return -1;
    const int E = oracle_out_dim(H, R, stride, pad);
    const int F = oracle_out_dim(W, S, stride, pad);
    for (int n = 0; n < N; ++n)
        for (int m = 0; m < M; ++m)
            for (int e = 0; e < E; ++e)
                for (int f = 0; f < F; ++f) {
                    double acc = 0.0, mag = 0.0;
                    for (int c = 0; c < C; ++c)
                        for (int r = 0; r < R; ++r)
                            for (int s = 0; s < S; ++s) {
                                const int h = e * stride + r - pad;
                                const int v = f * stride + s - pad;
                                if (h < 0 || h >= H || v < 0 || v >= W) continue;  /* zero pad */
                                const double p = w[(((size_t)m * C + c) * R + r) * S + s] *
                                                 x[(((size_t)n * C + c) * H + h) * W + v];
                                acc += p;
                                mag += fabs(p);
                            }
                    const size_t o = (((size_t)n * M + m) * E + e) * F + f;
                    y[o] = acc;
                    if (abs_sum) abs_sum[o] = mag;
                }
    return 0;
}

/* ---- CSR walker (Escoin Algorithm 2; Tuteja et al. Eq.(3)) ---- */

typedef struct {
    int N, C, H, W, M, R, S, stride, pad, E, F;
    const int32_t *rowptr, *colidx;
    const double *value, *x;
    double *y, *abs_sum;
    int64_t next;          /* next (n, m) work item, taken under the lock */
    pthread_mutex_t lock;
} csr_job;

static void csr_one_row(const csr_job *J, int n, int m)
{
    const int E = J->E, F = J->F, H = J->H, W = J->W, R = J->R, S = J->S;
    double *yo = J->y + ((size_t)n * J->M + m) * E * F;
    double *ao = J->abs_sum ? J->abs_sum + ((size_t)n * J->M + m) * E * F : NULL;
    for (int i = 0; i < E * F; ++i) {
        yo[i] = 0.0;
        if (ao) ao[i] = 0.0;
    }
    for (int32_t j = J->rowptr[m]; j < J->rowptr[m + 1]; ++j) {
        const int col = J->colidx[j];
        const int c = col / (R * S);
        const int r = (col / S) % R;
        const int s = col % S;
        const double v = J->value[j];
        const double *xc = J->x + ((size_t)n * J->C + c) * H * W;
        for (int e = 0; e < E; ++e) {
            const int h = e * J->stride + r - J->pad;
            if (h < 0 || h >= H) continue;               /* outside N(oc,h,w) */
            for (int f = 0; f < F; ++f) {
                const int q = f * J->stride + s - J->pad;
                if (q < 0 || q >= W) continue;
                const double p = v * xc[(size_t)h * W + q];
                yo[e * F + f] += p;
                if (ao) ao[e * F + f] += fabs(p);
            }
        }
    }
}

static void *csr_worker(void *arg)
{
    csr_job *J = (csr_job *)arg;
    const int64_t total = (int64_t)J->N * J->M;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t it = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (it >= total) break;
        csr_one_row(J, (int)(it / J->M), (int)(it % J->M));
    }
    return NULL;
}

static int check_csr(int M, int CRS, const int32_t *rowptr, const int32_t *colidx)
{
    if (rowptr[0] != 0) return -2;
    for (int m = 0; m < M; ++m) {
        if (rowptr[m + 1] < rowptr[m]) return -2;
        for (int32_t j = rowptr[m]; j < rowptr[m + 1]; ++j)
            if (colidx[j] < 0 || colidx[j] >= CRS) return -2;
    }
    return 0;
}

/* nthreads <= 0 -> one thread per online CPU.  Returns the thread count used
 * (>= 1) on success, a negative value on bad arguments. */
int oracle_csr(int N, int C, int H, int W, int M, int R, int S, int stride, int pad,
               const int32_t *rowptr, const int32_t *colidx, const double *value,
               const double *x, double *y, double *abs_sum, int nthreads)
{
    if (check_dims(N, C, H, W, M, R, S, stride, pad)) return -1;
    if (check_csr(M, C * R * S, rowptr, colidx)) return -2;
    csr_job J;
    J.N = N; J.C = C; J.H = H; J.W = W; J.M = M; J.R = R; J.S = S;
    J.stride = stride; J.pad = pad;
    J.E = oracle_out_dim(H, R, stride, pad);
    J.F = oracle_out_dim(W, S, stride, pad);
    J.rowptr = rowptr; J.colidx = colidx; J.value = value; J.x = x;
    J.y = y; J.abs_sum = abs_sum; J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads <= 0) nthreads = oracle_num_cpus();
    if ((int64_t)nthreads > (int64_t)N * M) nthreads = (int)((int64_t)N * M > 0 ? (int64_t)N * M : 1);
    if (nthreads <= 1) {
        csr_worker(&J);
        nthreads = 1;
    } else {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        int started = 0;
        for (int t = 0; t < nthreads; ++t)
            if (pthread_create(&tid[t], NULL, csr_worker, &J) == 0) ++started;
        if (started == 0) csr_worker(&J);
        for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
        free(tid);
        nthreads = started > 0 ? started : 1;
    }
    pthread_mutex_destroy(&J.lock);
    return nthreads;
}

/* One output element at a time, straight from Eq.(3): for each requested flat
 * index o = ((n*M + m)*E + e)*F + f, sum v_j * X[n, c_j, e*s + r_j - P,
 * f*s + s_j - P] over the nonzeros j of row m that land inside the image. */
int oracle_csr_points(int N, int C, int H, int W, int M, int R, int S, int stride, int pad,
                      const int32_t *rowptr, const int32_t *colidx, const double *value,
                      const double *x, int64_t npts, const int64_t *flat, double *y,
                      double *abs_sum)
{
    if (check_dims(N, C, H, W, M, R, S, stride, pad)) return -1;
    if (check_csr(M, C * R * S, rowptr, colidx)) return -2;
    const int E = oracle_out_dim(H, R, stride, pad);
    const int F = oracle_out_dim(W, S, stride, pad);
    const int64_t total = (int64_t)N * M * E * F;
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t o = flat[i];
        if (o < 0 || o >= total) return -1;
        const int f = (int)(o % F);
        const int e = (int)((o / F) % E);
        const int m = (int)((o / ((int64_t)E * F)) % M);
        const int n = (int)(o / ((int64_t)M * E * F));
        double acc = 0.0, mag = 0.0;
        for (int32_t j = rowptr[m]; j < rowptr[m + 1]; ++j) {
            const int col = colidx[j];
            const int c = col / (R * S), r = (col / S) % R, s = col % S;
            const int h = e * stride + r - pad, q = f * stride + s - pad;
            if (h < 0 || h >= H || q < 0 || q >= W) continue;
            const double p = value[j] * x[(((size_t)n * C + c) * H + h) * W + q];
            acc += p;
            mag += fabs(p);
        }
        y[i] = acc;
        if (abs_sum) abs_sum[i] = mag;
    }
    return 0;
}
