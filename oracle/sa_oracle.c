/*
 * sa_oracle.c -- plain FP64 CPU oracle of the Stable Audio 3 attention core.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  It shares no code, header,
 * table or constant with the CUDA path; the two meet only in the seeded input
 * bytes produced by the `synth` module.
 *
 * What it computes (slow, obviously correct, in the order the pages describe):
 *
 *   1. Decode the fp16/bf16 input bits exactly to double (or the FP32 bits of
 *      the FP32-input form, SAME-L's FP32 attention projections, HF
 *      discussion #6 "sm_120 SAME-L", "How the kernels differ").
 *   2. RoPE on every q and k row (rotate-half over the full head dim, base
 *      10000): theta_{p,i} = p * base^(-2i/d) for i < d/2, and
 *      x'_i = x_i cos - x_{i+d/2} sin,  x'_{i+d/2} = x_{i+d/2} cos + x_i sin.
 *      The pages say RoPE runs in FP32 and casts back to the autocast dtype
 *      (apply_rotary_pos_emb finishes with a cast to the output dtype, and the
 *      exported graph multiplies in FP32 before two casts to fp16; HF discussion
 *      #3 "fp16mixed attention-core fix", sections "The bug" and "The fix").  Here the rotation is FP64 and,
 *      in the default "method" cast mode, the rotated q/k are rounded to the
 *      storage dtype (round to nearest even) and decoded back to double.
 *      Cast mode "exact" skips that rounding.  For FP32 inputs the storage
 *      dtype is FP32, so the method's cast rounds to FP32.  The TF32 rounding
 *      of the tensor-core products is part of the method's kernel, not of
 *      what it computes, and is not modelled.
 *   3. Scaled dot-product attention per row with the exact two-pass softmax:
 *      s_j = q.k_j / sqrt(d) over the allowed keys, m = max s_j,
 *      e_j = exp(s_j - m), l = sum e_j, o = sum (e_j / l) v_j
 *      (F.scaled_dot_product_attention(q, k, v), same page, "The bug").
 *   4. Differential attention (two softmax maps sharing V, the second weighted
 *      by lambda and subtracted, HF discussion #6 "sm_120 SAME-L" section
 *      "How the kernels differ"): o = o(Q1,K1) - lambda_h * o(Q2,K2).
 *   5. Sliding window: key j is allowed for query i iff |i - j| <= window
 *      (the SAME-L window of +-17 in the same page's "Three gotchas" is
 *      symmetric); window < 0 means full attention.  Only keys in
 *      [max(0, i-w), min(L-1, i+w)] are visited; masked keys contribute
 *      exp(-inf) = 0, so this is exact.
 *   6. Optional QK-RMSNorm before RoPE (the pages run RMSNorm and RoPE next
 *      to attention in FP32, so that variances cannot overflow fp16; sa3_trt
 *      README "Notes on the design" and the encoder/decoder page's "Where the
 *      quantization goes, per tier"): every q and k row of d values becomes
 *      x_c * gamma_c / sqrt(mean_c(x_c^2) + eps), with one learned gamma[d]
 *      for q and one for k, then RoPE, then the single cast-back of step 2.
 *
 * Layouts (C order): q, k [B][H][nmaps][L][d]; v [B][H][L][dv];
 * output rows [nrows][dv] in double.  Input elements are 2-byte fp16/bf16 bits,
 * or 4-byte FP32 bits for dtype 2.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_FP16 0
#define OR_BF16 1
#define OR_FP32 2
#define OR_CAST_METHOD 0
#define OR_CAST_EXACT 1

/* ---------------------------------------------------------------- bits -> double */

double sa_oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25);    /* (1024+m) * 2^(e-15-10) */
    return sign ? -v : v;
}

double sa_oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);                /* subnormal: m * 2^(-126-7) */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x80), e - 134);    /* (128+m) * 2^(e-127-7) */
    return sign ? -v : v;
}

double sa_oracle_fp32_to_double(uint32_t f)
{
    int sign = (f >> 31) & 1;
    int e = (f >> 23) & 0xff;
    uint32_t m = f & 0x7fffff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -149);                /* subnormal: m * 2^(-126-23) */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x800000), e - 150); /* (2^23+m) * 2^(e-127-23) */
    return sign ? -v : v;
}

/* Element i of an input array of the given dtype (2-byte bits, or 4-byte FP32 bits). */
static double elem_to_double(const void* p, size_t i, int dtype)
{
    if (dtype == OR_FP32)
        return sa_oracle_fp32_to_double(((const uint32_t*)p)[i]);
    uint16_t x = ((const uint16_t*)p)[i];
    return dtype == OR_BF16 ? sa_oracle_bf16_to_double(x) : sa_oracle_fp16_to_double(x);
}

/* --------------------------------------------------- double -> dtype (RNE) -> double */

/* Round |x| to a multiple of the quantum of its binade (sig_bits significant
 * bits, normal exponents down to emin, below that the subnormal quantum of
 * emin), ties to even; above max_finite the result is infinity. */
static double round_generic(double x, int sig_bits, int emin, double max_finite)
{
    if (isnan(x) || isinf(x) || x == 0.0)
        return x;
    double a = fabs(x);
    int E;
    frexp(a, &E);              /* a in [2^(E-1), 2^E) */
    int e = E - 1;
    if (e < emin)
        e = emin;
    double quantum = ldexp(1.0, e - (sig_bits - 1));
    double r = nearbyint(a / quantum) * quantum;    /* default mode: ties to even */
    if (r > max_finite)
        r = INFINITY;
    return copysign(r, x);
}

double sa_oracle_round(double x, int dtype)
{
    if (dtype == OR_FP32)   /* 24 significant bits, emin -126, max (2-2^-23)*2^127 */
        return round_generic(x, 24, -126, ldexp(16777215.0, 104));
    if (dtype == OR_BF16)   /* 8 significant bits, emin -126, max (2-2^-7)*2^127 */
        return round_generic(x, 8, -126, ldexp(255.0, 120));
    /* fp16: 11 significant bits, emin -14, max 65504 */
    return round_generic(x, 11, -14, 65504.0);
}

void sa_oracle_round_array(const double* x, int64_t n, int dtype, double* y)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = sa_oracle_round(x[i], dtype);
}

/* ---------------------------------------------------------------- RoPE (FP64) */

/* Rotate one row x[d] at position p (rotate-half pairs (i, i + d/2)). */
static void rope_row(const double* x, double* y, int d, double p, double base)
{
    int h = d / 2;
    for (int i = 0; i < h; ++i) {
        double inv_freq = pow(base, -2.0 * (double)i / (double)d);
        double theta = p * inv_freq;
        double c = cos(theta), s = sin(theta);
        double a = x[i], b = x[i + h];
        y[i] = a * c - b * s;
        y[i + h] = b * c + a * s;
    }
}

/* ---------------------------------------------------------------- RMSNorm (FP64) */

/* y = x * gamma / sqrt(mean(x^2) + eps) over one row of d values (gamma NULL: all ones).
 * y may alias x. */
static void rmsnorm_row(const double* x, double* y, int d, const double* gamma, double eps)
{
    double ss = 0.0;
    for (int c = 0; c < d; ++c)
        ss += x[c] * x[c];
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int c = 0; c < d; ++c)
        y[c] = x[c] * inv * (gamma ? gamma[c] : 1.0);
}

/* Public: RMSNorm of n rows of x[n][d]. */
int sa_oracle_rmsnorm(const double* x, int64_t n, int d, const double* gamma, double eps, double* y)
{
    if (d <= 0 || !(eps >= 0.0))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        rmsnorm_row(x + r * d, y + r * d, d, gamma, eps);
    return 0;
}

/* Public: rotate n rows of x[n][d] at positions pos[n] (NULL: 0..n-1). */
int sa_oracle_rope(const double* x, const int32_t* pos, int64_t n, int d, double base, double* y)
{
    if (d <= 0 || (d & 1))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        rope_row(x + r * d, y + r * d, d, pos ? (double)pos[r] : (double)r, base);
    return 0;
}

/* ---------------------------------------------------------------- attention */

typedef struct {
    /* inputs */
    const void *q, *k, *v;           /* uint16 bits (fp16, bf16) or uint32 bits (FP32) */
    const int32_t* positions;
    int B, H, L, d, nmaps, dv, window, dtype, cast_mode;
    const double* lambda;
    double base;
    int qk_norm;                    /* 1: RMSNorm of q and k rows before RoPE */
    const double *gamma_q, *gamma_k;
    double eps;
    const int64_t* rows;
    int64_t nrows;
    double* out;
    /* per-(b,h) prepared operands, filled lazily under the lock */
    double** kr;       /* [B*H] -> [nmaps][L][d] rotated (and cast) keys */
    double** vd;       /* [B*H] -> [L][dv] values */
    pthread_mutex_t* head_lock;
    /* work distribution */
    int64_t next;
    pthread_mutex_t lock;
    int failed;
} job_t;

static double cast_back(double x, const job_t* J)
{
    return J->cast_mode == OR_CAST_METHOD ? sa_oracle_round(x, J->dtype) : x;
}

static double pos_of(const job_t* J, int l)
{
    return J->positions ? (double)J->positions[l] : (double)l;
}

/* Rotate all keys of head bh once; decode its values. */
static int prepare_head(job_t* J, int64_t bh)
{
    pthread_mutex_lock(&J->head_lock[bh]);
    if (J->kr[bh]) {
        pthread_mutex_unlock(&J->head_lock[bh]);
        return 0;
    }
    int L = J->L, d = J->d, dv = J->dv, nm = J->nmaps;
    double* kr = (double*)malloc(sizeof(double) * (size_t)nm * L * d);
    double* vd = (double*)malloc(sizeof(double) * (size_t)L * dv);
    double* row = (double*)malloc(sizeof(double) * d);
    if (!kr || !vd || !row) {
        free(kr); free(vd); free(row);
        pthread_mutex_unlock(&J->head_lock[bh]);
        return -1;
    }
    for (int m = 0; m < nm; ++m) {
        size_t kbase = (((size_t)bh * nm + m) * L) * d;
        for (int l = 0; l < L; ++l) {
            for (int c = 0; c < d; ++c)
                row[c] = elem_to_double(J->k, kbase + (size_t)l * d + c, J->dtype);
            if (J->qk_norm)
                rmsnorm_row(row, row, d, J->gamma_k, J->eps);
            double* dst = kr + ((size_t)m * L + l) * d;
            rope_row(row, dst, d, pos_of(J, l), J->base);
            for (int c = 0; c < d; ++c)
                dst[c] = cast_back(dst[c], J);
        }
    }
    size_t vbase = (size_t)bh * L * dv;
    for (size_t i = 0; i < (size_t)L * dv; ++i)
        vd[i] = elem_to_double(J->v, vbase + i, J->dtype);
    free(row);
    J->vd[bh] = vd;
    J->kr[bh] = kr;   /* published last */
    pthread_mutex_unlock(&J->head_lock[bh]);
    return 0;
}

/* o[dv] = softmax(q . K^T / sqrt(d)) V over keys lo..hi (two-pass, exact). */
static void attend(const double* qr, const double* K, const double* V, int d, int dv,
                   int lo, int hi, double* s, double* o)
{
    double scale = 1.0 / sqrt((double)d);
    double m = -INFINITY;
    for (int j = lo; j <= hi; ++j) {
        const double* kj = K + (size_t)j * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += qr[c] * kj[c];
        s[j - lo] = acc * scale;
        if (s[j - lo] > m)
            m = s[j - lo];
    }
    double l = 0.0;
    for (int j = lo; j <= hi; ++j) {
        s[j - lo] = exp(s[j - lo] - m);
        l += s[j - lo];
    }
    for (int c = 0; c < dv; ++c)
        o[c] = 0.0;
    for (int j = lo; j <= hi; ++j) {
        double w = s[j - lo] / l;
        const double* vj = V + (size_t)j * dv;
        for (int c = 0; c < dv; ++c)
            o[c] += w * vj[c];
    }
}

static void* worker(void* arg)
{
    job_t* J = (job_t*)arg;
    int L = J->L, d = J->d, dv = J->dv, nm = J->nmaps;
    double* qraw = (double*)malloc(sizeof(double) * d);
    double* qr = (double*)malloc(sizeof(double) * d);
    double* s = (double*)malloc(sizeof(double) * L);
    double* o = (double*)malloc(sizeof(double) * dv);
    if (!qraw || !qr || !s || !o) {
        pthread_mutex_lock(&J->lock); J->failed = 1; pthread_mutex_unlock(&J->lock);
        free(qraw); free(qr); free(s); free(o);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t t = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (t >= J->nrows)
            break;
        int64_t flat = J->rows ? J->rows[t] : t;   /* (b*H + h)*L + i */
        int64_t bh = flat / L;
        int i = (int)(flat % L);
        if (prepare_head(J, bh) != 0) {
            pthread_mutex_lock(&J->lock); J->failed = 1; pthread_mutex_unlock(&J->lock);
            break;
        }
        int lo = 0, hi = L - 1;
        if (J->window >= 0) {
            lo = i - J->window < 0 ? 0 : i - J->window;
            hi = i + J->window > L - 1 ? L - 1 : i + J->window;
        }
        double* dst = J->out + t * dv;
        for (int c = 0; c < dv; ++c)
            dst[c] = 0.0;
        for (int m = 0; m < nm; ++m) {
            size_t qbase = ((((size_t)bh * nm + m) * L) + i) * d;
            for (int c = 0; c < d; ++c)
                qraw[c] = elem_to_double(J->q, qbase + c, J->dtype);
            if (J->qk_norm)
                rmsnorm_row(qraw, qraw, d, J->gamma_q, J->eps);
            rope_row(qraw, qr, d, pos_of(J, i), J->base);
            for (int c = 0; c < d; ++c)
                qr[c] = cast_back(qr[c], J);
            attend(qr, J->kr[bh] + (size_t)m * L * d, J->vd[bh], d, dv, lo, hi, s, o);
            /* map 0 enters with weight 1, map 1 with -lambda_h */
            double wgt = 1.0;
            if (m == 1)
                wgt = -J->lambda[bh % J->H];
            for (int c = 0; c < dv; ++c)
                dst[c] += wgt * o[c];
        }
    }
    free(qraw); free(qr); free(s); free(o);
    return NULL;
}

/*
 * Public entry with the optional QK-RMSNorm.  rows: flattened row ids
 * (b*H + h)*L + i, or NULL for all B*H*L rows in order.  lambda: [H] (required
 * when nmaps == 2).  qk_norm != 0: gamma_q, gamma_k [d] (NULL: all ones) and
 * eps >= 0 normalise every q and k row before RoPE.
 * Returns 0 on success, a negative code on bad arguments or allocation failure.
 */
int sa_oracle_rope_attn_qknorm(const void* q, const void* k, const void* v,
                               const int32_t* positions, int B, int H, int L, int d, int nmaps,
                               int dv, int window, const double* lambda, int dtype, int cast_mode,
                               double base, int qk_norm, const double* gamma_q,
                               const double* gamma_k, double eps, const int64_t* rows,
                               int64_t nrows, double* out, int nthreads)
{
    if (!q || !k || !v || !out || B <= 0 || H <= 0 || L <= 0 || d <= 0 || (d & 1) || dv <= 0)
        return -1;
    if (qk_norm && !(eps >= 0.0))
        return -8;
    if (nmaps != 1 && nmaps != 2)
        return -2;
    if (nmaps == 2 && !lambda)
        return -3;
    if (dtype != OR_FP16 && dtype != OR_BF16 && dtype != OR_FP32)
        return -4;
    int64_t total = (int64_t)B * H * L;
    if (!rows)
        nrows = total;
    for (int64_t t = 0; rows && t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= total)
            return -5;
    if (nthreads < 1)
        nthreads = 1;

    job_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.positions = positions;
    J.B = B; J.H = H; J.L = L; J.d = d; J.nmaps = nmaps; J.dv = dv;
    J.window = window; J.dtype = dtype; J.cast_mode = cast_mode; J.lambda = lambda;
    J.base = base; J.rows = rows; J.nrows = nrows; J.out = out;
    J.qk_norm = qk_norm != 0; J.gamma_q = gamma_q; J.gamma_k = gamma_k; J.eps = eps;
    int64_t nbh = (int64_t)B * H;
    J.kr = (double**)calloc((size_t)nbh, sizeof(double*));
    J.vd = (double**)calloc((size_t)nbh, sizeof(double*));
    J.head_lock = (pthread_mutex_t*)calloc((size_t)nbh, sizeof(pthread_mutex_t));
    if (!J.kr || !J.vd || !J.head_lock) {
        free(J.kr); free(J.vd); free(J.head_lock);
        return -6;
    }
    for (int64_t i = 0; i < nbh; ++i)
        pthread_mutex_init(&J.head_lock[i], NULL);
    pthread_mutex_init(&J.lock, NULL);

    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; th && t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, worker, &J) == 0)
            ++started;
    if (started == 0)
        worker(&J);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);

    for (int64_t i = 0; i < nbh; ++i) {
        free(J.kr[i]);
        free(J.vd[i]);
        pthread_mutex_destroy(&J.head_lock[i]);
    }
    free(J.kr); free(J.vd); free(J.head_lock);
    pthread_mutex_destroy(&J.lock);
    return J.failed ? -7 : 0;
}

/* Public entry without the QK-RMSNorm (the attention core as the pages describe it). */
int sa_oracle_rope_attn(const void* q, const void* k, const void* v,
                        const int32_t* positions, int B, int H, int L, int d, int nmaps,
                        int dv, int window, const double* lambda, int dtype, int cast_mode,
                        double base, const int64_t* rows, int64_t nrows, double* out,
                        int nthreads)
{
    return sa_oracle_rope_attn_qknorm(q, k, v, positions, B, H, L, d, nmaps, dv, window, lambda,
                                      dtype, cast_mode, base, 0, NULL, NULL, 0.0, rows, nrows,
                                      out, nthreads);
}
