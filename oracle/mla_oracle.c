/*
 * CPU oracle for the Multi-Head Latent Attention prolog.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load this
 * file's library.  The CUDA library never links, includes or calls it, and it
 * shares no code with the CUDA path.
 *
 * It computes the prolog of "aclnnMlaPrologV2WeightNz" (Function: Formula) as
 * the plain definition, in double precision, one token at a time:
 *
 *   c^Q  = RmsNorm(x . W^DQ)                  q^C = c^Q . W^UQ,  q^N = q^C . W^UK
 *   q^R  = ROPE(c^Q . W^QR)
 *   c^KV = RmsNorm(x . W^DKV),  k^C = Cache(c^KV)
 *   k^R  = Cache(ROPE(x . W^KR))
 *   dequantScaleQNope = RowMax(|q^N|) / 127,  q^N = round(q^N / dequantScaleQNope)
 *
 * with RmsNorm(x) = gamma * x_i / sqrt(mean(x^2) + eps)  (epsilon inside the root,
 * same page, Function: RmsNorm formula) and the "half" RoPE of "aclnnMlaPreprocess"
 * (Constraints: RoPE mode is half, interleave is not supported).
 *
 * The inputs are read as the exact bits the GPU reads (bf16 as uint16, int8, fp32
 * scales, int64 slots).  Nothing is rounded between steps except where the method
 * itself quantises (int8 codes) or writes a bf16 cache.  Readings of points the
 * pages leave open are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- scalars */

/* bf16 bit pattern -> double; exact. */
static double bf16_bits_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * double -> bf16 bits, round to nearest, ties to even, in ONE rounding step
 * (going through float first could round twice).  bf16 keeps 8 significant
 * bits; its smallest subnormal step is 2^-133; the largest finite value is
 * (2 - 2^-7) * 2^127.
 */
uint16_t mla_oracle_bf16_rne(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);            /* a = m * 2^e with m in [0.5, 1) */
    int qe = e - 8;                /* weight of the last kept bit */
    if (qe < -133)
        qe = -133;
    double r = nearbyint(ldexp(a, -qe));   /* default mode: nearest, ties to even */
    double rv = ldexp(r, qe);
    if (rv > 3.38953138925153547590470800371487866880e38)
        return (uint16_t)(sign | 0x7F80);
    float f = (float)rv;           /* exact: rv has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* Reading G6: "round" of the dynamic quantiser is round half away from zero,
 * and codes saturate to [-127, 127] (the scale maps the row maximum to 127). */
int8_t mla_oracle_round_i8(double v)
{
    double r = round(v);           /* C round(): halves away from zero */
    if (r > 127.0)
        r = 127.0;
    if (r < -127.0)
        r = -127.0;
    return (int8_t)r;
}

/* ------------------------------------------------------------------ steps */

/*
 * One row of a matrix product: out[j] = sum_k x[k] * W[k, col0 + j] for j < n,
 * W stored row-major with leading dimension ldw, in the (k, n) orientation of
 * "aclnnMlaPrologV2WeightNz" (Constraints: "when ... not transposed, the
 * representation of each dimension is (k, n)").  Each sum runs over k in
 * ascending order.
 */
void mla_oracle_row_times_bf16(const double* x, int64_t K, const uint16_t* W, int64_t ldw,
                               int64_t col0, int64_t n, double* out)
{
    for (int64_t j = 0; j < n; ++j)
        out[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double xv = x[k];
        const uint16_t* wr = W + k * ldw + col0;
        for (int64_t j = 0; j < n; ++j)
            out[j] += xv * bf16_bits_to_f64(wr[j]);
    }
}

/* The same for integer operands: an exact int64 sum (int8 x int8 products). */
void mla_oracle_row_times_i8(const int8_t* x, int64_t K, const int8_t* W, int64_t ldw,
                             int64_t col0, int64_t n, int64_t* out)
{
    for (int64_t j = 0; j < n; ++j)
        out[j] = 0;
    for (int64_t k = 0; k < K; ++k) {
        int64_t xv = x[k];
        const int8_t* wr = W + k * ldw + col0;
        for (int64_t j = 0; j < n; ++j)
            out[j] += xv * (int64_t)wr[j];
    }
}

/*
 * RmsNorm of "aclnnMlaPrologV2WeightNz" (Function: RmsNorm formula):
 *   RMS(y) = sqrt( (1/n) * sum_i y_i^2 + eps ),   out_i = gamma_i * y_i / RMS(y).
 * Reading G4: the "N" of the formula is the length of the normalised row
 * (Hcq for c^Q, Hckv for c^KV).  Epsilon sits inside the square root.
 */
void mla_oracle_rmsnorm(const double* y, int64_t n, const uint16_t* gamma, double eps, double* out)
{
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i)
        ss += y[i] * y[i];
    double rms = sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_bits_to_f64(gamma[i]) * y[i] / rms;
}

/*
 * "Half" RoPE ("aclnnMlaPreprocess", Constraints: RoPE mode), on a vector v of
 * even length dr with h = dr/2 and the full-width tables cos/sin of one token
 * ("aclnnMlaPrologV2WeightNz", Parameters: ropeSin, ropeCos of shape (T, Dr)):
 *   out = v * cos + rotate_half(v) * sin,   rotate_half(v) = [-v[h:], v[:h]]
 * i.e. out[j]   = v[j]   * cos[j]   - v[j+h] * sin[j]
 *      out[j+h] = v[j+h] * cos[j+h] + v[j]   * sin[j+h]      (j < h).
 */
void mla_oracle_rope_half(const double* v, int64_t dr, const uint16_t* cos_row,
                          const uint16_t* sin_row, double* out)
{
    int64_t h = dr / 2;
    for (int64_t j = 0; j < h; ++j) {
        double c0 = bf16_bits_to_f64(cos_row[j]), s0 = bf16_bits_to_f64(sin_row[j]);
        double c1 = bf16_bits_to_f64(cos_row[j + h]), s1 = bf16_bits_to_f64(sin_row[j + h]);
        out[j] = v[j] * c0 - v[j + h] * s0;
        out[j + h] = v[j + h] * c1 + v[j] * s1;
    }
}

/*
 * Dynamic quantisation of one row ("aclnnMlaPrologV2WeightNz", Function: Dequant
 * Scale Query Nope formula):  scale = RowMax(|v|) / 127,  code = round(v / scale).
 * Reading G7: an all-zero row gets scale 0 and all-zero codes (no division).
 * Returns the scale.
 */
double mla_oracle_dynamic_quant(const double* v, int64_t n, int8_t* codes)
{
    double m = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double a = fabs(v[i]);
        if (a > m)
            m = a;
    }
    double scale = m / 127.0;
    for (int64_t i = 0; i < n; ++i)
        codes[i] = (scale == 0.0) ? 0 : mla_oracle_round_i8(v[i] / scale);
    return scale;
}

/* ------------------------------------------------------------- whole prolog */

typedef struct {
    int64_t T, He, Hcq, N, D, Dr, Hckv, block_num, block_size;
    double eps_cq, eps_ckv;
    int32_t x_int8;     /* tokenX, weightDq, weightDkvKr are int8 (int8 full quantisation) */
    int32_t uqqr_int8;  /* weightUqQr is int8 (partial and full quantisation) */
    int32_t kv_int8;    /* kvCache holds int8 codes of c^KV * quantScaleCkv */
    int32_t kr_int8;    /* krCache holds int8 codes of k^R * quantScaleCkr */
    int32_t q_int8;     /* q^N is dynamically quantised to int8 */
    int32_t num_threads;
    /* inputs */
    const void* x;
    const void* w_dq;
    const void* w_uqqr;
    const uint16_t* w_uk;
    const void* w_dkvkr;
    const uint16_t* gamma_cq;
    const uint16_t* gamma_ckv;
    const uint16_t* rope_sin;
    const uint16_t* rope_cos;
    const int64_t* cache_index;
    const float* dequant_scale_x;       /* (T) */
    const float* dequant_scale_w_dq;    /* (Hcq) */
    const float* dequant_scale_w_uqqr;  /* (N*(D+Dr)) */
    const float* dequant_scale_w_dkvkr; /* (Hckv+Dr) */
    const float* quant_scale_ckv;       /* (Hckv) */
    const float* quant_scale_ckr;       /* (Dr) */
    const float* smooth_scales_cq;      /* (Hcq) or NULL */
    /* caches, updated in place at the rows named by cache_index */
    void* kv_cache;
    void* kr_cache;
    /* results before output rounding; any pointer may be NULL except q_nope, q_rope */
    double* q_nope;        /* (T, N, Hckv) */
    double* q_rope;        /* (T, N, Dr) */
    double* c_q;           /* (T, Hcq) */
    double* c_kv;          /* (T, Hckv) */
    double* k_r;           /* (T, Dr) */
    double* q_c;           /* (T, N, D) */
    int8_t* q_nope_i8;     /* (T, N, Hckv) when q_int8 */
    double* q_nope_scale;  /* (T, N) when q_int8 */
    int8_t* c_q_i8;        /* (T, Hcq) when uqqr_int8 */
    double* c_q_scale;     /* (T) when uqqr_int8 */
} mla_oracle_args;

enum { MLA_ORACLE_OK = 0, MLA_ORACLE_BAD_ARGS = 1, MLA_ORACLE_SLOT_RANGE = 2, MLA_ORACLE_SLOT_DUP = 3 };

/*
 * Checks the cache slots before anything is written.  "aclnnMlaPrologV2WeightNz"
 * (Parameters: cacheIndex) requires values in [0, BlockNum*BlockSize).
 * Reading G10: slots are distinct; the oracle refuses duplicates.
 */
static int check_slots(const mla_oracle_args* a)
{
    int64_t nslots = a->block_num * a->block_size;
    if (nslots == 0)
        return MLA_ORACLE_OK;   /* Skv = 0: caches are not updated */
    unsigned char* seen = (unsigned char*)calloc((size_t)nslots, 1);
    if (!seen)
        return MLA_ORACLE_BAD_ARGS;
    int rc = MLA_ORACLE_OK;
    for (int64_t t = 0; t < a->T; ++t) {
        int64_t s = a->cache_index[t];
        if (s < 0 || s >= nslots) { rc = MLA_ORACLE_SLOT_RANGE; break; }
        if (seen[s]) { rc = MLA_ORACLE_SLOT_DUP; break; }
        seen[s] = 1;
    }
    free(seen);
    return rc;
}

static int8_t quant_static(double v, double scale)
{
    /* Reading G12: a quantScale multiplies before rounding. */
    return mla_oracle_round_i8(v * scale);
}

/* One token: every step of the prolog in the order the page states them. */
static void prolog_token(const mla_oracle_args* a, int64_t t, double* buf)
{
    const int64_t He = a->He, Hcq = a->Hcq, N = a->N, D = a->D, Dr = a->Dr, Hckv = a->Hckv;
    const int64_t Wqr = N * (D + Dr);
    double* yq = buf;               /* Hcq   */
    double* ykv = yq + Hcq;         /* Hckv  */
    double* ykr = ykv + Hckv;       /* Dr    */
    double* cq = ykr + Dr;          /* Hcq   */
    double* ckv = cq + Hcq;         /* Hckv  */
    double* kr = ckv + Hckv;        /* Dr    */
    double* z = kr + Dr;            /* Wqr   */
    double* xr = z + Wqr;           /* He    */
    double* qn = xr + He;           /* Hckv  */
    double* u = qn + Hckv;          /* Hcq   */
    int64_t* acc = (int64_t*)(u + Hcq);            /* max(Hcq, Hckv+Dr, Wqr) */
    int8_t* cq8 = (int8_t*)(acc + (Wqr > Hcq + Hckv + Dr ? Wqr : Hcq + Hckv + Dr));  /* Hcq */

    /* 1. down-projections x.W^DQ and x.[W^DKV | W^KR] (Formula: c^Q, c^KV, k^R). */
    if (a->x_int8) {
        /* int8 full quantisation: int8 x int8 summed exactly, then scaled by the
         * per-token dequant scale of tokenX and the per-column scale of the weight
         * (scenario table: tokenX per-token, weights per-channel). */
        const int8_t* x8 = (const int8_t*)a->x + t * He;
        double sx = a->dequant_scale_x[t];
        mla_oracle_row_times_i8(x8, He, (const int8_t*)a->w_dq, Hcq, 0, Hcq, acc);
        for (int64_t j = 0; j < Hcq; ++j)
            yq[j] = (double)acc[j] * sx * (double)a->dequant_scale_w_dq[j];
        mla_oracle_row_times_i8(x8, He, (const int8_t*)a->w_dkvkr, Hckv + Dr, 0, Hckv + Dr, acc);
        for (int64_t j = 0; j < Hckv + Dr; ++j) {
            double v = (double)acc[j] * sx * (double)a->dequant_scale_w_dkvkr[j];
            if (j < Hckv) ykv[j] = v; else ykr[j - Hckv] = v;
        }
    } else {
        const uint16_t* xb = (const uint16_t*)a->x + t * He;
        for (int64_t k = 0; k < He; ++k)
            xr[k] = bf16_bits_to_f64(xb[k]);
        mla_oracle_row_times_bf16(xr, He, (const uint16_t*)a->w_dq, Hcq, 0, Hcq, yq);
        /* Reading G3: weightDkvKr columns are [Hckv of W^DKV | Dr of W^KR]. */
        mla_oracle_row_times_bf16(xr, He, (const uint16_t*)a->w_dkvkr, Hckv + Dr, 0, Hckv, ykv);
        mla_oracle_row_times_bf16(xr, He, (const uint16_t*)a->w_dkvkr, Hckv + Dr, Hckv, Dr, ykr);
    }

    /* 2. RmsNorm of both down-projected rows. */
    mla_oracle_rmsnorm(yq, Hcq, a->gamma_cq, a->eps_cq, cq);
    mla_oracle_rmsnorm(ykv, Hckv, a->gamma_ckv, a->eps_ckv, ckv);

    /* 3. k^R = ROPE(x.W^KR), no norm on this branch. */
    const uint16_t* cs = a->rope_cos + t * Dr;
    const uint16_t* sn = a->rope_sin + t * Dr;
    mla_oracle_rope_half(ykr, Dr, cs, sn, kr);

    /* 4. cache writes at slot cacheIndex[t]: row s of the (BlockNum*BlockSize, Nkv=1, H)
     * view, i.e. block s / BlockSize, offset s % BlockSize.  No other element changes. */
    int64_t nslots = a->block_num * a->block_size;
    if (nslots > 0) {
        int64_t s = a->cache_index[t];
        if (a->kv_int8) {
            int8_t* dst = (int8_t*)a->kv_cache + s * Hckv;
            for (int64_t j = 0; j < Hckv; ++j)
                dst[j] = quant_static(ckv[j], (double)a->quant_scale_ckv[j]);
        } else {
            uint16_t* dst = (uint16_t*)a->kv_cache + s * Hckv;
            for (int64_t j = 0; j < Hckv; ++j)
                dst[j] = mla_oracle_bf16_rne(ckv[j]);
        }
        if (a->kr_int8) {
            int8_t* dst = (int8_t*)a->kr_cache + s * Dr;
            for (int64_t j = 0; j < Dr; ++j)
                dst[j] = quant_static(kr[j], (double)a->quant_scale_ckr[j]);
        } else {
            uint16_t* dst = (uint16_t*)a->kr_cache + s * Dr;
            for (int64_t j = 0; j < Dr; ++j)
                dst[j] = mla_oracle_bf16_rne(kr[j]);
        }
    }

    /* 5. Q up-projection z = c^Q . [W^UQ | W^QR] (Formula: q^C and q^R).
     * Reading G2: the N*(D+Dr) columns hold, per head n, D columns of W^UQ and
     * then Dr columns of W^QR: column n*(D+Dr) + j. */
    if (a->uqqr_int8) {
        /* Reading G13: c^Q (times the smooth scales when given) is quantised per
         * token with RowMax/127 before the int8 product; the product is dequantised
         * by that scale and the per-column weight scale. */
        for (int64_t i = 0; i < Hcq; ++i)
            u[i] = cq[i] * (a->smooth_scales_cq ? (double)a->smooth_scales_cq[i] : 1.0);
        double scq = mla_oracle_dynamic_quant(u, Hcq, cq8);
        mla_oracle_row_times_i8(cq8, Hcq, (const int8_t*)a->w_uqqr, Wqr, 0, Wqr, acc);
        for (int64_t c = 0; c < Wqr; ++c)
            z[c] = (double)acc[c] * scq * (double)a->dequant_scale_w_uqqr[c];
        if (a->c_q_i8)
            memcpy(a->c_q_i8 + t * Hcq, cq8, (size_t)Hcq);
        if (a->c_q_scale)
            a->c_q_scale[t] = scq;
    } else {
        mla_oracle_row_times_bf16(cq, Hcq, (const uint16_t*)a->w_uqqr, Wqr, 0, Wqr, z);
    }

    /* 6. per head: q^R = ROPE(rope columns); q^N = q^C . W^UK[n]. */
    for (int64_t n = 0; n < N; ++n) {
        const double* zc = z + n * (D + Dr);            /* q^C of head n: D values */
        mla_oracle_rope_half(zc + D, Dr, cs, sn, a->q_rope + (t * N + n) * Dr);
        if (a->q_c)
            memcpy(a->q_c + (t * N + n) * D, zc, (size_t)D * sizeof(double));
        /* weightUk is (N, D, Hckv): q^N[c] = sum_d q^C[d] * W^UK[n, d, c]. */
        mla_oracle_row_times_bf16(zc, D, a->w_uk + n * D * Hckv, Hckv, 0, Hckv, qn);
        memcpy(a->q_nope + (t * N + n) * Hckv, qn, (size_t)Hckv * sizeof(double));
        /* 7. the fifth path: dynamic int8 quantisation of each (token, head) row. */
        if (a->q_int8) {
            double sc = mla_oracle_dynamic_quant(qn, Hckv, a->q_nope_i8 + (t * N + n) * Hckv);
            a->q_nope_scale[t * N + n] = sc;
        }
    }

    if (a->c_q)
        memcpy(a->c_q + t * Hcq, cq, (size_t)Hcq * sizeof(double));
    if (a->c_kv)
        memcpy(a->c_kv + t * Hckv, ckv, (size_t)Hckv * sizeof(double));
    if (a->k_r)
        memcpy(a->k_r + t * Dr, kr, (size_t)Dr * sizeof(double));
}

int mla_oracle_prolog(const mla_oracle_args* a)
{
    if (!a || a->T < 0 || a->He <= 0 || a->Hcq <= 0 || a->N <= 0 || a->D <= 0 || a->Dr <= 0 ||
        (a->Dr & 1) || a->Hckv <= 0 || !a->q_nope || !a->q_rope)
        return MLA_ORACLE_BAD_ARGS;
    if (a->q_int8 && (!a->q_nope_i8 || !a->q_nope_scale))
        return MLA_ORACLE_BAD_ARGS;
    if (a->T == 0)
        return MLA_ORACLE_OK;
    int rc = check_slots(a);
    if (rc != MLA_ORACLE_OK)
        return rc;

    const int64_t Wqr = a->N * (a->D + a->Dr);
    const int64_t accn = Wqr > a->Hcq + a->Hckv + a->Dr ? Wqr : a->Hcq + a->Hckv + a->Dr;
    const size_t per = sizeof(double) * (size_t)(2 * (a->Hcq + a->Hckv + a->Dr) + Wqr + a->He + a->Hckv + a->Hcq)
                     + sizeof(int64_t) * (size_t)accn + (size_t)a->Hcq + 64;
#ifdef _OPENMP
    if (a->num_threads > 0)
        omp_set_num_threads(a->num_threads);
#endif
    int failed = 0;
#pragma omp parallel
    {
        double* buf = (double*)malloc(per);
        if (!buf) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < a->T; ++t)
                prolog_token(a, t, buf);
            free(buf);
        }
    }
    return failed ? MLA_ORACLE_BAD_ARGS : MLA_ORACLE_OK;
}

int mla_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
