/*
 * ora.c -- fp64 CPU oracle for ring-chunked attention forward.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke check
 * and the benchmark's CPU-baseline / reference arm may load this library.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (MarkTechPost/mKernel page, table "Die fünf verschmolzenen
 * Kerne", row "Ring Attention": the local step is FlashAttention, i.e. exact
 * softmax attention; the KV sequence arrives block by block around a ring and
 * each received block is folded into the running result):
 *
 *   for batch b, query head h, query row s, KV head g = h / (H / Hkv):
 *     x_t   = scale * sum_d q[b,s,h,d] * k[b,t,g,d]       for allowed t
 *             (allowed: every t when non-causal, t <= s when causal)
 *     M     = max_t x_t,  L = sum_t exp(x_t - M)
 *     out   = sum_t exp(x_t - M) / L * v[b,t,g,:]
 *     lse   = M + ln L                                    (natural log)
 *
 * Layouts: q, out [B,S,H,D]; k, v [B,S,Hkv,D]; lse [B,H,S].  q/k/v arrive as
 * bf16 bit patterns (uint16) and are widened exactly to double; every
 * arithmetic step below is fp64.
 *
 * Four entry points, written independently of each other:
 *   ora_attn_direct -- the two-pass definition above (optionally also the
 *                      normalised weights p_st, for small cases);
 *   ora_attn_ring   -- the same result reached the way the method reaches it:
 *                      the keys are cut into P equal contiguous chunks, the
 *                      query row in chunk i visits chunks j = (i - t) mod P for
 *                      t = 0..P-1 (its own chunk first, then the block received
 *                      from the ring predecessor), causal chunks j > i hold no
 *                      allowed key, and each chunk's (max, sum, accumulator)
 *                      triple is folded into the running triple;
 *   ora_attn_block  -- one ring step: a query block against one key/value
 *                      block at given global positions (the partial that the
 *                      fold combines);
 *   ora_merge       -- combination of normalised partial results (O_k, lse_k)
 *                      computed over disjoint key sets: the fold above written
 *                      in log-sum-exp form;
 *   ora_attn_bwd    -- gradients of out with respect to q, k and v for a given
 *   ora_attn_bwd_dq    output gradient (the pages describe no backward pass;
 *                      this is the derivative of the definition above, see
 *                      the comment at bwd_row).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int B, H, Hkv, S, D, P, causal;
    double scale;
    const int64_t *rows; /* flat ids (b*H + h)*S + s, or NULL for all rows */
    int64_t n_rows;
    double *out;         /* [n_rows, D] */
    double *lse;         /* [n_rows] */
    double *weights;     /* [n_rows, S] or NULL (direct mode only) */
    int mode;            /* 0 direct, 1 ring */
    int64_t begin, end;  /* row range of this worker */
} job_t;

static void row_coords(const job_t *J, int64_t r, int *b, int *h, int *s)
{
    int64_t id = J->rows ? J->rows[r] : r;
    *s = (int)(id % J->S);
    id /= J->S;
    *h = (int)(id % J->H);
    *b = (int)(id / J->H);
}

/* score x_t = scale * <q[b,s,h,:], k[b,t,g,:]> in fp64 */
static double score(const job_t *J, int b, int h, int g, int s, int t)
{
    const uint16_t *qr = J->q + (((int64_t)b * J->S + s) * J->H + h) * J->D;
    const uint16_t *kr = J->k + (((int64_t)b * J->S + t) * J->Hkv + g) * J->D;
    double acc = 0.0;
    for (int d = 0; d < J->D; ++d)
        acc += widen_bf16(qr[d]) * widen_bf16(kr[d]);
    return J->scale * acc;
}

static const uint16_t *vrow(const job_t *J, int b, int g, int t)
{
    return J->v + (((int64_t)b * J->S + t) * J->Hkv + g) * J->D;
}

/* two-pass definition over all allowed keys */
static void direct_row(const job_t *J, int64_t r, double *x)
{
    int b, h, s;
    row_coords(J, r, &b, &h, &s);
    int g = h / (J->H / J->Hkv);
    int n_allowed = J->causal ? s + 1 : J->S;

    double M = -INFINITY;
    for (int t = 0; t < n_allowed; ++t) {
        x[t] = score(J, b, h, g, s, t);
        if (x[t] > M)
            M = x[t];
    }
    double L = 0.0;
    for (int t = 0; t < n_allowed; ++t)
        L += exp(x[t] - M);

    double *o = J->out + r * J->D;
    for (int d = 0; d < J->D; ++d)
        o[d] = 0.0;
    for (int t = 0; t < n_allowed; ++t) {
        double w = exp(x[t] - M) / L;
        const uint16_t *vr = vrow(J, b, g, t);
        for (int d = 0; d < J->D; ++d)
            o[d] += w * widen_bf16(vr[d]);
        if (J->weights)
            J->weights[r * J->S + t] = w;
    }
    if (J->weights)
        for (int t = n_allowed; t < J->S; ++t)
            J->weights[r * J->S + t] = 0.0;
    J->lse[r] = M + log(L);
}

/* fold over chunks in ring order */
static void ring_row(const job_t *J, int64_t r, double *x, double *oc)
{
    int b, h, s;
    row_coords(J, r, &b, &h, &s);
    int g = h / (J->H / J->Hkv);
    int C = J->S / J->P;
    int i = s / C;

    double m = -INFINITY, l = 0.0;
    double *o = J->out + r * J->D;
    for (int d = 0; d < J->D; ++d)
        o[d] = 0.0;

    for (int step = 0; step < J->P; ++step) {
        int j = ((i - step) % J->P + J->P) % J->P;
        int t0 = j * C, t1 = t0 + C;
        if (J->causal && t1 > s + 1)
            t1 = s + 1; /* keys past the query row are not allowed */
        if (t1 <= t0)
            continue;   /* the chunk holds no allowed key */

        /* this chunk's own triple (m_c, l_c, o_c) */
        double mc = -INFINITY;
        for (int t = t0; t < t1; ++t) {
            x[t - t0] = score(J, b, h, g, s, t);
            if (x[t - t0] > mc)
                mc = x[t - t0];
        }
        double lc = 0.0;
        for (int d = 0; d < J->D; ++d)
            oc[d] = 0.0;
        for (int t = t0; t < t1; ++t) {
            double e = exp(x[t - t0] - mc);
            lc += e;
            const uint16_t *vr = vrow(J, b, g, t);
            for (int d = 0; d < J->D; ++d)
                oc[d] += e * widen_bf16(vr[d]);
        }

        /* fold it into the running triple */
        double mn = m > mc ? m : mc;
        double a = (m == -INFINITY) ? 0.0 : exp(m - mn);
        double c = exp(mc - mn);
        l = l * a + lc * c;
        for (int d = 0; d < J->D; ++d)
            o[d] = o[d] * a + oc[d] * c;
        m = mn;
    }
    for (int d = 0; d < J->D; ++d)
        o[d] /= l;
    J->lse[r] = m + log(l);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *x = (double *)malloc(sizeof(double) * (size_t)J->S);
    double *oc = (double *)malloc(sizeof(double) * (size_t)J->D);
    if (!x || !oc) {
        free(x);
        free(oc);
        return (void *)1;
    }
    for (int64_t r = J->begin; r < J->end; ++r) {
        if (J->mode == 0)
            direct_row(J, r, x);
        else
            ring_row(J, r, x, oc);
    }
    free(x);
    free(oc);
    return NULL;
}

int ora_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int check_args(int B, int H, int Hkv, int S, int D, int P)
{
    if (B <= 0 || H <= 0 || Hkv <= 0 || S <= 0 || D <= 0 || P <= 0)
        return -1;
    if (H % Hkv != 0 || S % P != 0)
        return -1;
    return 0;
}

static int run(job_t *base, int n_threads)
{
    if (n_threads <= 0)
        n_threads = ora_default_threads();
    if (n_threads > base->n_rows)
        n_threads = base->n_rows > 0 ? (int)base->n_rows : 1;
    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    int rc = 0;
    for (int w = 0; w < n_threads; ++w) {
        jobs[w] = *base;
        jobs[w].begin = base->n_rows * w / n_threads;
        jobs[w].end = base->n_rows * (w + 1) / n_threads;
        if (pthread_create(&th[w], NULL, worker, &jobs[w]) != 0) {
            for (int u = 0; u < w; ++u)
                pthread_join(th[u], NULL);
            free(jobs);
            free(th);
            return -2;
        }
    }
    for (int w = 0; w < n_threads; ++w) {
        void *ret = NULL;
        pthread_join(th[w], &ret);
        if (ret)
            rc = -2;
    }
    free(jobs);
    free(th);
    return rc;
}

int ora_attn_direct(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int B, int H, int Hkv, int S, int D, int causal, double scale,
                    const int64_t *rows, int64_t n_rows,
                    double *out, double *lse, double *weights, int n_threads)
{
    if (check_args(B, H, Hkv, S, D, 1))
        return -1;
    job_t J = {q, k, v, B, H, Hkv, S, D, 1, causal, scale,
               rows, rows ? n_rows : (int64_t)B * H * S,
               out, lse, weights, 0, 0, 0};
    return run(&J, n_threads);
}

int ora_attn_ring(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  int B, int H, int Hkv, int S, int D, int P, int causal, double scale,
                  const int64_t *rows, int64_t n_rows,
                  double *out, double *lse, int n_threads)
{
    if (check_args(B, H, Hkv, S, D, P))
        return -1;
    job_t J = {q, k, v, B, H, Hkv, S, D, P, causal, scale,
               rows, rows ? n_rows : (int64_t)B * H * S,
               out, lse, NULL, 1, 0, 0};
    return run(&J, n_threads);
}

/*
 * One ring step: attention of a query block against one key/value block at
 * given global positions.  q [B,Sq,H,D] holds global rows q_pos0..q_pos0+Sq-1,
 * k/v [B,Sk,Hkv,D] hold global rows k_pos0..k_pos0+Sk-1; causal keeps key
 * position <= query position.  out [B,Sq,H,D] = the softmax-weighted mean of
 * the allowed value rows of this block, lse [B,H,Sq] = ln of the sum of their
 * exp(scores); a row with no allowed key gets out = 0 and lse = -inf.  This
 * is the per-block partial that the ring fold (and ora_merge) combines.
 */
int ora_attn_block(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   int B, int H, int Hkv, int Sq, int Sk, int D,
                   long long q_pos0, long long k_pos0, int causal, double scale,
                   double *out, double *lse)
{
    if (B <= 0 || H <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || D <= 0 || H % Hkv != 0)
        return -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)Sk);
    if (!x)
        return -2;
    const int G = H / Hkv;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int s = 0; s < Sq; ++s) {
                const int g = h / G;
                const uint16_t *qr = q + (((int64_t)b * Sq + s) * H + h) * D;
                double *o = out + (((int64_t)b * Sq + s) * H + h) * D;
                double *l = lse + ((int64_t)b * H + h) * Sq + s;
                double M = -INFINITY;
                int any = 0;
                for (int t = 0; t < Sk; ++t) {
                    if (causal && k_pos0 + t > q_pos0 + s) {
                        x[t] = -INFINITY;
                        continue;
                    }
                    const uint16_t *kr = k + (((int64_t)b * Sk + t) * Hkv + g) * D;
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += widen_bf16(qr[d]) * widen_bf16(kr[d]);
                    x[t] = scale * acc;
                    if (x[t] > M)
                        M = x[t];
                    any = 1;
                }
                for (int d = 0; d < D; ++d)
                    o[d] = 0.0;
                if (!any) {
                    *l = -INFINITY;
                    continue;
                }
                double L = 0.0;
                for (int t = 0; t < Sk; ++t)
                    if (x[t] != -INFINITY)
                        L += exp(x[t] - M);
                for (int t = 0; t < Sk; ++t) {
                    if (x[t] == -INFINITY)
                        continue;
                    const double w = exp(x[t] - M) / L;
                    const uint16_t *vr = v + (((int64_t)b * Sk + t) * Hkv + g) * D;
                    for (int d = 0; d < D; ++d)
                        o[d] += w * widen_bf16(vr[d]);
                }
                *l = M + log(L);
            }
    free(x);
    return 0;
}

/*
 * Merge n normalised partials.  o_parts [n,B,S,H,D], lse_parts [n,B,H,S];
 * out [B,S,H,D], lse [B,H,S].  Each partial k holds O_k = (sum over its keys of
 * e^{x_t} v_t) / (sum over its keys of e^{x_t}) and lse_k = ln(sum e^{x_t});
 * the union over all keys is lse = ln sum_k e^{lse_k} and
 * O = sum_k e^{lse_k - lse} O_k.  A partial with lse_k = -inf holds no key and
 * adds nothing; when every partial is empty, out = 0 and lse = -inf.
 */
int ora_merge(const double *o_parts, const double *lse_parts, int n,
              int B, int H, int S, int D, double *out, double *lse)
{
    if (n <= 0 || B <= 0 || H <= 0 || S <= 0 || D <= 0)
        return -1;
    int64_t o_stride = (int64_t)B * S * H * D;
    int64_t l_stride = (int64_t)B * H * S;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int s = 0; s < S; ++s) {
                int64_t li = ((int64_t)b * H + h) * S + s;
                int64_t oi = (((int64_t)b * S + s) * H + h) * D;
                double M = -INFINITY;
                for (int p = 0; p < n; ++p)
                    if (lse_parts[p * l_stride + li] > M)
                        M = lse_parts[p * l_stride + li];
                if (M == -INFINITY) {
                    for (int d = 0; d < D; ++d)
                        out[oi + d] = 0.0;
                    lse[li] = -INFINITY;
                    continue;
                }
                double Z = 0.0;
                for (int p = 0; p < n; ++p)
                    Z += exp(lse_parts[p * l_stride + li] - M);
                double L = M + log(Z);
                for (int d = 0; d < D; ++d)
                    out[oi + d] = 0.0;
                for (int p = 0; p < n; ++p) {
                    double lp = lse_parts[p * l_stride + li];
                    if (lp == -INFINITY)
                        continue;
                    double w = exp(lp - L);
                    for (int d = 0; d < D; ++d)
                        out[oi + d] += w * o_parts[p * o_stride + oi + d];
                }
                lse[li] = L;
            }
    return 0;
}

/*
 * Backward pass: the derivative of the definition at the top of this file.
 * For the loss  sum_{b,s,h,d} out[b,s,h,d] * dout[b,s,h,d]  and one query row
 * (b, h, s) with KV head g, weights p_t = exp(x_t - M) / L over allowed t:
 *
 *   dp_t  = <dout[b,s,h,:], v[b,t,g,:]>            (d loss / d p_t)
 *   delta = sum_t p_t dp_t                        (= <dout, out> of the row)
 *   ds_t  = p_t (dp_t - delta)                    (softmax Jacobian applied)
 *   dq[b,s,h,:]  = scale * sum_t ds_t k[b,t,g,:]
 *   dk[b,t,g,:] += scale * ds_t q[b,s,h,:]        (summed over rows and over
 *   dv[b,t,g,:] += p_t dout[b,s,h,:]               the query heads of group g)
 *
 * Every step in fp64 on exactly widened bf16 inputs.
 *
 * delta can also be taken from a given forward output: when `out` (bf16,
 * [B,S,H,D], or one row per sampled query in the dq-rows mode) is passed,
 * delta = <dout[b,s,h,:], out[b,s,h,:]> on that output, which is how a
 * backward pass that receives the forward's stored (rounded) output defines
 * it.  With out == NULL delta is the exact sum above.
 */
typedef struct {
    const uint16_t *q, *k, *v, *dout;
    const uint16_t *out;        /* optional: [B,S,H,D] (full) or [n_rows,D] (dq rows) */
    int B, H, Hkv, S, D, causal;
    double scale;
    double *dq, *dk, *dv;       /* full mode: [B,S,H,D], [B,S,Hkv,D] x2 */
    const int64_t *rows;        /* dq-rows mode: flat ids (b*H + h)*S + s */
    int64_t begin, end;         /* range of (b,g) groups or of rows */
    int mode;                   /* 0: full gradients per (b,g), 1: dq rows */
} bjob_t;

/* one query row: dq row, and (when dk/dv are given) its share of dk, dv */
static void bwd_row(const bjob_t *J, int b, int h, int s, const uint16_t *outr, double *x,
                    double *dqr, double *dk, double *dv)
{
    const int D = J->D, g = h / (J->H / J->Hkv);
    const int n_allowed = J->causal ? s + 1 : J->S;
    const uint16_t *qr = J->q + (((int64_t)b * J->S + s) * J->H + h) * D;
    const uint16_t *dor = J->dout + (((int64_t)b * J->S + s) * J->H + h) * D;

    double M = -INFINITY;
    for (int t = 0; t < n_allowed; ++t) {
        const uint16_t *kr = J->k + (((int64_t)b * J->S + t) * J->Hkv + g) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += widen_bf16(qr[d]) * widen_bf16(kr[d]);
        x[t] = J->scale * acc;
        if (x[t] > M)
            M = x[t];
    }
    double L = 0.0;
    for (int t = 0; t < n_allowed; ++t)
        L += exp(x[t] - M);

    /* x[t] becomes p_t; dp kept in x[S + t] */
    double *dp = x + J->S;
    double delta = 0.0;
    for (int t = 0; t < n_allowed; ++t) {
        x[t] = exp(x[t] - M) / L;
        const uint16_t *vr = J->v + (((int64_t)b * J->S + t) * J->Hkv + g) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += widen_bf16(dor[d]) * widen_bf16(vr[d]);
        dp[t] = acc;
        delta += x[t] * acc;
    }
    if (outr) {  /* delta from the given forward output row instead */
        delta = 0.0;
        for (int d = 0; d < D; ++d)
            delta += widen_bf16(dor[d]) * widen_bf16(outr[d]);
    }
    for (int d = 0; d < D; ++d)
        dqr[d] = 0.0;
    for (int t = 0; t < n_allowed; ++t) {
        const double ds = x[t] * (dp[t] - delta);
        const int64_t kv = (((int64_t)b * J->S + t) * J->Hkv + g) * D;
        const uint16_t *kr = J->k + kv;
        for (int d = 0; d < D; ++d)
            dqr[d] += J->scale * ds * widen_bf16(kr[d]);
        if (dk) {
            for (int d = 0; d < D; ++d) {
                dk[kv + d] += J->scale * ds * widen_bf16(qr[d]);
                dv[kv + d] += x[t] * widen_bf16(dor[d]);
            }
        }
    }
}

static void *bwd_worker(void *arg)
{
    bjob_t *J = (bjob_t *)arg;
    double *x = (double *)malloc(sizeof(double) * 2 * (size_t)J->S);
    if (!x)
        return (void *)1;
    const int G = J->H / J->Hkv;
    for (int64_t w = J->begin; w < J->end; ++w) {
        if (J->mode == 0) {
            /* group (b, g): every row of its query heads; this worker owns
               dk/dv of the group, so the accumulation needs no lock */
            const int b = (int)(w / J->Hkv), g = (int)(w % J->Hkv);
            for (int hh = 0; hh < G; ++hh)
                for (int s = 0; s < J->S; ++s) {
                    const int h = g * G + hh;
                    const int64_t ri = (((int64_t)b * J->S + s) * J->H + h) * J->D;
                    bwd_row(J, b, h, s, J->out ? J->out + ri : NULL, x, J->dq + ri, J->dk, J->dv);
                }
        } else {
            int64_t id = J->rows[w];
            const int s = (int)(id % J->S);
            id /= J->S;
            const int h = (int)(id % J->H), b = (int)(id / J->H);
            bwd_row(J, b, h, s, J->out ? J->out + w * J->D : NULL, x, J->dq + w * J->D, NULL,
                    NULL);
        }
    }
    free(x);
    return NULL;
}

static int bwd_run(const bjob_t *base, int64_t n_units, int n_threads)
{
    if (n_threads <= 0)
        n_threads = ora_default_threads();
    if (n_threads > n_units)
        n_threads = n_units > 0 ? (int)n_units : 1;
    bjob_t *jobs = (bjob_t *)calloc((size_t)n_threads, sizeof(bjob_t));
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    int rc = 0, started = 0;
    for (int w = 0; w < n_threads; ++w) {
        jobs[w] = *base;
        jobs[w].begin = n_units * w / n_threads;
        jobs[w].end = n_units * (w + 1) / n_threads;
        if (pthread_create(&th[w], NULL, bwd_worker, &jobs[w]) != 0) {
            rc = -2;
            break;
        }
        ++started;
    }
    for (int w = 0; w < started; ++w) {
        void *ret = NULL;
        pthread_join(th[w], &ret);
        if (ret)
            rc = -2;
    }
    free(jobs);
    free(th);
    return rc;
}

/* Full gradients: dq [B,S,H,D], dk and dv [B,S,Hkv,D] (overwritten); out may
   be NULL (exact delta) or the forward output [B,S,H,D] that delta is taken from. */
int ora_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                 const uint16_t *out, int B, int H, int Hkv, int S, int D, int causal,
                 double scale, double *dq, double *dk, double *dv, int n_threads)
{
    if (check_args(B, H, Hkv, S, D, 1))
        return -1;
    const size_t nkv = (size_t)B * S * Hkv * D;
    memset(dk, 0, nkv * sizeof(double));
    memset(dv, 0, nkv * sizeof(double));
    bjob_t J = {q, k, v, dout, out, B, H, Hkv, S, D, causal, scale, dq, dk, dv, NULL, 0, 0, 0};
    return bwd_run(&J, (int64_t)B * Hkv, n_threads);
}

/* dq of selected query rows only: dq [n_rows, D] for flat ids (b*H + h)*S + s;
   out_rows may be NULL (exact delta) or the forward output rows [n_rows, D]. */
int ora_attn_bwd_dq(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                    const uint16_t *out_rows, int B, int H, int Hkv, int S, int D, int causal,
                    double scale, const int64_t *rows, int64_t n_rows, double *dq, int n_threads)
{
    if (check_args(B, H, Hkv, S, D, 1) || !rows || n_rows <= 0)
        return -1;
    bjob_t J = {q, k, v, dout, out_rows, B, H, Hkv, S, D, causal, scale, dq, NULL, NULL,
                rows, 0, 0, 1};
    return bwd_run(&J, n_rows, n_threads);
}
