/*
 * zg_oracle.c -- plain fp64 CPU oracle for the ZGCM-1 attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA library and includes nothing from it.
 *
 * What it computes (sources, by page title and section):
 *   - "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ"
 *     (architecture): 27 of 32 layers are gated sliding-window attention over
 *     the most recent 128 tokens, 5 layers are global (full causal) attention;
 *     GatedSWA(h) = o_proj(A_SWA(q,k,v) ⊙ σ(g_proj(h))); q and k get QK
 *     RMSNorm and partial RoPE with rotary ratio 0.33; global layers are not
 *     gated.  KV cache: SWA layers keep a fixed 128 tokens, global layers keep
 *     the whole sequence.
 *   - "ZGCM-1: A Fully Open and Extremely Efficient Foundation Model for Math
 *     and Agentic Search" (jaehun.me review), section "게이트형 SWA의 동작"
 *     (how gated SWA works): a window of W tokens includes the query token
 *     itself; the gate multiplies the attention output element-wise.
 *   - hyper.ai summary (papers/2609.13356), section "方法" (method), the
 *     GatedSWA equation.
 *
 * Everything is evaluated in double precision straight from the definition:
 *   1. qh = RoPE_r(RMSNorm(q; w_q, eps), pos),  kh likewise with w_k
 *   2. s_j = <qh, kh_j> / sqrt(d) for j in J(i)
 *        SWA:    J(i) = { max(0, i-W+1) .. i }   (sequence index, self included)
 *        global: J(i) = { 0 .. i }
 *   3. p_j = exp(s_j - max s) / sum,  A = sum_j p_j v_j
 *   4. out = A * sigmoid(gate) (SWA)   or   out = A (global)
 *
 * Readings taken where the pages are silent (the same readings are stated in
 * the design notes of the repository):
 *   - RMSNorm: x * (mean_d(x^2) + eps)^(-1/2) * w, over one head's d values,
 *     weights [d] shared by all heads, separate for q and k.
 *   - RMSNorm before RoPE.
 *   - RoPE acts on dims [0, r) with rotate-half pairing (j, j + r/2) and angle
 *     pos * theta^(-2j/r); dims [r, d) pass through unchanged.
 *   - softmax scale 1/sqrt(d); sigmoid(x) = 1 / (1 + exp(-x)).
 *   - GQA: query head h reads KV head floor(h * Hkv / Hq).
 *   - decode caches hold post-norm post-RoPE keys and raw values; a global
 *     cache keeps position t in slot t, a ring keeps position t in slot t mod W.
 *
 * Inputs arrive as bf16 bit patterns (converted exactly to double), float32
 * or float64, chosen per call; outputs are double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element types an input array may hold */
enum { ZGO_BF16 = 0, ZGO_F64 = 1, ZGO_F32 = 2 };

typedef struct {
    const void *p;
    int dt;
} zgo_arr;

static double zgo_ld(zgo_arr a, size_t i)
{
    if (a.dt == ZGO_F64) return ((const double *)a.p)[i];
    if (a.dt == ZGO_F32) return (double)((const float *)a.p)[i];
    uint32_t u = (uint32_t)((const uint16_t *)a.p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- elementary steps (exported so the tests can pin them one by one) ---- */

/* y = x * (mean(x^2) + eps)^(-1/2) * w   over d values */
void zgo_rmsnorm(const double *x, const double *w, int d, double eps, double *y)
{
    double ss = 0.0;
    for (int t = 0; t < d; ++t) ss += x[t] * x[t];
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int t = 0; t < d; ++t) y[t] = x[t] * inv * w[t];
}

/* in-place partial RoPE on dims [0, r): pairs (j, j + r/2), angle pos*theta^(-2j/r) */
void zgo_rope(double *x, int r, double pos, double theta)
{
    int half = r / 2;
    for (int j = 0; j < half; ++j) {
        double freq = pow(theta, -2.0 * (double)j / (double)r);
        double ang = pos * freq;
        double c = cos(ang), s = sin(ang);
        double a = x[j], b = x[j + half];
        x[j] = a * c - b * s;
        x[j + half] = b * c + a * s;
    }
}

double zgo_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* softmax-weighted sum of nk value rows for one query:
 *   s_j = <qh, keys[j]> * scale ; out = sum_j softmax(s)_j * vals[j]
 * keys / vals are arrays of row pointers of length d. */
static void zgo_attend(const double *qh, const double *const *keys, const double *const *vals,
                       int nk, int d, double scale, double *s_buf, double *out)
{
    double m = -INFINITY;
    for (int j = 0; j < nk; ++j) {
        double s = 0.0;
        for (int t = 0; t < d; ++t) s += qh[t] * keys[j][t];
        s *= scale;
        s_buf[j] = s;
        if (s > m) m = s;
    }
    for (int t = 0; t < d; ++t) out[t] = 0.0;
    double l = 0.0;
    for (int j = 0; j < nk; ++j) {
        double p = exp(s_buf[j] - m);
        l += p;
        for (int t = 0; t < d; ++t) out[t] += p * vals[j][t];
    }
    for (int t = 0; t < d; ++t) out[t] /= l;
}

/* normalised + rotated copy of one head vector */
static void zgo_qk_transform(zgo_arr src, size_t off, const double *w, int d, int r,
                             double pos, double theta, double eps, double *tmp, double *dst)
{
    for (int t = 0; t < d; ++t) tmp[t] = zgo_ld(src, off + (size_t)t);
    zgo_rmsnorm(tmp, w, d, eps, dst);
    zgo_rope(dst, r, pos, theta);
}

/* ------------------------------- prefill --------------------------------- */

typedef struct {
    zgo_arr q, k, v, gate; /* gate.p == NULL: ungated */
    const int32_t *pos;
    const double *wq, *wk;
    int B, L, Hq, Hkv, d, window, r;
    double theta, eps;
    const int64_t *rows;
    int64_t nrows;
    double *out;
    /* global mode: per-batch precomputed kh and v as double [L][Hkv][d] (NULL where unused) */
    double **kh_all, **v_all;
    int64_t *kh_len;
    /* work split */
    int nthreads;
    int tid;
} zgo_prefill_job;

static void *zgo_prefill_worker(void *arg)
{
    zgo_prefill_job *J = (zgo_prefill_job *)arg;
    const int d = J->d, Hq = J->Hq, Hkv = J->Hkv, L = J->L;
    const int global = (J->window <= 0 || J->window >= L);
    const int W = global ? L : J->window;
    const double scale = 1.0 / sqrt((double)d);

    double *tmp = malloc(sizeof(double) * (size_t)d);
    double *qh = malloc(sizeof(double) * (size_t)d);
    double *acc = malloc(sizeof(double) * (size_t)d);
    double *s_buf = malloc(sizeof(double) * (size_t)(global ? L : W));
    const double **keys = malloc(sizeof(double *) * (size_t)(global ? L : W));
    const double **vals = malloc(sizeof(double *) * (size_t)(global ? L : W));
    /* SWA mode: keys/values of the window, for every KV head */
    double *kwin = global ? NULL : malloc(sizeof(double) * (size_t)W * (size_t)Hkv * (size_t)d);
    double *vwin = global ? NULL : malloc(sizeof(double) * (size_t)W * (size_t)Hkv * (size_t)d);

    for (int64_t n = J->tid; n < J->nrows; n += J->nthreads) {
        int64_t flat = J->rows[n];
        int b = (int)(flat / L), i = (int)(flat % L);
        int j0 = global ? 0 : (i - W + 1 > 0 ? i - W + 1 : 0);
        int nk = i - j0 + 1;
        /* values of the key range, all KV heads (global mode: precomputed) */
        for (int j = 0; j < (global ? 0 : nk); ++j)
            for (int g = 0; g < Hkv; ++g) {
                size_t off = (((size_t)b * L + (size_t)(j0 + j)) * Hkv + (size_t)g) * (size_t)d;
                for (int t = 0; t < d; ++t)
                    vwin[((size_t)j * Hkv + g) * d + t] = zgo_ld(J->v, off + (size_t)t);
            }
        if (!global) {
            for (int j = 0; j < nk; ++j) {
                int jj = j0 + j;
                double kp = (double)J->pos[(size_t)b * L + (size_t)jj];
                for (int g = 0; g < Hkv; ++g) {
                    size_t off = (((size_t)b * L + (size_t)jj) * Hkv + (size_t)g) * (size_t)d;
                    zgo_qk_transform(J->k, off, J->wk, d, J->r, kp, J->theta, J->eps, tmp,
                                     kwin + ((size_t)j * Hkv + g) * d);
                }
            }
        }
        double qp = (double)J->pos[(size_t)b * L + (size_t)i];
        for (int h = 0; h < Hq; ++h) {
            int g = (int)(((int64_t)h * Hkv) / Hq);
            size_t qoff = (((size_t)b * L + (size_t)i) * Hq + (size_t)h) * (size_t)d;
            zgo_qk_transform(J->q, qoff, J->wq, d, J->r, qp, J->theta, J->eps, tmp, qh);
            for (int j = 0; j < nk; ++j) {
                if (global) {
                    keys[j] = J->kh_all[b] + ((size_t)(j0 + j) * Hkv + g) * d;
                    vals[j] = J->v_all[b] + ((size_t)(j0 + j) * Hkv + g) * d;
                } else {
                    keys[j] = kwin + ((size_t)j * Hkv + g) * d;
                    vals[j] = vwin + ((size_t)j * Hkv + g) * d;
                }
            }
            zgo_attend(qh, keys, vals, nk, d, scale, s_buf, acc);
            double *o = J->out + ((size_t)n * Hq + (size_t)h) * (size_t)d;
            for (int t = 0; t < d; ++t) {
                double gt = 1.0;
                if (J->gate.p) gt = zgo_sigmoid(zgo_ld(J->gate, qoff + (size_t)t));
                o[t] = acc[t] * gt;
            }
        }
    }
    free(tmp); free(qh); free(acc); free(s_buf); free(keys); free(vals); free(kwin); free(vwin);
    return NULL;
}

typedef struct {
    zgo_arr k, v;
    const int32_t *pos;
    const double *wk;
    int L, Hkv, d, r, b;
    double theta, eps;
    int64_t len;
    double *dst, *vdst;
    int nthreads, tid;
} zgo_khat_job;

static void *zgo_khat_worker(void *arg)
{
    zgo_khat_job *J = (zgo_khat_job *)arg;
    double *tmp = malloc(sizeof(double) * (size_t)J->d);
    for (int64_t j = J->tid; j < J->len; j += J->nthreads) {
        double kp = (double)J->pos[(size_t)J->b * J->L + (size_t)j];
        for (int g = 0; g < J->Hkv; ++g) {
            size_t off = (((size_t)J->b * J->L + (size_t)j) * J->Hkv + (size_t)g) * (size_t)J->d;
            zgo_qk_transform(J->k, off, J->wk, J->d, J->r, kp, J->theta, J->eps, tmp,
                             J->dst + ((size_t)j * J->Hkv + g) * J->d);
            for (int t = 0; t < J->d; ++t)
                J->vdst[((size_t)j * J->Hkv + g) * J->d + t] = zgo_ld(J->v, off + (size_t)t);
        }
    }
    free(tmp);
    return NULL;
}

static int zgo_run(void *(*fn)(void *), void *jobs, size_t job_size, int nthreads)
{
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
    int rc = 0;
    for (int t = 0; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, fn, (char *)jobs + (size_t)t * job_size)) rc = -1;
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    return rc;
}

/*
 * Prefill output for a list of query rows (flattened b*L + i), every query head.
 *   q, gate [B,L,Hq,d]; k, v [B,L,Hkv,d]; pos [B,L]; wq, wk [d] (float32)
 *   window <= 0 or >= L selects global (full causal) attention, else a causal
 *   window of `window` tokens, self included.  gate == NULL: no gate.
 *   out [nrows, Hq, d] double.  Returns 0, or -1 on a bad argument.
 */
int zgo_prefill_rows(const void *q, const void *k, const void *v, const void *gate, int dt,
                     const int32_t *pos, const float *wq, const float *wk,
                     int B, int L, int Hq, int Hkv, int d, int window, int rotary_dim,
                     double theta, double eps, const int64_t *rows, int64_t nrows,
                     double *out, int nthreads)
{
    if (!q || !k || !v || !pos || !wq || !wk || !rows || !out) return -1;
    if (B <= 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv) return -1;
    if (rotary_dim < 0 || rotary_dim > d || rotary_dim % 2) return -1;
    if (nthreads < 1) nthreads = 1;
    for (int64_t n = 0; n < nrows; ++n)
        if (rows[n] < 0 || rows[n] >= (int64_t)B * L) return -1;

    double *wqd = malloc(sizeof(double) * (size_t)d), *wkd = malloc(sizeof(double) * (size_t)d);
    for (int t = 0; t < d; ++t) { wqd[t] = wq[t]; wkd[t] = wk[t]; }
    const int global = (window <= 0 || window >= L);

    double **kh_all = calloc((size_t)B, sizeof(double *));
    double **v_all = calloc((size_t)B, sizeof(double *));
    int64_t *kh_len = calloc((size_t)B, sizeof(int64_t));
    if (global) {
        /* keys 0 .. max requested row of each batch, transformed once */
        for (int64_t n = 0; n < nrows; ++n) {
            int b = (int)(rows[n] / L);
            int64_t need = rows[n] % L + 1;
            if (need > kh_len[b]) kh_len[b] = need;
        }
        for (int b = 0; b < B; ++b) {
            if (!kh_len[b]) continue;
            kh_all[b] = malloc(sizeof(double) * (size_t)kh_len[b] * (size_t)Hkv * (size_t)d);
            v_all[b] = malloc(sizeof(double) * (size_t)kh_len[b] * (size_t)Hkv * (size_t)d);
            if (!kh_all[b] || !v_all[b]) return -2;
            zgo_khat_job *kj = calloc((size_t)nthreads, sizeof(zgo_khat_job));
            for (int t = 0; t < nthreads; ++t) {
                zgo_khat_job x = {{k, dt}, {v, dt}, pos, wkd, L, Hkv, d, rotary_dim, b, theta, eps,
                                  kh_len[b], kh_all[b], v_all[b], nthreads, t};
                kj[t] = x;
            }
            zgo_run(zgo_khat_worker, kj, sizeof(zgo_khat_job), nthreads);
            free(kj);
        }
    }
    zgo_prefill_job *jobs = calloc((size_t)nthreads, sizeof(zgo_prefill_job));
    for (int t = 0; t < nthreads; ++t) {
        zgo_prefill_job x = {{q, dt}, {k, dt}, {v, dt}, {gate, dt}, pos, wqd, wkd,
                             B, L, Hq, Hkv, d, window, rotary_dim, theta, eps,
                             rows, nrows, out, kh_all, v_all, kh_len, nthreads, t};
        jobs[t] = x;
    }
    int rc = zgo_run(zgo_prefill_worker, jobs, sizeof(zgo_prefill_job), nthreads);
    free(jobs);
    for (int b = 0; b < B; ++b) { free(kh_all[b]); free(v_all[b]); }
    free(kh_all); free(v_all); free(kh_len); free(wqd); free(wkd);
    return rc;
}

/* -------------------------------- decode --------------------------------- */

typedef struct {
    zgo_arr q, kn, vn, gate, kg, vg, kr, vr;
    const float *wq, *wk;
    const uint8_t *is_global;
    const int *gidx, *sidx;
    int NL, Hq, Hkv, d, W, r, p;
    int64_t S;
    double theta, eps;
    double *out, *khat_new;
    int nthreads, tid;
} zgo_decode_job;

static void *zgo_decode_worker(void *arg)
{
    zgo_decode_job *J = (zgo_decode_job *)arg;
    const int d = J->d, Hq = J->Hq, Hkv = J->Hkv, p = J->p;
    const double scale = 1.0 / sqrt((double)d);
    const int64_t maxk = (int64_t)p + 1;
    double *tmp = malloc(sizeof(double) * (size_t)d), *w = malloc(sizeof(double) * (size_t)d);
    double *qh = malloc(sizeof(double) * (size_t)d), *acc = malloc(sizeof(double) * (size_t)d);
    double *kh = malloc(sizeof(double) * (size_t)d), *vnew = malloc(sizeof(double) * (size_t)d);
    double *s_buf = malloc(sizeof(double) * (size_t)maxk);
    const double **keys = malloc(sizeof(double *) * (size_t)maxk);
    const double **vals = malloc(sizeof(double *) * (size_t)maxk);
    double *kbuf = malloc(sizeof(double) * (size_t)maxk * (size_t)d);
    double *vbuf = malloc(sizeof(double) * (size_t)maxk * (size_t)d);

    /* one work item = (layer, kv head) */
    for (int item = J->tid; item < J->NL * Hkv; item += J->nthreads) {
        int l = item / Hkv, g = item % Hkv;
        int glob = J->is_global[l] != 0;
        /* the new token's key: normalised and rotated at position p */
        for (int t = 0; t < d; ++t) w[t] = J->wk[(size_t)l * d + t];
        zgo_qk_transform(J->kn, ((size_t)l * Hkv + g) * d, w, d, J->r, (double)p, J->theta,
                         J->eps, tmp, kh);
        for (int t = 0; t < d; ++t) {
            J->khat_new[((size_t)l * Hkv + g) * d + t] = kh[t];
            vnew[t] = zgo_ld(J->vn, ((size_t)l * Hkv + g) * d + (size_t)t);
        }
        /* key set: positions first..p, position p is the new token */
        int64_t first = glob ? 0 : ((int64_t)p - J->W + 1 > 0 ? (int64_t)p - J->W + 1 : 0);
        int nk = (int)(maxk - first);
        for (int j = 0; j < nk; ++j) {
            int64_t t_pos = first + j;
            if (t_pos == p) {
                keys[j] = kh;
                vals[j] = vnew;
                continue;
            }
            size_t off;
            zgo_arr ka, va;
            if (glob) {
                off = (((size_t)J->gidx[l] * Hkv + g) * (size_t)J->S + (size_t)t_pos) * d;
                ka = J->kg; va = J->vg;
            } else {
                off = (((size_t)J->sidx[l] * Hkv + g) * (size_t)J->W + (size_t)(t_pos % J->W)) * d;
                ka = J->kr; va = J->vr;
            }
            for (int t = 0; t < d; ++t) {
                kbuf[(size_t)j * d + t] = zgo_ld(ka, off + (size_t)t);
                vbuf[(size_t)j * d + t] = zgo_ld(va, off + (size_t)t);
            }
            keys[j] = kbuf + (size_t)j * d;
            vals[j] = vbuf + (size_t)j * d;
        }
        for (int t = 0; t < d; ++t) w[t] = J->wq[(size_t)l * d + t];
        for (int h = 0; h < Hq; ++h) {
            if ((int)(((int64_t)h * Hkv) / Hq) != g) continue;
            size_t qoff = ((size_t)l * Hq + h) * d;
            zgo_qk_transform(J->q, qoff, w, d, J->r, (double)p, J->theta, J->eps, tmp, qh);
            zgo_attend(qh, keys, vals, nk, d, scale, s_buf, acc);
            double *o = J->out + qoff;
            for (int t = 0; t < d; ++t)
                o[t] = glob ? acc[t] : acc[t] * zgo_sigmoid(zgo_ld(J->gate, qoff + (size_t)t));
        }
    }
    free(tmp); free(w); free(qh); free(acc); free(kh); free(vnew); free(s_buf);
    free(keys); free(vals); free(kbuf); free(vbuf);
    return NULL;
}

/*
 * One decode step of one sequence through an NL-layer hybrid stack.
 *   q, gate [NL,Hq,d]; k_new, v_new [NL,Hkv,d]; wq, wk [NL,d] float32
 *   is_global [NL]; global layers are numbered in order of appearance into
 *   k_glob, v_glob [NG,Hkv,S,d], SWA layers into k_ring, v_ring [NS,Hkv,W,d].
 *   The caches are read as they are before the step (the slot of position p
 *   is replaced by the new token).  p < S.
 *   out [NL,Hq,d] and khat_new [NL,Hkv,d] (key written into the cache), double.
 */
int zgo_decode_seq(const void *q, const void *k_new, const void *v_new, const void *gate, int dt,
                   const float *wq, const float *wk, const uint8_t *is_global,
                   const void *k_glob, const void *v_glob, const void *k_ring, const void *v_ring,
                   int cache_dt, int NL, int Hq, int Hkv, int d, int64_t S, int W, int rotary_dim,
                   double theta, double eps, int p, double *out, double *khat_new, int nthreads)
{
    if (!q || !k_new || !v_new || !gate || !wq || !wk || !is_global || !out || !khat_new) return -1;
    if (NL <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || W <= 0 || p < 0 || p >= S) return -1;
    if (rotary_dim < 0 || rotary_dim > d || rotary_dim % 2) return -1;
    if (nthreads < 1) nthreads = 1;
    int *gidx = malloc(sizeof(int) * (size_t)NL), *sidx = malloc(sizeof(int) * (size_t)NL);
    int ng = 0, ns = 0;
    for (int l = 0; l < NL; ++l) {
        gidx[l] = is_global[l] ? ng++ : -1;
        sidx[l] = is_global[l] ? -1 : ns++;
    }
    if ((ng && (!k_glob || !v_glob)) || (ns && (!k_ring || !v_ring))) {
        free(gidx); free(sidx);
        return -1;
    }
    zgo_decode_job *jobs = calloc((size_t)nthreads, sizeof(zgo_decode_job));
    for (int t = 0; t < nthreads; ++t) {
        zgo_decode_job x = {{q, dt}, {k_new, dt}, {v_new, dt}, {gate, dt},
                            {k_glob, cache_dt}, {v_glob, cache_dt}, {k_ring, cache_dt}, {v_ring, cache_dt},
                            wq, wk, is_global, gidx, sidx, NL, Hq, Hkv, d, W, rotary_dim, p, S,
                            theta, eps, out, khat_new, nthreads, t};
        jobs[t] = x;
    }
    int rc = zgo_run(zgo_decode_worker, jobs, sizeof(zgo_decode_job), nthreads);
    free(jobs); free(gidx); free(sidx);
    return rc;
}
