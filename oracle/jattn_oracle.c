/*
 * jattn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU reference for jagged attention, forward and backward.
 * Only the tests, the smoke check and the bench's CPU-baseline leg may call it;
 * the library's CUDA path never links or calls it, and this file shares no
 * header, helper or constant with that path.
 *
 * What it computes ("Training GEM at LLM scale", section "Jagged Sequence Flash
 * Attention": attention directly on variable-length jagged tensors, with custom
 * attention biases, asymmetric query/key-value lengths and a backward pass;
 * section "Generalized Dot-Product Attention (GDPA)": two matmuls with a
 * pointwise GELU or SiLU in place of softmax; section "BlockAttention": each
 * 64-token query block attends only to its own key/value block):
 *
 *   for every sequence b and head h, local rows i < Lq_b, keys j < Lk_b,
 *     s_ij   = scale * <q_i, k_j> + T[h, min(|i - j|, NB - 1)]   (bias optional, not scaled)
 *     softmax:  P_ij = exp(s_ij - m_i) / l_i,  m_i = max_j s_ij,  l_i = sum_j exp(s_ij - m_i)
 *               O_i = sum_j P_ij v_j,          lse_i = m_i + ln l_i
 *     act:      O_i = sum_j act(s_ij) v_j      (SiLU or tanh-GELU, no normalisation)
 *     block:    j restricted to the 64-block of i (floor(j/64) == floor(i/64))
 *     window W: j restricted to |i - j| < W (sliding-window attention, section
 *               "BlockAttention": each token attends only to nearby events;
 *               the band is symmetric, like the relative-position bias)
 *
 *   backward (chain rule of the above):
 *     dP_ij = <dO_i, v_j>
 *     softmax: dS_ij = P_ij (dP_ij - Delta_i),  Delta_i = <dO_i, O_i>  (fp64 O)
 *     act:     dS_ij = act'(s_ij) dP_ij
 *     dq_i = scale * sum_j dS_ij k_j ; dk_j = scale * sum_i dS_ij q_i
 *     dv_j = sum_i P_ij dO_i   (act: act(s_ij)) ; dT[h, bucket(i,j)] += dS_ij
 *
 * Layout: q/out/dout/dq are [Tq, H, D] and k/v/dk/dv are [Tk, H, D], row-major,
 * token-major, all float64; offsets are int32 exclusive prefix sums of length
 * B + 1; the bias table is [H, NB]; lse is [H, Tq].
 *
 * Readings where the pages are silent: the layout above; positions i, j are
 * local to the sequence (also in cross-attention); a sequence with Lk = 0 gives
 * O_i = 0 and lse_i = -inf; blocks start at local position 0 and the last one
 * is partial; no causal mask.
 *
 * Work is split over (b, h) pairs with plain POSIX threads; every (b, h) pair
 * owns its output rows, and the bias-gradient partials are summed in pair order,
 * so the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ACT_SOFTMAX = 0, ACT_SILU = 1, ACT_GELU_TANH = 2 };

typedef struct {
    int act, block, window, B, H, D, nb;
    const int32_t *q_off, *kv_off;
    const double *q, *k, *v, *bias, *dout;
    double scale;
    double *out, *lse;                 /* forward outputs */
    double *dq, *dk, *dv, *dbias_part; /* backward outputs; dbias_part is [B*H, nb] */
    int backward;
    long next;                         /* shared task counter */
    int err;
} job_t;

/* SiLU(x) = x * sigmoid(x) */
static double silu(double x) { return x / (1.0 + exp(-x)); }
static double silu_grad(double x) {
    double sg = 1.0 / (1.0 + exp(-x));
    return sg * (1.0 + x * (1.0 - sg));
}

/* tanh-GELU (Hendrycks & Gimpel): 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
static const double GELU_A = 0.044715;
static double gelu_c(void) { return sqrt(2.0 / M_PI); }
static double gelu_tanh(double x) {
    double u = gelu_c() * (x + GELU_A * x * x * x);
    return 0.5 * x * (1.0 + tanh(u));
}
static double gelu_tanh_grad(double x) {
    double c = gelu_c();
    double t = tanh(c * (x + GELU_A * x * x * x));
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * c * (1.0 + 3.0 * GELU_A * x * x);
}

static double act_f(int act, double x) { return act == ACT_SILU ? silu(x) : gelu_tanh(x); }
static double act_g(int act, double x) { return act == ACT_SILU ? silu_grad(x) : gelu_tanh_grad(x); }

static double dot(const double *a, const double *b, int n) {
    double s = 0.0;
    for (int d = 0; d < n; ++d) s += a[d] * b[d];
    return s;
}

static int bucket(const job_t *J, int i, int j) {
    int r = i > j ? i - j : j - i;
    return r < J->nb - 1 ? r : J->nb - 1;
}

/* allowed key range [*j0, *j1) for local query row i */
static void key_range(const job_t *J, int i, int Lk, int *j0, int *j1) {
    if (J->block > 0) {
        int blk = i / J->block;
        *j0 = blk * J->block;
        *j1 = (blk + 1) * J->block < Lk ? (blk + 1) * J->block : Lk;
        if (*j0 > Lk) *j0 = Lk;
    } else if (J->window > 0) {
        int lo = i - J->window + 1, hi = i + J->window; /* |i - j| < W */
        *j0 = lo > 0 ? lo : 0;
        *j1 = hi < Lk ? hi : Lk;
        if (*j0 > *j1) *j0 = *j1;
    } else {
        *j0 = 0;
        *j1 = Lk;
    }
}

/* one (b, h) pair; s, p are scratch rows of length >= Lk */
static void pair_task(job_t *J, int b, int h, double *s, double *p, double *orow) {
    const int H = J->H, D = J->D, rs = H * D;
    const int q0 = J->q_off[b], Lq = J->q_off[b + 1] - q0;
    const int k0 = J->kv_off[b], Lk = J->kv_off[b + 1] - k0;
    double *dbp = J->dbias_part ? J->dbias_part + ((long)b * H + h) * J->nb : NULL;

    for (int i = 0; i < Lq; ++i) {
        const double *qi = J->q + (long)(q0 + i) * rs + h * D;
        int j0, j1;
        key_range(J, i, Lk, &j0, &j1);
        /* scores */
        for (int j = j0; j < j1; ++j) {
            const double *kj = J->k + (long)(k0 + j) * rs + h * D;
            s[j] = J->scale * dot(qi, kj, D);
            if (J->bias) s[j] += J->bias[h * J->nb + bucket(J, i, j)];
        }
        /* probabilities (softmax) or activations */
        double lse_i = -INFINITY;
        if (J->act == ACT_SOFTMAX) {
            if (j1 > j0) {
                double m = -INFINITY, l = 0.0;
                for (int j = j0; j < j1; ++j) m = s[j] > m ? s[j] : m;
                for (int j = j0; j < j1; ++j) { p[j] = exp(s[j] - m); l += p[j]; }
                for (int j = j0; j < j1; ++j) p[j] /= l;
                lse_i = m + log(l);
            }
        } else {
            for (int j = j0; j < j1; ++j) p[j] = act_f(J->act, s[j]);
        }
        /* O_i */
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        for (int j = j0; j < j1; ++j) {
            const double *vj = J->v + (long)(k0 + j) * rs + h * D;
            for (int d = 0; d < D; ++d) orow[d] += p[j] * vj[d];
        }
        if (!J->backward) {
            double *oi = J->out + (long)(q0 + i) * rs + h * D;
            memcpy(oi, orow, sizeof(double) * D);
            if (J->lse) J->lse[(long)h * J->q_off[J->B] + q0 + i] = lse_i;
            continue;
        }
        /* backward for row i */
        const double *doi = J->dout + (long)(q0 + i) * rs + h * D;
        double delta = dot(doi, orow, D);
        double *dqi = J->dq + (long)(q0 + i) * rs + h * D;
        for (int j = j0; j < j1; ++j) {
            const double *kj = J->k + (long)(k0 + j) * rs + h * D;
            const double *vj = J->v + (long)(k0 + j) * rs + h * D;
            double *dkj = J->dk + (long)(k0 + j) * rs + h * D;
            double *dvj = J->dv + (long)(k0 + j) * rs + h * D;
            double dp = dot(doi, vj, D);
            double ds = J->act == ACT_SOFTMAX ? p[j] * (dp - delta) : act_g(J->act, s[j]) * dp;
            for (int d = 0; d < D; ++d) {
                dqi[d] += J->scale * ds * kj[d];
                dkj[d] += J->scale * ds * qi[d];
                dvj[d] += p[j] * doi[d];
            }
            if (dbp) dbp[bucket(J, i, j)] += ds;
        }
    }
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    int maxL = 1;
    for (int b = 0; b < J->B; ++b) {
        int lk = J->kv_off[b + 1] - J->kv_off[b];
        if (lk > maxL) maxL = lk;
    }
    double *s = (double *)malloc(sizeof(double) * maxL);
    double *p = (double *)malloc(sizeof(double) * maxL);
    double *o = (double *)malloc(sizeof(double) * J->D);
    if (!s || !p || !o) {
        __atomic_store_n(&J->err, 1, __ATOMIC_SEQ_CST);
        free(s); free(p); free(o);
        return NULL;
    }
    const long ntask = (long)J->B * J->H;
    for (;;) {
        long t = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (t >= ntask) break;
        pair_task(J, (int)(t / J->H), (int)(t % J->H), s, p, o);
    }
    free(s); free(p); free(o);
    return NULL;
}

static int run(job_t *J, int nthreads) {
    if (J->window < 0 || (J->window > 0 && J->block > 0)) return 4;
    for (int b = 0; b < J->B; ++b) {
        if (J->q_off[b + 1] < J->q_off[b] || J->kv_off[b + 1] < J->kv_off[b]) return 2;
        if (J->block > 0 && (J->q_off[b + 1] - J->q_off[b]) != (J->kv_off[b + 1] - J->kv_off[b])) return 3;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    J->next = 0;
    J->err = 0;
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[started], NULL, worker, J) == 0) ++started;
    }
    worker(J);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    return J->err;
}

int jattn_oracle_fwd(int act, int block, int window, int B, int H, int D, const int32_t *q_off,
                     const int32_t *kv_off, const double *q, const double *k, const double *v, const double *bias,
                     int nb, double scale, double *out, double *lse, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof(J));
    J.act = act; J.block = block; J.window = window; J.B = B; J.H = H; J.D = D; J.nb = bias ? nb : 1;
    J.q_off = q_off; J.kv_off = kv_off; J.q = q; J.k = k; J.v = v; J.bias = bias;
    J.scale = scale; J.out = out; J.lse = lse; J.backward = 0;
    return run(&J, nthreads);
}

/* dq, dk, dv must be zero-filled by the caller; dbias (if given) is [H, nb]. */
int jattn_oracle_bwd(int act, int block, int window, int B, int H, int D, const int32_t *q_off,
                     const int32_t *kv_off, const double *q, const double *k, const double *v, const double *bias,
                     int nb, double scale, const double *dout, double *dq, double *dk, double *dv, double *dbias,
                     int nthreads) {
    job_t J;
    memset(&J, 0, sizeof(J));
    J.act = act; J.block = block; J.window = window; J.B = B; J.H = H; J.D = D; J.nb = bias ? nb : 1;
    J.q_off = q_off; J.kv_off = kv_off; J.q = q; J.k = k; J.v = v; J.bias = bias;
    J.scale = scale; J.dout = dout; J.dq = dq; J.dk = dk; J.dv = dv; J.backward = 1;
    double *part = NULL;
    if (dbias && bias) {
        part = (double *)calloc((size_t)B * H * nb, sizeof(double));
        if (!part) return 1;
        J.dbias_part = part;
    }
    int rc = run(&J, nthreads);
    if (part) {
        for (int h = 0; h < H; ++h)
            for (int n = 0; n < nb; ++n) dbias[h * nb + n] = 0.0;
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h)
                for (int n = 0; n < nb; ++n) dbias[h * nb + n] += part[((long)b * H + h) * nb + n];
        free(part);
    }
    return rc;
}

/* Pointwise activations, exported so tests can pin them against library routines. */
double jattn_oracle_act(int act, double x) { return act_f(act, x); }
double jattn_oracle_act_grad(int act, double x) { return act_g(act, x); }
