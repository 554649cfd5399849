/*
 * kda_oracle.c -- plain, slow, fp64 CPU oracle for the Kimi Delta Attention
 * (KDA) layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "Kimi K3 / Architecture" (lei.chat), panel "Kimi Delta Attention .
 *        one head at token t" and panel "KDA short convolution . one channel c
 *        at token t".
 *   [P2] "Animated Kimi K3 architecture diagram", section "LOCAL MEMORY: A
 *        FIXED MATRIX THAT PREDICTS, FORGETS, AND CORRECTS" (the four moves
 *        PROBE / CORRECT / DECAY / WRITE, and the NOTEBOOK TRACE line
 *        "sequential ~ chunkwise, state shape stays fixed").
 *
 * All arithmetic is IEEE fp64 in the order the definitions state.  Inputs may
 * arrive as fp32 containers: every bf16 or fp32 input value is exactly
 * representable there, and it is widened to fp64 before any arithmetic.
 * Threads only split independent (sequence, head) units; no sum is reordered.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes as well):
 *   - tap w[0] multiplies x[t-3] and tap w[3] multiplies x[t]; no conv bias;
 *     inputs before a sequence start are zero, or come from the rolling conv
 *     state (3 values per channel, oldest first);
 *   - SiLU follows the conv on q, k and v alike;
 *   - L2 normalisation of q and k per head: x / sqrt(sum x^2 + eps_l2);
 *   - decay comes before the probe: S_bar = Diag(exp(g_t)) S_{t-1};
 *   - beta_t is one scalar per (token, head); the log-decay g_t is an input;
 *   - the readout o_t = scale * S_t^T q_t uses the state after the write;
 *   - head RMSNorm o / sqrt(mean o^2 + eps_rms) * w_rms, then times
 *     sigmoid(gate).
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu_d(double x) { return x * sigmoid_d(x); }

/* ------------------------------------------------------------------------ */
/* Short convolution, [P1] "KDA short convolution": causal window of width 4 */
/* over one channel (x[t-3], x[t-2], x[t-1], x[t] times w0..w3), only time    */
/* is mixed, left padding keeps the length, then SiLU ("Sigma 4 taps, SiLU    */
/* Swish").  The rolling state keeps the previous 3 raw values per channel.   */
/* ------------------------------------------------------------------------ */

/* value of the raw stream at local position s (s may be -3..-1: the state) */
static double raw_at(int64_t s, const float* x, int64_t xs, const double prev[3])
{
    return s >= 0 ? (double)x[s * xs] : prev[3 + s];
}

/* One channel over one sequence of L tokens.  prev = 3 values before t=0,
 * oldest first.  y (may be NULL) receives the conv output (after SiLU if
 * apply_silu), last3 (may be NULL) the last 3 raw values of the stream. */
static void conv_one_channel(int64_t L, const float* x, int64_t xs, const double w[4],
                             const double prev[3], double* y, int64_t ys, int apply_silu,
                             double last3[3])
{
    if (y) {
        for (int64_t t = 0; t < L; ++t) {
            double acc = 0.0;
            for (int j = 0; j < 4; ++j) acc += w[j] * raw_at(t - 3 + j, x, xs, prev);
            y[t * ys] = apply_silu ? silu_d(acc) : acc;
        }
    }
    if (last3) {
        for (int m = 0; m < 3; ++m) last3[m] = raw_at(L - 3 + m, x, xs, prev);
    }
}

/* Depthwise conv (+ SiLU) of every channel of a packed varlen buffer.
 * x: [T_total][x_stride] (the first n_ch entries of each row are used),
 * w: [n_ch][4], cu_seqlens: [N+1] host, state_in: [N][n_ch][3] or NULL,
 * y: [T_total][y_stride] or NULL, state_out: [N][n_ch][3] or NULL. */
int kda_oracle_conv_silu(int64_t T_total, int n_ch, const float* x, int64_t x_stride,
                         const float* w, const int32_t* cu_seqlens, int N,
                         const float* state_in, double* y, int64_t y_stride,
                         double* state_out, int apply_silu)
{
    if (!x || !w || !cu_seqlens || N < 0 || n_ch <= 0) return 1;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total) return 1;
    for (int n = 0; n < N; ++n) {
        int64_t t0 = cu_seqlens[n], L = (int64_t)cu_seqlens[n + 1] - t0;
        if (L < 0) return 1;
        for (int c = 0; c < n_ch; ++c) {
            double prev[3] = {0.0, 0.0, 0.0}, wd[4], last3[3];
            if (state_in)
                for (int m = 0; m < 3; ++m) prev[m] = state_in[((int64_t)n * n_ch + c) * 3 + m];
            for (int j = 0; j < 4; ++j) wd[j] = w[(int64_t)c * 4 + j];
            conv_one_channel(L, x + t0 * x_stride + c, x_stride, wd, prev,
                             y ? y + t0 * y_stride + c : NULL, y_stride, apply_silu, last3);
            if (state_out)
                for (int m = 0; m < 3; ++m) state_out[((int64_t)n * n_ch + c) * 3 + m] = last3[m];
        }
    }
    return 0;
}

/* [P1] KDA panel: q and k are L2-normalised after the activation, per 128-channel
 * head: x <- x / sqrt(sum x^2 + eps). */
static void l2norm_vec(int d, double* x, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < d; ++i) x[i] *= inv;
}

void kda_oracle_l2norm(int64_t n_rows, int d, double* x, int64_t row_stride, double eps)
{
    for (int64_t r = 0; r < n_rows; ++r) l2norm_vec(d, x + r * row_stride, eps);
}

/* [P1] KDA panel: RMSNorm per head, then a sigmoid output gate with one value per channel:
 * y = o / sqrt(mean(o^2) + eps) * w * sigmoid(gate); w NULL = ones, gate NULL = no gate. */
static void rmsnorm_gate_vec(int d, const double* o, const double* gate, const double* w,
                             double eps, double* y)
{
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += o[i] * o[i];
    double inv = 1.0 / sqrt(ss / d + eps);
    for (int i = 0; i < d; ++i) {
        double v = o[i] * inv;
        if (w) v *= w[i];
        if (gate) v *= sigmoid_d(gate[i]);
        y[i] = v;
    }
}

void kda_oracle_rmsnorm_gate(int64_t n_rows, int d, const double* o, const double* gate,
                             const double* w, double eps, double* y)
{
    for (int64_t r = 0; r < n_rows; ++r)
        rmsnorm_gate_vec(d, o + r * d, gate ? gate + r * d : NULL, w, eps, y + r * d);
}

/* ------------------------------------------------------------------------ */
/* Token-sequential gated delta rule, [P2] four moves, [P1] readout S_t^T q_t. */
/* S: [Dk][Dv] row-major (row = key channel), updated in place.               */
/*   DECAY   S_bar = Diag(alpha_t) S,  alpha_t = exp(g_t)                      */
/*   PROBE   k_t reads S_bar:  S_bar^T k_t                                     */
/*   CORRECT e_t = v_t - S_bar^T k_t                                           */
/*   WRITE   S_t = S_bar + beta_t k_t e_t^T                                    */
/*   READ    o_t = scale * S_t^T q_t                                           */
/* ------------------------------------------------------------------------ */
static void delta_step(int Dk, int Dv, const double* q, const double* k, const double* v,
                       const double* g, double beta, double scale, double* S, double* e,
                       double* o)
{
    for (int c = 0; c < Dk; ++c) {
        double a = exp(g[c]);
        for (int j = 0; j < Dv; ++j) S[c * Dv + j] *= a;
    }
    for (int j = 0; j < Dv; ++j) {
        double p = 0.0;
        for (int c = 0; c < Dk; ++c) p += S[c * Dv + j] * k[c];
        e[j] = v[j] - p;
    }
    for (int c = 0; c < Dk; ++c) {
        double bk = beta * k[c];
        for (int j = 0; j < Dv; ++j) S[c * Dv + j] += bk * e[j];
    }
    for (int j = 0; j < Dv; ++j) {
        double r = 0.0;
        for (int c = 0; c < Dk; ++c) r += S[c * Dv + j] * q[c];
        o[j] = scale * r;
    }
}

/* One (sequence, head) unit on already convolved/normalised inputs.
 * q,k,g: [L][*] with row strides; v: [L][*]; beta: [L] with stride bs;
 * S: [Dk][Dv] in/out; o: [L][os]. */
int kda_oracle_recurrence(int64_t L, int Dk, int Dv, const double* q, int64_t qs,
                          const double* k, int64_t ks, const double* v, int64_t vs,
                          const double* g, int64_t gs, const double* beta, int64_t bs,
                          double scale, double* S, double* o, int64_t os)
{
    double* e = (double*)malloc(sizeof(double) * (size_t)Dv);
    if (!e) return 2;
    for (int64_t t = 0; t < L; ++t)
        delta_step(Dk, Dv, q + t * qs, k + t * ks, v + t * vs, g + t * gs, beta[t * bs], scale,
                   S, e, o + t * os);
    free(e);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Chunkwise form, [P1] KDA panel: the state recurs from chunk to chunk while */
/* the tokens of a chunk are taken together; [P2] the state is carried across */
/* chunks.  A second, independent fp64 form of the same                       */
/* recurrence.  Within a chunk of Lc tokens, local index r, with             */
/* G_r = sum_{s<=r} g_s (per key channel) and w_i = beta_i e_i:              */
/*   S_r   = Diag(e^{G_r}) S0 + sum_{i<=r} Diag(e^{G_r - G_i}) k_i w_i^T      */
/*   A_ri  = beta_r sum_c k_rc k_ic e^{G_rc - G_ic}            (i < r)        */
/*   M_ri  = sum_c q_rc k_ic e^{G_rc - G_ic}                   (i <= r)       */
/*   w_r   = beta_r (v_r - S0^T (k_r . e^{G_r})) - sum_{i<r} A_ri w_i         */
/*           (forward substitution of (I + A) W = Diag(beta)(V - (K.Gamma)S0)) */
/*   o_r   = scale ((q_r . e^{G_r})^T S0 + sum_{i<=r} M_ri w_i)               */
/*   S_end = Diag(e^{G_last}) S0 + sum_i Diag(e^{G_last - G_i}) k_i w_i^T     */
/* Every ratio is formed as exp of a difference, never as a quotient.         */
/* chunk_states (may be NULL): [n_chunks][Dk][Dv], the state at each chunk    */
/* start.                                                                     */
/* ------------------------------------------------------------------------ */
int kda_oracle_chunkwise(int64_t L, int Dk, int Dv, int C, const double* q, int64_t qs,
                         const double* k, int64_t ks, const double* v, int64_t vs,
                         const double* g, int64_t gs, const double* beta, int64_t bs,
                         double scale, double* S, double* o, int64_t os, double* chunk_states)
{
    if (C <= 0) return 1;
    double* G = (double*)malloc(sizeof(double) * (size_t)C * Dk);
    double* A = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* M = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* W = (double*)malloc(sizeof(double) * (size_t)C * Dv);
    double* Sn = (double*)malloc(sizeof(double) * (size_t)Dk * Dv);
    if (!G || !A || !M || !W || !Sn) {
        free(G); free(A); free(M); free(W); free(Sn);
        return 2;
    }
    int64_t n_chunk = 0;
    for (int64_t s0 = 0; s0 < L; s0 += C, ++n_chunk) {
        int Lc = (int)((L - s0) < C ? (L - s0) : C);
        const double* qc = q + s0 * qs;
        const double* kc = k + s0 * ks;
        const double* vc = v + s0 * vs;
        const double* gc = g + s0 * gs;
        const double* bc = beta + s0 * bs;
        if (chunk_states) memcpy(chunk_states + n_chunk * Dk * Dv, S, sizeof(double) * Dk * Dv);
        for (int c = 0; c < Dk; ++c) {
            double acc = 0.0;
            for (int r = 0; r < Lc; ++r) {
                acc += gc[r * gs + c];
                G[r * Dk + c] = acc;
            }
        }
        for (int r = 0; r < Lc; ++r)
            for (int i = 0; i < Lc; ++i) {
                double a = 0.0, m = 0.0;
                if (i <= r)
                    for (int c = 0; c < Dk; ++c) {
                        double dec = exp(G[r * Dk + c] - G[i * Dk + c]);
                        a += kc[r * ks + c] * kc[i * ks + c] * dec;
                        m += qc[r * qs + c] * kc[i * ks + c] * dec;
                    }
                A[r * C + i] = (i < r) ? bc[r * bs] * a : 0.0;
                M[r * C + i] = (i <= r) ? m : 0.0;
            }
        for (int r = 0; r < Lc; ++r)
            for (int j = 0; j < Dv; ++j) {
                double p = 0.0;
                for (int c = 0; c < Dk; ++c) p += kc[r * ks + c] * exp(G[r * Dk + c]) * S[c * Dv + j];
                double w = bc[r * bs] * (vc[r * vs + j] - p);
                for (int i = 0; i < r; ++i) w -= A[r * C + i] * W[i * Dv + j];
                W[r * Dv + j] = w;
            }
        for (int r = 0; r < Lc; ++r)
            for (int j = 0; j < Dv; ++j) {
                double inter = 0.0, intra = 0.0;
                for (int c = 0; c < Dk; ++c) inter += qc[r * qs + c] * exp(G[r * Dk + c]) * S[c * Dv + j];
                for (int i = 0; i <= r; ++i) intra += M[r * C + i] * W[i * Dv + j];
                o[(s0 + r) * os + j] = scale * (inter + intra);
            }
        const double* Gl = G + (int64_t)(Lc - 1) * Dk;
        for (int c = 0; c < Dk; ++c)
            for (int j = 0; j < Dv; ++j) {
                double acc = exp(Gl[c]) * S[c * Dv + j];
                for (int i = 0; i < Lc; ++i) acc += kc[i * ks + c] * exp(Gl[c] - G[i * Dk + c]) * W[i * Dv + j];
                Sn[c * Dv + j] = acc;
            }
        memcpy(S, Sn, sizeof(double) * Dk * Dv);
    }
    free(G); free(A); free(M); free(W); free(Sn);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Whole layer: conv + SiLU + L2 -> recurrence -> RMSNorm + gate, per         */
/* (sequence, head), threaded over the independent units.                    */
/* ------------------------------------------------------------------------ */
typedef struct {
    int64_t T_total;
    int N, H, D;            /* heads in the arrays below; Dk = Dv = D */
    const int32_t* cu;      /* [N+1] host */
    const float *q, *k, *v; /* [T_total][H][D] raw (before the conv) */
    const float* conv_w;    /* [3][H*D][4] */
    const float* cs_in;     /* [N][3*H*D][3] or NULL */
    const float* g;         /* [T_total][H][D] */
    const float* beta;      /* [T_total][H] */
    const float* gate;      /* [T_total][H][D] or NULL */
    const float* rms_w;     /* [D] or NULL */
    double eps_l2, eps_rms, scale;
    const double* S0;       /* [N][H][D][D] or NULL */
    double* out;            /* [T_total][H][D] or NULL */
    double* o_pre;          /* [T_total][H][D] or NULL: o before RMSNorm/gate */
    double* S_fin;          /* [N][H][D][D] or NULL */
    double* cs_out;         /* [N][3*H*D][3] or NULL */
    int64_t next;           /* unit counter */
    int err;
} fwd_job;

static int fwd_unit(fwd_job* J, int n, int h)
{
    const int D = J->D, H = J->H;
    const int64_t HD = (int64_t)H * D, row = HD;
    const int64_t t0 = J->cu[n], L = (int64_t)J->cu[n + 1] - t0;
    double* buf = (double*)malloc(sizeof(double) * (size_t)(D * D + 9 * D + 3 * 3 * D));
    if (!buf) return 2;
    double* S = buf;
    double *qt = S + D * D, *kt = qt + D, *vt = kt + D, *gt = vt + D, *e = gt + D, *o = e + D,
           *gate = o + D, *y = gate + D, *wr = y + D;
    double* win = wr + D; /* [3 tensors][D][3] rolling raw window, oldest first */
    if (J->rms_w)
        for (int j = 0; j < D; ++j) wr[j] = J->rms_w[j];
    for (int c = 0; c < D; ++c)
        for (int j = 0; j < D; ++j)
            S[c * D + j] = J->S0 ? J->S0[(((int64_t)n * H + h) * D + c) * D + j] : 0.0;
    const float* src[3] = {J->q, J->k, J->v};
    for (int x = 0; x < 3; ++x)
        for (int d = 0; d < D; ++d)
            for (int m = 0; m < 3; ++m)
                win[(x * D + d) * 3 + m] =
                    J->cs_in ? (double)J->cs_in[((int64_t)n * 3 * HD + x * HD + (int64_t)h * D + d) * 3 + m]
                             : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t tt = t0 + t;
        double* dst[3] = {qt, kt, vt};
        for (int x = 0; x < 3; ++x)
            for (int d = 0; d < D; ++d) {
                const int64_t ch = (int64_t)h * D + d;
                double* wdw = win + (x * D + d) * 3;
                double xt = (double)src[x][tt * row + ch];
                const float* wp = J->conv_w + ((int64_t)x * HD + ch) * 4;
                double acc = (double)wp[0] * wdw[0] + (double)wp[1] * wdw[1] + (double)wp[2] * wdw[2] +
                             (double)wp[3] * xt;
                dst[x][d] = silu_d(acc);
                wdw[0] = wdw[1];
                wdw[1] = wdw[2];
                wdw[2] = xt;
            }
        l2norm_vec(D, qt, J->eps_l2);
        l2norm_vec(D, kt, J->eps_l2);
        for (int c = 0; c < D; ++c) gt[c] = (double)J->g[(tt * H + h) * D + c];
        delta_step(D, D, qt, kt, vt, gt, (double)J->beta[tt * H + h], J->scale, S, e, o);
        if (J->o_pre)
            for (int j = 0; j < D; ++j) J->o_pre[(tt * H + h) * D + j] = o[j];
        if (J->out) {
            if (J->gate)
                for (int j = 0; j < D; ++j) gate[j] = (double)J->gate[(tt * H + h) * D + j];
            rmsnorm_gate_vec(D, o, J->gate ? gate : NULL, J->rms_w ? wr : NULL, J->eps_rms, y);
            for (int j = 0; j < D; ++j) J->out[(tt * H + h) * D + j] = y[j];
        }
    }
    if (J->S_fin)
        for (int c = 0; c < D; ++c)
            for (int j = 0; j < D; ++j) J->S_fin[(((int64_t)n * H + h) * D + c) * D + j] = S[c * D + j];
    if (J->cs_out)
        for (int x = 0; x < 3; ++x)
            for (int d = 0; d < D; ++d)
                for (int m = 0; m < 3; ++m)
                    J->cs_out[((int64_t)n * 3 * HD + x * HD + (int64_t)h * D + d) * 3 + m] =
                        win[(x * D + d) * 3 + m];
    free(buf);
    return 0;
}

static void* fwd_worker(void* arg)
{
    fwd_job* J = (fwd_job*)arg;
    const int64_t units = (int64_t)J->N * J->H;
    for (;;) {
        int64_t u = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (u >= units) break;
        int rc = fwd_unit(J, (int)(u / J->H), (int)(u % J->H));
        if (rc) __atomic_store_n(&J->err, rc, __ATOMIC_RELAXED);
    }
    return NULL;
}

/* Full KDA layer forward (prefill, or decode when every sequence has one
 * token and the states are carried in).  Returns 0 on success.  n_threads
 * <= 0 uses every online core. */
int kda_oracle_forward(int64_t T_total, int N, int H, int D, const int32_t* cu_seqlens,
                       const float* q, const float* k, const float* v, const float* conv_w,
                       const float* conv_state_in, const float* g, const float* beta,
                       const float* gate, const float* rms_w, double eps_l2, double eps_rms,
                       double scale, const double* initial_state, double* out, double* o_pre,
                       double* final_state, double* conv_state_out, int n_threads)
{
    if (!cu_seqlens || !q || !k || !v || !conv_w || !g || !beta || N < 0 || H <= 0 || D <= 0)
        return 1;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total) return 1;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    fwd_job J = {T_total, N, H, D, cu_seqlens, q, k, v, conv_w, conv_state_in, g, beta, gate,
                 rms_w, eps_l2, eps_rms, scale, initial_state, out, o_pre, final_state,
                 conv_state_out, 0, 0};
    if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    int64_t units = (int64_t)N * H;
    if (n_threads > units) n_threads = (int)(units > 0 ? units : 1);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) return 2;
    int started = 0;
    for (int i = 1; i < n_threads; ++i) {
        pthread_t t;
        if (pthread_create(&t, NULL, fwd_worker, &J) == 0) th[started++] = t;
    }
    /* the calling thread works too */
    fwd_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return J.err;
}

/* ------------------------------------------------------------------------ */
/* Backward pass of the whole layer (reverse-mode derivatives of the forward  */
/* above), token-sequential and in fp64.  For one (sequence, head) unit the   */
/* forward is recomputed keeping every intermediate (the convolved and        */
/* activated q, k, v, their norms, the states S_0 .. S_L, o, the RMSNorm      */
/* factors), then the derivatives of loss = sum dy . y + sum dS_L . S_L run   */
/* backwards through the same steps:                                          */
/*   y = n w sig(z), n = o r, r = (mean o^2 + eps)^-1/2:                       */
/*     dz = dy n w sig(1 - sig);  dw += dy n sig;  dn = dy w sig;              */
/*     do = r dn - r^3 o (dn . o) / D                                         */
/*   o_t = scale S_t^T q_t:  dS += scale q_t do_t^T;  dq_t = scale S_t do_t    */
/*   S_t = P + beta k e^T, e = v - P^T k, P = Diag(alpha_t) S_{t-1}:           */
/*     w = dS^T k;  dv_t = beta w;  dbeta_t = w . e;                           */
/*     dk_t = beta (dS e - P w);  dP = dS - beta k w^T;                        */
/*     dg_t[c] = sum_j dP[c][j] P[c][j]  (d/dg of alpha = e^g);               */
/*     dS_{t-1} = Diag(alpha_t) dP                                            */
/*   x = a / sqrt(|a|^2 + eps):  da = (dx - x (x . dx)) / sqrt(|a|^2 + eps)    */
/*   a = u sig(u):  du = da sig(u) (1 + u (1 - sig(u)))                       */
/*   u_t = sum_j w_j x_{t-3+j}:  dx_{t-3+j} += w_j du_t;  dw_j += x_{t-3+j} du_t */
/*     (positions before the sequence belong to the rolling conv state).     */
/* ------------------------------------------------------------------------ */
typedef struct {
    fwd_job f;               /* the forward's inputs (outputs unused) */
    const double* dy;        /* [T_total][H][D] */
    const double* dS_fin;    /* [N][H][D][D] or NULL */
    double *dq, *dk, *dv;    /* [T_total][H][D]: d/d raw projections */
    double* dcw_part;        /* [N*H][3][D][4] per-unit conv-tap partials */
    double* dcs_in;          /* [N][3*H*D][3] or NULL */
    double *dg, *dbeta;      /* [T_total][H][D], [T_total][H] */
    double* dgate;           /* [T_total][H][D] or NULL */
    double* drms_part;       /* [N*H][D] per-unit RMSNorm-weight partials */
    double* dS0;             /* [N][H][D][D] or NULL */
} bwd_job;

static int bwd_unit(bwd_job* B, int n, int h)
{
    fwd_job* J = &B->f;
    const int D = J->D, H = J->H;
    const int64_t HD = (int64_t)H * D, DD = (int64_t)D * D;
    const int64_t t0 = J->cu[n], L = (int64_t)J->cu[n + 1] - t0;
    const int64_t u = (int64_t)n * H + h;
    const size_t LD = (size_t)(L > 0 ? L : 1) * D;
    /* per token: raw x, pre-activation u, activation a (3 parts each), q^, k^, norms, alpha,
       o, r, sig; states S_0..S_L */
    double* xr = (double*)calloc(3 * LD + 3 * 3 * D, sizeof(double)); /* [3][3 + L][D] incl. the window */
    double* ua = (double*)malloc(sizeof(double) * 3 * LD);
    double* aa = (double*)malloc(sizeof(double) * 3 * LD);
    double* qh = (double*)malloc(sizeof(double) * LD);
    double* kh = (double*)malloc(sizeof(double) * LD);
    double* rq = (double*)malloc(sizeof(double) * (size_t)(L + 1));
    double* rk = (double*)malloc(sizeof(double) * (size_t)(L + 1));
    double* al = (double*)malloc(sizeof(double) * LD);
    double* oo = (double*)malloc(sizeof(double) * LD);
    double* rr = (double*)malloc(sizeof(double) * (size_t)(L + 1));
    double* sg = (double*)malloc(sizeof(double) * LD);
    double* SS = (double*)malloc(sizeof(double) * (size_t)(L + 1) * DD);
    double* dS = (double*)malloc(sizeof(double) * DD);
    double* dP = (double*)malloc(sizeof(double) * DD);
    double* vec = (double*)malloc(sizeof(double) * 8 * D);
    double* da = (double*)calloc(3 * LD, sizeof(double)); /* d/d activation, then d/d u */
    if (!xr || !ua || !aa || !qh || !kh || !rq || !rk || !al || !oo || !rr || !sg || !SS || !dS || !dP || !vec || !da) {
        free(xr); free(ua); free(aa); free(qh); free(kh); free(rq); free(rk); free(al); free(oo); free(rr);
        free(sg); free(SS); free(dS); free(dP); free(vec); free(da);
        return 2;
    }
    const float* src[3] = {J->q, J->k, J->v};
    const int64_t XS = (L + 3) * D; /* stride of one part in xr: 3 window rows then L token rows */
    for (int x = 0; x < 3; ++x)
        for (int d = 0; d < D; ++d) {
            for (int m = 0; m < 3; ++m)
                xr[x * XS + m * D + d] =
                    J->cs_in ? (double)J->cs_in[((int64_t)n * 3 * HD + x * HD + (int64_t)h * D + d) * 3 + m] : 0.0;
            for (int64_t t = 0; t < L; ++t) xr[x * XS + (3 + t) * D + d] = (double)src[x][(t0 + t) * HD + (int64_t)h * D + d];
        }
    /* ---- forward, keeping everything */
    for (int c = 0; c < D; ++c)
        for (int j = 0; j < D; ++j) SS[c * D + j] = J->S0 ? J->S0[(u * D + c) * D + j] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t tt = t0 + t;
        for (int x = 0; x < 3; ++x)
            for (int d = 0; d < D; ++d) {
                const float* wp = J->conv_w + ((int64_t)x * HD + (int64_t)h * D + d) * 4;
                double acc = 0.0;
                for (int j = 0; j < 4; ++j) acc += (double)wp[j] * xr[x * XS + (t + j) * D + d];
                ua[x * LD + t * D + d] = acc;
                aa[x * LD + t * D + d] = silu_d(acc);
            }
        double sq = 0.0, sk = 0.0;
        for (int d = 0; d < D; ++d) {
            sq += aa[t * D + d] * aa[t * D + d];
            sk += aa[LD + t * D + d] * aa[LD + t * D + d];
        }
        rq[t] = sqrt(sq + J->eps_l2);
        rk[t] = sqrt(sk + J->eps_l2);
        for (int d = 0; d < D; ++d) {
            qh[t * D + d] = aa[t * D + d] / rq[t];
            kh[t * D + d] = aa[LD + t * D + d] / rk[t];
            al[t * D + d] = exp((double)J->g[(tt * H + h) * D + d]);
        }
        const double* Sp = SS + t * DD;
        double* Sn = SS + (t + 1) * DD;
        const double bt = (double)J->beta[tt * H + h];
        double* e = vec;
        for (int c = 0; c < D; ++c)
            for (int j = 0; j < D; ++j) Sn[c * D + j] = al[t * D + c] * Sp[c * D + j];
        for (int j = 0; j < D; ++j) {
            double p = 0.0;
            for (int c = 0; c < D; ++c) p += Sn[c * D + j] * kh[t * D + c];
            e[j] = aa[2 * LD + t * D + j] - p;
        }
        for (int c = 0; c < D; ++c)
            for (int j = 0; j < D; ++j) Sn[c * D + j] += bt * kh[t * D + c] * e[j];
        double ms = 0.0;
        for (int j = 0; j < D; ++j) {
            double r = 0.0;
            for (int c = 0; c < D; ++c) r += Sn[c * D + j] * qh[t * D + c];
            oo[t * D + j] = J->scale * r;
            ms += oo[t * D + j] * oo[t * D + j];
        }
        rr[t] = 1.0 / sqrt(ms / D + J->eps_rms);
        for (int j = 0; j < D; ++j) sg[t * D + j] = J->gate ? sigmoid_d((double)J->gate[(tt * H + h) * D + j]) : 1.0;
    }
    /* ---- backward */
    double* drms = B->drms_part + u * D;
    double* dcw = B->dcw_part + u * 3 * D * 4;
    for (int c = 0; c < D; ++c)
        for (int j = 0; j < D; ++j) dS[c * D + j] = B->dS_fin ? B->dS_fin[(u * D + c) * D + j] : 0.0;
    double *dn = vec, *dov = vec + D, *w = vec + 2 * D, *e = vec + 3 * D, *dqh = vec + 4 * D, *dkh = vec + 5 * D;
    for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t tt = t0 + t;
        const double* dyt = B->dy + (tt * H + h) * D;
        /* RMSNorm and gate */
        double dno = 0.0;
        for (int j = 0; j < D; ++j) {
            const double wj = J->rms_w ? (double)J->rms_w[j] : 1.0;
            const double nj = oo[t * D + j] * rr[t], s = sg[t * D + j];
            if (B->dgate) B->dgate[(tt * H + h) * D + j] = J->gate ? dyt[j] * nj * wj * s * (1.0 - s) : 0.0;
            drms[j] += dyt[j] * nj * s;
            dn[j] = dyt[j] * wj * s;
            dno += dn[j] * oo[t * D + j];
        }
        const double r = rr[t];
        for (int j = 0; j < D; ++j) dov[j] = r * dn[j] - r * r * r * oo[t * D + j] * dno / D;
        /* readout o_t = scale S_t^T q_t */
        const double* St = SS + (t + 1) * DD;
        for (int c = 0; c < D; ++c) {
            double acc = 0.0;
            for (int j = 0; j < D; ++j) {
                dS[c * D + j] += J->scale * qh[t * D + c] * dov[j];
                acc += St[c * D + j] * dov[j];
            }
            dqh[c] = J->scale * acc;
        }
        /* write S_t = P + beta k e^T with P = Diag(alpha_t) S_{t-1} */
        const double* Sp = SS + t * DD;
        const double bt = (double)J->beta[tt * H + h];
        for (int j = 0; j < D; ++j) {
            double pw = 0.0, ww = 0.0;
            for (int c = 0; c < D; ++c) {
                pw += al[t * D + c] * Sp[c * D + j] * kh[t * D + c];
                ww += dS[c * D + j] * kh[t * D + c];
            }
            e[j] = aa[2 * LD + t * D + j] - pw;
            w[j] = ww;
        }
        double db = 0.0;
        for (int j = 0; j < D; ++j) {
            da[2 * LD + t * D + j] = bt * w[j]; /* dv (v is the activation itself) */
            db += w[j] * e[j];
        }
        B->dbeta[tt * H + h] = db;
        for (int c = 0; c < D; ++c) {
            double de = 0.0, pw = 0.0, dgc = 0.0;
            for (int j = 0; j < D; ++j) {
                const double P = al[t * D + c] * Sp[c * D + j];
                de += dS[c * D + j] * e[j];
                pw += P * w[j];
                const double d = dS[c * D + j] - bt * kh[t * D + c] * w[j];
                dP[c * D + j] = d;
                dgc += d * P;
            }
            dkh[c] = bt * (de - pw);
            B->dg[(tt * H + h) * D + c] = dgc;
        }
        for (int c = 0; c < D; ++c)
            for (int j = 0; j < D; ++j) dS[c * D + j] = al[t * D + c] * dP[c * D + j];
        /* L2 norms */
        double xq = 0.0, xk = 0.0;
        for (int d = 0; d < D; ++d) {
            xq += qh[t * D + d] * dqh[d];
            xk += kh[t * D + d] * dkh[d];
        }
        for (int d = 0; d < D; ++d) {
            da[t * D + d] = (dqh[d] - qh[t * D + d] * xq) / rq[t];
            da[LD + t * D + d] = (dkh[d] - kh[t * D + d] * xk) / rk[t];
        }
    }
    if (B->dS0)
        for (int64_t i = 0; i < DD; ++i) B->dS0[u * DD + i] = dS[i];
    /* SiLU, then the conv: d/d raw x and d/d taps; positions before the sequence -> conv state */
    double* dxw = (double*)calloc((size_t)3 * XS, sizeof(double)); /* [3][3 + L][D] */
    if (!dxw) {
        free(xr); free(ua); free(aa); free(qh); free(kh); free(rq); free(rk); free(al); free(oo); free(rr);
        free(sg); free(SS); free(dS); free(dP); free(vec); free(da);
        return 2;
    }
    for (int x = 0; x < 3; ++x)
        for (int64_t t = 0; t < L; ++t)
            for (int d = 0; d < D; ++d) {
                const double uu = ua[x * LD + t * D + d], s = sigmoid_d(uu);
                const double du = da[x * LD + t * D + d] * s * (1.0 + uu * (1.0 - s));
                const float* wp = J->conv_w + ((int64_t)x * HD + (int64_t)h * D + d) * 4;
                for (int j = 0; j < 4; ++j) {
                    dxw[x * XS + (t + j) * D + d] += (double)wp[j] * du;
                    dcw[(x * D + d) * 4 + j] += xr[x * XS + (t + j) * D + d] * du;
                }
            }
    double* dst[3] = {B->dq, B->dk, B->dv};
    for (int x = 0; x < 3; ++x)
        for (int d = 0; d < D; ++d) {
            for (int64_t t = 0; t < L; ++t) dst[x][(t0 + t) * HD + (int64_t)h * D + d] = dxw[x * XS + (3 + t) * D + d];
            if (B->dcs_in)
                for (int m = 0; m < 3; ++m)
                    B->dcs_in[((int64_t)n * 3 * HD + x * HD + (int64_t)h * D + d) * 3 + m] = dxw[x * XS + m * D + d];
        }
    free(dxw);
    free(xr); free(ua); free(aa); free(qh); free(kh); free(rq); free(rk); free(al); free(oo); free(rr);
    free(sg); free(SS); free(dS); free(dP); free(vec); free(da);
    return 0;
}

typedef struct {
    bwd_job* B;
    int64_t next;
    int err;
} bwd_pool;

static void* bwd_worker(void* arg)
{
    bwd_pool* P = (bwd_pool*)arg;
    const int64_t units = (int64_t)P->B->f.N * P->B->f.H;
    for (;;) {
        int64_t u = __atomic_fetch_add(&P->next, 1, __ATOMIC_RELAXED);
        if (u >= units) break;
        int rc = bwd_unit(P->B, (int)(u / P->B->f.H), (int)(u % P->B->f.H));
        if (rc) __atomic_store_n(&P->err, rc, __ATOMIC_RELAXED);
    }
    return NULL;
}

/* Gradients of loss = sum dy . y + sum dS_fin . S_fin with respect to every input of
 * kda_oracle_forward.  dconv_w ([3][H*D][4]) and drms_w ([D]) are overwritten with sums over
 * all units (in unit order, so the result does not depend on the thread count); every other
 * output has one writer.  Optional outputs may be NULL: dconv_state_in, dgate, drms_w,
 * dinitial_state; d_final_state may be NULL (zero). */
int kda_oracle_backward(int64_t T_total, int N, int H, int D, const int32_t* cu_seqlens,
                        const float* q, const float* k, const float* v, const float* conv_w,
                        const float* conv_state_in, const float* g, const float* beta,
                        const float* gate, const float* rms_w, double eps_l2, double eps_rms,
                        double scale, const double* initial_state, const double* dy,
                        const double* d_final_state, double* dq, double* dk, double* dv,
                        double* dconv_w, double* dconv_state_in, double* dg, double* dbeta,
                        double* dgate, double* drms_w, double* dinitial_state, int n_threads)
{
    if (!cu_seqlens || !q || !k || !v || !conv_w || !g || !beta || !dy || !dq || !dk || !dv || !dconv_w ||
        !dg || !dbeta || N < 0 || H <= 0 || D <= 0)
        return 1;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T_total) return 1;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    const int64_t units = (int64_t)N * H;
    double* dcw_part = (double*)calloc((size_t)(units > 0 ? units : 1) * 3 * D * 4, sizeof(double));
    double* drms_part = (double*)calloc((size_t)(units > 0 ? units : 1) * D, sizeof(double));
    if (!dcw_part || !drms_part) {
        free(dcw_part);
        free(drms_part);
        return 2;
    }
    bwd_job B = {{T_total, N, H, D, cu_seqlens, q, k, v, conv_w, conv_state_in, g, beta, gate, rms_w, eps_l2,
                  eps_rms, scale, initial_state, NULL, NULL, NULL, NULL, 0, 0},
                 dy, d_final_state, dq, dk, dv, dcw_part, dconv_state_in, dg, dbeta, dgate, drms_part,
                 dinitial_state};
    bwd_pool P = {&B, 0, 0};
    if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > units) n_threads = (int)(units > 0 ? units : 1);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) {
        free(dcw_part);
        free(drms_part);
        return 2;
    }
    int started = 0;
    for (int i = 1; i < n_threads; ++i) {
        pthread_t t;
        if (pthread_create(&t, NULL, bwd_worker, &P) == 0) th[started++] = t;
    }
    bwd_worker(&P);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    const int64_t HD = (int64_t)H * D;
    for (int64_t i = 0; i < 3 * HD * 4; ++i) dconv_w[i] = 0.0;
    if (drms_w)
        for (int d = 0; d < D; ++d) drms_w[d] = 0.0;
    for (int64_t uu = 0; uu < units; ++uu) {
        const int h = (int)(uu % H);
        for (int x = 0; x < 3; ++x)
            for (int d = 0; d < D; ++d)
                for (int j = 0; j < 4; ++j)
                    dconv_w[((int64_t)x * HD + (int64_t)h * D + d) * 4 + j] += dcw_part[((uu * 3 + x) * D + d) * 4 + j];
        if (drms_w)
            for (int d = 0; d < D; ++d) drms_w[d] += drms_part[uu * D + d];
    }
    free(dcw_part);
    free(drms_part);
    return P.err;
}

int kda_oracle_num_cores(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }
