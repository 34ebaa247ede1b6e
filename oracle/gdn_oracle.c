/*
 * Frame-wise Gated DeltaNet forward and backward -- fp64 CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path must compute.  Only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or helper with the CUDA library and includes nothing of it.
 *
 * What it follows
 * ---------------
 * SANA-WM article (davidborish.com), section "The Architecture": the GDN is a
 * recurrent layer that consumes one whole latent frame per step and keeps a
 * fixed-size state matrix that is updated by a decay gate and a delta-rule
 * correction.  wispaper summary, "Methodology" section 1: frames are scanned
 * one by one while a compact state is updated.  The pages give the update in
 * words only; the exact form used here is the frame-wise gated delta rule
 *
 *     A_f = K_f^T B_f K_f            = sum_n beta_n k_n k_n^T      (dk x dk)
 *     U_f = V_f^T B_f K_f            = sum_n beta_n v_n k_n^T      (dv x dk)
 *     S_f = alpha_f * S_{f-1} (I - A_f) + U_f                      (dv x dk)
 *     O_f = Q_f S_f^T,  i.e.  o_n = S_f q_n  for every token n of frame f
 *
 * with one state S per (batch b, head h), fp64 throughout, S_0 = state_in or 0.
 * Readings taken where the pages are silent:
 *   - the decay alpha multiplies only the carried state, not the new write U_f;
 *   - every token of frame f reads the state AFTER frame f's update;
 *   - no 1/sqrt(d) scaling, output norm or gate: those belong to the block.
 *
 * Layouts (row-major, contiguous):
 *   q, k : bf16 bits  [B, F, N, H, dk]        v : bf16 bits [B, F, N, H, dv]
 *   alpha: fp32 [B, F, H]    beta: fp32 [B, F, N, H]
 *   state_in: fp32 [B, H, dv, dk] (may be NULL -> zero state)
 *   out: fp64 [B, F, N, H, dv]   state_out: fp64 [B, H, dv, dk]
 * bf16 inputs are decoded exactly (bf16 -> fp64 is exact), so the oracle sees
 * precisely the values the GPU sees.
 *
 * mode (oracle-internal switches, used only by the self-pins):
 *   ORACLE_MODE_GDN      the method above
 *   ORACLE_MODE_NODELTA  drop the delta correction: S_f = alpha_f S_{f-1} + U_f
 *                        (with alpha = 1 this is the cumulative linear attention
 *                        that the article contrasts GDN with)
 *   ORACLE_MODE_REVERSE  scan the frames in reverse order (f = F-1 .. 0); the
 *                        state after frame f is used for frame f's tokens
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MODE_GDN 0
#define ORACLE_MODE_NODELTA 1
#define ORACLE_MODE_REVERSE 2

static double bf16_to_f64(uint16_t bits)
{
    union { uint32_t u; float f; } c;
    c.u = ((uint32_t)bits) << 16;
    return (double)c.f;
}

/* Inputs come either as bf16 bit patterns with fp32 gates and state (the
 * values the GPU library receives) or as fp64 arrays (used to state the
 * folded prologue exactly). */
typedef struct {
    const uint16_t *q16, *k16, *v16;
    const double *q64, *k64, *v64;
    const float *alpha32, *beta32, *s0_32;
    const double *alpha64, *beta64, *s0_64;
} Inputs;

static double in_q(const Inputs* in, size_t i) { return in->q64 ? in->q64[i] : bf16_to_f64(in->q16[i]); }
static double in_k(const Inputs* in, size_t i) { return in->k64 ? in->k64[i] : bf16_to_f64(in->k16[i]); }
static double in_v(const Inputs* in, size_t i) { return in->v64 ? in->v64[i] : bf16_to_f64(in->v16[i]); }
static double in_alpha(const Inputs* in, size_t i) { return in->alpha64 ? in->alpha64[i] : (double)in->alpha32[i]; }
static double in_beta(const Inputs* in, size_t i) { return in->beta64 ? in->beta64[i] : (double)in->beta32[i]; }
static int has_s0(const Inputs* in) { return in->s0_64 != NULL || in->s0_32 != NULL; }
static double in_s0(const Inputs* in, size_t i) { return in->s0_64 ? in->s0_64[i] : (double)in->s0_32[i]; }

/* One (b, h) sequence.  Work arrays are allocated per call so that (b, h)
 * pairs can run on separate threads. */
static int run_head(const Inputs* in,
                    double* out, double* state_out, double* states_all,
                    const int64_t* sample_tok, int64_t n_samples, double* sample_out,
                    int b, int h, int B, int H, int F, int N, int dk, int dv, int mode)
{
    (void)B;
    double* S = (double*)calloc((size_t)dv * dk, sizeof(double));
    double* A = (double*)malloc((size_t)dk * dk * sizeof(double));
    double* U = (double*)malloc((size_t)dv * dk * sizeof(double));
    double* T = (double*)malloc((size_t)dv * dk * sizeof(double));
    double* kn = (double*)malloc((size_t)dk * sizeof(double));
    double* vn = (double*)malloc((size_t)dv * sizeof(double));
    double* qn = (double*)malloc((size_t)dk * sizeof(double));
    if (!S || !A || !U || !T || !kn || !vn || !qn) {
        free(S); free(A); free(U); free(T); free(kn); free(vn); free(qn);
        return 1;
    }

    /* S_0 */
    if (has_s0(in)) {
        const size_t s0 = ((size_t)b * H + h) * dv * dk;
        for (size_t e = 0; e < (size_t)dv * dk; ++e) S[e] = in_s0(in, s0 + e);
    }

    for (int step = 0; step < F; ++step) {
        const int f = (mode == ORACLE_MODE_REVERSE) ? (F - 1 - step) : step;
        const size_t frame = (size_t)b * F + f;

        /* A_f = sum_n beta_n k_n k_n^T ,  U_f = sum_n beta_n v_n k_n^T */
        memset(A, 0, (size_t)dk * dk * sizeof(double));
        memset(U, 0, (size_t)dv * dk * sizeof(double));
        for (int n = 0; n < N; ++n) {
            const size_t tok = frame * N + n;
            const double bn = in_beta(in, tok * H + h);
            for (int j = 0; j < dk; ++j) kn[j] = in_k(in, (tok * H + h) * dk + j);
            for (int i = 0; i < dv; ++i) vn[i] = in_v(in, (tok * H + h) * dv + i);
            for (int i = 0; i < dk; ++i) {
                const double w = bn * kn[i];
                double* row = A + (size_t)i * dk;
                for (int j = 0; j < dk; ++j) row[j] += w * kn[j];
            }
            for (int i = 0; i < dv; ++i) {
                const double w = bn * vn[i];
                double* row = U + (size_t)i * dk;
                for (int j = 0; j < dk; ++j) row[j] += w * kn[j];
            }
        }

        /* S_f = alpha_f (S_{f-1} - S_{f-1} A_f) + U_f */
        const double af = in_alpha(in, frame * H + h);
        if (mode == ORACLE_MODE_NODELTA) {
            for (size_t e = 0; e < (size_t)dv * dk; ++e) S[e] = af * S[e] + U[e];
        } else {
            for (int i = 0; i < dv; ++i) {
                double* trow = T + (size_t)i * dk;
                const double* srow = S + (size_t)i * dk;
                for (int j = 0; j < dk; ++j) trow[j] = 0.0;
                for (int m = 0; m < dk; ++m) {
                    const double s = srow[m];
                    const double* arow = A + (size_t)m * dk;
                    for (int j = 0; j < dk; ++j) trow[j] += s * arow[j];
                }
            }
            for (size_t e = 0; e < (size_t)dv * dk; ++e) S[e] = af * (S[e] - T[e]) + U[e];
        }

        if (states_all) {
            double* dst = states_all + (((size_t)b * H + h) * F + f) * dv * dk;
            memcpy(dst, S, (size_t)dv * dk * sizeof(double));
        }

        /* O_f = Q_f S_f^T : o_n[i] = sum_j S[i][j] q_n[j] */
        if (out) {
            for (int n = 0; n < N; ++n) {
                const size_t tok = frame * N + n;
                for (int j = 0; j < dk; ++j) qn[j] = in_q(in, (tok * H + h) * dk + j);
                double* op = out + (tok * H + h) * dv;
                for (int i = 0; i < dv; ++i) {
                    const double* srow = S + (size_t)i * dk;
                    double acc = 0.0;
                    for (int j = 0; j < dk; ++j) acc += srow[j] * qn[j];
                    op[i] = acc;
                }
            }
        }
        if (sample_out) {
            for (int64_t s = 0; s < n_samples; ++s) {
                const int64_t tok = sample_tok[s];
                if (tok / N != (int64_t)frame) continue;
                for (int j = 0; j < dk; ++j) qn[j] = in_q(in, ((size_t)tok * H + h) * dk + j);
                double* op = sample_out + ((size_t)s * H + h) * dv;
                for (int i = 0; i < dv; ++i) {
                    const double* srow = S + (size_t)i * dk;
                    double acc = 0.0;
                    for (int j = 0; j < dk; ++j) acc += srow[j] * qn[j];
                    op[i] = acc;
                }
            }
        }
    }

    if (state_out)
        memcpy(state_out + ((size_t)b * H + h) * dv * dk, S, (size_t)dv * dk * sizeof(double));

    free(S); free(A); free(U); free(T); free(kn); free(vn); free(qn);
    return 0;
}

/*
 * Full frame-wise forward.
 *   out         fp64 [B,F,N,H,dv]   every output, or NULL
 *   state_out   fp64 [B,H,dv,dk]    final state S_F, or NULL
 *   states_all  fp64 [B,H,F,dv,dk]  state after every frame, or NULL
 *   sample_tok / n_samples / sample_out: outputs of selected tokens only;
 *               sample_tok holds flat token indices (b*F + f)*N + n and
 *               sample_out is fp64 [n_samples, H, dv].  May be NULL / 0.
 *   n_threads   OpenMP threads over the (b, h) pairs (<= 0: library default).
 * Returns 0 on success, 1 on allocation failure, 2 on bad arguments.
 */
static int forward(const Inputs* in, int need_q, double* out, double* state_out, double* states_all,
                   const int64_t* sample_tok, int64_t n_samples, double* sample_out,
                   int B, int H, int F, int N, int dk, int dv, int mode, int n_threads)
{
    if (B < 1 || H < 1 || F < 0 || N < 0 || dk < 1 || dv < 1) return 2;
    if ((out || sample_out) && !need_q) return 2;
    if (mode < 0 || mode > 2) return 2;
    for (int64_t s = 0; s < n_samples; ++s)
        if (sample_tok[s] < 0 || sample_tok[s] >= (int64_t)B * F * N) return 2;

    const int pairs = B * H;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = 0;
    #pragma omp parallel for schedule(dynamic, 1) reduction(|:failed) num_threads(n_threads > 0 ? n_threads : omp_get_max_threads())
#endif
    for (int p = 0; p < pairs; ++p) {
        const int b = p / H, h = p % H;
        failed |= run_head(in, out, state_out, states_all, sample_tok, n_samples, sample_out,
                           b, h, B, H, F, N, dk, dv, mode);
    }
    return failed ? 1 : 0;
}

/*
 * Full frame-wise forward on the GPU library's input types (bf16 q/k/v,
 * fp32 alpha/beta/state_in).
 *   out         fp64 [B,F,N,H,dv]   every output, or NULL
 *   state_out   fp64 [B,H,dv,dk]    final state S_F, or NULL
 *   states_all  fp64 [B,H,F,dv,dk]  state after every frame, or NULL
 *   sample_tok / n_samples / sample_out: outputs of selected tokens only;
 *               sample_tok holds flat token indices (b*F + f)*N + n and
 *               sample_out is fp64 [n_samples, H, dv].  May be NULL / 0.
 *   n_threads   OpenMP threads over the (b, h) pairs (<= 0: library default).
 * Returns 0 on success, 1 on allocation failure, 2 on bad arguments.
 */
int oracle_gdn_frame_forward(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             const float* alpha, const float* beta, const float* state_in,
                             double* out, double* state_out, double* states_all,
                             const int64_t* sample_tok, int64_t n_samples, double* sample_out,
                             int B, int H, int F, int N, int dk, int dv, int mode, int n_threads)
{
    if (!alpha || !beta || !k || !v) return 2;
    Inputs in = {q, k, v, NULL, NULL, NULL, alpha, beta, state_in, NULL, NULL, NULL};
    return forward(&in, q != NULL, out, state_out, states_all, sample_tok, n_samples, sample_out,
                   B, H, F, N, dk, dv, mode, n_threads);
}

/* The same forward on fp64 inputs of the same layouts (q, k, v, alpha, beta,
 * state_in all fp64; state_in may be NULL). */
int oracle_gdn_frame_forward_f64(const double* q, const double* k, const double* v,
                                 const double* alpha, const double* beta, const double* state_in,
                                 double* out, double* state_out, double* states_all,
                                 const int64_t* sample_tok, int64_t n_samples, double* sample_out,
                                 int B, int H, int F, int N, int dk, int dv, int mode, int n_threads)
{
    if (!alpha || !beta || !k || !v) return 2;
    Inputs in = {NULL, NULL, NULL, q, k, v, NULL, NULL, NULL, alpha, beta, state_in};
    return forward(&in, q != NULL, out, state_out, states_all, sample_tok, n_samples, sample_out,
                   B, H, F, N, dk, dv, mode, n_threads);
}

/*
 * Backward of the forward above (reverse-mode derivatives), fp64, all arrays
 * fp64 in the forward's layouts.
 *
 * Given dL/dO (d_out, [B,F,N,H,dv]) and dL/dS_F (d_state_out, [B,H,dv,dk], or
 * NULL for zero), returns dL/dq, dL/dk, dL/dv (token layouts), dL/dalpha
 * [B,F,H], dL/dbeta [B,F,N,H] and dL/dS_0 [B,H,dv,dk] (d_state_in, may be
 * NULL).  The chain rule applied to the forward's steps, per (b, h):
 *
 *   G_f = dL/dS_f (everything that depends on S_f):
 *       G_{F-1} = dS_F + M_{F-1},   G_{f-1} = M_{f-1} + alpha_f G_f (I - A_f)
 *       with M_f = sum_n do_n q_n^T over frame f's tokens (o_n = S_f q_n),
 *       and dL/dS_0 = alpha_0 G_0 (I - A_0)       (A is symmetric)
 *   from S_f = alpha_f (S_{f-1} - S_{f-1} A_f) + U_f, with P_f = S_{f-1}^T G_f:
 *       dU_f = G_f,   dA_f = -alpha_f P_f,   dalpha_f = tr(P_f) - <P_f, A_f>
 *   from A_f = sum_n beta_n k_n k_n^T and U_f = sum_n beta_n v_n k_n^T:
 *       dk_n = beta_n ((dA_f + dA_f^T) k_n + G_f^T v_n),   dv_n = beta_n G_f k_n,
 *       dbeta_n = k_n^T dA_f k_n + v_n^T G_f k_n
 *   from o_n = S_f q_n:  dq_n = S_f^T do_n.
 * Returns 0 on success, 1 on allocation failure, 2 on bad arguments.
 */
static int backward_head(const double* q, const double* k, const double* v, const double* alpha,
                         const double* beta, const double* state_in, const double* d_out,
                         const double* d_state_out, double* dq, double* dkv_k, double* dkv_v,
                         double* d_alpha, double* d_beta, double* d_state_in,
                         int b, int h, int H, int F, int N, int dk, int dv)
{
    const size_t SD = (size_t)dv * dk, AD = (size_t)dk * dk;
    double* Sprev = (double*)malloc((size_t)(F + 1) * SD * sizeof(double)); /* Sprev[f] = S before frame f; Sprev[F] = S_F */
    double* Af = (double*)malloc((size_t)(F > 0 ? F : 1) * AD * sizeof(double));
    double* G = (double*)malloc(SD * sizeof(double));
    double* T = (double*)malloc(SD * sizeof(double));
    double* P = (double*)malloc(AD * sizeof(double));
    double* W = (double*)malloc(AD * sizeof(double));
    if (!Sprev || !Af || !G || !T || !P || !W) {
        free(Sprev); free(Af); free(G); free(T); free(P); free(W);
        return 1;
    }
    /* forward, keeping every state and every A_f */
    for (size_t e = 0; e < SD; ++e) Sprev[e] = state_in ? state_in[((size_t)b * H + h) * SD + e] : 0.0;
    for (int f = 0; f < F; ++f) {
        const size_t frame = (size_t)b * F + f;
        double* A = Af + (size_t)f * AD;
        double* S = Sprev + (size_t)(f + 1) * SD;
        const double* S0 = Sprev + (size_t)f * SD;
        memset(A, 0, AD * sizeof(double));
        memset(T, 0, SD * sizeof(double));       /* T = U_f */
        for (int n = 0; n < N; ++n) {
            const size_t th = (frame * N + n) * H + h;
            const double bn = beta[th];
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dk; ++j) A[(size_t)i * dk + j] += bn * k[th * dk + i] * k[th * dk + j];
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) T[(size_t)i * dk + j] += bn * v[th * dv + i] * k[th * dk + j];
        }
        const double af = alpha[frame * H + h];
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) {
                double sa = 0.0;
                for (int m = 0; m < dk; ++m) sa += S0[(size_t)i * dk + m] * A[(size_t)m * dk + j];
                S[(size_t)i * dk + j] = af * (S0[(size_t)i * dk + j] - sa) + T[(size_t)i * dk + j];
            }
    }
    /* reverse */
    for (size_t e = 0; e < SD; ++e) G[e] = d_state_out ? d_state_out[((size_t)b * H + h) * SD + e] : 0.0;
    for (int f = F - 1; f >= 0; --f) {
        const size_t frame = (size_t)b * F + f;
        const double* A = Af + (size_t)f * AD;
        const double* Sf = Sprev + (size_t)(f + 1) * SD;
        const double* S0 = Sprev + (size_t)f * SD;
        /* G_f = G (carried from frame f+1) + M_f;  dq_n = S_f^T do_n */
        for (int n = 0; n < N; ++n) {
            const size_t th = (frame * N + n) * H + h;
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) G[(size_t)i * dk + j] += d_out[th * dv + i] * q[th * dk + j];
            for (int j = 0; j < dk; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dv; ++i) acc += Sf[(size_t)i * dk + j] * d_out[th * dv + i];
                dq[th * dk + j] = acc;
            }
        }
        /* P_f = S_{f-1}^T G_f, dalpha_f, dA_f = -alpha_f P_f, W = dA_f + dA_f^T */
        const double af = alpha[frame * H + h];
        double tr = 0.0, pa = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dk; ++j) {
                double acc = 0.0;
                for (int m = 0; m < dv; ++m) acc += S0[(size_t)m * dk + i] * G[(size_t)m * dk + j];
                P[(size_t)i * dk + j] = acc;
            }
        for (int i = 0; i < dk; ++i) {
            tr += P[(size_t)i * dk + i];
            for (int j = 0; j < dk; ++j) pa += P[(size_t)i * dk + j] * A[(size_t)i * dk + j];
        }
        d_alpha[frame * H + h] = tr - pa;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dk; ++j) W[(size_t)i * dk + j] = -af * (P[(size_t)i * dk + j] + P[(size_t)j * dk + i]);
        /* token gradients of frame f */
        for (int n = 0; n < N; ++n) {
            const size_t th = (frame * N + n) * H + h;
            const double bn = beta[th];
            double kdak = 0.0, vgk = 0.0;
            for (int j = 0; j < dk; ++j) {
                double wk = 0.0, gv = 0.0;
                for (int m = 0; m < dk; ++m) wk += W[(size_t)j * dk + m] * k[th * dk + m];
                for (int i = 0; i < dv; ++i) gv += G[(size_t)i * dk + j] * v[th * dv + i];
                dkv_k[th * dk + j] = bn * (wk + gv);
                kdak += 0.5 * k[th * dk + j] * wk;   /* k^T dA k = k^T W k / 2 */
            }
            for (int i = 0; i < dv; ++i) {
                double gk = 0.0;
                for (int j = 0; j < dk; ++j) gk += G[(size_t)i * dk + j] * k[th * dk + j];
                dkv_v[th * dv + i] = bn * gk;
                vgk += v[th * dv + i] * gk;
            }
            d_beta[th] = kdak + vgk;
        }
        /* carry to S_{f-1}: alpha_f G_f (I - A_f) */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) {
                double ga = 0.0;
                for (int m = 0; m < dk; ++m) ga += G[(size_t)i * dk + m] * A[(size_t)m * dk + j];
                T[(size_t)i * dk + j] = af * (G[(size_t)i * dk + j] - ga);
            }
        memcpy(G, T, SD * sizeof(double));
    }
    if (d_state_in) memcpy(d_state_in + ((size_t)b * H + h) * SD, G, SD * sizeof(double));
    free(Sprev); free(Af); free(G); free(T); free(P); free(W);
    return 0;
}

int oracle_gdn_frame_backward_f64(const double* q, const double* k, const double* v,
                                  const double* alpha, const double* beta, const double* state_in,
                                  const double* d_out, const double* d_state_out,
                                  double* dq, double* dk_out, double* dv_out, double* d_alpha, double* d_beta,
                                  double* d_state_in, int B, int H, int F, int N, int dk, int dv, int n_threads)
{
    if (!q || !k || !v || !alpha || !beta || !d_out || !dq || !dk_out || !dv_out || !d_alpha || !d_beta) return 2;
    if (B < 1 || H < 1 || F < 0 || N < 0 || dk < 1 || dv < 1) return 2;
    const int pairs = B * H;
    int failed = 0;
#ifdef _OPENMP
    #pragma omp parallel for schedule(dynamic, 1) reduction(|:failed) num_threads(n_threads > 0 ? n_threads : omp_get_max_threads())
#endif
    for (int p = 0; p < pairs; ++p)
        failed |= backward_head(q, k, v, alpha, beta, state_in, d_out, d_state_out, dq, dk_out, dv_out,
                                d_alpha, d_beta, d_state_in, p / H, p % H, H, F, N, dk, dv);
    (void)n_threads;
    return failed ? 1 : 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
