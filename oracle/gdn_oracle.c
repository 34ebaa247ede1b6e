/*
 * Frame-wise Gated DeltaNet forward -- fp64 CPU ORACLE.
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

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
