/*
 * gdn.h -- C ABI of the B300-native frame-wise Gated DeltaNet (GDN) forward.
 *
 * The operation (SANA-WM article, davidborish.com, section "The Architecture":
 * a recurrent layer that processes one entire latent frame per step and keeps
 * a fixed-size state matrix updated by a decay gate and a delta-rule
 * correction; wispaper summary, "Methodology" 1: frames are scanned one by
 * one).  Per batch row b and head h, with K_f, Q_f (N x dk) and V_f (N x dv)
 * the N tokens of latent frame f, B_f = diag(beta) and alpha_f the frame's
 * decay:
 *
 *     S_f = alpha_f * S_{f-1} * (I - K_f^T B_f K_f) + V_f^T B_f K_f
 *     O_f = Q_f * S_f^T                 (every token of frame f reads S_f)
 *
 * S is an fp32 dv x dk matrix, S_0 = state_in (or zero).
 *
 * Layouts (all contiguous, row-major, tokens frame-major):
 *     q, k        bf16  [B, F, N, H, dk]
 *     v, out      bf16  [B, F, N, H, dv]
 *     alpha       fp32  [B, F, H]
 *     beta        fp32  [B, F, N, H]
 *     state_in,
 *     state_out   fp32  [B, H, dv, dk]      S[i][j], i in dv, j in dk
 *
 * Ownership: every pointer is caller-owned DEVICE memory on the current CUDA
 * device; the library never frees it.  The library owns its workspace
 * (per-frame A_f, U_f and the bf16 per-frame states, see
 * gdn_workspace_bytes), taken with stream-ordered allocation on `stream` from
 * a library memory pool and returned on the same stream, so calls on
 * different streams do not share scratch.
 *
 * Semantics: every entry point validates its arguments on the host first and
 * launches nothing if they are bad.  A launched call is asynchronous on
 * `stream`; kernel-side failures (a bounded wait that ran out) are recorded
 * on the device and reported by gdn_sync_status().  No entry point throws,
 * exits or aborts.  Results are deterministic: no atomics take part in any
 * sum, and every reduction runs in a fixed order.
 *
 * Supported sizes: B, H, F, N >= 1; dk and dv multiples of 16 in [16, 128];
 * B*F*N*H*max(dk,dv) < 2^31 elements per tensor.  Pointers must be 16-byte
 * aligned (tensor-memory-accelerator copies require it).
 */
#ifndef GDN_B300_H
#define GDN_B300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_NULL_PTR = 1,     /* a required pointer is NULL                       */
    GDN_ERR_BAD_DIM = 2,      /* B, H, F or N < 1, or a tensor too large           */
    GDN_ERR_UNSUPPORTED = 3,  /* dk or dv not a multiple of 16 in [16,128]        */
    GDN_ERR_MISALIGNED = 4,   /* a pointer is not 16-byte aligned                 */
    GDN_ERR_ALLOC = 5,        /* workspace allocation failed                       */
    GDN_ERR_LAUNCH = 6,       /* a kernel launch or CUDA runtime call failed       */
    GDN_ERR_TIMEOUT = 7,      /* a device-side bounded wait ran out (sync_status) */
    GDN_ERR_ALIAS = 8,        /* out overlaps an input                             */
    GDN_ERR_NO_DEVICE = 9,    /* no usable sm_103 device is current               */
    GDN_ERR_TOO_LARGE = 10,   /* needs more than the fixed no-alloc scratch       */
    GDN_ERR_RANGE = 11        /* an input value outside the entry point's range
                                 (device-reported, via gdn_sync_status)           */
} gdn_status;

/*
 * Whole-sequence forward: runs all F frames of every (b, h) and writes every
 * O_f to `out` and S_F to `state_out`.
 *   state_in   may be NULL (S_0 = 0).
 *   state_out  may be NULL (final state not wanted) or equal to state_in
 *              (in-place resident state); it must not partially overlap it.
 *   out        must not overlap q, k, v, alpha, beta or the states.
 * Phases: frame-parallel contractions A_f = K_f^T B_f K_f and
 * U_f = V_f^T B_f K_f on tcgen05 tensor cores; the sequential scan
 * S_f = alpha_f (S_{f-1} - S_{f-1} A_f) + U_f; the frame-parallel output
 * O_f = Q_f S_f^T on tcgen05 tensor cores.  By default the three run side by
 * side in one launch (gdn_set_single_pass); otherwise in stream order.
 */
gdn_status gdn_frame_forward(const void* q, const void* k, const void* v,
                             const float* alpha, const float* beta,
                             const float* state_in, void* out, float* state_out,
                             int B, int H, int F, int N, int dk, int dv,
                             gdn_stream_t stream);

/*
 * Reverse-direction forward for the bidirectional stage (WorldFoundry model
 * card, "What it is for": the quality profile keeps a bidirectional stage):
 * the same recurrence with the frames scanned from F-1 down to 0,
 *     S_f = alpha_f * S_{f+1} * (I - K_f^T B_f K_f) + V_f^T B_f K_f,  S_F = state_in
 *     O_f = Q_f * S_f^T
 * so state_out holds the state after frame 0.  Same arguments, layouts,
 * validation and results as gdn_frame_forward applied to the frame-reversed
 * sequence; how the two directions of a bidirectional layer are combined is
 * left to the caller.
 */
gdn_status gdn_frame_forward_reverse(const void* q, const void* k, const void* v,
                                     const float* alpha, const float* beta,
                                     const float* state_in, void* out, float* state_out,
                                     int B, int H, int F, int N, int dk, int dv,
                                     gdn_stream_t stream);

/*
 * Forward with the per-token prologue of a GDN block folded into the kernels,
 * for callers whose projections emit raw queries, keys and gate logits:
 *     q <- q / max(|q|, 1e-12),  k <- k / max(|k|, 1e-12)   per (token, head)
 *     beta  = sigmoid(b_logit)                               [B, F, N, H]
 *     alpha = exp(-softplus(a_logit) * alpha_scale)          [B, F, H]
 * followed by exactly the gdn_frame_forward recurrence.  q and k are read
 * once: the contraction kernel normalizes k rows as it scales them by beta,
 * the output kernel divides each output row by |q_n|, and the scan applies the
 * decay gate.  Same layouts, validation and ownership as gdn_frame_forward
 * (a_logit and b_logit take the places of alpha and beta).
 */
gdn_status gdn_frame_forward_gated(const void* q, const void* k, const void* v,
                                   const float* a_logit, const float* b_logit, float alpha_scale,
                                   const float* state_in, void* out, float* state_out,
                                   int B, int H, int F, int N, int dk, int dv,
                                   gdn_stream_t stream);

/* gdn_frame_step with the same folded prologue as gdn_frame_forward_gated. */
gdn_status gdn_frame_step_gated(const void* q, const void* k, const void* v,
                                const float* a_logit, const float* b_logit, float alpha_scale,
                                const float* state_in, void* out, float* state_out,
                                int B, int H, int N, int dk, int dv,
                                gdn_stream_t stream);

/*
 * Forward with 8-bit inputs.  The SANA-WM article ("NVIDIA's New 2.6B World
 * Model...", intro) deploys a distilled variant with NVFP4 quantization; the
 * pages do not say which tensors are quantized or how.  This entry point
 * takes q, k and v as OCP FP8 E4M3 bytes (1 sign, 4 exponent bits with bias
 * 7, 3 mantissa bits; code 0x7F/0xFF is NaN) with one fp32 scale per tensor:
 * the value of element x is scale * e4m3(x).  Layouts as gdn_frame_forward
 * with one byte per element (q, k: [B, F, N, H, dk]; v: [B, F, N, H, dv]);
 * out stays bf16 and the state fp32.  The recurrence is exactly that of
 * gdn_frame_forward on the decoded values.  The kernels decode in shared
 * memory (exactly) and fold the scales into A, U and out, so HBM carries one
 * byte per input element.  The contraction scales k and v by sqrt(beta) in
 * f16 arithmetic, so every beta must lie in [0, 16384]; a value outside (or
 * NaN) is reported as GDN_ERR_RANGE by gdn_sync_status.  Validation and
 * other errors as gdn_frame_forward (q, k, v, out 16-byte aligned).
 */
gdn_status gdn_frame_forward_fp8(const void* q, const void* k, const void* v,
                                 float q_scale, float k_scale, float v_scale,
                                 const float* alpha, const float* beta,
                                 const float* state_in, void* out, float* state_out,
                                 int B, int H, int F, int N, int dk, int dv,
                                 gdn_stream_t stream);

/*
 * Backward of gdn_frame_forward, for training (the SANA-WM pages train the
 * model, wispaper "Methodology"; they give no gradient formulas).  Given the
 * forward's inputs and the upstream gradients d_out = dL/dout [B, F, N, H, dv]
 * (bf16) and d_state_out = dL/dstate_out [B, H, dv, dk] (fp32, NULL = 0), it
 * writes dq, dk [B, F, N, H, dk] and dv [B, F, N, H, dv] (bf16), d_alpha
 * [B, F, H] and d_beta [B, F, N, H] (fp32), and d_state_in [B, H, dv, dk]
 * (fp32, may be NULL).  The chain rule of the forward's steps:
 *     G_{f-1} = M_{f-1} + alpha_f G_f (I - A_f),  G_{F-1} = dS_F + M_{F-1},
 *     M_f = dO_f^T Q_f,  P_f = S_{f-1}^T G_f,  dA_f = -alpha_f P_f,
 *     dalpha_f = tr P_f - <P_f, A_f>,  dS_0 = alpha_0 G_0 (I - A_0),
 *     dq_n = S_f^T do_n,  dk_n = beta_n ((dA_f + dA_f^T) k_n + G_f^T v_n),
 *     dv_n = beta_n G_f k_n,  dbeta_n = k_n^T dA_f k_n + v_n^T G_f k_n.
 * It recomputes the forward states (phase 1 and the scan), runs the state
 * gradient recurrence on the same scan kernel in reverse, then two
 * frame-parallel tcgen05 kernels form the gradients.  Outputs must not
 * overlap inputs or each other (GDN_ERR_ALIAS); otherwise validation and
 * errors as gdn_frame_forward.  Batch rows run one after another on the
 * stream with one workspace of about (F + 1) * H * (2 dk^2 + 12 dv dk) bytes.
 */
gdn_status gdn_frame_backward(const void* q, const void* k, const void* v,
                              const float* alpha, const float* beta, const float* state_in,
                              const void* d_out, const float* d_state_out,
                              void* dq_out, void* dk_out, void* dv_out, float* d_alpha, float* d_beta,
                              float* d_state_in,
                              int B, int H, int F, int N, int dk, int dv,
                              gdn_stream_t stream);

/*
 * Forward with NVFP4 inputs, the format of the distilled SANA-WM variant (the
 * SANA-WM article, "NVIDIA's New 2.6B World Model...", intro: four sampling
 * steps with NVFP4 quantization; the pages say no more).  Each of q, k, v is
 *   codes   uint8 [B, F, N, H, d/2]   two FP4 E2M1 codes per byte, element 2i
 *                                     in the low nibble (1 sign, 2 exponent
 *                                     bits with bias 1, 1 mantissa bit)
 *   scales  uint8 [B, F, N, H, d/16]  one OCP FP8 E4M3 block scale per 16
 *                                     consecutive elements of a token's head
 *   gs      one fp32 scale per tensor
 * and element i of a row is gs * e4m3(scale[i / 16]) * e2m1(code i).  The
 * recurrence is exactly that of gdn_frame_forward on the decoded values; out
 * stays bf16 and the state fp32.  The kernels decode in shared memory (the
 * product of a code and its block scale is exact in f16) and fold the
 * per-tensor scales into A, U and out, so HBM carries half a byte per input
 * element plus one byte per 16.  Head sizes dk, dv must be 64 or 128
 * (GDN_ERR_UNSUPPORTED otherwise); codes and scales 16-byte aligned; every
 * beta in [0, 512] (the contraction forms sqrt(beta) times values up to
 * 6 * 448 in f16), anything else is reported as GDN_ERR_RANGE by
 * gdn_sync_status.  Other validation and errors as gdn_frame_forward.
 */
gdn_status gdn_frame_forward_nvfp4(const void* q4, const void* k4, const void* v4,
                                   const void* q_sf, const void* k_sf, const void* v_sf,
                                   float q_gs, float k_gs, float v_gs,
                                   const float* alpha, const float* beta,
                                   const float* state_in, void* out, float* state_out,
                                   int B, int H, int F, int N, int dk, int dv,
                                   gdn_stream_t stream);

/* gdn_frame_step with the NVFP4 inputs of gdn_frame_forward_nvfp4. */
gdn_status gdn_frame_step_nvfp4(const void* q4, const void* k4, const void* v4,
                                const void* q_sf, const void* k_sf, const void* v_sf,
                                float q_gs, float k_gs, float v_gs,
                                const float* alpha, const float* beta,
                                const float* state_in, void* out, float* state_out,
                                int B, int H, int N, int dk, int dv,
                                gdn_stream_t stream);

/*
 * Forward that keeps the activations its backward needs, for training: the
 * same results as gdn_frame_forward, and in addition
 *   saved_A  bf16 [B, F, H, dk, dk]   A_f = K_f^T B_f K_f of every frame
 *   saved_S  bf16 [B, F, H, dv, dk]   the state after every frame, rounded to bf16
 * (B*F*H*(dk*dk + dv*dk)*2 bytes, 127 MB at the 60 s shape), written by the
 * kernels as they go (phase 1, then the scan and output pass).  Caller-owned
 * device memory, 16-byte aligned, clear of every other argument.  Pass both to
 * gdn_frame_backward_saved, which then skips recomputing them.
 */
gdn_status gdn_frame_forward_save(const void* q, const void* k, const void* v,
                                  const float* alpha, const float* beta,
                                  const float* state_in, void* out, float* state_out,
                                  void* saved_A, void* saved_S,
                                  int B, int H, int F, int N, int dk, int dv,
                                  gdn_stream_t stream);

/*
 * gdn_frame_backward from the activations of gdn_frame_forward_save (same
 * inputs, same shapes): the per-frame A_f and state images are copied from
 * saved_A, saved_S instead of being recomputed (phase 1 and the forward scan
 * are skipped).  The gradients are bit-identical to gdn_frame_backward's.
 */
gdn_status gdn_frame_backward_saved(const void* q, const void* k, const void* v,
                                    const float* alpha, const float* beta, const float* state_in,
                                    const void* saved_A, const void* saved_S,
                                    const void* d_out, const float* d_state_out,
                                    void* dq_out, void* dk_out, void* dv_out, float* d_alpha, float* d_beta,
                                    float* d_state_in,
                                    int B, int H, int F, int N, int dk, int dv,
                                    gdn_stream_t stream);

/* gdn_frame_step with the 8-bit inputs of gdn_frame_forward_fp8. */
gdn_status gdn_frame_step_fp8(const void* q, const void* k, const void* v,
                              float q_scale, float k_scale, float v_scale,
                              const float* alpha, const float* beta,
                              const float* state_in, void* out, float* state_out,
                              int B, int H, int N, int dk, int dv,
                              gdn_stream_t stream);

/*
 * One-frame step for interactive rollout (WorldFoundry model card, "What it
 * is for": a resident pipeline that advances in native 8k+1 windows): the same
 * operation with F = 1 on a resident state.
 *   q, k   bf16 [B, N, H, dk];  v, out bf16 [B, N, H, dv];
 *   alpha  fp32 [B, H];         beta fp32 [B, N, H];
 *   state_in / state_out fp32 [B, H, dv, dk]; state_out may equal state_in.
 * By default (gdn_set_fused_step) the frame runs as one kernel, launched with
 * programmatic dependent launch: its prologue (barriers, tensor memory) may
 * overlap the end of the previous kernel in the stream, and it touches no
 * global memory before that kernel has completed.  Every sum is taken in a
 * fixed order, so the result is deterministic.
 */
gdn_status gdn_frame_step(const void* q, const void* k, const void* v,
                          const float* alpha, const float* beta,
                          const float* state_in, void* out, float* state_out,
                          int B, int H, int N, int dk, int dv,
                          gdn_stream_t stream);

/*
 * gdn_frame_forward with per-phase timing: records the caller's CUDA events
 * phase_events[0..3] (cudaEvent_t handles, created by the caller) on `stream`
 * before phase 1, before phase 2, before phase 3 and after phase 3, so that
 * cudaEventElapsedTime gives each kernel's duration.  Same contract and
 * results as gdn_frame_forward.  NULL events -> GDN_ERR_NULL_PTR.
 */
gdn_status gdn_frame_forward_timed(const void* q, const void* k, const void* v,
                                   const float* alpha, const float* beta,
                                   const float* state_in, void* out, float* state_out,
                                   int B, int H, int F, int N, int dk, int dv,
                                   gdn_stream_t stream, void* const* phase_events);

/*
 * gdn_frame_forward on HOST buffers (same layouts): the sequence is processed
 * in chunks of frames (about F/8 each; gdn_set_host_chunk_frames), double-
 * buffered in library-owned device memory.  Chunk i's inputs are copied in on
 * a library copy stream while chunk i-1 runs on `stream` and chunk i-2's
 * outputs are copied out on a second library copy stream, so both directions
 * of the host link and the kernels overlap; the state is carried on the
 * device from chunk to chunk (exactly: the result is bit-identical to one
 * gdn_frame_forward over the whole sequence).  Returns after synchronising
 * `stream`, with `out` and (if not NULL) `state_out` written.  Page-locked
 * host buffers make the copies run at full link speed and asynchronously.
 */
gdn_status gdn_frame_forward_host(const void* q, const void* k, const void* v,
                                  const float* alpha, const float* beta,
                                  const float* state_in, void* out, float* state_out,
                                  int B, int H, int F, int N, int dk, int dv,
                                  gdn_stream_t stream);

/*
 * Phase 1 on head pairs.  on != 0 (default): with bf16 inputs, dk = dv = 128,
 * an even number of heads and N a multiple of 8, the contraction takes two
 * heads of a frame at a time, its copies covering the 512 contiguous bytes
 * both heads occupy per token (about twice the copy rate of one head's 256
 * bytes).  on = 0: one head at a time.  Results are identical.  Applies to
 * calls made after it returns.  A scheduling control of this library; the
 * pages have no counterpart.
 */
void gdn_set_contract_pairs(int on);

/* Frames per chunk of gdn_frame_forward_host (0: automatic, about F / 8).
 * Applies to calls made after it returns. */
void gdn_set_host_chunk_frames(int frames);

/* Bytes of library workspace one gdn_frame_forward call of this shape takes
 * on the current device (0 for invalid shapes; with no usable device, an
 * upper bound). */
size_t gdn_workspace_bytes(int B, int H, int F, int N, int dk, int dv);

/* Bytes of library workspace one gdn_frame_step call of this shape takes on
 * the three-phase step path (gdn_set_fused_step(0)), computed with the work
 * plan that call would launch on the current device (with no usable device:
 * an upper bound). */
size_t gdn_step_workspace_bytes(int B, int H, int N, int dk, int dv);

/* Static, human-readable name of a status code. */
const char* gdn_status_string(gdn_status s);

/*
 * Synchronises `stream`, then returns the first error any kernel of this
 * library recorded on the current device since the last call (for example
 * GDN_ERR_TIMEOUT from a bounded wait), or GDN_ERR_LAUNCH if the stream
 * reports a CUDA error; clears the recorded device error.
 */
gdn_status gdn_sync_status(gdn_stream_t stream);

/*
 * Upper bound, in nanoseconds, of every device-side wait (mbarrier phase
 * waits) in this library's kernels; a wait that runs out records
 * GDN_ERR_TIMEOUT and the kernel returns early.  Default 2e9 (2 s).
 * Values < 1000 are raised to 1000.  Applies to launches after the call.
 */
void gdn_set_wait_limit_ns(unsigned long long limit_ns);

/*
 * Schedule of phases 2 and 3.  mode 1 (default): when the device supports
 * cooperative launches and the heads leave most SMs free, the scan and the
 * output pass run as one cooperative launch in which output CTAs consume each
 * frame's state as soon as the scan CTAs publish it.  mode 16, 32 or 64: the
 * same, with that many state rows per scan CTA (if dv allows it).  mode 0:
 * the scan and the output pass run as two ordinary launches.  All schedules
 * give identical results.  Applies to calls made after it returns.
 */
void gdn_set_fused_scan(int mode);

/*
 * Work plan of phase 1.  Phase 1 runs (b, f, h) items round-robin over one CTA
 * per SM.  The items left over after the last full round can be split into
 * token ranges, one CTA each, whose fp32 partial sums are then added in split
 * order (the launch is then cooperative).  max_split 0 (default): split only
 * items of at least 32 chunks of 64 tokens, into as many ranges as the free
 * CTAs and the chunks allow; 1: never split; k > 1: split the leftover items
 * into up to k ranges whatever their length.  Results are deterministic for
 * every setting; different settings round the split items' sums in a
 * different order.  Applies to calls made after it returns.  A scheduling
 * control of this library; the pages have no counterpart.
 */
void gdn_set_contract_split(int max_split);

/*
 * The one-launch step.  on != 0 (default): gdn_frame_step and
 * gdn_frame_step_noalloc run a frame with bf16 inputs as one kernel: one
 * thread-block cluster of 4 CTAs per head splits the frame's contraction by
 * its columns (two CTAs form A, two form U, each over all tokens), the U CTAs
 * advance the state rows with A received through distributed shared memory,
 * and all four write outputs for a quarter of the frame's 128-token tiles,
 * with no workspace in HBM and no cross-CTA sums.  on = 0: the three-phase
 * path (two launches and a workspace).  The two agree to bf16 rounding: the
 * one-launch step rounds the product beta k (or beta v) on the other factor
 * of each contraction term than phase 1 does.  Applies to calls made after it
 * returns.  A scheduling control of this library; the pages have no
 * counterpart.
 */
void gdn_set_fused_step(int on);

/*
 * The single-pass forward.  on != 0 (default): gdn_frame_forward and its
 * reverse, folded-prologue and 8-bit variants run a sequence of F >= 2
 * frames as ONE cooperative launch when the device allows it and B*H is at
 * most a quarter of the SMs: one CTA per head runs the scan, about half of
 * the other SMs (48.5 % for bf16, 57.5 % fp8, 60.5 % NVFP4, 60.6 % with the
 * folded prologue) run the frame-parallel contractions and the rest the output
 * pass, each frame handed on through small ring buffers of the workspace
 * that stay in L2 (per-slot counts raised with release semantics, bounded
 * acquire waits), so HBM carries only the layer's own inputs and outputs.
 * on = 0: phase 1 as its own launch followed by phases 2 and 3
 * (gdn_set_fused_scan).  contract_ctas > 0 fixes the number of contraction
 * CTAs and ring_frames > 0 the ring depth in frames (0: automatic; a
 * forced depth is raised to at least 2 and capped at F).  The
 * schedules differ only in the order of rounding of the scan's S * A_f
 * product (the single pass multiplies by A_f's rows, the other schedules by
 * its columns; A_f is symmetric): results agree to bf16 rounding.  Applies
 * to calls made after it returns.  A scheduling control of this library; the
 * pages have no counterpart.
 */
void gdn_set_single_pass(int on, int contract_ctas, int ring_frames);

/*
 * Schedule gdn_frame_forward takes for this shape on the current device:
 * 2 single pass, 1 phase 1 then phases 2 and 3 in one cooperative launch,
 * 0 three launches, -1 invalid shape or no usable device.
 */
int gdn_forward_schedule(int B, int H, int F, int N, int dk, int dv);

/*
 * Schedule phases 2 and 3 take for this shape on the current device: +R when
 * they run as one cooperative launch with R rows of S per scan CTA, -R when
 * they run as two launches, 0 for invalid shapes or no usable device.
 */
int gdn_scan_schedule(int B, int H, int dv);

/*
 * Self-test of the bounded-wait machinery: launches one small kernel that
 * waits on a shared-memory barrier that nothing ever completes, with a wait
 * limit of `limit_ns`; the wait runs out, the kernel records GDN_ERR_TIMEOUT
 * and returns.  No fault, trap or hang is involved.  Read the result with
 * gdn_sync_status().
 */
gdn_status gdn_selftest_wait_timeout(unsigned long long limit_ns, gdn_stream_t stream);

/*
 * Diagnostics of the bounded waits: copies to info[0..4] where the first wait
 * that ran out since the last call gave up -- {site, block index, thread
 * index, value seen, value awaited} (site 0: no wait ran out; site codes are
 * role * 10000 + step or unit, for example 1320000 + f: a scan CTA waiting
 * for frame f's contraction) -- and clears the record.  Synchronous; call it
 * after gdn_sync_status reported GDN_ERR_TIMEOUT.
 */
gdn_status gdn_debug_last_timeout(int* info);

/* Library version string. */
const char* gdn_version(void);

/*
 * Allocation-free variant of gdn_frame_step.  No counterpart in the SANA-WM
 * pages: it exists for callers that cannot allocate device memory when they
 * advance the state -- for example a resident interactive rollout that
 * reserved (nearly) all device memory up front for its models, or a runtime
 * whose allocator must not be entered from this code path -- so the
 * stream-ordered workspace allocation of gdn_frame_step is not an option.
 *
 * Same arguments, layouts, results and validation as gdn_frame_step.  The
 * workspace lives instead in one fixed array of GDN_STEP_NOALLOC_SCRATCH_BYTES
 * bytes in the library's device image: every GPU that loads the library
 * holds it until the process exits.  No call allocates or frees memory.
 *   - With the one-launch step on (gdn_set_fused_step, the default) the call
 *     uses no scratch at all.  Otherwise it uses the array: a shape whose
 *     workspace (gdn_step_workspace_bytes, the same work plan) exceeds it
 *     returns GDN_ERR_TOO_LARGE before anything is launched.
 *   - The first call on each device, whichever step path it takes, looks up
 *     the array's device address (cudaGetSymbolAddress) with that device
 *     current; make that first call before any stream capture starts.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents; each call clears the counters it uses with a stream-ordered
 *     memset and writes every other scratch byte before reading it.  Calls
 *     that may overlap on the GPU (different streams, or unordered host
 *     threads) race on the array: order them, for example by issuing them on
 *     one stream.
 *   - The looked-up address (like the library's other per-device state) is
 *     kept for the life of the process: resetting a device
 *     (cudaDeviceReset) while the library is loaded is not supported.
 */
#define GDN_STEP_NOALLOC_SCRATCH_BYTES (32u << 20)
gdn_status gdn_frame_step_noalloc(const void* q, const void* k, const void* v,
                                  const float* alpha, const float* beta,
                                  const float* state_in, void* out, float* state_out,
                                  int B, int H, int N, int dk, int dv,
                                  gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_B300_H */
