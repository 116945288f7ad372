/*
 * kdn.h -- C ABI of the GB300 (sm_103a) Kalman Delta Network mixer library.
 *
 * The library computes the forward mixer of a Kalman Delta Network (KDN):
 * "Kalman Delta Networks: Uncertainty-aware Associative Memory" (Bui, Huang,
 * Ying, arXiv:2609.07816v1).  Per head it keeps a memory S (d_k x d_v, row =
 * key channel) and an uncertainty state (d_k variances for the Diagonal
 * variant, one scalar for the Isotropic variant), and for every token t:
 *
 *   predict   S_hat = diag(a_t) S,   a_t = exp(log_alpha_t)         (Sec. 3.2 Eq. 12)
 *             Diagonal:  p_hat = a_t^2 * p + omega_t                (Sec. 4.1 Eq. 23)
 *             Isotropic: b_hat = mean_i(a_t,i^2) * b + omega_t      (Sec. 4.2 Eq. 40)
 *   gain      Diagonal:  kappa = p_hat * k / (r_t + sum_i p_hat_i k_i^2)   (Eq. 24-27)
 *             Isotropic: kappa = k * b_hat / (r_t + b_hat ||k||^2)
 *   write     S = S_hat + kappa (v_t - S_hat^T k_t)^T               (Eq. 13-16, 38-39)
 *   read      o_t = S^T q_t            (after the write)            (Eq. 17)
 *   update    Diagonal:  p = p_hat / (1 + (mu / r_t) k^2 * p_hat)   (Eq. 60-65)
 *             Isotropic: b = b_hat / (1 + mu ||k||^2 / (d_k r_t) * b_hat)   (App. C)
 *
 * The uncertainty recurrence is a Moebius map evaluated as a 2x2 associative
 * scan (Eq. 32-37); the memory write is evaluated chunk by chunk in the
 * compact-WY / UT form (App. D).  Results do not depend on the chunk length
 * beyond floating-point rounding.
 *
 * The same memory machinery also runs the preconditioned delta rule with
 * per-channel decay (PKDA; "Preconditioned DeltaNet", arXiv:2604.21100v1,
 * Sec. 2.4 Eq. 9 and Sec. 2.5), whose write key is the read key rescaled per
 * channel by a bounded function of a decayed key statistic; see
 * kdn_pkda_forward.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains them and keeps no global mutable state
 *     (re-entrant; concurrent calls on different streams with disjoint buffers
 *     are safe).  The one exception is kdn_forward_noalloc, which uses a
 *     library-owned static device array and a per-device cache of its address
 *     (see that entry point for the sharing rules).
 *   - Layouts are dense row-major with the feature dimension innermost:
 *       q, k, log_alpha       [B, T, H, d_k]
 *       v, o                  [B, T, H, d_v]
 *       omega                 [B, T, H, d_k] (Diagonal) or [B, T, H] (Isotropic)
 *       r                     [B, T, H]   observation-noise VARIANCE, > 0
 *       S0, S_T, S            [B, H, d_k, d_v] fp32
 *       p0, p_T, p            [B, H, d_k] (Diagonal) or [B, H] (Isotropic) fp32
 *     q, k, v and o are stored as io_dtype (KDN_F32 or KDN_BF16); every other
 *     tensor is fp32.  Arithmetic is fp32 (tensor-core operands bf16 on the
 *     bf16 path, fp32 accumulation and fp32 state).
 *   - Every pointer must be 16-byte aligned.
 *   - Outputs must not overlap inputs, except S_T == S0 and p_T == p0 (resume
 *     in place), which are allowed.
 *   - mu < 0 selects mu = d_k (the paper's default information scale).
 *   - Host-side validation runs before anything is enqueued and returns
 *     synchronously.  Kernels are enqueued on `stream`; the call returns
 *     without synchronising.  A launch failure returns KDN_ERR_CUDA.
 *   - Conditions found on the device (a bounded wait that gave up, a chunk
 *     whose cumulative log-decay is outside the safe range) are recorded in a
 *     status word at the start of the workspace; kdn_read_device_status()
 *     returns it.  No kernel traps, asserts, prints or spins without bound.
 *   - Nothing throws across the ABI.
 */
#ifndef KDN_H
#define KDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *kdn_stream_t;

typedef enum {
    KDN_OK = 0,
    KDN_ERR_NULL = 1,         /* a required pointer is NULL                          */
    KDN_ERR_SHAPE = 2,        /* a size is negative, or sizes are inconsistent       */
    KDN_ERR_DTYPE = 3,        /* io_dtype is not KDN_F32 or KDN_BF16                 */
    KDN_ERR_ALIGN = 4,        /* a pointer is not 16-byte aligned                    */
    KDN_ERR_WORKSPACE = 5,    /* workspace NULL or smaller than kdn_workspace_size() */
    KDN_ERR_UNSUPPORTED = 6,  /* d_k, d_v or chunk outside the supported set         */
    KDN_ERR_CUDA = 7,         /* a CUDA runtime call or kernel launch failed         */
    KDN_ERR_TIMEOUT = 8,      /* device: a bounded wait gave up (results invalid)    */
    KDN_ERR_RANGE = 9,        /* device: a chunk's cumulative log-decay left the
                                 range the factored decay supports (results invalid) */
    KDN_ERR_ALIAS = 10        /* an output overlaps an input (other than S/p resume) */
} kdn_status;

typedef enum { KDN_F32 = 0, KDN_BF16 = 1 } kdn_dtype;
typedef enum { KDN_DIAG = 0, KDN_ISO = 1, KDN_PKDA = 2 } kdn_variant;

/* Flags for the forward calls (and kdn_step_ex). */
#define KDN_FLAG_PORTABLE 0x1u   /* force the CUDA-core (FFMA) chunk path */
#define KDN_FLAG_NO_SPLIT 0x2u   /* tensor-core path: never split sequences into segments */
/*
 * Test facility for the bounded-wait path; never set it in production.  The
 * kernels that wait on asynchronous copies (the tensor-core forward and the
 * d_k = d_v = 128 decode kernel) first wait, with a short bound (a few
 * milliseconds), on a barrier that nothing completes, while their first
 * copies are in flight.  The wait gives up, the status word records
 * KDN_ERR_TIMEOUT, and each CTA takes its abort path: it issues no further
 * work, lets the copies already issued land and exits.  The outputs of such
 * a call are undefined; the stream and the device stay usable.  Other paths
 * (CUDA-core forward, other decode shapes, the dense filter) ignore the flag.
 */
#define KDN_FLAG_TIMEOUT_PROBE 0x100u

/*
 * Sequence split (tensor-core path).  When B*H sequences would leave most of
 * the GPU idle (2*B*H <= N_SM, the SM count of the current device: 152 on
 * GB300, and 152 when no device can be queried) and each is long
 * (T >= 2048), every sequence is cut into nseg = min(N_SM / (B*H), T / 1024)
 * segments of a multiple of 256 tokens that run on separate SMs.  The plan,
 * and therefore kdn_workspace_size() and kdn_forward_kernel_count(), depend on
 * the device that is current when they are called: query them with the same
 * device current as the forward call.  The method's state map over a segment is
 * affine, S_out = Phi S_in + S_loc, for the segment's gains, which depend only
 * on the uncertainty (statistic) recurrence: a scan over the whole sequence
 * gives each segment's initial uncertainty; one pass from S = 0 gives every
 * segment's S_loc and its outputs o_loc, one from S = I with zero values gives
 * Phi and the transformed queries Phi_t^T q_t; a short serial pass chains the
 * maps into each segment's initial state S_in and the final state, and the
 * outputs are completed as o_t = o_loc,t + S_in^T (Phi_t^T q_t).  The result is
 * the same recurrence up to rounding (the correction term is formed with bf16
 * operands); the cost is about twice the arithmetic on nseg times the SMs.
 * kdn_workspace_size() includes the per-segment states and the transformed
 * queries (2 bytes per token-head-channel); KDN_FLAG_NO_SPLIT keeps one CTA per
 * sequence.
 */

/*
 * Supported sizes: d_k, d_v in {16, 32, 64, 128}; chunk in {16, 32, 64}
 * (0 selects 64, or T rounded up to 16 when T < 64); any T >= 0 (a ragged
 * tail chunk is masked; T == 0 copies the initial state to the outputs);
 * B, H >= 0.  The tensor-core path is used for bf16 io with d_k = d_v = 128
 * and chunk 64; every other supported case runs on the CUDA-core path.
 */

/*
 * Bytes of device workspace a forward (T > 0) or step (T == 1) call needs.
 * variant: KDN_DIAG, KDN_ISO or KDN_PKDA.  Returns 0 for unsupported arguments.  The
 * workspace is scratch owned by the caller, at least 256-byte aligned; its
 * first 256 bytes hold the device status word.  Calls that overlap in time
 * must use different workspaces.
 */
size_t kdn_workspace_size(int variant, int B, int T, int H, int dk, int dv, int chunk,
                          int io_dtype, uint32_t flags);

/*
 * Diagonal KDN forward over T tokens (KDN paper Sec. 4.1, Eq. 23-30 and
 * 60-65; Moebius scan Eq. 32-37; chunkwise form App. D).
 *
 * Inputs : q, k [B,T,H,dk] io_dtype; v [B,T,H,dv] io_dtype;
 *          log_alpha [B,T,H,dk] (log of the per-channel decay, <= 0 in use);
 *          omega [B,T,H,dk] process-noise variance >= 0; r [B,T,H] > 0;
 *          S0 [B,H,dk,dv] or NULL (zero memory); p0 [B,H,dk] or NULL (ones).
 * Outputs: o [B,T,H,dv] io_dtype (read after each token's write);
 *          S_T [B,H,dk,dv], p_T [B,H,dk]: the state after token T-1 (the
 *          mu-scaled posterior variances), the resume point for kdn_step or
 *          a later forward call.
 * mu     : information scale (< 0 selects d_k); chunk: see above.
 * Errors : KDN_ERR_* from validation, KDN_ERR_CUDA on a launch failure.
 */
kdn_status kdn_diag_forward(int B, int T, int H, int dk, int dv, int chunk, float mu,
                            int io_dtype, uint32_t flags,
                            const void *q, const void *k, const void *v,
                            const float *log_alpha, const float *omega, const float *r,
                            const float *S0, const float *p0,
                            void *o, float *S_T, float *p_T,
                            void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * Isotropic KDN forward (KDN paper Sec. 4.2, Eq. 40; App. C): one
 * uncertainty scalar per head, omega [B,T,H], p0 and p_T [B,H].  The mean
 * path keeps the per-channel transition diag(a_t).  Everything else as
 * kdn_diag_forward.
 */
kdn_status kdn_iso_forward(int B, int T, int H, int dk, int dv, int chunk, float mu,
                           int io_dtype, uint32_t flags,
                           const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *omega, const float *r,
                           const float *S0, const float *p0,
                           void *o, float *S_T, float *p_T,
                           void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * KDN forward driven by the layer's gate pre-activations (the fused gate
 * prologue).  KDN reading notes Sec. 5.1: the end-to-end network produces
 *
 *   alpha_t = sigma(a_t),  omega_t = softplus(w_t),  r_t = r_min + softplus(rho_t),
 *
 * where a, w, rho are the projections W x + b of the layer input (computing
 * them is the caller's GEMM).  This call takes a, w, rho and runs the forward of
 * kdn_diag_forward / kdn_iso_forward on log alpha = log sigma(a) = -softplus(-a),
 * omega and r.  Optionally it also writes the effective write strength of every
 * token (reading notes Sec. 3.2; the paper's App. B, Eq. 58-61)
 *
 *   beta_eff_t = k_t^T kappa_t = z_t / (r_t + z_t),   z_t = k_t^T P_hat_t k_t,
 *
 * the fraction of the innovation along k_t that the write removes, in [0, 1).
 *
 * variant: KDN_DIAG or KDN_ISO (other values: KDN_ERR_SHAPE).
 * Inputs : q, k, v, S0, p0, mu, chunk, flags as kdn_diag_forward / kdn_iso_forward;
 *          alpha_logit [B,T,H,dk] io_dtype; omega_logit [B,T,H,dk] (diagonal) or
 *          [B,T,H] (isotropic) io_dtype; r_logit [B,T,H] io_dtype.
 *          r_min: floor of the observation-noise variance (< 0 selects the notes'
 *          0.01; NaN or infinity returns KDN_ERR_SHAPE).
 * Outputs: o, S_T, p_T as the ungated forward; beta_eff [B,T,H] fp32, or NULL.
 * Paths  : one elementwise kernel over every SM evaluates the three branches from
 *          the logits into fp32 log alpha, omega and r in the workspace; the
 *          ungated forward path for these sizes (see "Supported sizes") then runs on
 *          them.  beta_eff comes from the gains that path forms: on the tensor-core
 *          path from the diagonal of the chunk's gain system, z_t = r_t +
 *          k_t^T P_hat_t k_t (requesting it keeps one CTA per sequence: no sequence
 *          split), on the CUDA-core path as k^T kappa from the gain scan.  (The
 *          branches evaluated inside the fused kernel's gain pass instead were measured
 *          slower: that pass is serial per token and the transcendentals lengthen it.)
 * Workspace: kdn_gated_workspace_size() bytes (at least kdn_workspace_size() of
 *          the same arguments).
 * Errors : as kdn_diag_forward; KDN_ERR_ALIAS also when beta_eff overlaps an
 *          input or another output.
 */
size_t kdn_gated_workspace_size(int variant, int B, int T, int H, int dk, int dv, int chunk,
                                int io_dtype, uint32_t flags);
kdn_status kdn_gated_forward(int variant, int B, int T, int H, int dk, int dv, int chunk, float mu,
                             float r_min, int io_dtype, uint32_t flags,
                             const void *q, const void *k, const void *v,
                             const void *alpha_logit, const void *omega_logit, const void *r_logit,
                             const float *S0, const float *p0,
                             void *o, float *S_T, float *p_T, float *beta_eff,
                             void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * Preconditioned delta rule with per-channel decay, PKDA ("Preconditioned
 * DeltaNet", arXiv:2604.21100v1: Sec. 2.4 Eq. 9, the write key; Sec. 2.5, the
 * decayed state; Sec. 2.6, its chunkwise form).  PGDN is the special case of
 * a log_alpha equal across channels, PDN the case log_alpha = 0.  Per head,
 * memory S (d_k x d_v, row = key channel) and key statistic A (d_k), and for
 * every token t:
 *
 *   A      = alpha_p_t A + beta_p_t (k_t * k_t)           (this token included)
 *   rho    = log(max(A, 1e-20)) - center_h                (centred in log space)
 *   k_til  = exp(-log(x) rho / (1 + |rho|)) * k_t         (softsign; scale in [1/x, x])
 *   S_hat  = diag(exp(log_alpha_t)) S
 *   S      = S_hat + beta_t k_til (v_t - S_hat^T k_t)^T   (residual with the read key)
 *   o_t    = S^T q_t                                      (after the write)
 *
 * Inputs : q, k [B,T,H,dk] io_dtype; v [B,T,H,dv] io_dtype;
 *          log_alpha [B,T,H,dk] (log of the per-channel state decay);
 *          beta [B,T,H] write strength; alpha_p [B,T,H] statistic decay in
 *          [0, 1]; beta_p [B,T,H] statistic weight >= 0; center [H] the
 *          per-head log-space centre (the pages' mu > 0);
 *          S0 [B,H,dk,dv] or NULL (zero memory); A0 [B,H,dk] or NULL (zero
 *          statistic).
 * Outputs: o [B,T,H,dv] io_dtype; S_T [B,H,dk,dv]; A_T [B,H,dk] (the state
 *          after token T-1, the resume point of kdn_pkda_step or a later call).
 * x      : bound of the write scale (the pages use 1.5); x <= 0 selects 1.5.
 * Sizes, paths, workspace (variant KDN_PKDA), flags, aliasing (S_T == S0 and
 * A_T == A0 allowed) and errors: as kdn_diag_forward.
 */
kdn_status kdn_pkda_forward(int B, int T, int H, int dk, int dv, int chunk, float x,
                            int io_dtype, uint32_t flags,
                            const void *q, const void *k, const void *v,
                            const float *log_alpha, const float *beta, const float *alpha_p,
                            const float *beta_p, const float *center,
                            const float *S0, const float *A0,
                            void *o, float *S_T, float *A_T,
                            void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * Single-token decode for B independent sequences (the recurrent form of
 * the same recurrence; KDN paper Sec. 5.1 and App. C): one token per
 * (sequence, head), state updated IN PLACE.
 *
 * variant: KDN_DIAG or KDN_ISO.
 * Inputs : q, k [B,H,dk] io_dtype; v [B,H,dv] io_dtype; log_alpha [B,H,dk];
 *          omega [B,H,dk] (Diagonal) or [B,H] (Isotropic); r [B,H].
 * In/out : S [B,H,dk,dv], p [B,H,dk] or [B,H] (fp32).
 * Output : o [B,H,dv] io_dtype.
 * Workspace: kdn_workspace_size(variant, B, 1, H, dk, dv, 0, io_dtype, 0) bytes.
 */
kdn_status kdn_step(int variant, int B, int H, int dk, int dv, float mu, int io_dtype,
                    const void *q, const void *k, const void *v,
                    const float *log_alpha, const float *omega, const float *r,
                    float *S, float *p, void *o,
                    void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * kdn_step with flags: the same call, arguments and workspace.  flags may be 0
 * or KDN_FLAG_TIMEOUT_PROBE (see above); other bits return
 * KDN_ERR_UNSUPPORTED.
 */
kdn_status kdn_step_ex(int variant, int B, int H, int dk, int dv, float mu, int io_dtype, uint32_t flags,
                       const void *q, const void *k, const void *v,
                       const float *log_alpha, const float *omega, const float *r,
                       float *S, float *p, void *o,
                       void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * Single-token PKDA decode (one token of kdn_pkda_forward per sequence and
 * head), state updated IN PLACE.
 * Inputs : q, k [B,H,dk] io_dtype; v [B,H,dv] io_dtype; log_alpha [B,H,dk];
 *          beta, alpha_p, beta_p [B,H]; center [H].
 * In/out : S [B,H,dk,dv], A [B,H,dk] (fp32).
 * Output : o [B,H,dv] io_dtype.
 * Workspace: kdn_workspace_size(KDN_PKDA, B, 1, H, dk, dv, 0, io_dtype, 0) bytes.
 */
kdn_status kdn_pkda_step(int B, int H, int dk, int dv, float x, int io_dtype,
                         const void *q, const void *k, const void *v,
                         const float *log_alpha, const float *beta, const float *alpha_p,
                         const float *beta_p, const float *center,
                         float *S, float *A, void *o,
                         void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * Dense-covariance (exact) Kalman memory forward (KDN paper Sec. 3.2, Eq. 12-17):
 * the filter that the Diagonal and Isotropic KDN approximate.  Per head a
 * memory S (d x d) and a full key covariance P (d x d); for every token, with
 * a_t = exp(log_alpha_t):
 *
 *   P_hat = diag(a_t) P diag(a_t) + diag(omega_t),  u = P_hat k_t,
 *   kappa = u / (r_t + k_t^T u),  P = P_hat - kappa u^T  (= (I - kappa k^T) P_hat),
 *   S_hat = diag(a_t) S,  S = S_hat + kappa (v_t - S_hat^T k_t)^T,  o_t = S^T q_t.
 *
 * Inputs : q, k, v [B,T,H,d] io_dtype; log_alpha, omega [B,T,H,d] fp32;
 *          r [B,T,H] fp32 > 0; S0 [B,H,d,d] or NULL (zero memory);
 *          P0 [B,H,d,d] or NULL (identity), symmetric positive semi-definite.
 * Outputs: o [B,T,H,d] io_dtype; S_T, P_T [B,H,d,d] fp32 (the state after token
 *          T-1; S_T == S0 and P_T == P0 are allowed).
 * Sizes  : d in {32, 64, 128} (d_k = d_v = d); any T >= 0; B, H >= 0.
 * Two passes.  The covariance recurrence runs in token order, one CTA per head,
 * and writes the gains kappa_t [B,T,H,d] fp32 into the workspace.  The decay is
 * held outside P (P = G Ptil G for a diagonal G of decay factors), so a token
 * costs one matrix-vector product and one rank-1 downdate, 2 d^2 multiply-adds.
 * For d = 128 the tokens go in blocks of up to 16 with Ptil in shared memory:
 * the block's products run on tensor cores (3xTF32, fp32-level accuracy) and a
 * 16 x 16 elimination gives every token's gain from the block-start covariance.
 * A block ends early where a channel's log decay within it would exceed 40.  For
 * d = 32 and 64 the tokens go in pairs with Ptil in registers, and G is folded
 * into Ptil whenever a channel's running decay would fall below 2^-20.  Given
 * the gains, the mean
 * S = diag(a) S + kappa (v - (diag(a) S)^T k)^T is the delta rule with write
 * key kappa and runs chunkwise: on the fused tensor-core kernel (bf16 io,
 * d = 128, T > 32) or on the CUDA-core chunk path.
 * Workspace: kdn_dense_workspace_size() bytes (its first 256 bytes hold the
 *          device status word; then kappa, 4 B T H d bytes).
 * Alignment, aliasing and errors as kdn_diag_forward.
 */
size_t kdn_dense_workspace_size(int B, int T, int H, int d, int io_dtype);
kdn_status kdn_dense_forward(int B, int T, int H, int d, int io_dtype,
                             const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *omega, const float *r,
                             const float *S0, const float *P0,
                             void *o, float *S_T, float *P_T,
                             void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * Backward pass of the Diagonal or Isotropic KDN forward: the gradients of
 *
 *     L = sum(dO * o) + sum(dS_T * S_T) + sum(dp_T * p_T)
 *
 * with respect to every input of kdn_diag_forward / kdn_iso_forward.  The pages
 * define the forward recurrence only (KDN paper Sec. 4.1 Eq. 23-27 and 60-65, Sec.
 * 4.2 Eq. 40 and App. C); these are the exact adjoint of that recurrence (its
 * training scans, Sec. 5.1), evaluated in the compact-WY chunk form of App. D with
 * the gains from the forward's Moebius gain scan (Eq. 32-37), on CUDA cores in fp32.
 *
 * variant: KDN_DIAG or KDN_ISO.  Inputs q, k, v, log_alpha, omega, r, S0, p0, mu
 * and io_dtype exactly as for the forward call being differentiated (S0, p0 may be
 * NULL: zero memory, unit variances).  Upstream gradients: dO [B,T,H,dv] in
 * io_dtype, dS_T [B,H,dk,dv] and dp_T ([B,H,dk] or [B,H]) fp32; each may be NULL
 * (zero).  Outputs, all fp32, all required: grad_q, grad_k [B,T,H,dk]; grad_v
 * [B,T,H,dv]; grad_log_alpha [B,T,H,dk]; grad_omega [B,T,H,dk] (Diagonal) or
 * [B,T,H] (Isotropic); grad_r [B,T,H]; grad_S0 [B,H,dk,dv]; grad_p0 [B,H,dk] or
 * [B,H] (the gradients with respect to S0 and p0, or to their defaults when those
 * are NULL).  Outputs must not overlap each other, the inputs or the workspace.
 * Sizes: dk, dv in {16, 32, 64, 128}; any T >= 0; B, H >= 0.
 * Workspace: kdn_backward_workspace_size() bytes (gains, the state at every
 * 16-token chunk start -- 4 dk dv bytes per chunk and head -- and the gain
 * gradients); its first 256 bytes hold the device status word.
 * Errors: as kdn_diag_forward; KDN_ERR_RANGE in the status word when a chunk's
 * cumulative log-decay leaves the supported range.
 */
size_t kdn_backward_workspace_size(int variant, int B, int T, int H, int dk, int dv, int io_dtype);

kdn_status kdn_backward(int variant, int B, int T, int H, int dk, int dv, float mu, int io_dtype,
                        const void *q, const void *k, const void *v,
                        const float *log_alpha, const float *omega, const float *r,
                        const float *S0, const float *p0,
                        const void *dO, const float *dS_T, const float *dp_T,
                        float *grad_q, float *grad_k, float *grad_v, float *grad_log_alpha,
                        float *grad_omega, float *grad_r, float *grad_S0, float *grad_p0,
                        void *workspace, size_t workspace_bytes, kdn_stream_t stream);

/*
 * Forward without a caller workspace.  The paper has no counterpart: this is
 * a convenience of the library for callers that cannot allocate device
 * memory at the point where they run the mixer -- for example code inside a
 * host framework that owns every device allocation and forbids cudaMalloc in
 * its execution callbacks, or a latency-critical loop that must not pay for
 * cudaMalloc/cudaFree, which can synchronise the whole device.
 *
 * The scratch the forward needs (per-token gains, Moebius chunk summaries,
 * the status word) comes from a library-owned static device array of
 * KDN_STATIC_SCRATCH_BYTES, which every GPU that loads the library holds
 * until the process exits.  This entry point calls no cudaMalloc, cudaFree
 * or other allocating routine.
 *
 * variant: KDN_DIAG or KDN_ISO (PKDA has no allocation-free entry point).
 * Every other argument means what it means for kdn_diag_forward / kdn_iso_forward; inputs and outputs are still
 * caller-owned device buffers.  status_out: NULL, or a caller-owned device
 * uint32_t (4-byte aligned) that receives this call's device status word on
 * `stream` (the codes kdn_read_device_status returns).
 *
 * Set-up: the first call on a device looks up the device address of the
 * static array, with that device current; make that first call before any
 * stream capture begins on the device.  The address is cached per device for
 * the life of the process: after cudaDeviceReset (or any teardown of the
 * device's primary context) the cached address is stale, so do not call this
 * entry point again in a process that has reset the device.
 *
 * Sharing: all calls in the process share the one array per device and it
 * keeps the last call's contents; each call clears what must start at zero
 * (the status word) and writes everything else before reading it.  Calls
 * whose work overlaps on the GPU (other streams, other host threads on the
 * same device) race on the array and corrupt each other's results: order
 * them on one stream or synchronise between them.
 *
 * Errors: KDN_ERR_WORKSPACE when the problem needs more scratch than
 * KDN_STATIC_SCRATCH_BYTES (kdn_workspace_size() gives the need; with
 * flags = 0 a bf16 forward with d_k = d_v = 128 needs about
 * 4 * B * T * H * d_k bytes on the CUDA-core path); otherwise as
 * kdn_diag_forward.
 */
#define KDN_STATIC_SCRATCH_BYTES (32u << 20)

kdn_status kdn_forward_noalloc(int variant, int B, int T, int H, int dk, int dv, int chunk,
                               float mu, int io_dtype, uint32_t flags,
                               const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *omega, const float *r,
                               const float *S0, const float *p0,
                               void *o, float *S_T, float *p_T, uint32_t *status_out,
                               kdn_stream_t stream);

/*
 * Synchronise `stream` and return the device status word the last call that
 * used `workspace` left there: KDN_OK, KDN_ERR_TIMEOUT or KDN_ERR_RANGE (or
 * KDN_ERR_CUDA if the copy itself fails, KDN_ERR_NULL for a NULL workspace).
 */
kdn_status kdn_read_device_status(const void *workspace, kdn_stream_t stream);

/*
 * Number of kernels one forward call with these arguments enqueues on its
 * stream (the status-word memset is not a kernel).  0 for rejected arguments
 * or an empty batch.  For capture into CUDA graphs and for launch accounting.
 */
int kdn_forward_kernel_count(int variant, int B, int T, int H, int dk, int dv, int chunk,
                             int io_dtype, uint32_t flags);

/* Static description of a status code (never NULL). */
const char *kdn_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
int kdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDN_H */
