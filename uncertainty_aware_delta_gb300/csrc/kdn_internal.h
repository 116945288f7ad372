// Internal launchers of the KDN library (host side; not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kdn {

struct ForwardArgs {
    int variant;  // 0 diagonal, 1 isotropic, 2 PKDA (preconditioned delta rule)
    int B, T, H, dk, dv, chunk;
    float mu;
    int io;       // 0 fp32, 1 bf16
    const void *q, *k, *v;
    const float *log_alpha, *omega, *r, *S0, *p0;   // PKDA: p0 is the initial key statistic
    void* o;
    float *S_T, *p_T;                               // PKDA: p_T is the final key statistic
    uint32_t* status;  // device status word
    // PKDA only: beta, alpha_p, beta_p [B,T,H], center [H], -log2(x)
    const float *beta, *alpha_p, *beta_p, *center;
    float neg_log2x;
    uint32_t flags;    // KDN_FLAG_* of the call
    // KDN: effective write strength k^T kappa [B,T,H] fp32, or null (not written).
    // The tensor-core path writes it only when it runs whole sequences.
    float* beta_eff;
};

// Gate branches on pre-activations into fp32 log_alpha [B,T,H,dk], omega
// [B,T,H,dk] (diagonal) or [B,T,H] (isotropic) and r [B,T,H], for the paths that
// take fp32 gates.  gates.cu
cudaError_t launch_gate_expand(int variant, int B, int T, int H, int dk, int io, float r_min,
                               const void* alpha_logit, const void* omega_logit, const void* r_logit,
                               float* log_alpha, float* omega, float* r, cudaStream_t s);
// beta_eff [B,T,H] = sum_i k_i kappa_i from the gain scan's kappa [B,T,H,dk].  gates.cu
cudaError_t launch_beta_from_kappa(int B, int T, int H, int dk, int io, const void* k, const float* kappa,
                                   float* beta_eff, cudaStream_t s);

// Gain-scan workspace (CUDA-core path): gains and Moebius chunk summaries.
struct ScanWorkspace {
    float* kappa;      // [B,T,H,dk]
    float* summary;    // [B*H, nG, nu, 4]
    float* carry;      // [B*H, nG, nu]
    int chunk_g;       // tokens per gain chunk
    int n_chunks_g;
};

constexpr int kGainChunk = 256;

// Moebius 2x2 gain scan (KDN), or the key-statistic scan and write keys
// (PKDA): writes kappa [B,T,H,dk] and p_T.  scan.cu
cudaError_t launch_gain_scan(const ForwardArgs& a, const ScanWorkspace& w, cudaStream_t s);

// CUDA-core chunkwise memory pass (compact-WY/UT form, fp32 FFMA).  chunk_simt.cu
cudaError_t launch_chunk_simt(const ForwardArgs& a, const float* kappa, cudaStream_t s);

// Single-token decode, state in place.  step.cu
struct StepArgs {
    int variant, B, H, dk, dv, io;
    float mu;
    const void *q, *k, *v;
    const float *log_alpha, *omega, *r;
    float *S, *p;       // PKDA: p is the key statistic
    void* o;
    uint32_t* status;
    const float *beta, *alpha_p, *beta_p, *center;   // PKDA only
    float neg_log2x;
    uint32_t flags;     // KDN_FLAG_* of the call
};
cudaError_t launch_step(const StepArgs& a, cudaStream_t s);

// Chunk summaries and exclusive carries only (no replay) of the gain scan (KDN)
// or the statistic scan (PKDA): w.carry [B*H, n_chunks_g, nu] holds the
// recurrence's value at the start of every gain chunk.  scan.cu
cudaError_t launch_scan_carries(const ForwardArgs& a, const ScanWorkspace& w, cudaStream_t s);

// Fused tensor-core forward (gain scan + compact-WY chunk pass).  chunk_tc.cu
bool tc_path_supported(int io, int dk, int dv, int chunk);

// Sequence split of the tensor-core forward for few long sequences: nseg
// segments of seg_len tokens (a multiple of kGainChunk) per sequence run on
// separate SMs.  The state map of a segment is affine, S_out = Phi S_in + S_loc;
// one pass gives every segment's S_loc and outputs o_loc (from S = 0), one its
// Phi and transformed queries Phi_t^T q_t (from S = I, values zero), a short
// serial pass chains the maps into each segment's initial state and the final
// state, and o_t = o_loc,t + S_in^T (Phi_t^T q_t) completes the outputs.
struct TcSplit {
    int nseg = 1, seg_len = 0;          // nseg == 1: no split
    float* summary = nullptr;           // scan workspace (gain chunks of kGainChunk tokens)
    float* carry = nullptr;
    int n_chunks_g = 0;
    float* S_loc = nullptr;             // [B*H*nseg][dk][dv] each
    float* Phi = nullptr;
    float* S_in = nullptr;              // chained initial states, held as bf16 S_in^T [j][i]
    void* qt = nullptr;                 // [B][T][H][dk] bf16: q~_t = Phi_t^T q_t of each segment
};
TcSplit tc_split_plan(int B, int T, int H, uint32_t flags);   // nseg and seg_len only
cudaError_t launch_forward_tc(const ForwardArgs& a, const TcSplit& sp, cudaStream_t s);
int tc_kernel_count(int nseg);
// Sequence split, after the two map passes: chained initial states S_in (as bf16
// S_in^T) and the final state, then o += S_in^T q~ per segment.  split.cu
cudaError_t launch_segment_states(const ForwardArgs& a, const TcSplit& sp, cudaStream_t s);
cudaError_t launch_segment_correction(const ForwardArgs& a, const TcSplit& sp, cudaStream_t s);

// Dense-covariance (exact) Kalman memory forward.
struct DenseArgs {
    int B, T, H, d, io;
    const void *q, *k, *v;
    const float *log_alpha, *omega, *r, *S0, *P0;
    void* o;
    float *S_T, *P_T;
};
// The covariance recurrence token by token: kappa [B,T,H,d] fp32 and P_T.  dense.cu
cudaError_t launch_dense_covariance(const DenseArgs& a, float* kappa, cudaStream_t s);

// Copy the initial state to the outputs (T == 0).  chunk_simt.cu
cudaError_t launch_state_copy(const ForwardArgs& a, cudaStream_t s);

// Backward pass (gradients of sum(dO o) + sum(dS_T S_T) + sum(dp_T p_T)).  backward.cu
struct BackwardArgs {
    int variant, B, T, H, dk, dv, io;   // variant: 0 diagonal, 1 isotropic
    float mu;
    const void *q, *k, *v, *dO;
    const float *log_alpha, *omega, *r, *S0, *p0, *dS_T, *dp_T;
    float *dq, *dk_out, *dv_out, *dla, *domega, *dr, *dS0, *dp0;
    uint32_t* status;
};
struct BackwardWorkspace {
    float* kappa;      // [B,T,H,dk] gains from the gain scan
    float* summary;    // gain-scan chunk summaries and carries
    float* carry;
    int n_chunks_g;
    float* p_scratch;  // [B*H, nu] (the scan's final variances, unused)
    float* ckpt;       // [B*H][ceil(T / chunk) + 1][dk][dv] states at memory-chunk starts
    float* dkappa;     // [B,T,H,dk]
    float* pck;        // [B*H][ceil(T / block)][nu] variances at gain-adjoint block starts
};
cudaError_t launch_backward(const BackwardArgs& a, const BackwardWorkspace& w, cudaStream_t s);
size_t backward_mem_smem_bytes(int dk, int dv);
int backward_chunk();   // tokens per memory-adjoint chunk
int backward_block();   // tokens per gain-adjoint checkpoint block

}  // namespace kdn
