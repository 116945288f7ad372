// C ABI of the KDN mixer library: argument validation, workspace carving and
// kernel dispatch.  See include/kdn.h for the contract of every entry point.

#include <cmath>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "kdn.h"
#include "kdn_internal.h"

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kStatusBytes = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool supported_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

int resolve_chunk(int chunk, int T) {
    if (chunk != 0) return chunk;
    if (T >= 64) return 64;
    if (T > 32) return 64;
    if (T > 16) return 32;
    return 16;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    const void* p;
    size_t n;
};

bool overlaps(Range a, Range b) {
    if (!a.p || !b.p || a.n == 0 || b.n == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Tensor-core path availability (set by chunk_tc.cu when compiled in).
bool use_tc_path(int io, int dk, int dv, int chunk, uint32_t flags) {
    if (flags & KDN_FLAG_PORTABLE) return false;
    return kdn::tc_path_supported(io, dk, dv, chunk);
}

struct WsLayout {
    size_t total;
    size_t kappa_off, summary_off, carry_off;
    int nG;
    // tensor-core sequence split: per-segment state maps and initial states
    kdn::TcSplit split;
    size_t sloc_off, phi_off, sin_off, qt_off;
};

WsLayout ws_layout(int variant, int B, int T, int H, int dk, int dv, int chunk, int io,
                   uint32_t flags) {
    WsLayout w;
    memset(&w, 0, sizeof(w));
    size_t off = kStatusBytes;
    if (T > 0 && !use_tc_path(io, dk, dv, chunk, flags)) {
        const int nu = variant == KDN_ISO ? 1 : dk;
        const size_t BH = (size_t)B * H;
        w.nG = (T + kdn::kGainChunk - 1) / kdn::kGainChunk;
        w.kappa_off = off;
        off = align_up(off + sizeof(float) * (size_t)B * T * H * dk);
        w.summary_off = off;
        off = align_up(off + sizeof(float) * 4 * BH * w.nG * nu);
        w.carry_off = off;
        off = align_up(off + sizeof(float) * BH * w.nG * nu);
    } else if (T > 0) {
        w.split = kdn::tc_split_plan(B, T, H, flags);
        if (w.split.nseg > 1) {
            const int nu = variant == KDN_ISO ? 1 : dk;
            const size_t BH = (size_t)B * H, nst = BH * w.split.nseg * dk * dv;
            w.nG = (T + kdn::kGainChunk - 1) / kdn::kGainChunk;
            w.summary_off = off;
            off = align_up(off + sizeof(float) * 4 * BH * w.nG * nu);
            w.carry_off = off;
            off = align_up(off + sizeof(float) * BH * w.nG * nu);
            w.sloc_off = off;
            off = align_up(off + sizeof(float) * nst);
            w.phi_off = off;
            off = align_up(off + sizeof(float) * nst);
            w.sin_off = off;
            off = align_up(off + sizeof(float) * nst);
            w.qt_off = off;   // bf16 [B, T, H, dk]
            off = align_up(off + 2 * (size_t)B * T * H * dk);
        }
    }
    w.total = off;
    return w;
}

kdn_status validate_common(int variant, int B, int T, int H, int dk, int dv, int chunk, int io) {
    if (variant != KDN_DIAG && variant != KDN_ISO && variant != KDN_PKDA) return KDN_ERR_SHAPE;
    if (io != KDN_F32 && io != KDN_BF16) return KDN_ERR_DTYPE;
    if (B < 0 || T < 0 || H < 0) return KDN_ERR_SHAPE;
    if (!supported_dim(dk) || !supported_dim(dv)) return KDN_ERR_UNSUPPORTED;
    if (chunk != 0 && chunk != 16 && chunk != 32 && chunk != 64) return KDN_ERR_UNSUPPORTED;
    // keep every element index of a [B,T,H,d] tensor below 2^40
    if ((double)B * (double)T * (double)H * 128.0 > 1.0e12) return KDN_ERR_SHAPE;
    if ((double)B * (double)H > 2.0e9) return KDN_ERR_SHAPE;
    return KDN_OK;
}

// Inputs of the preconditioned delta rule (PKDA) that KDN does not have.
struct PkdaInputs {
    const float *beta, *alpha_p, *beta_p, *center;
    float x;
};

float resolve_x(float x) { return x > 0.f ? x : 1.5f; }

kdn_status forward_impl(int variant, int B, int T, int H, int dk, int dv, int chunk, float mu,
                        int io, uint32_t flags, const void* q, const void* k, const void* v,
                        const float* log_alpha, const float* omega, const float* r,
                        const float* S0, const float* p0, void* o, float* S_T, float* p_T,
                        void* workspace, size_t workspace_bytes, kdn_stream_t stream,
                        const PkdaInputs& pk, float* beta_eff = nullptr) {
    kdn_status st = validate_common(variant, B, T, H, dk, dv, chunk, io);
    if (st != KDN_OK) return st;
    chunk = resolve_chunk(chunk, T);
    const bool is_pk = variant == KDN_PKDA;
    const size_t BH = (size_t)B * H;
    const size_t esz = io == KDN_BF16 ? 2 : 4;
    const size_t ntok = (size_t)B * T * H;
    const size_t nu = variant == KDN_ISO ? 1 : (size_t)dk;
    if (!workspace) return KDN_ERR_WORKSPACE;
    if (BH > 0 && (!S_T || !p_T)) return KDN_ERR_NULL;
    if (ntok > 0 && (!q || !k || !v || !log_alpha || !o)) return KDN_ERR_NULL;
    if (ntok > 0 && !is_pk && (!omega || !r)) return KDN_ERR_NULL;
    if (ntok > 0 && is_pk && (!pk.beta || !pk.alpha_p || !pk.beta_p || !pk.center)) return KDN_ERR_NULL;
    const void* ptrs[] = {q, k, v, log_alpha, omega, r, S0, p0, o, S_T, p_T, workspace,
                          pk.beta, pk.alpha_p, pk.beta_p, pk.center};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDN_ERR_ALIGN;
    const WsLayout w = ws_layout(variant, B, T, H, dk, dv, chunk, io, flags);
    if (workspace_bytes < w.total) return KDN_ERR_WORKSPACE;

    const Range in[] = {{q, ntok * dk * esz}, {k, ntok * dk * esz}, {v, ntok * dv * esz},
                        {log_alpha, ntok * dk * 4}, {omega, ntok * nu * 4}, {r, ntok * 4},
                        {S0, BH * dk * dv * 4}, {p0, BH * nu * 4},
                        {pk.beta, ntok * 4}, {pk.alpha_p, ntok * 4}, {pk.beta_p, ntok * 4},
                        {pk.center, (size_t)H * 4}};
    const Range ro = {o, ntok * dv * esz}, rs = {S_T, BH * dk * dv * 4}, rp = {p_T, BH * nu * 4};
    const Range rw = {workspace, w.total};
    for (const Range& x : in) {
        if (overlaps(ro, x) || overlaps(rw, x)) return KDN_ERR_ALIAS;
        if (x.p != S0 && overlaps(rs, x)) return KDN_ERR_ALIAS;
        if (x.p != p0 && overlaps(rp, x)) return KDN_ERR_ALIAS;
    }
    if (overlaps(ro, rs) || overlaps(ro, rp) || overlaps(rs, rp) || overlaps(rw, ro) ||
        overlaps(rw, rs) || overlaps(rw, rp))
        return KDN_ERR_ALIAS;
    if (S0 && S0 != (const float*)S_T && overlaps(rs, Range{S0, BH * dk * dv * 4})) return KDN_ERR_ALIAS;
    if (p0 && p0 != (const float*)p_T && overlaps(rp, Range{p0, BH * nu * 4})) return KDN_ERR_ALIAS;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t* status = static_cast<uint32_t*>(workspace);
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return KDN_ERR_CUDA;
    if (BH == 0) return KDN_OK;

    kdn::ForwardArgs a;
    a.variant = variant; a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.chunk = chunk;
    a.mu = mu < 0.f ? (float)dk : mu;
    a.io = io; a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.omega = omega; a.r = r;
    a.S0 = S0; a.p0 = p0; a.o = o; a.S_T = S_T; a.p_T = p_T; a.status = status;
    a.beta = pk.beta; a.alpha_p = pk.alpha_p; a.beta_p = pk.beta_p; a.center = pk.center;
    a.neg_log2x = -log2f(resolve_x(pk.x));
    a.flags = flags;
    a.beta_eff = beta_eff;

    cudaError_t e;
    if (T == 0) {
        e = kdn::launch_state_copy(a, s);
    } else if (use_tc_path(io, dk, dv, chunk, flags)) {
        kdn::TcSplit sp = w.split;
        if (sp.nseg > 1) {
            char* base = static_cast<char*>(workspace);
            sp.summary = reinterpret_cast<float*>(base + w.summary_off);
            sp.carry = reinterpret_cast<float*>(base + w.carry_off);
            sp.n_chunks_g = w.nG;
            sp.S_loc = reinterpret_cast<float*>(base + w.sloc_off);
            sp.Phi = reinterpret_cast<float*>(base + w.phi_off);
            sp.S_in = reinterpret_cast<float*>(base + w.sin_off);
            sp.qt = base + w.qt_off;
        }
        e = kdn::launch_forward_tc(a, sp, s);
    } else {
        char* base = static_cast<char*>(workspace);
        kdn::ScanWorkspace sw;
        sw.kappa = reinterpret_cast<float*>(base + w.kappa_off);
        sw.summary = reinterpret_cast<float*>(base + w.summary_off);
        sw.carry = reinterpret_cast<float*>(base + w.carry_off);
        sw.chunk_g = kdn::kGainChunk;
        sw.n_chunks_g = w.nG;
        e = kdn::launch_gain_scan(a, sw, s);
        if (e == cudaSuccess) e = kdn::launch_chunk_simt(a, sw.kappa, s);
        // effective write strength k^T kappa from the scan's gains
        if (e == cudaSuccess && beta_eff) e = kdn::launch_beta_from_kappa(B, T, H, dk, io, k, sw.kappa, beta_eff, s);
    }
    return e == cudaSuccess ? KDN_OK : KDN_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t kdn_workspace_size(int variant, int B, int T, int H, int dk, int dv, int chunk,
                          int io_dtype, uint32_t flags) {
    if (validate_common(variant, B, T, H, dk, dv, chunk, io_dtype) != KDN_OK) return 0;
    chunk = resolve_chunk(chunk, T);
    return ws_layout(variant, B, T, H, dk, dv, chunk, io_dtype, flags).total;
}

kdn_status kdn_diag_forward(int B, int T, int H, int dk, int dv, int chunk, float mu,
                            int io_dtype, uint32_t flags, const void* q, const void* k,
                            const void* v, const float* log_alpha, const float* omega,
                            const float* r, const float* S0, const float* p0, void* o,
                            float* S_T, float* p_T, void* workspace, size_t workspace_bytes,
                            kdn_stream_t stream) {
    return forward_impl(KDN_DIAG, B, T, H, dk, dv, chunk, mu, io_dtype, flags, q, k, v,
                        log_alpha, omega, r, S0, p0, o, S_T, p_T, workspace, workspace_bytes,
                        stream, PkdaInputs{});
}

kdn_status kdn_iso_forward(int B, int T, int H, int dk, int dv, int chunk, float mu,
                           int io_dtype, uint32_t flags, const void* q, const void* k,
                           const void* v, const float* log_alpha, const float* omega,
                           const float* r, const float* S0, const float* p0, void* o, float* S_T,
                           float* p_T, void* workspace, size_t workspace_bytes,
                           kdn_stream_t stream) {
    return forward_impl(KDN_ISO, B, T, H, dk, dv, chunk, mu, io_dtype, flags, q, k, v, log_alpha,
                        omega, r, S0, p0, o, S_T, p_T, workspace, workspace_bytes, stream,
                        PkdaInputs{});
}

kdn_status kdn_pkda_forward(int B, int T, int H, int dk, int dv, int chunk, float x, int io_dtype,
                            uint32_t flags, const void* q, const void* k, const void* v,
                            const float* log_alpha, const float* beta, const float* alpha_p,
                            const float* beta_p, const float* center, const float* S0,
                            const float* A0, void* o, float* S_T, float* A_T, void* workspace,
                            size_t workspace_bytes, kdn_stream_t stream) {
    return forward_impl(KDN_PKDA, B, T, H, dk, dv, chunk, 0.f, io_dtype, flags, q, k, v, log_alpha,
                        nullptr, nullptr, S0, A0, o, S_T, A_T, workspace, workspace_bytes, stream,
                        PkdaInputs{beta, alpha_p, beta_p, center, x});
}

}  // extern "C"

namespace {

// Gated forward: the ungated path's workspace first, then the fp32 gates
// (log alpha [B,T,H,dk], omega [B,T,H,dk] or [B,T,H], r [B,T,H]) the gate prologue
// writes and that path reads.
struct GatedLayout {
    size_t base;                 // the ungated path's workspace (kdn_workspace_size)
    size_t la_off, om_off, r_off, total;
};

GatedLayout gated_layout(int variant, int B, int T, int H, int dk, int dv, int chunk, int io, uint32_t flags) {
    GatedLayout g;
    memset(&g, 0, sizeof(g));
    g.base = align_up(ws_layout(variant, B, T, H, dk, dv, chunk, io, flags).total);
    size_t off = g.base;
    if (T > 0) {
        const size_t ntok = (size_t)B * T * H, nu = variant == KDN_ISO ? 1 : (size_t)dk;
        g.la_off = off;
        off = align_up(off + 4 * ntok * dk);
        g.om_off = off;
        off = align_up(off + 4 * ntok * nu);
        g.r_off = off;
        off = align_up(off + 4 * ntok);
    }
    g.total = off;
    return g;
}

}  // namespace

extern "C" {

size_t kdn_gated_workspace_size(int variant, int B, int T, int H, int dk, int dv, int chunk,
                                int io_dtype, uint32_t flags) {
    if (variant != KDN_DIAG && variant != KDN_ISO) return 0;
    if (validate_common(variant, B, T, H, dk, dv, chunk, io_dtype) != KDN_OK) return 0;
    chunk = resolve_chunk(chunk, T);
    return gated_layout(variant, B, T, H, dk, dv, chunk, io_dtype, flags).total;
}

kdn_status kdn_gated_forward(int variant, int B, int T, int H, int dk, int dv, int chunk, float mu,
                             float r_min, int io_dtype, uint32_t flags, const void* q, const void* k,
                             const void* v, const void* alpha_logit, const void* omega_logit,
                             const void* r_logit, const float* S0, const float* p0, void* o, float* S_T,
                             float* p_T, float* beta_eff, void* workspace, size_t workspace_bytes,
                             kdn_stream_t stream) {
    if (variant != KDN_DIAG && variant != KDN_ISO) return KDN_ERR_SHAPE;
    kdn_status st = validate_common(variant, B, T, H, dk, dv, chunk, io_dtype);
    if (st != KDN_OK) return st;
    if (std::isnan(r_min) || std::isinf(r_min)) return KDN_ERR_SHAPE;
    if (r_min < 0.f) r_min = 0.01f;
    chunk = resolve_chunk(chunk, T);
    const size_t BH = (size_t)B * H, ntok = (size_t)B * T * H, esz = io_dtype == KDN_BF16 ? 2 : 4;
    const size_t nu = variant == KDN_ISO ? 1 : (size_t)dk;
    if (!workspace) return KDN_ERR_WORKSPACE;
    if (BH > 0 && (!S_T || !p_T)) return KDN_ERR_NULL;
    if (ntok > 0 && (!q || !k || !v || !alpha_logit || !omega_logit || !r_logit || !o)) return KDN_ERR_NULL;
    const void* ptrs[] = {q, k, v, alpha_logit, omega_logit, r_logit, S0, p0, o, S_T, p_T, beta_eff, workspace};
    for (const void* x : ptrs)
        if (x && !aligned16(x)) return KDN_ERR_ALIGN;
    const GatedLayout g = gated_layout(variant, B, T, H, dk, dv, chunk, io_dtype, flags);
    if (workspace_bytes < g.total) return KDN_ERR_WORKSPACE;
    const Range in[] = {{q, ntok * dk * esz}, {k, ntok * dk * esz}, {v, ntok * dv * esz},
                        {alpha_logit, ntok * dk * esz}, {omega_logit, ntok * nu * esz}, {r_logit, ntok * esz},
                        {S0, BH * dk * dv * 4}, {p0, BH * nu * 4}};
    const Range out[] = {{o, ntok * dv * esz}, {S_T, BH * dk * dv * 4}, {p_T, BH * nu * 4},
                         {beta_eff, ntok * 4}, {workspace, g.total}};
    const int nout = sizeof(out) / sizeof(out[0]);
    for (int o1 = 0; o1 < nout; ++o1) {
        for (const Range& x : in) {
            // resuming in place: S_T may be S0 and p_T may be p0
            if ((o1 == 1 && x.p == S0 && S0 == (const float*)S_T) || (o1 == 2 && x.p == p0 && p0 == (const float*)p_T))
                continue;
            if (overlaps(out[o1], x)) return KDN_ERR_ALIAS;
        }
        for (int o2 = o1 + 1; o2 < nout; ++o2)
            if (overlaps(out[o1], out[o2])) return KDN_ERR_ALIAS;
    }

    // fp32 gates into the workspace (one elementwise kernel over all SMs), then the
    // ungated path on them, its own scratch at the start of the workspace.  With
    // beta_eff requested the tensor-core path keeps one CTA per sequence (the split
    // path does not form it); its workspace is then no larger.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(workspace);
    float* la = reinterpret_cast<float*>(base + g.la_off);
    float* om = reinterpret_cast<float*>(base + g.om_off);
    float* rr = reinterpret_cast<float*>(base + g.r_off);
    if (T > 0 && BH > 0 &&
        kdn::launch_gate_expand(variant, B, T, H, dk, io_dtype, r_min, alpha_logit, omega_logit, r_logit, la, om, rr,
                                s) != cudaSuccess)
        return KDN_ERR_CUDA;
    const bool on = T > 0;
    return forward_impl(variant, B, T, H, dk, dv, chunk, mu, io_dtype, beta_eff ? (flags | KDN_FLAG_NO_SPLIT) : flags,
                        q, k, v, on ? la : nullptr, on ? om : nullptr, on ? rr : nullptr, S0, p0, o, S_T, p_T,
                        workspace, g.base, stream, PkdaInputs{}, on ? beta_eff : nullptr);
}

}  // extern "C"

namespace {

kdn_status step_impl(int variant, int B, int H, int dk, int dv, float mu, int io_dtype,
                     const void* q, const void* k, const void* v, const float* log_alpha,
                     const float* omega, const float* r, float* S, float* p, void* o,
                     void* workspace, size_t workspace_bytes, kdn_stream_t stream,
                     const PkdaInputs& pk, uint32_t flags) {
    kdn_status st = validate_common(variant, B, 1, H, dk, dv, 0, io_dtype);
    if (st != KDN_OK) return st;
    if (!workspace) return KDN_ERR_WORKSPACE;
    if (workspace_bytes < kStatusBytes) return KDN_ERR_WORKSPACE;
    const bool is_pk = variant == KDN_PKDA;
    const size_t BH = (size_t)B * H;
    if (BH > 0 && (!q || !k || !v || !log_alpha || !S || !p || !o)) return KDN_ERR_NULL;
    if (BH > 0 && !is_pk && (!omega || !r)) return KDN_ERR_NULL;
    if (BH > 0 && is_pk && (!pk.beta || !pk.alpha_p || !pk.beta_p || !pk.center)) return KDN_ERR_NULL;
    const void* ptrs[] = {q, k, v, log_alpha, omega, r, S, p, o, workspace,
                          pk.beta, pk.alpha_p, pk.beta_p, pk.center};
    for (const void* x : ptrs)
        if (x && !aligned16(x)) return KDN_ERR_ALIGN;
    const size_t esz = io_dtype == KDN_BF16 ? 2 : 4;
    const size_t nu = variant == KDN_ISO ? 1 : (size_t)dk;
    const Range in[] = {{q, BH * dk * esz}, {k, BH * dk * esz}, {v, BH * dv * esz},
                        {log_alpha, BH * dk * 4}, {omega, BH * nu * 4}, {r, BH * 4},
                        {pk.beta, BH * 4}, {pk.alpha_p, BH * 4}, {pk.beta_p, BH * 4},
                        {pk.center, (size_t)H * 4}};
    const Range rs = {S, BH * dk * dv * 4}, rp = {p, BH * nu * 4}, ro = {o, BH * dv * esz};
    const Range rw = {workspace, kStatusBytes};
    for (const Range& x : in)
        if (overlaps(rs, x) || overlaps(rp, x) || overlaps(ro, x) || overlaps(rw, x))
            return KDN_ERR_ALIAS;
    if (overlaps(rs, rp) || overlaps(rs, ro) || overlaps(rp, ro) || overlaps(rw, rs) ||
        overlaps(rw, rp) || overlaps(rw, ro))
        return KDN_ERR_ALIAS;
    kdn::StepArgs a;
    a.variant = variant; a.B = B; a.H = H; a.dk = dk; a.dv = dv; a.io = io_dtype;
    a.mu = mu < 0.f ? (float)dk : mu;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.omega = omega; a.r = r;
    a.S = S; a.p = p; a.o = o; a.status = static_cast<uint32_t*>(workspace);
    a.beta = pk.beta; a.alpha_p = pk.alpha_p; a.beta_p = pk.beta_p; a.center = pk.center;
    a.neg_log2x = -log2f(resolve_x(pk.x));
    a.flags = flags;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the status word is cleared here, in stream order, so no CTA of the step can
    // clear a condition another CTA has already recorded
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return KDN_ERR_CUDA;
    if (BH == 0) return KDN_OK;
    return kdn::launch_step(a, s) == cudaSuccess ? KDN_OK : KDN_ERR_CUDA;
}

}  // namespace

extern "C" {

kdn_status kdn_step(int variant, int B, int H, int dk, int dv, float mu, int io_dtype,
                    const void* q, const void* k, const void* v, const float* log_alpha,
                    const float* omega, const float* r, float* S, float* p, void* o,
                    void* workspace, size_t workspace_bytes, kdn_stream_t stream) {
    if (variant != KDN_DIAG && variant != KDN_ISO) return KDN_ERR_SHAPE;
    return step_impl(variant, B, H, dk, dv, mu, io_dtype, q, k, v, log_alpha, omega, r, S, p, o,
                     workspace, workspace_bytes, stream, PkdaInputs{}, 0u);
}

kdn_status kdn_step_ex(int variant, int B, int H, int dk, int dv, float mu, int io_dtype, uint32_t flags,
                       const void* q, const void* k, const void* v, const float* log_alpha,
                       const float* omega, const float* r, float* S, float* p, void* o,
                       void* workspace, size_t workspace_bytes, kdn_stream_t stream) {
    if (variant != KDN_DIAG && variant != KDN_ISO) return KDN_ERR_SHAPE;
    if (flags & ~KDN_FLAG_TIMEOUT_PROBE) return KDN_ERR_UNSUPPORTED;
    return step_impl(variant, B, H, dk, dv, mu, io_dtype, q, k, v, log_alpha, omega, r, S, p, o,
                     workspace, workspace_bytes, stream, PkdaInputs{}, flags);
}

kdn_status kdn_pkda_step(int B, int H, int dk, int dv, float x, int io_dtype, const void* q,
                         const void* k, const void* v, const float* log_alpha, const float* beta,
                         const float* alpha_p, const float* beta_p, const float* center, float* S,
                         float* A, void* o, void* workspace, size_t workspace_bytes,
                         kdn_stream_t stream) {
    return step_impl(KDN_PKDA, B, H, dk, dv, 0.f, io_dtype, q, k, v, log_alpha, nullptr, nullptr, S,
                     A, o, workspace, workspace_bytes, stream,
                     PkdaInputs{beta, alpha_p, beta_p, center, x}, 0u);
}

size_t kdn_dense_workspace_size(int B, int T, int H, int d, int io_dtype) {
    if (io_dtype != KDN_F32 && io_dtype != KDN_BF16) return 0;
    if (B < 0 || T < 0 || H < 0 || (d != 32 && d != 64 && d != 128)) return 0;
    if ((double)B * (double)T * (double)H * 128.0 > 1.0e12 || (double)B * (double)H > 2.0e9) return 0;
    return kStatusBytes + align_up(sizeof(float) * (size_t)B * T * H * d);
}

kdn_status kdn_dense_forward(int B, int T, int H, int d, int io_dtype, const void* q, const void* k,
                             const void* v, const float* log_alpha, const float* omega, const float* r,
                             const float* S0, const float* P0, void* o, float* S_T, float* P_T,
                             void* workspace, size_t workspace_bytes, kdn_stream_t stream) {
    if (io_dtype != KDN_F32 && io_dtype != KDN_BF16) return KDN_ERR_DTYPE;
    if (B < 0 || T < 0 || H < 0) return KDN_ERR_SHAPE;
    if (d != 32 && d != 64 && d != 128) return KDN_ERR_UNSUPPORTED;
    if ((double)B * (double)T * (double)H * 128.0 > 1.0e12 || (double)B * (double)H > 2.0e9)
        return KDN_ERR_SHAPE;
    const size_t BH = (size_t)B * H, ntok = (size_t)B * T * H, esz = io_dtype == KDN_BF16 ? 2 : 4;
    if (BH > 0 && (!S_T || !P_T)) return KDN_ERR_NULL;
    if (ntok > 0 && (!q || !k || !v || !log_alpha || !omega || !r || !o)) return KDN_ERR_NULL;
    if (!workspace) return KDN_ERR_WORKSPACE;
    const void* ptrs[] = {q, k, v, log_alpha, omega, r, S0, P0, o, S_T, P_T, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDN_ERR_ALIGN;
    const size_t need = kdn_dense_workspace_size(B, T, H, d, io_dtype);
    if (workspace_bytes < need) return KDN_ERR_WORKSPACE;
    const size_t nd = ntok * d, ns = BH * d * d;
    const Range in[] = {{q, nd * esz}, {k, nd * esz}, {v, nd * esz}, {log_alpha, nd * 4},
                        {omega, nd * 4}, {r, ntok * 4}, {S0, ns * 4}, {P0, ns * 4}};
    const Range ro = {o, nd * esz}, rs = {S_T, ns * 4}, rp = {P_T, ns * 4}, rw = {workspace, need};
    for (const Range& x : in) {
        if (overlaps(ro, x) || overlaps(rw, x)) return KDN_ERR_ALIAS;
        if (x.p != S0 && overlaps(rs, x)) return KDN_ERR_ALIAS;
        if (x.p != P0 && overlaps(rp, x)) return KDN_ERR_ALIAS;
    }
    if (overlaps(ro, rs) || overlaps(ro, rp) || overlaps(rs, rp) || overlaps(rw, ro) || overlaps(rw, rs) ||
        overlaps(rw, rp))
        return KDN_ERR_ALIAS;
    if (S0 && S0 != (const float*)S_T && overlaps(rs, Range{S0, ns * 4})) return KDN_ERR_ALIAS;
    if (P0 && P0 != (const float*)P_T && overlaps(rp, Range{P0, ns * 4})) return KDN_ERR_ALIAS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t* status = static_cast<uint32_t*>(workspace);
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return KDN_ERR_CUDA;
    if (BH == 0) return KDN_OK;
    float* kappa = reinterpret_cast<float*>(static_cast<char*>(workspace) + kStatusBytes);

    // (1) the covariance recurrence, token by token: kappa and P_T
    kdn::DenseArgs a;
    a.B = B; a.T = T; a.H = H; a.d = d; a.io = io_dtype;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.omega = omega; a.r = r;
    a.S0 = S0; a.P0 = P0; a.o = o; a.S_T = S_T; a.P_T = P_T;
    if (kdn::launch_dense_covariance(a, kappa, s) != cudaSuccess) return KDN_ERR_CUDA;
    // (2) the mean with the gains given
    if (T == 0) {
        cudaError_t e = S0 ? (S0 == (const float*)S_T ? cudaSuccess
                                                        : cudaMemcpyAsync(S_T, S0, ns * 4, cudaMemcpyDeviceToDevice, s))
                           : cudaMemsetAsync(S_T, 0, ns * 4, s);
        return e == cudaSuccess ? KDN_OK : KDN_ERR_CUDA;
    }
    kdn::ForwardArgs f;
    memset(&f, 0, sizeof(f));
    f.B = B; f.T = T; f.H = H; f.dk = d; f.dv = d; f.io = io_dtype;
    f.chunk = resolve_chunk(0, T);
    f.q = q; f.k = k; f.v = v; f.log_alpha = log_alpha; f.omega = kappa;
    f.S0 = S0; f.o = o; f.S_T = S_T; f.status = status;
    cudaError_t e;
    if (use_tc_path(io_dtype, d, d, f.chunk, 0)) {
        f.variant = 3;   // the fused kernel's given-gains instance (whole sequences)
        e = kdn::launch_forward_tc(f, kdn::TcSplit{}, s);
    } else {
        f.variant = KDN_DIAG;   // (the chunk pass reads only the gains)
        e = kdn::launch_chunk_simt(f, kappa, s);
    }
    return e == cudaSuccess ? KDN_OK : KDN_ERR_CUDA;
}

}  // extern "C"

namespace {

struct BwLayout {
    size_t total, kappa_off, summary_off, carry_off, pscr_off, ckpt_off, dkappa_off, pck_off;
    int nG;
};

BwLayout bw_layout(int variant, int B, int T, int H, int dk, int dv) {
    BwLayout w;
    memset(&w, 0, sizeof(w));
    const size_t BH = (size_t)B * H, nu = variant == KDN_ISO ? 1 : (size_t)dk, ntok = (size_t)B * T * H;
    const size_t nch = (T + kdn::backward_chunk() - 1) / kdn::backward_chunk();
    const size_t nblk = (T + kdn::backward_block() - 1) / kdn::backward_block();
    w.nG = (T + kdn::kGainChunk - 1) / kdn::kGainChunk;
    size_t off = kStatusBytes;
    w.kappa_off = off;
    off = align_up(off + 4 * ntok * dk);
    w.summary_off = off;
    off = align_up(off + 4 * 4 * BH * w.nG * nu);
    w.carry_off = off;
    off = align_up(off + 4 * BH * w.nG * nu);
    w.pscr_off = off;
    off = align_up(off + 4 * BH * nu);
    w.ckpt_off = off;
    off = align_up(off + 4 * BH * (nch + 1) * dk * dv);
    w.dkappa_off = off;
    off = align_up(off + 4 * ntok * dk);
    w.pck_off = off;
    off = align_up(off + 4 * BH * nblk * nu);
    w.total = off;
    return w;
}

}  // namespace

extern "C" {

size_t kdn_backward_workspace_size(int variant, int B, int T, int H, int dk, int dv, int io_dtype) {
    if (variant != KDN_DIAG && variant != KDN_ISO) return 0;
    if (validate_common(variant, B, T, H, dk, dv, 0, io_dtype) != KDN_OK) return 0;
    return bw_layout(variant, B, T, H, dk, dv).total;
}

kdn_status kdn_backward(int variant, int B, int T, int H, int dk, int dv, float mu, int io_dtype,
                        const void* q, const void* k, const void* v, const float* log_alpha,
                        const float* omega, const float* r, const float* S0, const float* p0,
                        const void* dO, const float* dS_T, const float* dp_T, float* dq, float* dk_out,
                        float* dv_out, float* dlog_alpha, float* domega, float* dr, float* dS0,
                        float* dp0, void* workspace, size_t workspace_bytes, kdn_stream_t stream) {
    if (variant != KDN_DIAG && variant != KDN_ISO) return KDN_ERR_SHAPE;
    kdn_status st = validate_common(variant, B, T, H, dk, dv, 0, io_dtype);
    if (st != KDN_OK) return st;
    const size_t BH = (size_t)B * H, ntok = (size_t)B * T * H, esz = io_dtype == KDN_BF16 ? 2 : 4;
    const size_t nu = variant == KDN_ISO ? 1 : (size_t)dk;
    if (!workspace) return KDN_ERR_WORKSPACE;
    if (BH > 0 && (!dS0 || !dp0)) return KDN_ERR_NULL;
    if (ntok > 0 && (!q || !k || !v || !log_alpha || !omega || !r || !dq || !dk_out || !dv_out ||
                     !dlog_alpha || !domega || !dr))
        return KDN_ERR_NULL;
    const void* ptrs[] = {q, k, v, log_alpha, omega, r, S0, p0, dO, dS_T, dp_T, dq, dk_out, dv_out,
                          dlog_alpha, domega, dr, dS0, dp0, workspace};
    for (const void* x : ptrs)
        if (x && !aligned16(x)) return KDN_ERR_ALIGN;
    const BwLayout w = bw_layout(variant, B, T, H, dk, dv);
    if (workspace_bytes < w.total) return KDN_ERR_WORKSPACE;
    const Range in[] = {{q, ntok * dk * esz}, {k, ntok * dk * esz}, {v, ntok * dv * esz},
                        {log_alpha, ntok * dk * 4}, {omega, ntok * nu * 4}, {r, ntok * 4},
                        {S0, BH * dk * dv * 4}, {p0, BH * nu * 4}, {dO, ntok * dv * esz},
                        {dS_T, BH * dk * dv * 4}, {dp_T, BH * nu * 4}};
    const Range out[] = {{dq, ntok * dk * 4}, {dk_out, ntok * dk * 4}, {dv_out, ntok * dv * 4},
                         {dlog_alpha, ntok * dk * 4}, {domega, ntok * nu * 4}, {dr, ntok * 4},
                         {dS0, BH * dk * dv * 4}, {dp0, BH * nu * 4}, {workspace, w.total}};
    const int nout = sizeof(out) / sizeof(out[0]);
    for (int o1 = 0; o1 < nout; ++o1) {
        for (const Range& x : in)
            if (overlaps(out[o1], x)) return KDN_ERR_ALIAS;
        for (int o2 = o1 + 1; o2 < nout; ++o2)
            if (overlaps(out[o1], out[o2])) return KDN_ERR_ALIAS;
    }
    if (kdn::backward_mem_smem_bytes(dk, dv) > 232448) return KDN_ERR_UNSUPPORTED;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t* status = static_cast<uint32_t*>(workspace);
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return KDN_ERR_CUDA;
    if (BH == 0) return KDN_OK;
    if (T == 0) {   // nothing between the initial and the final state
        const size_t nS = BH * dk * dv * 4, np = BH * nu * 4;
        cudaError_t e = dS_T ? cudaMemcpyAsync(dS0, dS_T, nS, cudaMemcpyDeviceToDevice, s)
                             : cudaMemsetAsync(dS0, 0, nS, s);
        if (e == cudaSuccess)
            e = dp_T ? cudaMemcpyAsync(dp0, dp_T, np, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(dp0, 0, np, s);
        return e == cudaSuccess ? KDN_OK : KDN_ERR_CUDA;
    }
    kdn::BackwardArgs a;
    a.variant = variant; a.B = B; a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.io = io_dtype;
    a.mu = mu < 0.f ? (float)dk : mu;
    a.q = q; a.k = k; a.v = v; a.dO = dO; a.log_alpha = log_alpha; a.omega = omega; a.r = r;
    a.S0 = S0; a.p0 = p0; a.dS_T = dS_T; a.dp_T = dp_T;
    a.dq = dq; a.dk_out = dk_out; a.dv_out = dv_out; a.dla = dlog_alpha; a.domega = domega; a.dr = dr;
    a.dS0 = dS0; a.dp0 = dp0; a.status = status;
    char* base = static_cast<char*>(workspace);
    kdn::BackwardWorkspace bw;
    bw.kappa = reinterpret_cast<float*>(base + w.kappa_off);
    bw.summary = reinterpret_cast<float*>(base + w.summary_off);
    bw.carry = reinterpret_cast<float*>(base + w.carry_off);
    bw.n_chunks_g = w.nG;
    bw.p_scratch = reinterpret_cast<float*>(base + w.pscr_off);
    bw.ckpt = reinterpret_cast<float*>(base + w.ckpt_off);
    bw.dkappa = reinterpret_cast<float*>(base + w.dkappa_off);
    bw.pck = reinterpret_cast<float*>(base + w.pck_off);
    return kdn::launch_backward(a, bw, s) == cudaSuccess ? KDN_OK : KDN_ERR_CUDA;
}

kdn_status kdn_read_device_status(const void* workspace, kdn_stream_t stream) {
    if (!workspace) return KDN_ERR_NULL;
    uint32_t word = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDN_ERR_CUDA;
    return static_cast<kdn_status>(word);
}

int kdn_forward_kernel_count(int variant, int B, int T, int H, int dk, int dv, int chunk,
                             int io_dtype, uint32_t flags) {
    if (validate_common(variant, B, T, H, dk, dv, chunk, io_dtype) != KDN_OK) return 0;
    if ((size_t)B * H == 0) return 0;
    if (T == 0) return 1;
    chunk = resolve_chunk(chunk, T);
    return use_tc_path(io_dtype, dk, dv, chunk, flags)
               ? kdn::tc_kernel_count(kdn::tc_split_plan(B, T, H, flags).nseg)
               : 4;
}

const char* kdn_status_string(int status) {
    switch (status) {
        case KDN_OK: return "ok";
        case KDN_ERR_NULL: return "a required pointer is NULL";
        case KDN_ERR_SHAPE: return "invalid or inconsistent sizes";
        case KDN_ERR_DTYPE: return "io dtype must be KDN_F32 or KDN_BF16";
        case KDN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case KDN_ERR_WORKSPACE: return "workspace missing or too small";
        case KDN_ERR_UNSUPPORTED: return "d_k, d_v or chunk outside the supported set";
        case KDN_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case KDN_ERR_TIMEOUT: return "a bounded device wait gave up";
        case KDN_ERR_RANGE: return "a chunk's cumulative log-decay is outside the supported range";
        case KDN_ERR_ALIAS: return "an output overlaps an input";
        default: return "unknown status";
    }
}

int kdn_abi_version(void) { return 106; }

}  // extern "C"
