// Sequence split of the tensor-core forward: chaining of the segments' state maps
// and the output correction (sm_103a).
//
// The KDN state update (KDN paper Sec. 3.2, Eq. 12-17: S_hat = D S, S = S_hat +
// kappa delta^T with delta = v - S_hat^T k, o = S^T q) is affine in the state once
// the gains are fixed, and the gains depend only on the uncertainty recurrence
// (Sec. 4.1 / 4.2), never on S.  So a segment of a sequence maps its initial state
// to S_out = Phi S_in + S_loc, and its outputs are o_t = o_loc,t + S_in^T q~_t with
// q~_t = Phi_t^T q_t.  The fused kernel produces S_loc and o_loc (from S = 0) and
// Phi and q~ (from S = I with zero values) for every segment in parallel; the
// kernels here chain the maps into each segment's initial state and the final
// state, and add the correction term to the outputs.

#include <cuda_bf16.h>

#include "common.cuh"
#include "kdn_internal.h"
#include "sm100.cuh"

namespace kdn {
namespace {

using namespace sm100;

constexpr int kD = 128;   // d_k = d_v on the tensor-core path

// Chain the segment maps of each sequence: S_in(0) = S0 (zero when NULL) and
// S_in(s + 1) = Phi_s S_in(s) + S_loc(s), all [B*H*nseg][128][128] fp32.  Grid
// (B*H, 128 / 16), 256 threads: a CTA owns 16 value columns of the state and walks
// the segments in order; thread (row i, 8 columns) forms its part of each product.
// Each segment's initial state goes out transposed in bf16, S_in^T [j][i] (the B
// operand of the output correction); after the last segment the CTA writes the
// sequence's final state (S_T may be S0: a CTA reads its columns of S0 before it
// writes them).
__global__ void __launch_bounds__(256) segment_states_kernel(const float* S0,
                                                              const float* __restrict__ Phi,
                                                              const float* __restrict__ S_loc,
                                                              __nv_bfloat16* __restrict__ S_inT, float* S_T,
                                                              int nseg) {
    __shared__ float cur[kD][17];
    const int bh = blockIdx.x, cb = blockIdx.y * 16, tid = threadIdx.x;
    for (int e = tid; e < kD * 16; e += 256) {
        const int i = e >> 4, j = e & 15;
        cur[i][j] = S0 ? S0[(static_cast<size_t>(bh) * kD + i) * kD + cb + j] : 0.0f;
    }
    __syncthreads();
    const int i = tid >> 1, j0 = (tid & 1) * 8;
    for (int sg = 0; sg < nseg; ++sg) {
        const size_t mb = (static_cast<size_t>(bh) * nseg + sg) * kD * kD;
        {   // thread -> column cb + (tid >> 4), channels 8 (tid & 15) .. + 7: one 16-byte store
            const int jl = tid >> 4, ic = (tid & 15) * 8;
            const uint4 pk = make_uint4(pack_bf16(cur[ic][jl], cur[ic + 1][jl]), pack_bf16(cur[ic + 2][jl], cur[ic + 3][jl]),
                                        pack_bf16(cur[ic + 4][jl], cur[ic + 5][jl]), pack_bf16(cur[ic + 6][jl], cur[ic + 7][jl]));
            *reinterpret_cast<uint4*>(S_inT + mb + static_cast<size_t>(cb + jl) * kD + ic) = pk;
        }
        float acc[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) acc[jj] = S_loc[mb + static_cast<size_t>(i) * kD + cb + j0 + jj];
        const float4* phi = reinterpret_cast<const float4*>(Phi + mb + static_cast<size_t>(i) * kD);
#pragma unroll 4
        for (int k4 = 0; k4 < kD / 4; ++k4) {
            const float4 f = phi[k4];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                acc[jj] = fmaf(f.x, cur[4 * k4][j0 + jj],
                               fmaf(f.y, cur[4 * k4 + 1][j0 + jj],
                                    fmaf(f.z, cur[4 * k4 + 2][j0 + jj], fmaf(f.w, cur[4 * k4 + 3][j0 + jj], acc[jj]))));
        }
        if (sg == nseg - 1) {
            float* st = S_T + (static_cast<size_t>(bh) * kD + i) * kD + cb + j0;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) st[jj] = acc[jj];
            break;
        }
        __syncthreads();
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) cur[i][j0 + jj] = acc[jj];
        __syncthreads();
    }
}

// Output correction of a split sequence.  The outputs of a segment are linear in
// its initial state: o_t = S_t^T q_t with S_t = Phi_t S_in + S_loc,t, so
// o_t = o_loc,t + S_in^T (Phi_t^T q_t).  The pass from S = 0 writes o_loc into o;
// the pass from S = I with zero values writes q~_t = Phi_t^T q_t (its own outputs);
// this kernel adds S_in^T q~_t once the chained initial states S_in are known.
// CTA: (group of kCorrTiles 128-token tiles, segment, b*h), 256 threads; warp w owns
// rows 16w..16w+15 of a tile and all 128 value columns.  bf16 operands (S_in rounded
// to bf16 as in the state's bf16 copy that the fused kernel multiplies by), fp32
// accumulation, warp-level m16n8k16 MMAs from shared memory.
constexpr int kCorrRows = 128, kCorrTiles = 8, kCorrLd = kD + 8;   // +8: conflict-free ldmatrix rows
constexpr int kCorrSmem = 5 * kCorrRows * kCorrLd * 2;   // S_in^T, two q~ tiles, two o tiles

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const __nv_bfloat16* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

__global__ void __launch_bounds__(256, 1) segment_output_correction_kernel(const __nv_bfloat16* __restrict__ S_inT,
                                                                           const __nv_bfloat16* __restrict__ qt,
                                                                           __nv_bfloat16* __restrict__ o, int T,
                                                                           int H, int nseg, int seg_len,
                                                                           int skip_first) {
    extern __shared__ __align__(16) unsigned char corr_smem[];
    __nv_bfloat16* Bs = reinterpret_cast<__nv_bfloat16*>(corr_smem);   // S_in^T [j][i]
    __nv_bfloat16* As = Bs + kCorrRows * kCorrLd;                       // q~ rows [t][i], two buffers
    __nv_bfloat16* Os = As + 2 * kCorrRows * kCorrLd;                   // o rows [t][j], two buffers
    const int bh = blockIdx.z, seg = blockIdx.y, b = bh / H, h = bh % H;
    if (seg == 0 && skip_first) return;   // the first segment starts from S = 0
    const int tb = seg * seg_len, Ts = min(seg_len, T - tb);
    const int r0 = blockIdx.x * kCorrTiles * kCorrRows;
    if (r0 >= Ts) return;
    const int ntiles = min(kCorrTiles, (Ts - r0 + kCorrRows - 1) / kCorrRows);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t ts = static_cast<size_t>(H) * kD;   // token stride of [B, T, H, d]
    const size_t row0 = (static_cast<size_t>(b) * T + tb) * ts + static_cast<size_t>(h) * kD;
    // q~ and o rows of tile k into buffers k & 1 (q~ rows past the segment read as zero)
    auto load_tile = [&](int k) {
        const int rt = r0 + k * kCorrRows;
        __nv_bfloat16* dq = As + (k & 1) * kCorrRows * kCorrLd;
        __nv_bfloat16* dout = Os + (k & 1) * kCorrRows * kCorrLd;
        for (int e = tid; e < kCorrRows * (kD / 8); e += 256) {   // 16-byte pieces, 16 per row
            const int r = e >> 4, c = (e & 15) * 8;
            if (rt + r < Ts) {
                cp_async16(dq + r * kCorrLd + c, qt + row0 + (rt + r) * ts + c);
                cp_async16(dout + r * kCorrLd + c, o + row0 + (rt + r) * ts + c);
            } else {
                *reinterpret_cast<uint4*>(dq + r * kCorrLd + c) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    load_tile(0);
    const __nv_bfloat16* St = S_inT + (static_cast<size_t>(bh) * nseg + seg) * kD * kD;
    for (int e = tid; e < kD * (kD / 8); e += 256) {
        const int j = e >> 4, c = (e & 15) * 8;
        *reinterpret_cast<uint4*>(Bs + j * kCorrLd + c) = __ldg(reinterpret_cast<const uint4*>(St + j * kD + c));
    }
    const int g = lane >> 2, q = lane & 3;
    for (int tile = 0; tile < ntiles; ++tile) {
        const int rt = r0 + tile * kCorrRows;
        if (tile + 1 < ntiles) {   // the next tile's rows land while this one is multiplied
            load_tile(tile + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();   // this tile's rows (and S_in^T) are in shared memory for every warp
        const __nv_bfloat16* A = As + (tile & 1) * kCorrRows * kCorrLd;
        float acc[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t a[4];
            ldmatrix_x4(a, A + (16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8) * kCorrLd + 16 * ks + (lane >> 4) * 8);
#pragma unroll
            for (int np = 0; np < 8; ++np) {   // value columns 16 np .. 16 np + 15
                uint32_t bb[4];
                ldmatrix_x4(bb, Bs + (16 * np + (lane & 7) + (lane >> 4) * 8) * kCorrLd + 16 * ks + ((lane >> 3) & 1) * 8);
                mma_bf16_16816(acc[2 * np], a, bb[0], bb[1]);
                mma_bf16_16816(acc[2 * np + 1], a, bb[2], bb[3]);
            }
        }
        // o rows += the product, in shared memory (each element has one owner), then
        // written back row by row in 16-byte pieces
        __nv_bfloat16* Ot = Os + (tile & 1) * kCorrRows * kCorrLd;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = 16 * warp + g + 8 * hr;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                __nv_bfloat162* pp = reinterpret_cast<__nv_bfloat162*>(Ot + r * kCorrLd + 8 * nt + 2 * q);
                const float2 cur = __bfloat1622float2(*pp);
                *pp = __floats2bfloat162_rn(cur.x + acc[nt][2 * hr], cur.y + acc[nt][2 * hr + 1]);
            }
        }
        __syncthreads();
        for (int e = tid; e < kCorrRows * (kD / 8); e += 256) {
            const int r = e >> 4, c = (e & 15) * 8;
            if (rt + r < Ts)
                *reinterpret_cast<uint4*>(o + row0 + (rt + r) * ts + c) =
                    *reinterpret_cast<const uint4*>(Ot + r * kCorrLd + c);
        }
        __syncthreads();   // every warp has read buffers tile & 1 before they are refilled
    }
}

}  // namespace

cudaError_t launch_segment_states(const ForwardArgs& a, const TcSplit& sp, cudaStream_t s) {
    __nv_bfloat16* S_inT = reinterpret_cast<__nv_bfloat16*>(sp.S_in);   // bf16 in the fp32 slot
    segment_states_kernel<<<dim3(a.B * a.H, kD / 16), 256, 0, s>>>(a.S0, sp.Phi, sp.S_loc, S_inT, a.S_T,
                                                                      sp.nseg);
    return cudaGetLastError();
}

cudaError_t launch_segment_correction(const ForwardArgs& a, const TcSplit& sp, cudaStream_t s) {
    const cudaError_t e = cudaFuncSetAttribute(segment_output_correction_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kCorrSmem);
    if (e != cudaSuccess) return e;
    const int groups = (sp.seg_len + kCorrTiles * kCorrRows - 1) / (kCorrTiles * kCorrRows);
    segment_output_correction_kernel<<<dim3(groups, sp.nseg, a.B * a.H), 256, kCorrSmem, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(sp.S_in), static_cast<const __nv_bfloat16*>(sp.qt),
        static_cast<__nv_bfloat16*>(a.o), a.T, a.H, sp.nseg, sp.seg_len, a.S0 == nullptr ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace kdn
