// Warp-level fp32-accurate products on tensor cores, and 16-byte async copies
// (shared by the CUDA-core chunk pass and the backward's memory adjoint).
#pragma once

#include <stdint.h>

namespace kdn {

// C(r, c) (+)= alpha sum_k A(r, k) B(k, c) on shared-memory operands with arbitrary
// strides: A(r, k) = A[r ar + k ak], B(k, c) = B[k bk + c bc], C(r, c) = C[r cr + c];
// R a multiple of 16, N of 8 NT, K of 8.  Warp-level m16n8k8 TF32 tensor-core MMAs
// (fp32 accumulation) in the 3xTF32 split: each operand x = hi + lo with hi and lo
// TF32 (round to nearest), and the product takes lo*hi + hi*lo + hi*hi, which keeps
// fp32-level accuracy (the dropped lo*lo term is below 2^-22 of the product).  A warp
// computes one 16-row tile of NT 8-column tiles at a time; every warp of the block
// takes part.  Fragment layouts (m16n8k8, A row-major, B column-major): lane = 4 g + q;
// A: (g, q), (g + 8, q), (g, q + 4), (g + 8, q + 4); B: (k = q, n = g), (k = q + 4, n = g);
// C: (g, 2 q), (g, 2 q + 1), (g + 8, 2 q), (g + 8, 2 q + 1).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = to_tf32(x);
    lo = to_tf32(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_m16n8k8_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte asynchronous copy global -> shared (L2 only), or 16 zero bytes when !valid
// (no global read then); completion by cp_async_wait_all() and a barrier.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gsrc), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// (wofs rotates the units over the warps, so small products issued back to back
//  without a barrier can land on different warps)
template <int NT>
__device__ void smem_gemm(int R, int N, int K, const float* A, int ar, int ak, const float* B, int bk, int bc,
                          float* C, int cr, float alpha, bool accumulate, int wofs = 0) {
    const int lane = threadIdx.x & 31, nw = blockDim.x >> 5, warp = ((threadIdx.x >> 5) + wofs) % nw;
    const int g = lane >> 2, q = lane & 3;
    const int nrt = R / 16, nct = N / (8 * NT);
    for (int u = warp; u < nrt * nct; u += nw) {
        const int r0 = (u / nct) * 16, c0 = (u % nct) * 8 * NT;
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
        const float* ap = A + (r0 + g) * ar + q * ak;
        for (int k0 = 0; k0 < K; k0 += 8) {
            uint32_t ah[4], al[4];
            split_tf32(ap[k0 * ak], ah[0], al[0]);
            split_tf32(ap[8 * ar + k0 * ak], ah[1], al[1]);
            split_tf32(ap[(k0 + 4) * ak], ah[2], al[2]);
            split_tf32(ap[8 * ar + (k0 + 4) * ak], ah[3], al[3]);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const float* bp = B + (k0 + q) * bk + (c0 + 8 * n + g) * bc;
                uint32_t bh0, bl0, bh1, bl1;
                split_tf32(bp[0], bh0, bl0);
                split_tf32(bp[4 * bk], bh1, bl1);
                mma_m16n8k8_tf32(acc[n], al, bh0, bh1);
                mma_m16n8k8_tf32(acc[n], ah, bl0, bl1);
                mma_m16n8k8_tf32(acc[n], ah, bh0, bh1);
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float* d0 = C + (r0 + g) * cr + c0 + 8 * n + 2 * q;
            float* d1 = d0 + 8 * cr;
            if (accumulate) {
                d0[0] = fmaf(alpha, acc[n][0], d0[0]);
                d0[1] = fmaf(alpha, acc[n][1], d0[1]);
                d1[0] = fmaf(alpha, acc[n][2], d1[0]);
                d1[1] = fmaf(alpha, acc[n][3], d1[1]);
            } else {
                d0[0] = alpha * acc[n][0];
                d0[1] = alpha * acc[n][1];
                d1[0] = alpha * acc[n][2];
                d1[1] = alpha * acc[n][3];
            }
        }
    }
}

}  // namespace kdn
