// gdn_mma.cuh -- CTA-wide dense contraction on the tensor cores (TF32 in, fp32
// accumulate) with the mma.sync instruction, for the chunked backward's kernels at the
// shapes and dtypes the tcgen05 kernels do not take (fp32 inputs, dv != 128, dk < 128).
//
// cta_gemm_tc(split, M, N, K, A, as0, as1, B, bs0, bs1, f) computes
//     C(m, n) = sum_k A(m, k) B(k, n),  A(m, k) = A[m*as0 + k*as1],  B(k, n) = B[k*bs0 + n*bs1]
// over fp32 operands in shared (or global) memory, with M a multiple of 16, N of
// 16 and K of 8.  Each warp owns 16 x (8*nb) output tiles and issues
// mma.sync.m16n8k8 TF32 instructions over k in increasing order; every output
// element is produced exactly once, by one thread, through f(m, n, value), so
// callers can fuse any elementwise epilogue.  With split (a CTA-uniform flag), each operand is
// split into a TF32 high part and a TF32 remainder and three products
// (hi*hi + hi*lo + lo*hi) are accumulated, which keeps about fp32 accuracy.
// Results are deterministic (fixed tile ownership and k order).  cta_gemm_tc_rmw is the same
// product for epilogues that update a value held elsewhere (C += A B into global memory).
//
// Fragment layout of m16n8k8 (PTX ISA): with g = lane / 4 and t = lane % 4,
//   A (16 x 8, row):  a0 = A[g][t], a1 = A[g+8][t], a2 = A[g][t+4], a3 = A[g+8][t+4]
//   B (8 x 8, col):   b0 = B[t][g], b1 = B[t+4][g]
//   C (16 x 8):       c0 = C[g][2t], c1 = C[g][2t+1], c2 = C[g+8][2t], c3 = C[g+8][2t+1]
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One warp's 16 x (8*nb) tile of the product, k in increasing order, into acc[j][0..3]
// (the C fragment layout above, one 8-column sub-tile per j).
__device__ __forceinline__ void warp_tile_tc(bool split, int m0, int n0, int nb, int K, const float* __restrict__ A,
                                             int as0, int as1, const float* __restrict__ B, int bs0, int bs1,
                                             float (&acc)[4][4]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    const float* a_r0 = A + (size_t)(m0 + g) * as0;
    const float* a_r1 = A + (size_t)(m0 + g + 8) * as0;
    for (int k0 = 0; k0 < K; k0 += 8) {
        const float af[4] = {a_r0[(size_t)(k0 + t) * as1], a_r1[(size_t)(k0 + t) * as1],
                             a_r0[(size_t)(k0 + t + 4) * as1], a_r1[(size_t)(k0 + t + 4) * as1]};
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ah[i] = tf32_rna(af[i]);
            if (split) al[i] = tf32_rna(af[i] - __uint_as_float(ah[i]));
        }
        const float* b_k0 = B + (size_t)(k0 + t) * bs0;
        const float* b_k1 = B + (size_t)(k0 + t + 4) * bs0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < nb) {
                const size_t col = (size_t)(n0 + 8 * j + g) * bs1;
                const float b0f = b_k0[col], b1f = b_k1[col];
                const uint32_t bh0 = tf32_rna(b0f), bh1 = tf32_rna(b1f);
                mma_tf32_16x8x8(acc[j], ah, bh0, bh1);
                if (split) {
                    const uint32_t bl0 = tf32_rna(b0f - __uint_as_float(bh0));
                    const uint32_t bl1 = tf32_rna(b1f - __uint_as_float(bh1));
                    mma_tf32_16x8x8(acc[j], ah, bl0, bl1);
                    mma_tf32_16x8x8(acc[j], al, bh0, bh1);
                }
            }
        }
    }
}

template <typename F>
__device__ __forceinline__ void cta_gemm_tc(bool split, int M, int N, int K, const float* __restrict__ A, int as0, int as1,
                                            const float* __restrict__ B, int bs0, int bs1, F&& f) {
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nb = N >= 32 ? 4 : N / 8;  // n sub-tiles of 8 per warp tile
    const int tiles_m = M >> 4, tiles_n = N / (8 * nb);
    for (int tile = warp; tile < tiles_m * tiles_n; tile += nw) {
        const int tm = tile / tiles_n, tn = tile - tm * tiles_n;
        const int m0 = tm * 16, n0 = tn * 8 * nb;
        float acc[4][4];
        warp_tile_tc(split, m0, n0, nb, K, A, as0, as1, B, bs0, bs1, acc);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < nb) {
                const int n = n0 + 8 * j + 2 * t;
                f(m0 + g, n, acc[j][0]);
                f(m0 + g, n + 1, acc[j][1]);
                f(m0 + g + 8, n, acc[j][2]);
                f(m0 + g + 8, n + 1, acc[j][3]);
            }
        }
    }
}

// The same product with a read-modify-write epilogue: prior(m, n) fetches the value an output
// element updates, f(m, n, value, prior value) writes it.  Every prior of a warp tile is fetched
// before any element of it is written, so the fetches (from global memory, say) are in flight
// together instead of one after another behind each write.  prior and f must touch only the
// element (m, n) they are given.
template <typename P, typename F>
__device__ __forceinline__ void cta_gemm_tc_rmw(bool split, int M, int N, int K, const float* __restrict__ A, int as0,
                                                int as1, const float* __restrict__ B, int bs0, int bs1, P&& prior,
                                                F&& f) {
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nb = N >= 32 ? 4 : N / 8;
    const int tiles_m = M >> 4, tiles_n = N / (8 * nb);
    for (int tile = warp; tile < tiles_m * tiles_n; tile += nw) {
        const int tm = tile / tiles_n, tn = tile - tm * tiles_n;
        const int m0 = tm * 16, n0 = tn * 8 * nb;
        float acc[4][4], old[4][4];
        warp_tile_tc(split, m0, n0, nb, K, A, as0, as1, B, bs0, bs1, acc);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < nb) {
                const int n = n0 + 8 * j + 2 * t;
                old[j][0] = prior(m0 + g, n);
                old[j][1] = prior(m0 + g, n + 1);
                old[j][2] = prior(m0 + g + 8, n);
                old[j][3] = prior(m0 + g + 8, n + 1);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < nb) {
                const int n = n0 + 8 * j + 2 * t;
                f(m0 + g, n, acc[j][0], old[j][0]);
                f(m0 + g, n + 1, acc[j][1], old[j][1]);
                f(m0 + g + 8, n, acc[j][2], old[j][2]);
                f(m0 + g + 8, n + 1, acc[j][3], old[j][3]);
            }
        }
    }
}

}  // namespace gdn
