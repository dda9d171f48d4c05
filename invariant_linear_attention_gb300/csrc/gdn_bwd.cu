// gdn_bwd.cu -- chunked (WY-form) backward of the gated delta rule.
//
// On the pages the chunked form is used only for gradients, which need no
// batch invariance ("Defending Against the Training-Inference Numeric
// Mismatch in RL (Especially Linear Attention)", section 3.2).  The
// chunk form used here (chunk C = 64 tokens, restarting at every sequence
// start, last chunk partial) is the WY / UT representation of the delta rule
// (Yang et al. 2024; Gated Delta Networks, ICLR 2025).  Within a chunk with
// start state S0 (dv x dk) and in-chunk positions r:
//     gam = cumsum(g), Gam = exp(gam), E[r,s] = exp(gam_r - gam_s), b_s = exp(gam_last - gam_s)
//     A = strict_lower(diag(beta) (E * K K^T)),  T = (I + A)^-1
//     W = T diag(beta Gam) K,   U~ = T diag(beta) V,   U = U~ - W S0^T
//     O = diag(Gam) Q S0^T + (lower(E) * Q K^T) U,      S_end = Gam_last S0 + U^T diag(b) K
// Backward, for D = dL/dS_end and dO:
//     dU   = P^T dO + diag(b) K D^T                  (P = lower(E) * Q K^T)
//     dS0  = Gam_last D + dO^T diag(Gam) Q - dU^T W   (the D of the previous chunk)
//     dQ   = diag(Gam) dO S0 + dQK K,  dK = dQK^T Q + diag(b) U D + diag(beta Gam) T^T dW + (dKK + dKK^T) K
//     dW = -dU S0, dV = diag(beta) T^T dU, dA = -T^T dT T^T, dT = dW (beta Gam K)^T + dU (beta V)^T
//     plus the dbeta and dgam terms; dg = reverse cumsum of dgam inside the chunk.
// Dense products run on the tensor cores in TF32 with fp32 accumulation.  For bf16
// inputs with dv = 128 the serial state passes, and at dk = dv = 128 every contracting
// stage, use the fifth-generation tensor cores (tcgen05: operands in shared memory,
// accumulators in TMEM; gdn_umma.cuh) in *_tc kernels; there bwd_intra_s and bwd_intra_c
// are one kernel, bwd_intra_tc, and the operands that come from memory unchanged arrive by
// tensor copies.  Products that produce dk- or dv-wide results are laid out with that
// index as their 128 rows; the C x C ones use M = 64.  Other shapes and fp32 inputs go
// through one CTA-wide mma.sync helper (m16n8k8; 3xTF32 split for fp32 inputs, about
// fp32 accuracy), or the fp32 SIMT loop below when built with GDN_BWD_SIMT.  Kernels:
//     bwd_offsets   chunk offsets per sequence (+ cu_seqlens validation)
//     bwd_norm      q^, k^ and 1/|.| per (token, k-head)
//     bwd_wy        per (chunk, head): gam, T, W, U~, Q K^T (+ diag(b) K, diag(Gam) Q off tcgen05)
//     bwd_state_fwd per (sequence, head, dv slice): chunk-start states S_c and U   [sequential]
//     bwd_state_bwd per (sequence, head, dv slice): D_c (end-of-chunk grads) and dU; d_init_state
//     bwd_intra_s   per (chunk, head): the products with S0 and D (dQ_S, dW, U D)  [chunk-parallel]
//     bwd_intra_c   per (chunk, head): the C x C products, dV, dbeta, dg          [chunk-parallel]
//     bwd_fold      per (token, k-head): sum over the value heads of a k-head, L2-norm backward;
//                   in bwd_intra_tc the last value-head CTA of each (chunk, k-head) does it on chip
// Gradients are deterministic (fixed orders everywhere, no atomics on data: the one atomic counts
// arrivals for the on-chip fold and decides which CTA sums, not the order of the sum).
#include <algorithm>
#include <cuda_fp16.h>

#include "gdn_async.cuh"
#include "gdn_host.h"
#include "gdn_mma.cuh"
#include "gdn_step.cuh"
#include "gdn_umma.cuh"

namespace gdn {

constexpr int kC = 64;        // chunk length
#ifndef STAGGER_INTRA_CYCLES
#define STAGGER_INTRA_CYCLES 100000
#endif
constexpr int kMaxD = 128;    // max dk, dv
// smem leading dims = 4 (mod 32): row-major tensor-core fragment loads hit 32 distinct banks
constexpr int kLdD = kMaxD + 4;  // C x d and d x d matrices
constexpr int kLdC = kC + 4;     // C x C matrices
#ifndef GDN_BWD_NT
#define GDN_BWD_NT 1024
#endif
constexpr int kNT = GDN_BWD_NT;  // threads of the chunk-parallel kernels (32 warps hide their latency)
#ifndef GDN_BWD_NT_WY
#define GDN_BWD_NT_WY 512
#endif
// threads of bwd_wy: its ~103 KB of shared memory fits two CTAs per SM, which 512 threads allow
constexpr int kNTwy = GDN_BWD_NT_WY;
#ifndef GDN_BWD_NTS
#define GDN_BWD_NTS 1024
#endif
constexpr int kNTs = GDN_BWD_NTS;  // threads of the state-pass kernels (one CTA holds all dv rows)

struct BwdParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const float* init_state;
    const int32_t* cu;
    const void* dout;
    const float* dfinal;
    void* dq_out;
    void* dk_out;
    void* dv_out;
    float* dg;
    float* dbeta;
    float* dinit;
    unsigned* err;
    int32_t* coff;     // [N+1] chunk offsets
    float* qn;         // [T, HK, dk]
    float* kn;         // [T, HK, dk]
    float* qinv;       // [T, HK]
    float* kinv;       // [T, HK]
    float* gam;        // [T, HV]
    float* Wb;         // per chunk-head C x dk  (W, later dW)
    float* Utb;        // per chunk-head C x dv  (U~)
    float* Tb;         // per chunk-head C x C
    float* QKb;        // per chunk-head C x C: Q K^T
    float* Pb;         // per chunk-head C x C: P = lower(E) * Q K^T (rows >= len zero)
    float* BKb;        // per chunk-head C x dk: diag(b) K, b_r = exp(gam_last - gam_r)
    float* GQb;        // per chunk-head C x dk: diag(Gam) Q
    float* Sb;         // per chunk-head dv x dk (chunk-start state)
    float* Db;         // per chunk-head dv x dk (dL/d state at chunk end)
    __half* Sh;        // dk = dv = 128 (bf16), in place of Sb: per chunk-head S^T, 128 x 128, as scaled fp16
    __half* Dh;        //   likewise D^T, in place of Db
    float* Ssc;        //   per chunk-head 16 factors of Sh, one per 32 x 32 tile: value = fp16 * factor
    float* Dsc;        //   likewise for Dh
    float* Ub;         // per chunk-head C x dv
    float* dUb;        // per chunk-head C x dv
    float* dgamA;      // per chunk-head C
    float* dqh;        // [T, HV, dk]
    unsigned* fcnt;    // [nchm, HK] arrivals of the value-head CTAs of bwd_intra_tc_kernel (zeroed per call)
    float* dkh;        // [T, HV, dk]
    int N, T, HK, HV, G, dk, dv, use_norm, nchm, dtype;
    int nsm;                 // SMs of the device
    long long stagger_intra; // first-wave start spread of bwd_intra_tc_kernel, SM cycles (0: none)
};

// Spread the start of a chunk kernel's first wave (its first nsm CTAs in launch order) evenly over
// `cycles` SM cycles.  Every CTA of these kernels takes about the same time, so without a spread
// the waves stay aligned and all SMs fetch their first operands in the same burst; spread over
// about two CTA lifetimes, the bursts of different SMs stop coinciding.  The wait is a bounded
// sleep loop; it changes no result.
__device__ __forceinline__ void stagger_first_wave(long long cycles, int nsm) {
    const long long lin = (long long)blockIdx.x + (long long)blockIdx.y * gridDim.x;
    if (cycles <= 0 || lin >= nsm) return;
    const long long t0 = clock64(), delay = lin * cycles / nsm;
    while (clock64() - t0 < delay) __nanosleep(100);
}

__device__ __forceinline__ size_t ch_index(const BwdParams& p, int c, int h) { return (size_t)c * p.HV + h; }

__device__ __forceinline__ float ld_any(const void* base, size_t i, int dtype) {
    return dtype == GDN_BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i])
                             : reinterpret_cast<const float*>(base)[i];
}
__device__ __forceinline__ void st_any(void* base, size_t i, int dtype, float x) {
    if (dtype == GDN_BF16) reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
    else reinterpret_cast<float*>(base)[i] = x;
}

// Locate global chunk c: sequence n (largest n with coff[n] <= c), token range [t0, t0 + len).
__device__ __forceinline__ bool chunk_of(const BwdParams& p, int c, int& n, int& t0, int& len) {
    if (c >= p.coff[p.N]) return false;
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.coff[mid] <= c) lo = mid;
        else hi = mid - 1;
    }
    n = lo;
    int bos = min(max(p.cu[n], 0), p.T), eos = min(max(p.cu[n + 1], bos), p.T);
    t0 = bos + (c - p.coff[n]) * kC;
    len = min(kC, eos - t0);
    return len > 0;
}

// CTA-wide C(m, n) = sum_k A(m, k) B(k, n) over fp32 operands (shared or global),
// A(m, k) = A[m * as0 + k * as1], B(k, n) = B[k * bs0 + n * bs1].  Every output is
// produced by exactly one thread, once, through f(m, n, value); the k order is
// increasing, so results are deterministic.  4 x 4 register micro-tiles with
// rows m = tm + i * TMc and columns n = tn + j * TNc.
template <typename F>
__device__ __forceinline__ void cta_gemm(int M, int N, int K, const float* __restrict__ A, int as0, int as1,
                                         const float* __restrict__ B, int bs0, int bs1, F&& f) {
    const int tmc = M >> 2, tnc = N >> 2;
    for (int tile = threadIdx.x; tile < tmc * tnc; tile += blockDim.x) {
        const int tm = tile / tnc, tn = tile - tm * tnc;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        const float* a0 = A + (size_t)tm * as0;
        const float* b0 = B + (size_t)tn * bs1;
        for (int kk = 0; kk < K; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = a0[(size_t)(i * tmc) * as0 + (size_t)kk * as1];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = b0[(size_t)kk * bs0 + (size_t)(j * tnc) * bs1];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) f(tm + i * tmc, tn + j * tnc, acc[i][j]);
    }
}

// The backward's product: tensor cores unless GDN_BWD_SIMT.  The operand
// precision follows the input dtype: bf16 inputs (8 significant bits) run
// plain TF32, fp32 inputs the 3xTF32 split (about fp32 accuracy).
template <typename F>
__device__ __forceinline__ void bgemm_impl(bool split, int M, int N, int K, const float* __restrict__ A, int as0,
                                           int as1, const float* __restrict__ B, int bs0, int bs1, F&& f) {
#ifdef GDN_BWD_SIMT
    cta_gemm(M, N, K, A, as0, as1, B, bs0, bs1, f);
#else
    cta_gemm_tc(split, M, N, K, A, as0, as1, B, bs0, bs1, f);
#endif
}
#define bgemm(...) bgemm_impl(p.dtype == GDN_F32, __VA_ARGS__)

// The product added onto values held elsewhere: prior(m, n) reads what f(m, n, x, prior) updates.
template <typename P, typename F>
__device__ __forceinline__ void bgemm_rmw_impl(bool split, int M, int N, int K, const float* __restrict__ A, int as0,
                                               int as1, const float* __restrict__ B, int bs0, int bs1, P&& prior,
                                               F&& f) {
#ifdef GDN_BWD_SIMT
    cta_gemm(M, N, K, A, as0, as1, B, bs0, bs1, [&](int m, int n, float x) { f(m, n, x, prior(m, n)); });
#else
    cta_gemm_tc_rmw(split, M, N, K, A, as0, as1, B, bs0, bs1, prior, f);
#endif
}
#define bgemm_rmw(...) bgemm_rmw_impl(p.dtype == GDN_F32, __VA_ARGS__)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Copy rows [0, len) of a global fp32 matrix (row r at base + r * gstride) into shared memory
// (leading dim ld), zero-filling rows len .. R-1.  cols, gstride and ld are multiples of 4 and
// both bases 16-byte aligned: the copy is 16-byte cp.async, all in flight at once, and each
// thread waits for its own copies before returning (callers still barrier before reading).
__device__ __forceinline__ void load_rows_f32(float* dst, int ld, const float* base, size_t gstride, int R, int len,
                                              int cols) {
    const int c4 = cols >> 2;
    for (int i = threadIdx.x; i < R * c4; i += blockDim.x) {
        const int r = i / c4, c = (i - r * c4) << 2;
        float* d = dst + r * ld + c;
        if (r < len) cp_async16(d, base + (size_t)r * gstride + c);
        else *reinterpret_cast<float4*>(d) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    cp_async_wait_all();
}

// load_rows_f32 without the final wait: the copies complete at the caller's cp_async_wait_all().
__device__ __forceinline__ void load_rows_f32_async(float* dst, int ld, const float* base, size_t gstride, int R,
                                                    int len, int cols) {
    const int c4 = cols >> 2;
    for (int i = threadIdx.x; i < R * c4; i += blockDim.x) {
        const int r = i / c4, c = (i - r * c4) << 2;
        float* d = dst + r * ld + c;
        if (r < len) cp_async16(d, base + (size_t)r * gstride + c);
        else *reinterpret_cast<float4*>(d) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Same for a bf16 or fp32 source widened to fp32 (4 elements per access, 4 accesses in flight).
__device__ __forceinline__ float4 ld4_any(const void* base, size_t i, int dtype) {
    if (dtype == GDN_BF16) {
        const uint2 raw = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + i);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
}
__device__ __forceinline__ void load_rows_any(float* dst, int ld, const void* base, size_t off, size_t gstride,
                                              int R, int len, int cols, int dtype) {
    const int c4 = cols >> 2, total = R * c4;
    for (int i0 = threadIdx.x; i0 < total; i0 += 4 * blockDim.x) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * blockDim.x;
            const int r = i / c4, c = (i - r * c4) << 2;
            v[u] = (i < total && r < len) ? ld4_any(base, off + (size_t)r * gstride + c, dtype)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * blockDim.x;
            if (i < total) {
                const int r = i / c4, c = (i - r * c4) << 2;
                *reinterpret_cast<float4*>(dst + r * ld + c) = v[u];
            }
        }
    }
}

// Store rows [0, R) of a shared matrix (leading dim ld) to global (row stride gstride), float4 at a time.
__device__ __forceinline__ void store_rows_f32(float* base, size_t gstride, const float* src, int ld, int R,
                                               int cols) {
    const int c4 = cols >> 2;
    for (int i = threadIdx.x; i < R * c4; i += blockDim.x) {
        const int r = i / c4, c = (i - r * c4) << 2;
        *reinterpret_cast<float4*>(base + (size_t)r * gstride + c) = *reinterpret_cast<const float4*>(src + r * ld + c);
    }
}

// ---------------------------------------------------------------------------
__global__ void bwd_offsets_kernel(BwdParams p) {
    if (threadIdx.x != 0) return;
    int acc = 0;
    for (int n = 0; n < p.N; ++n) {
        const int a = p.cu[n], b = p.cu[n + 1];
        if ((n == 0 && a != 0) || b < a || (n == p.N - 1 && b != p.T)) atomicOr(p.err, GDN_DEVERR_CU_SEQLENS);
        const int lo = min(max(a, 0), p.T), hi = min(max(b, lo), p.T);
        p.coff[n] = acc;
        acc += (hi - lo + kC - 1) / kC;
    }
    p.coff[p.N] = min(acc, p.nchm);
}

// one warp per (token, k-head): q^, k^ and the reciprocal norms
__global__ void bwd_norm_kernel(BwdParams p) {
    const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= (long long)p.T * p.HK) return;
    for (int which = 0; which < 2; ++which) {
        const void* src = which ? p.k : p.q;
        float x[4];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = lane + 32 * i;
            x[i] = j < p.dk ? ld_any(src, (size_t)w * p.dk + j, p.dtype) : 0.f;
            ss = fmaf(x[i], x[i], ss);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
        const float inv = p.use_norm ? __frsqrt_rn(ss + kNormEps) : 1.f;
        float* dst = (which ? p.kn : p.qn) + (size_t)w * p.dk;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = lane + 32 * i;
            if (j < p.dk) dst[j] = x[i] * inv;
        }
        if (lane == 0) (which ? p.kinv : p.qinv)[w] = inv;
    }
}

// ---------------------------------------------------------------------------
// per (chunk, head): gam, T = (I + A)^-1, W, U~, QK
__global__ void __launch_bounds__(kNTwy) bwd_wy_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int c = blockIdx.x, h = blockIdx.y;
    int n, t0, len;
    if (!chunk_of(p, c, n, t0, len)) return;
    const int hk = h / p.G, dk = p.dk, dv = p.dv;
    float* sK = sm;                  // C x kLdD
    float* sQ = sK + kC * kLdD;      // C x kLdD (later V)
    float* sA = sQ + kC * kLdD;      // C x kLdC
    float* sT = sA + kC * kLdC;      // C x kLdC
    float* sTt = sA;                 // C x kLdC, reuses A's space: written only after the solve has read A
    float* sg = sT + kC * kLdC;      // gam [C]
    float* sGb = sg + kC;            // beta * Gam [C]
    float* sb = sGb + kC;            // beta [C]

    load_rows_f32(sK, kLdD, p.kn + ((size_t)t0 * p.HK + hk) * dk, (size_t)p.HK * dk, kC, len, dk);
    load_rows_f32(sQ, kLdD, p.qn + ((size_t)t0 * p.HK + hk) * dk, (size_t)p.HK * dk, kC, len, dk);
    if (threadIdx.x < 32) {
        // inclusive cumsum of g over the chunk, one warp, fixed order (lane-serial blocks of 2)
        float g0 = 0.f, g1 = 0.f;
        const int r0 = 2 * threadIdx.x, r1 = r0 + 1;
        if (r0 < len) g0 = p.g[(size_t)(t0 + r0) * p.HV + h];
        if (r1 < len) g1 = p.g[(size_t)(t0 + r1) * p.HV + h];
        float s = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(kFull, s, off);
            if ((int)threadIdx.x >= off) s += y;
        }
        const float excl = s - (g0 + g1);
        const float c0 = excl + g0, c1 = c0 + g1;
        sg[r0] = c0;
        sg[r1] = c1;
        const float b0 = r0 < len ? p.beta[(size_t)(t0 + r0) * p.HV + h] : 0.f;
        const float b1 = r1 < len ? p.beta[(size_t)(t0 + r1) * p.HV + h] : 0.f;
        sb[r0] = b0;
        sb[r1] = b1;
        sGb[r0] = b0 * __expf(c0);
        sGb[r1] = b1 * __expf(c1);
        if (r0 < len) p.gam[(size_t)(t0 + r0) * p.HV + h] = c0;
        if (r1 < len) p.gam[(size_t)(t0 + r1) * p.HV + h] = c1;
    }
    __syncthreads();
    const size_t ci = ch_index(p, c, h);
    // A = strict_lower(beta_r E[r,s] (K K^T)[r,s]);  QK = Q K^T (stored)
    bgemm(kC, kC, dk, sK, kLdD, 1, sK, 1, kLdD, [&](int r, int s, float kk) {
        sA[r * kLdC + s] = (s < r) ? sb[r] * __expf(sg[r] - sg[s]) * kk : 0.f;
    });
    float* QK = p.QKb + ci * kC * kC;
    float* P = p.Pb + ci * kC * kC;
    bgemm(kC, kC, dk, sQ, kLdD, 1, sK, 1, kLdD, [&](int r, int s, float x) {
        QK[r * kC + s] = x;
        P[r * kC + s] = (s <= r && r < len) ? x * __expf(sg[r] - sg[s]) : 0.f;
    });
    {
        // diag(b) K and diag(Gam) Q for the sequential passes (rows >= len are zero already)
        const float gl = sg[len - 1];
        float* BK = p.BKb + ci * kC * dk;
        float* GQ = p.GQb + ci * kC * dk;
        const int c4 = dk >> 2;
        for (int i = threadIdx.x; i < kC * c4; i += blockDim.x) {
            const int r = i / c4, j = (i - r * c4) << 2;
            const float b = r < len ? __expf(gl - sg[r]) : 0.f, G = r < len ? __expf(sg[r]) : 0.f;
            const float4 k4 = *reinterpret_cast<const float4*>(sK + r * kLdD + j);
            const float4 q4 = *reinterpret_cast<const float4*>(sQ + r * kLdD + j);
            *reinterpret_cast<float4*>(BK + r * dk + j) = make_float4(b * k4.x, b * k4.y, b * k4.z, b * k4.w);
            *reinterpret_cast<float4*>(GQ + r * dk + j) = make_float4(G * q4.x, G * q4.y, G * q4.z, G * q4.w);
        }
    }
    __syncthreads();
    // T = (I + A)^-1: thread j solves column j by forward substitution (columns are independent)
    if (threadIdx.x < kC) {
        const int j = threadIdx.x;
        for (int r = 0; r < kC; ++r) {
            // x = delta_rj - sum_{j <= s < r} A[r][s] T[s][j], as four interleaved partial sums
            float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
            int s = j;
            for (; s + 3 < r; s += 4) {
                x0 = fmaf(sA[r * kLdC + s], sT[s * kLdC + j], x0);
                x1 = fmaf(sA[r * kLdC + s + 1], sT[(s + 1) * kLdC + j], x1);
                x2 = fmaf(sA[r * kLdC + s + 2], sT[(s + 2) * kLdC + j], x2);
                x3 = fmaf(sA[r * kLdC + s + 3], sT[(s + 3) * kLdC + j], x3);
            }
            for (; s < r; ++s) x0 = fmaf(sA[r * kLdC + s], sT[s * kLdC + j], x0);
            const float x = ((r == j) ? 1.f : 0.f) - ((x0 + x1) + (x2 + x3));
            sT[r * kLdC + j] = (r < j) ? 0.f : x;
        }
    }
    // V into sQ (Q is no longer needed)
    __syncthreads();
    load_rows_any(sQ, kLdD, p.v, ((size_t)t0 * p.HV + h) * dv, (size_t)p.HV * dv, kC, len, dv, p.dtype);
    float* Tg = p.Tb + ci * kC * kC;
    for (int i = threadIdx.x; i < kC * kC; i += blockDim.x) {
        const int r = i / kC, s = i - r * kC;
        Tg[i] = sT[r * kLdC + s];
        sTt[r * kLdC + s] = sT[r * kLdC + s] * sGb[s];
    }
    __syncthreads();
    float* W = p.Wb + ci * kC * dk;
    bgemm(kC, dk, kC, sTt, kLdC, 1, sK, kLdD, 1, [&](int r, int j, float x) { W[r * dk + j] = x; });
    __syncthreads();
    for (int i = threadIdx.x; i < kC * kC; i += blockDim.x) {
        const int r = i / kC, s = i - r * kC;
        sTt[r * kLdC + s] = sT[r * kLdC + s] * sb[s];
    }
    __syncthreads();
    float* Ut = p.Utb + ci * kC * dv;
    bgemm(kC, dv, kC, sTt, kLdC, 1, sQ, kLdD, 1, [&](int r, int j, float x) { Ut[r * dv + j] = x; });
}

// ---------------------------------------------------------------------------
// per (sequence, head, slice of R rows): S_c for every chunk, U = U~ - W S^T, S <- Gam_C S + U^T diag(b) K
__global__ void __launch_bounds__(kNTs) bwd_state_fwd_kernel(BwdParams p, int R) {
    extern __shared__ float sm[];
    const int n = blockIdx.x, h = blockIdx.y, r0 = blockIdx.z * R;
    const int dk = p.dk, dv = p.dv;
    float* sS = sm;                   // R x kLdD
    float* sW = sS + R * kLdD;        // C x kLdD
    float* sK = sW + kC * kLdD;       // C x kLdD: diag(b) K
    float* sU = sK + kC * kLdD;       // C x (R + 4)
    float* sUt = sU + kC * (R + 4);   // C x (R + 4): U~ slice
    const int ldU = R + 4;
    const float* s0 = p.init_state ? p.init_state + (((size_t)n * p.HV + h) * dv + r0) * dk : nullptr;
    for (int i = threadIdx.x; i < R * dk; i += blockDim.x) {
        const int r = i / dk, j = i - r * dk;
        sS[r * kLdD + j] = s0 ? s0[(size_t)r * dk + j] : 0.f;
    }
    const int bos = min(max(p.cu[n], 0), p.T), eos = min(max(p.cu[n + 1], bos), p.T);
    const int nch = (eos - bos + kC - 1) / kC;
    for (int j = 0; j < nch; ++j) {
        const int c = p.coff[n] + j;
        if (c >= p.nchm) break;
        const int t0 = bos + j * kC, len = min(kC, eos - t0);
        const size_t ci = ch_index(p, c, h);
        __syncthreads();
        // chunk-start state out; stage W, diag(b) K and the U~ slice
        store_rows_f32(p.Sb + ci * dv * dk + (size_t)r0 * dk, dk, sS, kLdD, R, dk);
        load_rows_f32_async(sW, kLdD, p.Wb + ci * kC * dk, dk, kC, kC, dk);
        load_rows_f32_async(sK, kLdD, p.BKb + ci * kC * dk, dk, kC, kC, dk);
        load_rows_f32_async(sUt, ldU, p.Utb + ci * kC * dv + r0, dv, kC, kC, R);
        const float Gl = __expf(p.gam[(size_t)(t0 + len - 1) * p.HV + h]);
        cp_async_wait_all();
        __syncthreads();
        // U = U~ - W S^T  (C x R)
        float* Ug = p.Ub + ci * kC * dv + r0;
        bgemm(kC, R, dk, sW, kLdD, 1, sS, 1, kLdD, [&](int r, int i, float x) {
            const float u = sUt[r * ldU + i] - x;
            sU[r * ldU + i] = u;
            Ug[(size_t)r * dv + i] = u;
        });
        __syncthreads();
        // S <- Gam_last S + U^T (b K)
        bgemm(R, dk, kC, sU, 1, ldU, sK, kLdD, 1,
              [&](int i, int jj, float x) { sS[i * kLdD + jj] = fmaf(Gl, sS[i * kLdD + jj], x); });
    }
}

// per (sequence, head, slice of R rows), chunks in reverse: D_c (gradient at chunk end), dU; d_init_state
__global__ void __launch_bounds__(kNTs) bwd_state_bwd_kernel(BwdParams p, int R) {
    extern __shared__ float sm[];
    const int n = blockIdx.x, h = blockIdx.y, r0 = blockIdx.z * R;
    const int dk = p.dk, dv = p.dv;
    const int ldR = R + 4;
    float* sD = sm;                    // R x kLdD
    float* sQ = sD + R * kLdD;         // C x kLdD: diag(Gam) Q
    float* sW = sQ + kC * kLdD;        // C x kLdD: diag(b) K, then W
    float* sP = sW + kC * kLdD;        // C x kLdC: P
    float* sO = sP + kC * kLdC;        // C x ldR:  dO slice
    float* sdU = sO + kC * ldR;        // C x ldR
    const float* df = p.dfinal ? p.dfinal + (((size_t)n * p.HV + h) * dv + r0) * dk : nullptr;
    for (int i = threadIdx.x; i < R * dk; i += blockDim.x) {
        const int r = i / dk, j = i - r * dk;
        sD[r * kLdD + j] = df ? df[(size_t)r * dk + j] : 0.f;
    }
    const int bos = min(max(p.cu[n], 0), p.T), eos = min(max(p.cu[n + 1], bos), p.T);
    const int nch = (eos - bos + kC - 1) / kC;
    for (int j = nch - 1; j >= 0; --j) {
        const int c = p.coff[n] + j;
        if (c >= p.nchm) continue;
        const int t0 = bos + j * kC, len = min(kC, eos - t0);
        const size_t ci = ch_index(p, c, h);
        __syncthreads();
        store_rows_f32(p.Db + ci * dv * dk + (size_t)r0 * dk, dk, sD, kLdD, R, dk);
        load_rows_f32_async(sQ, kLdD, p.GQb + ci * kC * dk, dk, kC, kC, dk);
        load_rows_f32_async(sW, kLdD, p.BKb + ci * kC * dk, dk, kC, kC, dk);
        load_rows_f32_async(sP, kLdC, p.Pb + ci * kC * kC, kC, kC, kC, kC);
        load_rows_any(sO, ldR, p.dout, ((size_t)t0 * p.HV + h) * dv + r0, (size_t)p.HV * dv, kC, len, R, p.dtype);
        const float Gl = __expf(p.gam[(size_t)(t0 + len - 1) * p.HV + h]);
        cp_async_wait_all();
        __syncthreads();
        // dU = P^T dO + (b K) D^T   (C x R)
        bgemm(kC, R, kC, sP, 1, kLdC, sO, ldR, 1, [&](int s, int i, float x) { sdU[s * ldR + i] = x; });
        __syncthreads();
        float* dUg = p.dUb + ci * kC * dv + r0;
        bgemm(kC, R, dk, sW, kLdD, 1, sD, 1, kLdD, [&](int s, int i, float x) {
            const float u = sdU[s * ldR + i] + x;
            sdU[s * ldR + i] = u;
            dUg[(size_t)s * dv + i] = u;
        });
        __syncthreads();
        // W into sW (overlapping the next product), then D <- Gam_last D + dO^T (Gam Q) - dU^T W
        load_rows_f32_async(sW, kLdD, p.Wb + ci * kC * dk, dk, kC, kC, dk);
        bgemm(R, dk, kC, sO, 1, ldR, sQ, kLdD, 1,
              [&](int i, int jj, float x) { sD[i * kLdD + jj] = fmaf(Gl, sD[i * kLdD + jj], x); });
        cp_async_wait_all();
        __syncthreads();
        bgemm(R, dk, kC, sdU, 1, ldR, sW, kLdD, 1, [&](int i, int jj, float x) { sD[i * kLdD + jj] -= x; });
    }
    __syncthreads();
    if (p.dinit) store_rows_f32(p.dinit + (((size_t)n * p.HV + h) * dv + r0) * dk, dk, sD, kLdD, R, dk);
}

// ---------------------------------------------------------------------------
// The serial state passes on the fifth-generation tensor cores (bf16 inputs, dv = 128, dk in
// {32, 64, 128}).  One CTA of 512 threads per (sequence, head).  Every product has the M = 128
// state rows as its rows, so thread (warp w, lane l) owns state row i = 32 (w mod 4) + l in
// every epilogue, and the column group w / 4 of it.  The fp32 state (or state gradient) stays in
// TMEM for the whole sequence (each kernel says where); the tensor core reads it there as an A
// operand, and every other operand as a TF32-rounded copy in shared memory in the K-major
// core-matrix layout of gdn_umma.cuh.
// Every *_tc kernel runs exactly kNTtc threads per CTA: their thread-to-element mappings (16
// warps = 4 TMEM lane quarters x 4 column groups, and the staging strides) assume it.
constexpr int kNTtc = 512;
// At dk = 128 the chunk states S_c and D_c go out transposed (dk x dv), the layout in which
// bwd_intra_tc_kernel takes them as K-major operands, and as fp16 of their TF32 values with a
// factor per 32 x 32 tile (store_state_f16); other dk keep the row-major fp32 layout.
template <int DK>
constexpr bool kStateTransposed = DK == 128;
constexpr uint32_t kSboC = kC * 32;  // 8 rows x 64 values x 4 bytes

// Staging of one operand: every thread first loads its items (all loads in flight together),
// then writes them, rounded to TF32, into the operand's K-major core-matrix layout.

// The thread-to-element map of an NN x KK row-major operand (rows n, four consecutive k per item):
// a warp covers 8 rows x 16 values, 64 contiguous bytes of each of 8 source rows and one 128-byte
// core-matrix block per quarter of the warp's 16-byte stores.
template <int NN, int KK>
struct RowsTc {
    static constexpr int kItems = NN * KK / 4 / kNTtc;
    __device__ __forceinline__ static int row(int it) {
        const int e = threadIdx.x + it * kNTtc, lane = e & 31, blk = e >> 5;
        return (blk / (KK / 16)) * 8 + (lane & 7);
    }
    __device__ __forceinline__ static int col(int it) {
        const int e = threadIdx.x + it * kNTtc, lane = e & 31, blk = e >> 5;
        return ((blk % (KK / 16)) * 4 + (lane >> 3)) * 4;
    }
};

// dst(n, k) = src[k * NN + n] (the transpose of a row-major KK x NN block).  Consecutive threads
// take consecutive n: coalesced loads, conflict-free 16-byte stores.
template <int NN, int KK>
struct ColsTc {
    static constexpr int kItems = NN * KK / 4 / kNTtc;
    float4 v[kItems];
    __device__ __forceinline__ void load(const float* __restrict__ src) {
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int e = threadIdx.x + it * kNTtc, n = e % NN, k = (e / NN) * 4;
            v[it] = make_float4(src[(size_t)k * NN + n], src[(size_t)(k + 1) * NN + n], src[(size_t)(k + 2) * NN + n],
                                src[(size_t)(k + 3) * NN + n]);
        }
    }
    __device__ __forceinline__ void put(uint8_t* dst) const {
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int e = threadIdx.x + it * kNTtc, n = e % NN, k = (e / NN) * 4;
            *reinterpret_cast<float4*>(dst + umma_koff(n, k, KK * 32)) = tf32_round4(v[it]);
        }
    }
    // The same copy by 4-byte cp.async (no registers); round_in_place once this thread's copies landed.
    __device__ __forceinline__ static void issue_async(uint8_t* dst, const float* __restrict__ src) {
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int e = threadIdx.x + it * kNTtc, n = e % NN, k = (e / NN) * 4;
#pragma unroll
            for (int t = 0; t < 4; ++t) cp_async4(dst + umma_koff(n, k + t, KK * 32), src + (size_t)(k + t) * NN + n);
        }
    }
    __device__ __forceinline__ static void round_in_place(uint8_t* dst) {
#pragma unroll
        for (int it = 0; it < kItems; ++it) {
            const int e = threadIdx.x + it * kNTtc, n = e % NN, k = (e / NN) * 4;
            float4* q = reinterpret_cast<float4*>(dst + umma_koff(n, k, KK * 32));
            *q = tf32_round4(*q);
        }
    }
};

// Issue-side barrier: shared-memory writes of every thread are visible to the tensor core and
// earlier TMEM reads are ordered before the next MMA.
__device__ __forceinline__ void tc_sync() {
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Bounded wait for the MMAs committed to bar; every thread gets the CTA-wide verdict.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t& phase) {
    const bool ok = __syncthreads_and(mbar_wait_bounded(bar, phase));
    phase ^= 1u;
    tc_fence_after();
    return ok;
}

// Store this thread's slice of a row-major 128 x DK fp32 matrix (row i, columns c0 ..) to global.
template <int NS>
__device__ __forceinline__ void store_slice(float* dst, const float (&x)[NS]) {
#pragma unroll
    for (int m = 0; m < NS; m += 4) *reinterpret_cast<float4*>(dst + m) = make_float4(x[m], x[m + 1], x[m + 2], x[m + 3]);
}
// Write this thread's slice (row i, columns c0 .. c0 + NS) as the TF32 operand copy (sbo per 8 rows).
template <int NS>
__device__ __forceinline__ void put_slice_tc(uint8_t* dst, int i, int c0, uint32_t sbo, const float (&x)[NS], float sign) {
#pragma unroll
    for (int m = 0; m < NS; m += 4)
        *reinterpret_cast<float4*>(dst + umma_koff(i, c0 + m, sbo)) =
            make_float4(tf32_round(sign * x[m]), tf32_round(sign * x[m + 1]), tf32_round(sign * x[m + 2]),
                        tf32_round(sign * x[m + 3]));
}

// This thread's slice of a 128 x 128 state (row i, columns 32 cg .. 32 cg + 31, in TMEM at t) out as
// the fp16 transpose dst[j][i].  Each value is first rounded to TF32, as a product reads it, then
// multiplied by a power of two 2^e shared by the warp's 32 x 32 tile (rows 32 (i / 32) .., the
// same columns), with e chosen so that the tile's largest magnitude lands in [2^14, 2^15).  fp16
// holds 10 mantissa bits like TF32, so every value within a factor 2^29 of the tile's largest
// (an fp16 normal number after scaling) is stored exactly; smaller ones keep an absolute error
// below 2^-40 of it.  The factor back, 2^-e, goes to fac[4 cg + i / 32].
__device__ __forceinline__ void store_state_f16(__half* dst, float* fac, uint32_t t, int i, int cg) {
    float m = 0.f;
#pragma unroll
    for (int c = 0; c < 32; c += 16) {
        float x[16];
        tmem_ld<2>(t + c, x);
#pragma unroll
        for (int u = 0; u < 16; ++u) m = fmaxf(m, fabsf(x[u]));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
    // m = 1.f * 2^(be - 127) for a normal m (be its biased exponent), so e = 14 - (be - 127); a
    // tile of zeros or of fp32 subnormals takes the largest factor, one with an inf the factor 1
    const int be = (int)((__float_as_uint(m) >> 23) & 255u);
    const int e = be == 255 ? 0 : min(141 - be, 126);
    const float up = __uint_as_float((uint32_t)(127 + e) << 23), down = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
    for (int c = 0; c < 32; c += 16) {
        float x[16];
        tmem_ld<2>(t + c, x);
#pragma unroll
        for (int u = 0; u < 16; ++u) dst[(size_t)(32 * cg + c + u) * 128 + i] = __float2half_rn(tf32_round(x[u]) * up);
    }
    if ((threadIdx.x & 31) == 0) fac[4 * cg + (i >> 5)] = down;
}

// per (sequence, head), chunks in order: S_c out, U = U~ - W S^T, S <- Gam_last S + U^T diag(b) K.
// The state lives in TMEM (fp32, row i in lane i, columns [0, DK)): it is the A operand of S W^T
// (read as TF32: the low 13 mantissa bits unused) and, scaled by Gam_last in place once that product
// is done, the accumulator of U^T diag(b) K, so no state epilogue or shared-memory copy of S sits
// between one chunk's last product and the next chunk's first.  While chunk j computes, chunk j+1's
// W arrives by 16-byte cp.async once the first product has read W, and its normalised keys come
// into registers; diag(b) K is formed when they are written as the operand.  U~ comes into
// registers while the first product runs.  At dk = 128 S_c goes out as fp16 with tile factors
// (store_state_f16), and the pass streams about 160 KB per chunk step (S_c and U out; W, U~ and K^
// in), so one CTA per SM already keeps HBM well loaded.
template <int DK>
__global__ void __launch_bounds__(kNTtc, 1) bwd_state_fwd_tc_kernel(BwdParams p) {
    constexpr int kDv = 128, kS = DK / 4, kSc = kS >= 16 ? 16 : 8;  // state columns per thread, per TMEM access
    constexpr uint32_t kSboD = DK * 32;
    constexpr bool kStateT = kStateTransposed<DK>;
    extern __shared__ __align__(128) uint8_t smb[];
    uint8_t* sW = smb;                          // B of U^T = S W^T:         64 x DK
    uint8_t* sUt = sW + kC * DK * 4;            // A of U^T diag(b) K:       128 x 64
    uint8_t* sBKt = sUt + kDv * kC * 4;         // B (transposed diag(b) K): DK x 64
    float* sfb = reinterpret_cast<float*>(sBKt + DK * kC * 4);  // b_r = exp(gam_last - gam_r) of the chunk in bk
    uint64_t* bar = reinterpret_cast<uint64_t*>(sfb + kC);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    const int i = (warp & 3) * 32 + (tid & 31), cg = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    using WRows = RowsTc<kC, DK>;
    // W of chunk ci into its operand layout (at dk = 128 already TF32, as bwd_wy_tc_kernel stores it)
    auto issue_w = [&](size_t ci) {
        const float* src = p.Wb + ci * kC * DK;
#pragma unroll
        for (int it = 0; it < WRows::kItems; ++it) {
            const int r = WRows::row(it), k = WRows::col(it);
            cp_async16(sW + umma_koff(r, k, kSboD), src + (size_t)r * DK + k);
        }
    };
    auto round_w = [&]() {
#pragma unroll
        for (int it = 0; it < WRows::kItems; ++it) {
            float4* q = reinterpret_cast<float4*>(sW + umma_koff(WRows::row(it), WRows::col(it), kSboD));
            *q = tf32_round4(*q);
        }
    };
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(slot, 256);
    const int bos = min(max(p.cu[n], 0), p.T), eos = min(max(p.cu[n + 1], bos), p.T);
    const int nch = (eos - bos + kC - 1) / kC;
    auto has = [&](int j) { return j < nch && p.coff[n] + j < p.nchm; };
    // K^T of the chunk about to run in registers (the normalised keys, rows >= len zero), and its
    // factors b_r in sfb; the product diag(b) K^ is taken when the operand is written (bk_put)
    const int hk = h / p.G;
    ColsTc<DK, kC> bk;
    float fb_gl = 0.f, fb_gr = 0.f;  // gam_last and gam_r (r = tid < 64) of the chunk in bk, or 0 past len
    bool fb_in = false;
    auto bk_load = [&](int jc) {
        const int t0c = bos + jc * kC, lenc = min(kC, eos - t0c);
        const float* kr = p.kn + ((size_t)t0c * p.HK + hk) * DK;
        const size_t st = (size_t)p.HK * DK;
#pragma unroll
        for (int it = 0; it < ColsTc<DK, kC>::kItems; ++it) {
            const int e = tid + it * kNTtc, nn = e % DK, k = (e / DK) * 4;
            bk.v[it] = make_float4(k < lenc ? kr[k * st + nn] : 0.f, k + 1 < lenc ? kr[(k + 1) * st + nn] : 0.f,
                                   k + 2 < lenc ? kr[(k + 2) * st + nn] : 0.f, k + 3 < lenc ? kr[(k + 3) * st + nn] : 0.f);
        }
        if (tid < kC) {  // used a chunk step later: no wait for these loads here
            fb_in = tid < lenc;
            fb_gl = p.gam[(size_t)(t0c + lenc - 1) * p.HV + h];
            fb_gr = fb_in ? p.gam[(size_t)(t0c + tid) * p.HV + h] : 0.f;
        }
    };
    auto bk_put = [&]() {
#pragma unroll
        for (int it = 0; it < ColsTc<DK, kC>::kItems; ++it) {
            const int e = tid + it * kNTtc, nn = e % DK, k = (e / DK) * 4;
            const float4 v = bk.v[it];
            *reinterpret_cast<float4*>(sBKt + umma_koff(nn, k, kC * 32)) = tf32_round4(
                make_float4(sfb[k] * v.x, sfb[k + 1] * v.y, sfb[k + 2] * v.z, sfb[k + 3] * v.w));
        }
    };
    if (has(0)) {
        issue_w(ch_index(p, p.coff[n], h));
        bk_load(0);
    }
    tc_sync();  // the TMEM address is in *slot
    const uint32_t tmem = *slot, tS = tmem + lane_base + cg * kS;
    {   // S_0 (this thread's kS columns of row i) into TMEM
        const float* s0 = p.init_state ? p.init_state + (((size_t)n * p.HV + h) * kDv + i) * DK + cg * kS : nullptr;
#pragma unroll
        for (int c = 0; c < kS; c += 8) {
            float x[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) x[m] = s0 ? s0[c + m] : 0.f;
            tmem_st<1>(tS + c, x);
        }
    }
    uint32_t phase = 0;
    bool ok = true;
    for (int j = 0; has(j) && ok; ++j) {
        const int c = p.coff[n] + j;
        const int t0 = bos + j * kC, len = min(kC, eos - t0);
        const size_t ci = ch_index(p, c, h), cn = ch_index(p, c + 1, h);
        const bool next = has(j + 1);
        cp_async_wait_all();  // this thread's copies of W (commits what is still open)
        if constexpr (DK != 128) round_w();
        if (tid < kC) sfb[tid] = fb_in ? __expf(fb_gl - fb_gr) : 0.f;
        __syncthreads();  // sfb of this chunk is complete
        bk_put();
        const float Gl = __expf(p.gam[(size_t)(t0 + len - 1) * p.HV + h]);
        tc_sync();
        if (tid == 0) {
            const uint32_t id = umma_idesc_tf32(kDv, kC);
            for (int s8 = 0; s8 < DK / 8; ++s8)
                umma_tf32_ts(tmem + 128, tmem + 8 * s8, umma_desc(smem_u32(sW) + 256u * s8, kSboD), id, s8 > 0);
            umma_commit(bar);
        }
        // chunk-start state out, U~ into registers and the next chunk's keys, while the product runs
        if constexpr (kStateT) {
            store_state_f16(p.Sh + ci * DK * kDv, p.Ssc + ci * 16, tS, i, cg);
        } else {
#pragma unroll
            for (int c8 = 0; c8 < kS; c8 += kSc) {
                float x[kSc];
                tmem_ld<kSc / 8>(tS + c8, x);
                float* dst = p.Sb + (ci * kDv + i) * DK + cg * kS + c8;
#pragma unroll
                for (int m = 0; m < kSc; m += 4)
                    *reinterpret_cast<float4*>(dst + m) = make_float4(x[m], x[m + 1], x[m + 2], x[m + 3]);
            }
        }
        float ut[16];
        {
            const float* ug = p.Utb + ci * kC * kDv + i;
#pragma unroll
            for (int m = 0; m < 16; ++m) ut[m] = ug[(size_t)(cg * 16 + m) * kDv];
        }
        if (next) bk_load(j + 1);
        if (!(ok = tc_wait(bar, phase))) break;
        if (next) issue_w(cn);
        // S <- Gam_last S in place: the first term of the state update
#pragma unroll
        for (int c8 = 0; c8 < kS; c8 += kSc) {
            float x[kSc];
            tmem_ld<kSc / 8>(tS + c8, x);
#pragma unroll
            for (int m = 0; m < kSc; ++m) x[m] *= Gl;
            tmem_st<kSc / 8>(tS + c8, x);
        }
        {   // U[r][i] = U~[r][i] - (S W^T)[i][r] for this thread's 16 values of r
            float x[16];
            tmem_ld<2>(tmem + lane_base + 128 + cg * 16, x);
            float* ug = p.Ub + ci * kC * kDv + i;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                x[m] = ut[m] - x[m];
                // at dk = 128 U only ever enters the tensor cores: stored already rounded to TF32
                ug[(size_t)(cg * 16 + m) * kDv] = DK == 128 ? tf32_round(x[m]) : x[m];
            }
            put_slice_tc<16>(sUt, i, cg * 16, kSboC, x, 1.f);
        }
        tc_sync();
        if (tid == 0) {  // S += U^T diag(b) K
            umma_tf32_k(tmem, smem_u32(sUt), kSboC, smem_u32(sBKt), kSboC, umma_idesc_tf32(kDv, DK), kC, true);
            umma_commit(bar);
        }
        if (!(ok = tc_wait(bar, phase))) break;
    }
    cp_async_wait_all();
    if (!ok && tid == 0) atomicOr(p.err, GDN_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// per (sequence, head), chunks in reverse: D_c out (gradient at chunk end), dU, d_init_state.
//   dU^T = dO^T P + D (diag(b) K)^T,   D <- Gam_last D + dO^T diag(Gam) Q - dU^T W
// D lives in TMEM (fp32, row i in lane i, columns [256, 256 + DK)): the A operand of D (diag(b) K)^T
// (read as TF32) and, scaled by Gam_last in place once the first product is done, the accumulator
// of the last two.  D_c goes out while the first product runs (at dk = 128 as fp16 with tile
// factors, store_state_f16).  W^T has a buffer of its own (loaded
// into registers during the first product).  The next chunk's P, and its k and q rows as given
// (bf16, into staging buffers), arrive by cp.async while the last two products run; at the top of
// its step they become diag(b) K^ and (diag(Gam) Q^)^T, scaled by 1/|k_r|, 1/|q_r| and the decay
// factors and rounded.  The next chunk's dO comes into registers meanwhile and takes dO^T's place
// once the products are done.
template <int DK>
__global__ void __launch_bounds__(kNTtc, 1) bwd_state_bwd_tc_kernel(BwdParams p) {
    constexpr int kDv = 128, kS = DK / 4, kSc = kS >= 16 ? 16 : 8;  // state columns per thread, per TMEM access
    constexpr int kStg = DK * 2 + 16;  // staging row pitch (bytes): 16-byte aligned, rows on different banks
    constexpr uint32_t kSboD = DK * 32;
    constexpr bool kStateT = kStateTransposed<DK>;
    extern __shared__ __align__(128) uint8_t smb[];
    uint8_t* sOt = smb;                         // A: dO^T                      128 x 64
    uint8_t* sW = sOt + kDv * kC * 4;           // B: W^T                       DK x 64
    uint8_t* sPt = sW + DK * kC * 4;            // B: P^T                       64 x 64
    uint8_t* sBK = sPt + kC * kC * 4;           // B: diag(b) K                 64 x DK
    uint8_t* sGQt = sBK + kC * DK * 4;          // B: (diag(Gam) Q)^T           DK x 64
    uint8_t* sdUt = sGQt + DK * kC * 4;         // A: -dU^T                     128 x 64
    uint8_t* sKs = sdUt + kDv * kC * 4;         // k rows of the next chunk, bf16, rows kStg bytes apart
    uint8_t* sQs = sKs + kC * kStg;             // q rows likewise
    float* sfb = reinterpret_cast<float*>(sQs + kC * kStg);  // b_r of the chunk in sBK (0 past len)
    float* sfg = sfb + kC;                                    // Gam_r of the chunk in sGQt (0 past len)
    float* skinv = sfg + kC;                                  // 1/|k_r|, 1/|q_r| of that chunk
    float* sqinv = skinv + kC;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sqinv + kC);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
    const int i = (warp & 3) * 32 + (tid & 31), cg = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    using PT = ColsTc<kC, kC>;
    using BK = RowsTc<kC, DK>;
    using GT = ColsTc<DK, kC>;
    constexpr int kOItems = kDv * kC / 4 / kNTtc;
    float4 o[kOItems];  // dO^T of the chunk about to run: (i, r) = dO[t0 + r][h][i], rows r >= len zero
    auto load_dO = [&](int t0, int len) {
        const size_t st = (size_t)p.HV * kDv;
#pragma unroll
        for (int it = 0; it < kOItems; ++it) {
            const int e = tid + it * kNTtc, ii = e % kDv, r = (e / kDv) * 4;
            const size_t base = ((size_t)(t0 + r) * p.HV + h) * kDv + ii;
            o[it] = make_float4(r < len ? ld_any(p.dout, base, p.dtype) : 0.f,
                                r + 1 < len ? ld_any(p.dout, base + st, p.dtype) : 0.f,
                                r + 2 < len ? ld_any(p.dout, base + 2 * st, p.dtype) : 0.f,
                                r + 3 < len ? ld_any(p.dout, base + 3 * st, p.dtype) : 0.f);
        }
    };
    auto put_dO = [&]() {
#pragma unroll
        for (int it = 0; it < kOItems; ++it) {
            const int e = tid + it * kNTtc, ii = e % kDv, r = (e / kDv) * 4;
            *reinterpret_cast<float4*>(sOt + umma_koff(ii, r, kSboC)) = tf32_round4(o[it]);
        }
    };
    const int hk = h / p.G;
    // P^T (by cp.async into its operand layout) and the k and q rows of chunk ci as given (bf16, by
    // 16-byte cp.async into the staging buffers; tokens t0c .., lenc of them, rows >= lenc zero), and
    // the factors b_r, Gam_r, 1/|k_r|, 1/|q_r| for the top of its step
    float fb_gl = 0.f, fb_gr = 0.f;  // gam_last and gam_r (r = tid < 64) of the chunk being copied
    float fb_kinv = 0.f, fb_qinv = 0.f;
    bool fb_in = false;
    auto issue_chunk = [&](size_t ci, int t0c, int lenc) {
        PT::issue_async(sPt, p.Pb + ci * kC * kC);
        const __nv_bfloat16* kr = static_cast<const __nv_bfloat16*>(p.k) + ((size_t)t0c * p.HK + hk) * DK;
        const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(p.q) + ((size_t)t0c * p.HK + hk) * DK;
        const size_t st = (size_t)p.HK * DK;
        constexpr int kPieces = DK / 8;  // 16-byte pieces per row
        for (int e = tid; e < kC * kPieces; e += kNTtc) {
            const int r = e / kPieces, c = (e % kPieces) * 8;
            uint8_t* dk_ = sKs + r * kStg + c * 2;
            uint8_t* dq_ = sQs + r * kStg + c * 2;
            if (r < lenc) {
                cp_async16(dk_, kr + r * st + c);
                cp_async16(dq_, qr + r * st + c);
            } else {
                *reinterpret_cast<uint4*>(dk_) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(dq_) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (tid < kC) {  // used a chunk step later: no wait for these loads here
            fb_in = tid < lenc;
            fb_gl = p.gam[(size_t)(t0c + lenc - 1) * p.HV + h];
            fb_gr = fb_in ? p.gam[(size_t)(t0c + tid) * p.HV + h] : 0.f;
            fb_kinv = fb_in ? p.kinv[(size_t)(t0c + tid) * p.HK + hk] : 0.f;
            fb_qinv = fb_in ? p.qinv[(size_t)(t0c + tid) * p.HK + hk] : 0.f;
        }
    };
    // diag(b) K^ and (diag(Gam) Q^)^T as TF32 from the staged rows: b_r (k_r 1/|k_r|) and
    // Gam_r (q_r 1/|q_r|), the same fp32 products as the normalised rows times the factors
    auto stage_in = [&]() {
        auto bf = [](uint32_t u, int hi) { return __uint_as_float(hi ? (u & 0xFFFF0000u) : (u << 16)); };
#pragma unroll
        for (int it = 0; it < BK::kItems; ++it) {
            const int r = BK::row(it), k = BK::col(it);
            const uint2 raw = *reinterpret_cast<const uint2*>(sKs + r * kStg + k * 2);
            const float f = sfb[r], iv = skinv[r];
            *reinterpret_cast<float4*>(sBK + umma_koff(r, k, DK * 32)) = tf32_round4(
                make_float4(f * (bf(raw.x, 0) * iv), f * (bf(raw.x, 1) * iv), f * (bf(raw.y, 0) * iv),
                            f * (bf(raw.y, 1) * iv)));
        }
#pragma unroll
        for (int it = 0; it < GT::kItems; ++it) {
            const int e = tid + it * kNTtc, nn = e % DK, k = (e / DK) * 4;
            float v[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float x = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sQs + (k + t) * kStg + nn * 2));
                v[t] = sfg[k + t] * (x * sqinv[k + t]);
            }
            *reinterpret_cast<float4*>(sGQt + umma_koff(nn, k, kC * 32)) = tf32_round4(make_float4(v[0], v[1], v[2], v[3]));
        }
    };
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(slot, 512);
    const int bos = min(max(p.cu[n], 0), p.T), eos = min(max(p.cu[n + 1], bos), p.T);
    const int nch = (eos - bos + kC - 1) / kC;
    const int jtop = min(nch, p.nchm - p.coff[n]) - 1;  // last chunk inside the workspace
    if (jtop >= 0) {
        const int t0 = bos + jtop * kC;
        issue_chunk(ch_index(p, p.coff[n] + jtop, h), t0, min(kC, eos - t0));
        load_dO(t0, min(kC, eos - t0));
        put_dO();
    }
    tc_sync();  // the TMEM address is in *slot
    const uint32_t tmem = *slot, tD = tmem + lane_base + 256 + cg * kS;
    {   // D at the sequence end (this thread's kS columns of row i) into TMEM
        const float* df = p.dfinal ? p.dfinal + (((size_t)n * p.HV + h) * kDv + i) * DK + cg * kS : nullptr;
#pragma unroll
        for (int c = 0; c < kS; c += 8) {
            float x[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) x[m] = df ? df[c + m] : 0.f;
            tmem_st<1>(tD + c, x);
        }
    }
    uint32_t phase = 0;
    bool ok = true;
    for (int j = jtop; j >= 0 && ok; --j) {
        const int c = p.coff[n] + j;
        const int t0 = bos + j * kC, len = min(kC, eos - t0);
        const size_t ci = ch_index(p, c, h);
        const bool prev = j > 0;
        const int tp = t0 - kC;  // the chunk before this one is always full
        cp_async_wait_all();  // this thread's copies of P and of the k and q rows
        if constexpr (DK != 128) PT::round_in_place(sPt);  // at dk = 128 bwd_wy_tc_kernel stores P as TF32
        if (tid < kC) {
            sfb[tid] = fb_in ? __expf(fb_gl - fb_gr) : 0.f;
            sfg[tid] = fb_in ? __expf(fb_gr) : 0.f;
            skinv[tid] = fb_kinv;
            sqinv[tid] = fb_qinv;
        }
        __syncthreads();  // the factors and every thread's staged rows are in shared memory
        stage_in();
        const float Gl = __expf(p.gam[(size_t)(t0 + len - 1) * p.HV + h]);
        tc_sync();
        if (tid == 0) {  // dU^T = dO^T P + D (diag(b) K)^T
            const uint32_t i1 = umma_idesc_tf32(kDv, kC);
            umma_tf32_k(tmem, smem_u32(sOt), kSboC, smem_u32(sPt), kSboC, i1, kC, false);
            for (int s8 = 0; s8 < DK / 8; ++s8)
                umma_tf32_ts(tmem, tmem + 256 + 8 * s8, umma_desc(smem_u32(sBK) + 256u * s8, kSboD), i1, true);
            umma_commit(bar);
        }
        // D_c out and W^T into registers while the product runs
        if constexpr (kStateT) {
            store_state_f16(p.Dh + ci * DK * kDv, p.Dsc + ci * 16, tD, i, cg);
        } else {
#pragma unroll
            for (int c8 = 0; c8 < kS; c8 += kSc) {
                float x[kSc];
                tmem_ld<kSc / 8>(tD + c8, x);
                float* dst = p.Db + (ci * kDv + i) * DK + cg * kS + c8;
#pragma unroll
                for (int m = 0; m < kSc; m += 4)
                    *reinterpret_cast<float4*>(dst + m) = make_float4(x[m], x[m + 1], x[m + 2], x[m + 3]);
            }
        }
        GT w;
        w.load(p.Wb + ci * kC * DK);
        if (!(ok = tc_wait(bar, phase))) break;
        // D <- Gam_last D in place: the first term of the update
#pragma unroll
        for (int c8 = 0; c8 < kS; c8 += kSc) {
            float x[kSc];
            tmem_ld<kSc / 8>(tD + c8, x);
#pragma unroll
            for (int m = 0; m < kSc; ++m) x[m] *= Gl;
            tmem_st<kSc / 8>(tD + c8, x);
        }
        {   // dU[s][i] for this thread's 16 values of s; -dU^T as the last product's A
            float x[16];
            tmem_ld<2>(tmem + lane_base + cg * 16, x);
            float* dug = p.dUb + ci * kC * kDv + i;
#pragma unroll
            for (int m = 0; m < 16; ++m)  // at dk = 128 only ever a TF32 operand: stored rounded
                dug[(size_t)(cg * 16 + m) * kDv] = DK == 128 ? tf32_round(x[m]) : x[m];
            put_slice_tc<16>(sdUt, i, cg * 16, kSboC, x, -1.f);
        }
        w.put(sW);
        tc_sync();
        if (tid == 0) {  // D += dO^T diag(Gam) Q - dU^T W
            const uint32_t i2 = umma_idesc_tf32(kDv, DK);
            umma_tf32_k(tmem + 256, smem_u32(sOt), kSboC, smem_u32(sGQt), kSboC, i2, kC, true);
            umma_tf32_k(tmem + 256, smem_u32(sdUt), kSboC, smem_u32(sW), kSboC, i2, kC, true);
            umma_commit(bar);
        }
        if (prev) {  // the next chunk's operands while they run
            issue_chunk(ci - p.HV, tp, kC);
            load_dO(tp, kC);
        }
        if (!(ok = tc_wait(bar, phase))) break;
        if (prev) put_dO();  // the last products have read dO^T
    }
    cp_async_wait_all();
    if (ok && p.dinit) {
        float* dst = p.dinit + (((size_t)n * p.HV + h) * kDv + i) * DK + cg * kS;
#pragma unroll
        for (int c8 = 0; c8 < kS; c8 += kSc) {
            float x[kSc];
            tmem_ld<kSc / 8>(tD + c8, x);
            store_slice<kSc>(dst + c8, x);
        }
    }
    if (!ok && tid == 0) atomicOr(p.err, GDN_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Deterministic CTA sum of one float per thread (fixed tree); all threads get the result.
__device__ __forceinline__ float cta_sum(float x, float* red) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[w] = x;
    __syncthreads();
    float s = 0.f;
    for (int i = 0; i < nw; ++i) s += red[i];
    return s;
}

// per (chunk, head): products with S0 and D.
//   dQ_S = diag(Gam) dO S0 -> dqh;  dgam_r += q^_r . dQ_S,r;  dW = -dU S0 -> Wb
//   dgam_last += Gam_last <D, S0>;  UD = U D: dkh = diag(b) UD, db_s = k^_s . UD_s
__global__ void __launch_bounds__(kNT) bwd_intra_s_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int c = blockIdx.x, h = blockIdx.y;
    int n, t0, len;
    if (!chunk_of(p, c, n, t0, len)) return;
    const int hk = h / p.G, dk = p.dk, dv = p.dv;
    float* sBig = sm;                   // dv x kLdD  (S0, then D)
    float* sA = sBig + kMaxD * kLdD;    // C x kLdD   (dO, then U)
    float* sB = sA + kC * kLdD;         // C x kLdD   (Q, then K)
    float* sC = sB + kC * kLdD;         // C x kLdD   (dU, then UD)
    float* sX = sC + kC * kLdD;         // C x kLdD   (dQ_S)
    float* sg = sX + kC * kLdD;         // gam [C]
    float* sdg = sg + kC;               // dgam [C]
    float* red = sdg + kC;              // [32]
    const size_t ci = ch_index(p, c, h);
    load_rows_f32(sBig, kLdD, p.Sb + ci * dv * dk, dk, dv, dv, dk);
    load_rows_any(sA, kLdD, p.dout, ((size_t)t0 * p.HV + h) * dv, (size_t)p.HV * dv, kC, len, dv, p.dtype);
    load_rows_f32(sB, kLdD, p.qn + ((size_t)t0 * p.HK + hk) * dk, (size_t)p.HK * dk, kC, len, dk);
    load_rows_f32(sC, kLdD, p.dUb + ci * kC * dv, dv, kC, kC, dv);
    for (int i = threadIdx.x; i < kC; i += blockDim.x) {
        // past the chunk's end gam stays at its last value (as the cumsum in bwd_wy_tc_kernel leaves it),
        // so gam is non-increasing over all 64 rows and exp(gam_r - gam_s), s <= r, never exceeds 1
        sg[i] = p.gam[(size_t)(t0 + min(i, len - 1)) * p.HV + h];
        sdg[i] = 0.f;
    }
    __syncthreads();
    const float gl = sg[len - 1];
    // dQ_S = diag(Gam) dO S0
    bgemm(kC, dk, dv, sA, kLdD, 1, sBig, kLdD, 1,
             [&](int r, int j, float x) { sX[r * kLdD + j] = (r < len) ? __expf(sg[r]) * x : 0.f; });
    // dW = -dU S0
    float* dW = p.Wb + ci * kC * dk;
    bgemm(kC, dk, dv, sC, kLdD, 1, sBig, kLdD, 1, [&](int r, int j, float x) { dW[r * dk + j] = -x; });
    __syncthreads();
    float* dq = p.dqh;
    for (int i = threadIdx.x; i < kC * dk; i += blockDim.x) {
        const int r = i / dk, j = i - r * dk;
        if (r < len) dq[((size_t)(t0 + r) * p.HV + h) * dk + j] = sX[r * kLdD + j];
    }
    // dgam_r += q^_r . dQ_S,r  (one warp per row, fixed order)
    {
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
        for (int r = w; r < len; r += nw) {
            float s = 0.f;
            for (int j = lane; j < dk; j += 32) s = fmaf(sB[r * kLdD + j], sX[r * kLdD + j], s);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
            if (lane == 0) sdg[r] += s;
        }
    }
    // <D, S0> with D read from global against S0 in shared memory
    const float* Dg = p.Db + ci * dv * dk;
    float part = 0.f;
    {
        const int c4 = dk >> 2, total = dv * c4;
        for (int i0 = threadIdx.x; i0 < total; i0 += 4 * blockDim.x) {
            float4 d4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * blockDim.x;
                d4[u] = i < total ? *reinterpret_cast<const float4*>(Dg + (size_t)4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * blockDim.x;
                if (i < total) {
                    const int r = i / c4, j = (i - r * c4) << 2;
                    const float* sp = sBig + r * kLdD + j;
                    part = fmaf(d4[u].x, sp[0], part);
                    part = fmaf(d4[u].y, sp[1], part);
                    part = fmaf(d4[u].z, sp[2], part);
                    part = fmaf(d4[u].w, sp[3], part);
                }
            }
        }
    }
    const float dS = cta_sum(part, red);
    __syncthreads();
    // D phase: D into sBig, U into sA, K into sB
    load_rows_f32(sBig, kLdD, Dg, dk, dv, dv, dk);
    load_rows_f32(sA, kLdD, p.Ub + ci * kC * dv, dv, kC, kC, dv);
    load_rows_f32(sB, kLdD, p.kn + ((size_t)t0 * p.HK + hk) * dk, (size_t)p.HK * dk, kC, len, dk);
    __syncthreads();
    bgemm(kC, dk, dv, sA, kLdD, 1, sBig, kLdD, 1, [&](int r, int j, float x) { sC[r * kLdD + j] = x; });
    __syncthreads();
    float* dkk = p.dkh;
    for (int i = threadIdx.x; i < kC * dk; i += blockDim.x) {
        const int r = i / dk, j = i - r * dk;
        if (r < len) dkk[((size_t)(t0 + r) * p.HV + h) * dk + j] = __expf(gl - sg[r]) * sC[r * kLdD + j];
    }
    __syncthreads();
    {
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
        for (int r = w; r < len; r += nw) {
            float s = 0.f;
            for (int j = lane; j < dk; j += 32) s = fmaf(sB[r * kLdD + j], sC[r * kLdD + j], s);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
            if (lane == 0) sX[r] = __expf(gl - sg[r]) * s;  // b_s db_s (sX reused as scratch)
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int r = 0; r < len; ++r) tot += sX[r];
        for (int r = 0; r < len; ++r) sdg[r] -= sX[r];
        sdg[len - 1] += tot + __expf(gl) * dS;
    }
    __syncthreads();
    float* dga = p.dgamA + ci * kC;
    for (int i = threadIdx.x; i < kC; i += blockDim.x) dga[i] = sdg[i];
}

// Sums over the 32 lanes of a warp of each of NV values (NV = 32 or 16), by a transpose-reduce
// butterfly in a fixed order; afterwards lane l holds the sum for value l % NV.
template <int NV>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[NV]) {
    const int lane = threadIdx.x & 31;
    if constexpr (NV == 16) {
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] += __shfl_xor_sync(kFull, v[k], 16);
    }
#pragma unroll
    for (int half = NV / 2; half >= 1; half >>= 1) {
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float send = upper ? v[k] : v[k + half];
            const float keep = upper ? v[k + half] : v[k];
            v[k] = keep + __shfl_xor_sync(kFull, send, half);
        }
    }
    return v[0];
}

// Sum over the 16 lanes of a half warp (xor butterfly, fixed order); every lane gets the sum.
// All 32 lanes of the warp must call it.
__device__ __forceinline__ float half_sum(float x) {
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}

// per (chunk, head), dk = dv = 128, bf16 inputs: bwd_wy_kernel on tcgen05.
//   [K; Q] K^T (M = 128: rows 0..63 give K K^T, rows 64..127 give Q K^T; the B operand is the
//   first 64 rows of the same shared-memory copy), A and P from them, T = (I + A)^-1 by
//   16 x 16 blocks (below), then W^T = K^T (T diag(beta Gam))^T
//   and U~^T = V^T (T diag(beta))^T with the dk / dv index as the M = 128 rows, so each epilogue
//   thread stores one column of W and U~: coalesced.
//   Shared memory is reused by phase: QK^T and P are staged where Q^ was and leave coalesced, and
//   V arrives by tensor copy into that space while the solve runs; K^T and V^T are then written
//   by columns, four values of s per 16-byte store.
//   Two CTAs share an SM (64 registers a thread, 97 KB of shared memory and 256 TMEM columns
//   each), so that one CTA's copies, solve and epilogues overlap the other's.
constexpr int kLdT = kC + 1;  // fp32 A and T in shared memory: row-per-lane writes hit distinct banks

// Staging of QK^T row r (64 fp32, sixteen 16-byte pieces) in the Q^ half of the swizzled [K^; Q^]
// copy: rows 0..31 in the first 32-value box, rows 32..63 in the second, 256 bytes a row; P's
// staging is 32 KB further on (the third and fourth boxes).  Piece pc sits at pc ^ (r mod 16), so
// that eight consecutive rows writing the same piece, or one row's pieces read in order, fall in
// distinct banks.
__device__ __forceinline__ uint8_t* qkp_stage(uint8_t* sX, int r, int pc) {
    return sX + 16384 * (r >> 5) + 8192 + 256 * (r & 31) + 16 * (pc ^ (r & 15));
}
constexpr int kWyCtasPerSm = 2;
constexpr size_t kWyTcSmem = (size_t)65536 + 2 * 4 * kC * kLdT + 4 * 3 * kC + 32;
// 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(kWyCtasPerSm * (kWyTcSmem + 1024) <= 228 * 1024, "two wy CTAs must fit on one SM");

__global__ void __launch_bounds__(kNTtc, kWyCtasPerSm)
    bwd_wy_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_v, BwdParams p) {
    constexpr int kD = 128;
    extern __shared__ __align__(1024) uint8_t smb_sw[];  // swizzled operands: 1 KB aligned
    uint8_t* const smb = smb_sw;
    uint8_t* sX = smb;  // A: [K; Q] 128 x 128 (swizzled, by tensor copies), then K^T | V^T (128 x 64 each)
    float* sAf = reinterpret_cast<float*>(sX + 65536);          // A (fp32, 64 x kLdT)
    float* sTf = sAf + kC * kLdT;                               // T (fp32, 64 x kLdT)
    uint8_t* sB2 = reinterpret_cast<uint8_t*>(sAf);             // B: T diag(beta Gam) 64 x 64, over A
    uint8_t* sB3 = reinterpret_cast<uint8_t*>(sTf);             // B: T diag(beta)     64 x 64, over T
    float* sg = sTf + kC * kLdT;                                // gam
    float* sGb = sg + kC;                                       // beta Gam
    float* sb = sGb + kC;                                       // beta
    uint64_t* bar = reinterpret_cast<uint64_t*>(sb + kC);
    uint64_t* bar_ld = bar + 1;  // the tensor copies of K^ and Q^
    uint64_t* bar_v = bar + 2;   // the tensor copy of V
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 3);
    // one CTA per (chunk, value head), the heads of a chunk adjacent in launch order (they copy the
    // same K^ and Q^ rows)
    const int h = (int)(blockIdx.x % (unsigned)p.HV), c = (int)(blockIdx.x / (unsigned)p.HV);
    int n, t0, len;
    if (!chunk_of(p, c, n, t0, len)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q = warp & 3, cg = warp >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int hk = h / p.G;
    const size_t ci = ch_index(p, c, h);
    if (smem_u32(smb) & 1023u) {  // the swizzled atoms need 1 KB alignment (the same for every CTA)
        if (tid == 0) atomicOr(p.err, GDN_DEVERR_SMEM_ALIGN);
        return;
    }
    // K^ (rows 0..63) and Q^ (rows 64..127) by tensor copies, four swizzled boxes of 32 values each,
    // in flight while warp 0 takes the cumsum
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_ld, 1);
        mbar_init(bar_v, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(bar_ld, 65536u);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            tma_load_2d(sX + 16384 * a, &tm_k, bar_ld, hk * kD + 32 * a, t0);
            tma_load_2d(sX + 16384 * a + 8192, &tm_q, bar_ld, hk * kD + 32 * a, t0);
        }
    }
    if (warp == 0) tmem_alloc(slot, 256);
    if (warp == 0) {
        // inclusive cumsum of g over the chunk, fixed order (lane-serial blocks of 2)
        float g0 = 0.f, g1 = 0.f;
        const int r0 = 2 * lane, r1 = r0 + 1;
        if (r0 < len) g0 = p.g[(size_t)(t0 + r0) * p.HV + h];
        if (r1 < len) g1 = p.g[(size_t)(t0 + r1) * p.HV + h];
        float s = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(kFull, s, off);
            if (lane >= off) s += y;
        }
        const float excl = s - (g0 + g1);
        const float c0 = excl + g0, c1 = c0 + g1;
        sg[r0] = c0;
        sg[r1] = c1;
        const float b0 = r0 < len ? p.beta[(size_t)(t0 + r0) * p.HV + h] : 0.f;
        const float b1 = r1 < len ? p.beta[(size_t)(t0 + r1) * p.HV + h] : 0.f;
        sb[r0] = b0;
        sb[r1] = b1;
        sGb[r0] = b0 * __expf(c0);
        sGb[r1] = b1 * __expf(c1);
        if (r0 < len) p.gam[(size_t)(t0 + r0) * p.HV + h] = c0;
        if (r1 < len) p.gam[(size_t)(t0 + r1) * p.HV + h] = c1;
    }
    __syncthreads();  // the barriers' initialisation is visible
    bool ok = __syncthreads_and(mbar_wait_bounded(bar_ld, 0));
    if (ok) {
        // TF32 rounding of the copy, and zero rows past the chunk (the copy fills them from the next
        // sequence): rows len..63 of K^ and of Q^, 128 bytes in each atom column
#pragma unroll
        for (int it = 0; it < 65536 / 16 / kNTtc; ++it) {
            float4* v = reinterpret_cast<float4*>(sX) + tid + it * kNTtc;
            *v = tf32_round4(*v);
        }
        if (len < kC) {
            __syncthreads();
            for (int e = tid; e < 2 * (kC - len) * 32; e += kNTtc) {
                const int u = e & 7, a = (e >> 3) & 3, rr = len + (e >> 5) % (kC - len), half = (e >> 5) / (kC - len);
                *reinterpret_cast<float4*>(sX + 16384 * a + 128 * (rr + kC * half) + 16 * u) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    } else if (tid == 0) {
        mbar_wait_bounded(bar_ld, 0);  // copies still in flight land before the CTA leaves
    }
    tc_sync();
    const uint32_t tmem = *slot;
    uint32_t phase = 0;
    bool v_pending = false;  // the copy of V is issued and not yet seen complete
    do {
        if (!ok) break;
        if (tid == 0) {
            const UmmaOp x = op_sw(smem_u32(sX), kD);
            umma_tf32_op(tmem, x, x, umma_idesc_tf32(kD, kC), kD, false);
            umma_commit(bar);
        }
        if (!(ok = tc_wait(bar, phase))) break;
        {
            // rows m < 64: A[r][s] = beta_r E[r][s] (K K^T)[r][s] for s < r;  rows m >= 64: Q K^T and P
            float x[16];
            tmem_ld<2>(tmem + lane_base + cg * 16, x);
            const int m = q * 32 + lane, r = m & (kC - 1);
            // gam of this thread's 16 columns and of its row, and beta_r, read before any store
            float gs[16];
#pragma unroll
            for (int t = 0; t < 16; t += 4) {
                const float4 g4 = *reinterpret_cast<const float4*>(sg + cg * 16 + t);
                gs[t] = g4.x, gs[t + 1] = g4.y, gs[t + 2] = g4.z, gs[t + 3] = g4.w;
            }
            const float gr = sg[r], br = sb[r];
            if (m < kC) {
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int s = cg * 16 + t;
                    sAf[r * kLdT + s] = s < r ? br * __expf(gr - gs[t]) * x[t] : 0.f;
                }
            } else {
                // QK^T and P rows staged where Q^ was (the first product has read it), and written
                // out coalesced once the CTA has staged them all
#pragma unroll
                for (int t = 0; t < 16; t += 4) {
                    uint8_t* qk = qkp_stage(sX, r, (cg * 16 + t) >> 2);
                    *reinterpret_cast<float4*>(qk) = make_float4(x[t], x[t + 1], x[t + 2], x[t + 3]);
                    float e[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int s = cg * 16 + t + u;
                        e[u] = (s <= r && r < len) ? x[t + u] * __expf(gr - gs[t + u]) : 0.f;
                    }
                    // P only ever enters the tensor cores (the backward state pass): stored as TF32
                    *reinterpret_cast<float4*>(qk + 32768) = tf32_round4(make_float4(e[0], e[1], e[2], e[3]));
                }
            }
        }
        tc_fence_before();
        __syncthreads();  // A complete; the first product has read sX
        {   // QK^T, then P: row-major 64 x 64 blocks of the (chunk, head), a warp writing two rows
            constexpr int kIt = 2 * kC * kC / 4 / kNTtc;
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, pc = e & 15, r = (e >> 4) & (kC - 1), isP = e >> 10;
                const float4 v = *reinterpret_cast<const float4*>(qkp_stage(sX, r, pc) + 32768 * isP);
                *reinterpret_cast<float4*>((isP ? p.Pb : p.QKb) + (ci * kC + r) * kC + 4 * pc) = v;
            }
        }
        {
            // K^T for after the solve: column j of four consecutive rows s .. s + 3 per item from the
            // copy in sX, consecutive threads on consecutive j, written into sX as K^T (j, s) in one
            // 16-byte store.  V comes by tensor copy during the solve and goes the same way (below).
            constexpr int kIt = kD * kC / 4 / kNTtc;
            float4 kr[kIt];
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, n = e % kD, s = (e / kD) * 4;
                float kv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) kv[u] = *reinterpret_cast<const float*>(sX + sw128_off(s + u, n, kD));
                kr[it] = make_float4(kv[0], kv[1], kv[2], kv[3]);
            }
            // T = (I + A)^-1 by 16 x 16 blocks (A is strictly lower).  The diagonal blocks
            // T_II = (I + A_II)^-1 by forward substitution: each half warp takes two columns of one
            // block, lane r of the half keeps the partial sums sigma_r = sum_{s < r} A[r][s] t[s] of
            // block row r, and at step s the owner of row s turns its final sigma_s into
            // t[s] = (s == j) - sigma_s, broadcasts it, and every lane adds A[r][s] t[s] (rows r <= s
            // add 0); at the end T[r][j] = (r == j) - sigma_r.  The blocks below follow from them.
            {
                const int w = tid >> 5, hf = lane >> 4, rr = lane & 15;
                const int I = w >> 2, ca = 4 * (w & 3) + 2 * hf;  // columns ca, ca + 1 of diagonal block I
                const int row = 16 * I + rr;
                float pa = 0.f, pb = 0.f;
#pragma unroll
                for (int sl = 0; sl < 16; ++sl) {
                    const float av = sAf[row * kLdT + 16 * I + sl];
                    const float ta = __shfl_sync(kFull, (sl == ca ? 1.f : 0.f) - pa, sl + 16 * hf);
                    const float tb = __shfl_sync(kFull, (sl == ca + 1 ? 1.f : 0.f) - pb, sl + 16 * hf);
                    pa = fmaf(av, ta, pa);
                    pb = fmaf(av, tb, pb);
                }
                sTf[row * kLdT + 16 * I + ca] = (rr == ca ? 1.f : 0.f) - pa;
                sTf[row * kLdT + 16 * I + ca + 1] = (rr == ca + 1 ? 1.f : 0.f) - pb;
                for (int e = tid; e < kC * kC; e += kNTtc) {  // the blocks above the diagonal are zero
                    const int r = e >> 6, c2 = e & 63;
                    if ((c2 >> 4) > (r >> 4)) sTf[r * kLdT + c2] = 0.f;
                }
            }
            __syncthreads();
            // V (bf16, two boxes of 64 values x 64 rows) by tensor copy into the halves of the first
            // two atom columns that held Q^ (free since QK^T and P went out), during the rest of the
            // solve
            if (tid == 0) {
                fence_async_smem();
                mbar_arrive_expect_tx(bar_v, 16384u);
                tma_load_2d(sX + 8192, &tm_v, bar_v, h * kD, t0);
                tma_load_2d(sX + 24576, &tm_v, bar_v, h * kD + 64, t0);
            }
            v_pending = true;
            {
                // M_IK = T_II A_IK for every K < I (six blocks, independent of each other), then block
                // rows I = 1, 2, 3: T_IJ = -sum_{K = J}^{I - 1} M_IK T_KJ.  Two accumulators per sum.
                float* M = reinterpret_cast<float*>(sX);  // scratch in the copy of K^ and Q^ (read into kr
                                                          // above): block (I, K) at 256 (I (I - 1) / 2 + K)
                for (int e = tid; e < 6 * 256; e += kNTtc) {
                    const int pb = e >> 8, r = (e >> 4) & 15, c2 = e & 15;
                    const int I = pb < 1 ? 1 : (pb < 3 ? 2 : 3), K = pb - I * (I - 1) / 2;
                    const float* tr = sTf + (16 * I + r) * kLdT + 16 * I;
                    const float* ac = sAf + 16 * I * kLdT + 16 * K + c2;
                    float x0 = 0.f, x1 = 0.f;
#pragma unroll
                    for (int k = 0; k < 16; k += 2) {
                        x0 = fmaf(tr[k], ac[k * kLdT], x0);
                        x1 = fmaf(tr[k + 1], ac[(k + 1) * kLdT], x1);
                    }
                    M[e] = x0 + x1;
                }
                __syncthreads();
#pragma unroll
                for (int I = 1; I < 4; ++I) {
                    for (int e = tid; e < I * 256; e += kNTtc) {
                        const int J = e >> 8, r = (e >> 4) & 15, c2 = e & 15;
                        float x0 = 0.f, x1 = 0.f;
                        for (int K = J; K < I; ++K) {
                            const float* mr = M + 256 * (I * (I - 1) / 2 + K) + 16 * r;
                            const float* tc = sTf + 16 * K * kLdT + 16 * J + c2;
#pragma unroll
                            for (int k = 0; k < 16; k += 2) {
                                x0 = fmaf(mr[k], tc[k * kLdT], x0);
                                x1 = fmaf(mr[k + 1], tc[(k + 1) * kLdT], x1);
                            }
                        }
                        sTf[(16 * I + r) * kLdT + 16 * J + c2] = -(x0 + x1);
                    }
                    __syncthreads();
                }
            }
            if (!(ok = __syncthreads_and(mbar_wait_bounded(bar_v, 0)))) break;
            v_pending = false;
            // V's column i = n of rows s .. s + 3 per item (the K^T mapping) from its copy: 128-byte
            // rows, 16-byte pieces swizzled; s >= len zero (the copy reads on into the next sequence)
            float4 vr[kIt];
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, n = e % kD, s = (e / kD) * 4;
                const uint8_t* box = sX + 8192 + 16384 * (n >> 6);
                float v4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int r = s + u;
                    const unsigned short b = *reinterpret_cast<const unsigned short*>(
                        box + 128 * r + ((((n & 63) >> 3) ^ (r & 7)) << 4) + (n & 7) * 2);
                    v4[u] = r < len ? __uint_as_float((uint32_t)b << 16) : 0.f;
                }
                vr[it] = make_float4(v4[0], v4[1], v4[2], v4[3]);
            }
            __syncthreads();  // every read of the copies of K^ and V is done
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, n = e % kD, s = (e / kD) * 4;
                *reinterpret_cast<float4*>(sX + umma_koff(n, s, kSboC)) = tf32_round4(kr[it]);
                *reinterpret_cast<float4*>(sX + 32768 + umma_koff(n, s, kSboC)) = tf32_round4(vr[it]);
            }
        }
        __syncthreads();
        {
            // T out, sixteen threads on a row (coalesced); B operands T diag(beta Gam) (over A, unused
            // since the blocks M were formed) and T diag(beta) (over T itself, once every thread holds
            // its values of T), rows r, k = s, consecutive threads on consecutive rows (the 16-byte
            // stores of a core matrix's eight rows then fill all banks)
            constexpr int kIt = kC * kC / 4 / kNTtc;
            float* Tg = p.Tb + ci * kC * kC;
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, r = e / (kC / 4), s = (e % (kC / 4)) * 4;
                const float* tr = sTf + r * kLdT + s;
                *reinterpret_cast<float4*>(Tg + r * kC + s) = make_float4(tr[0], tr[1], tr[2], tr[3]);
            }
            float4 tv[kIt];
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, r = e % kC, s = (e / kC) * 4;
                const float* tr = sTf + r * kLdT + s;
                tv[it] = make_float4(tr[0], tr[1], tr[2], tr[3]);
                *reinterpret_cast<float4*>(sB2 + umma_koff(r, s, kSboC)) = tf32_round4(make_float4(
                    tv[it].x * sGb[s], tv[it].y * sGb[s + 1], tv[it].z * sGb[s + 2], tv[it].w * sGb[s + 3]));
            }
            __syncthreads();  // T is read in full before T diag(beta) overwrites it
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, r = e % kC, s = (e / kC) * 4;
                *reinterpret_cast<float4*>(sB3 + umma_koff(r, s, kSboC)) = tf32_round4(
                    make_float4(tv[it].x * sb[s], tv[it].y * sb[s + 1], tv[it].z * sb[s + 2], tv[it].w * sb[s + 3]));
            }
        }
        tc_sync();
        if (tid == 0) {
            const uint32_t id = umma_idesc_tf32(kD, kC);
            umma_tf32_k(tmem + 64, smem_u32(sX), kSboC, smem_u32(sB2), kSboC, id, kC, false);
            umma_tf32_k(tmem + 128, smem_u32(sX) + 32768, kSboC, smem_u32(sB3), kSboC, id, kC, false);
            umma_commit(bar);
        }
        if (!(ok = tc_wait(bar, phase))) break;
        {
            // W[r][j] = (W^T)[j][r] and U~[r][i] = (U~^T)[i][r] for r = 16 cg + t, row-major into sX
            // (free once the products have read K^T and V^T), then out by one 32 KB bulk copy each
            const int jj = q * 32 + lane;
            float w[16], u[16];
            tmem_ld_pair(tmem + lane_base + 64 + cg * 16, w, tmem + lane_base + 128 + cg * 16, u);
            float* sWr = reinterpret_cast<float*>(sX);
            float* sUr = sWr + kC * kD;
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                sWr[(cg * 16 + t) * kD + jj] = tf32_round(w[t]);  // W only ever enters the tensor cores
                sUr[(cg * 16 + t) * kD + jj] = u[t];
            }
            __syncthreads();
            if (tid == 0) {
                fence_async_smem();
                bulk_store(p.Wb + ci * kC * kD, sWr, kC * kD * 4);
                bulk_store(p.Utb + ci * kC * kD, sUr, kC * kD * 4);
                bulk_commit();
                bulk_wait_read();  // the CTA's shared memory stays until the copies have read it
            }
        }
    } while (false);
    if (!ok && tid == 0) {
        atomicOr(p.err, GDN_DEVERR_TIMEOUT);
        if (v_pending) mbar_wait_bounded(bar_v, 0);  // the copy of V lands before the CTA leaves
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// per (chunk, head): the C x C part.
__global__ void __launch_bounds__(kNT) bwd_intra_c_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int c = blockIdx.x, h = blockIdx.y;
    int n, t0, len;
    if (!chunk_of(p, c, n, t0, len)) return;
    const int hk = h / p.G, dk = p.dk, dv = p.dv;
    float* sK = sm;                    // C x kLdD
    float* sA = sK + kC * kLdD;        // dO -> dW
    float* sB = sA + kC * kLdD;        // U -> V
    float* sCb = sB + kC * kLdD;       // Q -> dU
    float* s1 = sCb + kC * kLdD;       // QK -> F1 -> dT -> dA -> dKK
    float* s2 = s1 + kC * kLdC;        // dQK -> F2 -> Z -> KK -> dKK + dKK^T
    float* sT = s2 + kC * kLdC;        // T
    float* sE = sT + kC * kLdC;        // dE accumulator
    float* sg = sE + kC * kLdC;        // gam
    float* sbe = sg + kC;              // beta
    float* sdg = sbe + kC;             // dgam
    float* sdb = sdg + kC;             // dbeta
    const size_t ci = ch_index(p, c, h);
    load_rows_f32(sK, kLdD, p.kn + ((size_t)t0 * p.HK + hk) * dk, (size_t)p.HK * dk, kC, len, dk);
    load_rows_any(sA, kLdD, p.dout, ((size_t)t0 * p.HV + h) * dv, (size_t)p.HV * dv, kC, len, dv, p.dtype);
    load_rows_f32(sB, kLdD, p.Ub + ci * kC * dv, dv, kC, kC, dv);
    load_rows_f32(sCb, kLdD, p.qn + ((size_t)t0 * p.HK + hk) * dk, (size_t)p.HK * dk, kC, len, dk);
    load_rows_f32(s1, kLdC, p.QKb + ci * kC * kC, kC, kC, kC, kC);
    load_rows_f32(sT, kLdC, p.Tb + ci * kC * kC, kC, kC, kC, kC);
    const float* dga = p.dgamA + ci * kC;
    for (int i = threadIdx.x; i < kC; i += blockDim.x) {
        // past the chunk's end gam stays at its last value (as the cumsum in bwd_wy_tc_kernel leaves it),
        // so gam is non-increasing over all 64 rows and exp(gam_r - gam_s), s <= r, never exceeds 1
        sg[i] = p.gam[(size_t)(t0 + min(i, len - 1)) * p.HV + h];
        sbe[i] = i < len ? p.beta[(size_t)(t0 + i) * p.HV + h] : 0.f;
        sdg[i] = dga[i];
        sdb[i] = 0.f;
    }
    for (int i = threadIdx.x; i < kC * kLdC; i += blockDim.x) sE[i] = 0.f;
    __syncthreads();
    // c1: dP = dO U^T -> dQK = lower(dP) * E, dE = lower(dP) * QK
    bgemm(kC, kC, dv, sA, kLdD, 1, sB, 1, kLdD, [&](int r, int s, float x) {
        const bool in = (s <= r) && (r < len);
        const float e = in ? __expf(sg[r] - sg[s]) : 0.f;
        s2[r * kLdC + s] = in ? x * e : 0.f;
        sE[r * kLdC + s] = in ? x * s1[r * kLdC + s] : 0.f;
    });
    __syncthreads();
    float* dq = p.dqh;
    float* dkk = p.dkh;
    // The updates of dq and dk below are read-modify-writes of global memory: each output
    // element's old value comes in through the prior functor, all of a tile's at once.
    auto at = [&](int r, int j) { return ((size_t)(t0 + r) * p.HV + h) * dk + j; };
    auto dq_old = [&](int r, int j) { return r < len ? dq[at(r, j)] : 0.f; };
    auto dk_old = [&](int r, int j) { return r < len ? dkk[at(r, j)] : 0.f; };
    bgemm_rmw(kC, dk, kC, s2, kLdC, 1, sK, kLdD, 1, dq_old, [&](int r, int j, float x, float o) {
        if (r < len) dq[at(r, j)] = o + x;
    });
    __syncthreads();
    bgemm_rmw(kC, dk, kC, s2, 1, kLdC, sCb, kLdD, 1, dk_old, [&](int s, int j, float x, float o) {
        if (s < len) dkk[at(s, j)] = o + x;
    });
    __syncthreads();
    // c2: dW -> sA, V -> sB, dU -> sCb
    load_rows_f32(sA, kLdD, p.Wb + ci * kC * dk, dk, kC, kC, dk);
    load_rows_any(sB, kLdD, p.v, ((size_t)t0 * p.HV + h) * dv, (size_t)p.HV * dv, kC, len, dv, p.dtype);
    load_rows_f32(sCb, kLdD, p.dUb + ci * kC * dv, dv, kC, kC, dv);
    __syncthreads();
    // F1 = dW K^T, F2 = dU V^T
    bgemm(kC, kC, dk, sA, kLdD, 1, sK, 1, kLdD, [&](int s, int r, float x) { s1[s * kLdC + r] = x; });
    bgemm(kC, kC, dv, sCb, kLdD, 1, sB, 1, kLdD, [&](int s, int r, float x) { s2[s * kLdC + r] = x; });
    __syncthreads();
    // column dots with T: dbeta_r, dgam_r; then dT(s,r) = beta_r (Gam_r F1 + F2)
    for (int r = threadIdx.x >> 4; r < kC; r += blockDim.x >> 4) {
        const int l = threadIdx.x & 15;
        float a1 = 0.f, a2 = 0.f;
        for (int s = l; s < kC; s += 16) {
            a1 = fmaf(sT[s * kLdC + r], s1[s * kLdC + r], a1);
            a2 = fmaf(sT[s * kLdC + r], s2[s * kLdC + r], a2);
        }
        a1 = half_sum(a1);
        a2 = half_sum(a2);
        if (l == 0) {
            const float Gr = __expf(sg[r]);
            sdb[r] += Gr * a1 + a2;
            sdg[r] += Gr * sbe[r] * a1;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kC * kC; i += blockDim.x) {
        const int s = i / kC, r = i - s * kC;
        s1[s * kLdC + r] = sbe[r] * fmaf(__expf(sg[r]), s1[s * kLdC + r], s2[s * kLdC + r]);
    }
    __syncthreads();
    // dK += diag(beta Gam) T^T dW;  dV = diag(beta) T^T dU
    bgemm_rmw(kC, dk, kC, sT, 1, kLdC, sA, kLdD, 1, dk_old, [&](int r, int j, float x, float o) {
        if (r < len) dkk[at(r, j)] = o + sbe[r] * __expf(sg[r]) * x;
    });
    bgemm(kC, dv, kC, sT, 1, kLdC, sCb, kLdD, 1, [&](int r, int j, float x) {
        if (r < len) st_any(p.dv_out, ((size_t)(t0 + r) * p.HV + h) * dv + j, p.dtype, sbe[r] * x);
    });
    // c4: Z = dT T^T -> s2;  dA = -T^T Z (strictly lower) -> s1
    bgemm(kC, kC, kC, s1, kLdC, 1, sT, 1, kLdC, [&](int a, int b, float x) { s2[a * kLdC + b] = x; });
    __syncthreads();
    bgemm(kC, kC, kC, sT, 1, kLdC, s2, kLdC, 1,
             [&](int r, int s, float x) { s1[r * kLdC + s] = (s < r) ? -x : 0.f; });
    __syncthreads();
    // c5: KK = K K^T -> s2; dbeta_r += sum_s dA E KK; dKK = dA beta_r E -> s1; dE += dA beta_r KK
    bgemm(kC, kC, dk, sK, kLdD, 1, sK, 1, kLdD, [&](int r, int s, float x) { s2[r * kLdC + s] = x; });
    __syncthreads();
    for (int r = threadIdx.x >> 4; r < kC; r += blockDim.x >> 4) {
        const int l = threadIdx.x & 15;
        float acc = 0.f;
        for (int s = l; s < r; s += 16) {
            const float a = s1[r * kLdC + s], e = __expf(sg[r] - sg[s]), kk = s2[r * kLdC + s];
            acc = fmaf(a * e, kk, acc);
            s1[r * kLdC + s] = a * sbe[r] * e;
            sE[r * kLdC + s] = fmaf(a * sbe[r], kk, sE[r * kLdC + s]);
        }
        acc = half_sum(acc);
        if (l == 0) sdb[r] += acc;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kC * kC; i += blockDim.x) {
        const int r = i / kC, s = i - r * kC;
        s2[r * kLdC + s] = s1[r * kLdC + s] + s1[s * kLdC + r];
    }
    __syncthreads();
    bgemm_rmw(kC, dk, kC, s2, kLdC, 1, sK, kLdD, 1, dk_old, [&](int r, int j, float x, float o) {
        if (r < len) dkk[at(r, j)] = o + x;
    });
    // c6: dgam from E (row sums minus column sums of dE * E), then dg = reverse cumsum
    for (int r = threadIdx.x >> 4; r < kC; r += blockDim.x >> 4) {
        const int l = threadIdx.x & 15;
        float rs = 0.f, cs = 0.f;
        for (int s = l; s < kC; s += 16) {  // dE is lower triangular: exp only on its support
            rs = fmaf(sE[r * kLdC + s], s <= r ? __expf(sg[r] - sg[s]) : 0.f, rs);
            cs = fmaf(sE[s * kLdC + r], s >= r ? __expf(sg[s] - sg[r]) : 0.f, cs);
        }
        rs = half_sum(rs);
        cs = half_sum(cs);
        if (l == 0) sdg[r] += rs - cs;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float acc = 0.f;
        for (int r = len - 1; r >= 0; --r) {
            acc += sdg[r];
            p.dg[(size_t)(t0 + r) * p.HV + h] = acc;
            p.dbeta[(size_t)(t0 + r) * p.HV + h] = sdb[r];
        }
    }
}

// dst(n, k) = get(k, n) for n < NN, k < KK (a transpose), rounded to TF32; consecutive threads
// take consecutive n.
template <int NN, int KK, typename G>
__device__ __forceinline__ void stage_cols_fn(uint8_t* dst, G get) {
    constexpr int kItems = NN * KK / 4 / kNTtc;
    float4 v[kItems];
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const int e = threadIdx.x + it * kNTtc, n = e % NN, k = (e / NN) * 4;
        v[it] = make_float4(get(k, n), get(k + 1, n), get(k + 2, n), get(k + 3, n));
    }
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
        const int e = threadIdx.x + it * kNTtc, n = e % NN, k = (e / NN) * 4;
        *reinterpret_cast<float4*>(dst + umma_koff(n, k, KK * 32)) = tf32_round4(v[it]);
    }
}

// One warp per (token, k-head) w[u], NT of them at once: sum the G value heads' dq^ and dk^ rows in
// increasing head order, then the L2-norm backward, into dq and dk.  Tokens with on[u] false are
// skipped.  Every load of a head step (dq and dk of all NT tokens together) is issued before any
// is used, and the inverse norms with the first ones, so the NT tokens share their round trips;
// each element still sums the heads in increasing order.  The partial rows are read at L2
// (__ldcg): in bwd_intra_tc_kernel they were written by other CTAs of the same launch.
template <int NT>
__device__ __forceinline__ void fold_tokens(const BwdParams& p, const long long (&w)[NT], const bool (&on)[NT],
                                            int lane) {
    float dsum[NT][2][4], x[NT][2][4], inv[NT][2];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = lane + 32 * i;
            const bool in = on[u] && j < p.dk;
            x[u][0][i] = in ? p.qn[(size_t)w[u] * p.dk + j] : 0.f;
            x[u][1][i] = in ? p.kn[(size_t)w[u] * p.dk + j] : 0.f;
            dsum[u][0][i] = dsum[u][1][i] = 0.f;
        }
        inv[u][0] = on[u] ? p.qinv[w[u]] : 0.f;
        inv[u][1] = on[u] ? p.kinv[w[u]] : 0.f;
    }
    for (int g = 0; g < p.G; ++g) {
        float a[NT][4], b[NT][4];
#pragma unroll
        for (int u = 0; u < NT; ++u) {
            const int t = (int)(w[u] / p.HK), hk = (int)(w[u] - (long long)t * p.HK);
            const size_t base = ((size_t)t * p.HV + hk * p.G + g) * p.dk;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = lane + 32 * i;
                const bool in = on[u] && j < p.dk;
                a[u][i] = in ? __ldcg(p.dqh + base + j) : 0.f;
                b[u][i] = in ? __ldcg(p.dkh + base + j) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dsum[u][0][i] += a[u][i];
                dsum[u][1][i] += b[u][i];
            }
    }
#pragma unroll
    for (int u = 0; u < NT; ++u) {
        if (!on[u]) continue;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) dot = fmaf(x[u][which][i], dsum[u][which][i], dot);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(kFull, dot, off);
            void* dst = which ? p.dk_out : p.dq_out;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = lane + 32 * i;
                if (j < p.dk) {
                    const float gval = p.use_norm ? (dsum[u][which][i] - x[u][which][i] * dot) * inv[u][which]
                                                  : dsum[u][which][i];
                    st_any(dst, (size_t)w[u] * p.dk + j, p.dtype, gval);
                }
            }
        }
    }
}

// Eight fp16 values (one 16-byte piece of a stored state) times the factor of their tile, in fp32.
__device__ __forceinline__ void unpack_h8(const uint4& v, float fac, float (&x)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[u]));
        x[2 * u] = f.x * fac;
        x[2 * u + 1] = f.y * fac;
    }
}
// Values i = 8 pc .. 8 pc + 7 of row j of a K-half (128 rows x 64 fp32) in the 128-byte-swizzled
// K-major layout: atom column pc / 4 (32 values, 16 KB), 16-byte pieces 2 (pc % 4) and the next.
// The second atom column stores its two pieces in the other order, so that the eight threads of a
// row (pc = 0 .. 7) fill eight different bank groups with each store.
__device__ __forceinline__ void put_piece_sw128(uint8_t* half_base, int j, int pc, const float (&x)[8]) {
    uint8_t* row = half_base + 16384 * (pc >> 2) + 128 * j;
    const float4 lo = make_float4(x[0], x[1], x[2], x[3]), hi = make_float4(x[4], x[5], x[6], x[7]);
    const int sw = pc >> 2;
    *reinterpret_cast<float4*>(row + (((2 * (pc & 3) + sw) ^ (j & 7)) << 4)) = sw ? hi : lo;
    *reinterpret_cast<float4*>(row + (((2 * (pc & 3) + (sw ^ 1)) ^ (j & 7)) << 4)) = sw ? lo : hi;
}

// per (chunk, head), dk = dv = 128, bf16 inputs: bwd_intra_s_kernel and bwd_intra_c_kernel in one
// kernel on tcgen05.  The products with the chunk states come first, in transposed form (rows = the
// dk index j):
//   X_q = S0^T dO^T:  dQ_S[r][j] = Gam_r X_q[j][r]      X_w = S0^T dU^T:  dW[s][j] = -X_w[j][s]
//   Y = D^T U^T:      (diag(b) U D)[r][j] = b_r Y[j][r]  and dW = -(dU S0) once more with M = 64
// and dgam_r = q^_r . dQ_S,r - b_r k^_r . Y_r (+ sum_r b_r k^_r . Y_r + Gam_last <D, S0> on the last
// row).  Gam_r X_q and b_r Y go back into TMEM (tcgen05.st) as the first terms of the dq^T and
// dk^T accumulators; dW stays on chip, as F1's operand and, from X_w, as the transposed one.
// The C x C products (dP = dO U^T, K K^T, F1 = dW K^T, F2 = dU V^T, Z = dT T^T, T^T Z) use M = 64:
// row m of the result sits in TMEM lane 32 (m / 16) + m % 16, so lanes 0..15 of each warp quarter
// hold 16 rows, which the 16x256b loads (tmem_ld16) spread over all 32 threads of the warp.  The
// products that update dq, dk, dv are taken transposed with the dk / dv index as their 128 rows;
// dq's two and dk's five terms (dKK and dKK^T separately) accumulate in TMEM and meet global memory
// once.
//   TMEM columns: 0 dP, then Z | 64 K K^T | 128 X_q, then dq^T | 192 Y, then dk^T | 256 X_w, then
//   dv^T | 320 dU S0 (128 wide), then F1 | 384 F2 | 448 T^T Z
//   shared memory: five 32 KB operand buffers R1..R5 and two 16 KB ones C1, C2 (together one
//   32 KB buffer at first), reused by phase; S0^T and D^T enter in two K-halves of 32 KB.
// K^, U and dU arrive by tensor copies (one thread, one mbarrier) in the 128-byte-swizzled K-major
// layout (boxes of 32 values x rows, four atom columns per 128 values).  S0^T arrives the same way
// as stored (fp16, boxes of 64 values) and threads write it, times its tile factors, into that
// layout; D^T (fp16, through registers) takes the same layout.  Every other operand uses the layout
// of umma_koff.
// dE's row pitch in bwd_intra_tc_kernel: a warp's float2 accesses (rows lane / 4 and 8 on, column
// pairs 2 (lane % 4)) take two wavefronts, the least for 256 bytes
constexpr int kLdE = kC + 8;
constexpr size_t kIntraCTcSmem = (size_t)5 * 32768 + 2 * 16384 + 4 * kC * kLdE + 4 * (6 * kC + 3 * 4 * kC) + 32;
static_assert(kIntraCTcSmem <= 227 * 1024, "bwd_intra_tc_kernel's shared memory");

__global__ void __launch_bounds__(kNTtc, 1)
    bwd_intra_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_u,
                        const __grid_constant__ CUtensorMap tm_du, const __grid_constant__ CUtensorMap tm_s,
                        const __grid_constant__ CUtensorMap tm_qk, const __grid_constant__ CUtensorMap tm_t,
                        const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_do, BwdParams p) {
    constexpr int kD = 128;
    constexpr uint32_t kSboD = kD * 32;  // 128 values per row
    extern __shared__ __align__(1024) uint8_t smb_sw[];  // swizzled operands: 1 KB aligned
    uint8_t* const smb = smb_sw;
    uint8_t* R1 = smb;
    uint8_t* R2 = R1 + 32768;
    uint8_t* R3 = R2 + 32768;
    uint8_t* R4 = R3 + 32768;
    uint8_t* R5 = R4 + 32768;
    uint8_t* C1 = R5 + 32768;
    uint8_t* C2 = C1 + 16384;
    float* sE = reinterpret_cast<float*>(C2 + 16384);  // dE accumulator, 64 x kLdE
    float* sg = sE + kC * kLdE;                         // gam
    float* sbe = sg + kC;                               // beta
    float* sdg = sbe + kC;                              // dgam
    float* sdb = sdg + kC;                              // dbeta
    float* part1 = sdb + kC;                            // [4][64] partials: F1 column dots, then dE * E row sums
    float* part2 = part1 + 4 * kC;                      // [4][64] partials: F2 column dots, then dE * E column sums
    float* rowp = part2 + 4 * kC;                       // [4][64] row-loop partials
    float* sgE = rowp + 4 * kC;                         // exp(gam_r)
    float* sgL = sgE + kC;                              // exp(gam_last - gam_r)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sgL + kC);
    uint64_t* bar_ld = bar + 1;  // the tensor copies of phase A
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 2);
    uint32_t* s_last = slot + 1;  // this CTA folds the chunk's dq^, dk^ rows of its k-head
    // one CTA per (chunk, value head), the heads of a chunk adjacent in launch order
    const int h = (int)(blockIdx.x % (unsigned)p.HV), c = (int)(blockIdx.x / (unsigned)p.HV);
    int n, t0, len;
    if (!chunk_of(p, c, n, t0, len)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q = warp & 3, cg = warp >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int hk = h / p.G;
    const size_t ci = ch_index(p, c, h);
    // an M = 64 result comes in by 16x256b loads (tmem_ld16): this thread's rows ra and ra + 8, and
    // in each block of 8 columns the pair from cp on
    const int ra = 16 * q + (lane >> 2), cp = 2 * (lane & 3);
    const int jj = 32 * q + lane;          // the dk / dv index of an M = 128 result
    const size_t sk = (size_t)p.HK * kD;
    const float* kb = p.kn + ((size_t)t0 * p.HK + hk) * kD;  // K^ row s at kb + s * sk
    const float* qb = p.qn + ((size_t)t0 * p.HK + hk) * kD;
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    // the swizzled atoms need 1 KB alignment of the dynamic shared memory (the same for every CTA)
    if (smem_u32(smb) & 1023u) {
        if (tid == 0) atomicOr(p.err, GDN_DEVERR_SMEM_ALIGN);
        return;
    }
    stagger_first_wave(p.stagger_intra, p.nsm);
    // phase A: K^ -> R1, U -> R3, dU -> R5 (rows = chunk positions) by tensor copies (four boxes of 32
    // values per operand); S0^T (fp16, two boxes of 64 values) -> R4 + 16 KB and C2, and dO (bf16, two
    // boxes of 64 values) -> R2 + 16 KB, converted once they land: S0^T in two K-halves into R4 and
    // C1|C2 (rows j, k = i), dO into R2
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_ld, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(bar_ld, 4u * 32768u + 16384u);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            tma_load_2d(R1 + 8192 * a, &tm_k, bar_ld, hk * kD + 32 * a, t0);
            tma_load_2d(R3 + 8192 * a, &tm_u, bar_ld, 32 * a, (int)(ci * kC));
            tma_load_2d(R5 + 8192 * a, &tm_du, bar_ld, 32 * a, (int)(ci * kC));
        }
        // S0^T as stored (fp16, two boxes of 64 values x 128 rows) into the second halves of its
        // targets, R4 and C1|C2
        tma_load_2d(R4 + 16384, &tm_s, bar_ld, 0, (int)(ci * kD));
        tma_load_2d(C1 + 16384, &tm_s, bar_ld, 64, (int)(ci * kD));
        tma_load_2d(R2 + 16384, &tm_do, bar_ld, h * kD, t0);
        tma_load_2d(R2 + 24576, &tm_do, bar_ld, h * kD + 64, t0);
    }
    if (warp == 0) tmem_alloc(slot, 512);
    // D^T (fp16, row j = dk index, dv index i contiguous) into registers in pieces of 8 values, the
    // pieces where this thread converts S0^T below: piece f = tid + 512 it is K-half hb = f / 1024, row
    // j = (f / 8) % 128, values i = 64 hb + 8 (f % 8) ..; with each piece the factors of its tile of D
    // and of S0.  <D, S0> takes both as stored, and D^T lands in S0^T's layout.
    const __half* Dt = p.Dh + ci * kD * kD;
    uint4 dh[4];
    float dfac[4], sfac[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int f = tid + it * kNTtc, hb = f >> 10, j = (f >> 3) & (kD - 1), pc = f & 7;
        dh[it] = *reinterpret_cast<const uint4*>(Dt + j * kD + 64 * hb + 8 * pc);
        const int tile = 4 * (j >> 5) + 2 * hb + (pc >> 2);
        dfac[it] = p.Dsc[ci * 16 + tile];
        sfac[it] = p.Ssc[ci * 16 + tile];
    }
    for (int i = tid; i < kC; i += kNTtc) {
        // past the chunk's end gam stays at its last value (as the cumsum in bwd_wy_tc_kernel leaves it),
        // so gam is non-increasing over all 64 rows and exp(gam_r - gam_s), s <= r, never exceeds 1
        const float gi = p.gam[(size_t)(t0 + min(i, len - 1)) * p.HV + h];
        sg[i] = gi;
        sgE[i] = __expf(gi);
        sgL[i] = __expf(p.gam[(size_t)(t0 + len - 1) * p.HV + h] - gi);
        sbe[i] = i < len ? p.beta[(size_t)(t0 + i) * p.HV + h] : 0.f;
        sdb[i] = 0.f;
    }
    __syncthreads();  // the barriers' initialisation is visible
    bool ok = __syncthreads_and(mbar_wait_bounded(bar_ld, 0));
    int ld_pending = ok ? -1 : 0;  // parity of tensor copies issued and not yet seen complete
    float dot = 0.f;  // this thread's share of <D, S0>, in fp32
    if (ok) {
        // dO: its bf16 copy in R2 + 16 KB (two swizzled boxes of 64 rows x 64) -> R2 in fp32, rows
        // >= len zero; every read before any write
        {
            using RO = RowsTc<kC, kD>;
            float4 ov[RO::kItems];
#pragma unroll
            for (int u = 0; u < RO::kItems; ++u) {
                const int r = RO::row(u), k = RO::col(u);
                const uint2 b = *reinterpret_cast<const uint2*>(
                    R2 + 16384 + (k >> 6) * 8192 + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
                ov[u] = r < len ? make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                                              __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u))
                                : z4;
            }
            uint4 sv[4];  // S0^T's pieces (see dh) from its copy: 128-byte rows, 16-byte pieces swizzled
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int f = tid + it * kNTtc, hb = f >> 10, j = (f >> 3) & (kD - 1), pc = f & 7;
                sv[it] = *reinterpret_cast<const uint4*>((hb ? C1 : R4) + 16384 + 128 * j + ((pc ^ (j & 7)) << 4));
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < RO::kItems; ++u)
                *reinterpret_cast<float4*>(R2 + umma_koff(RO::row(u), RO::col(u), kSboD)) = tf32_round4(ov[u]);
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int f = tid + it * kNTtc, hb = f >> 10, j = (f >> 3) & (kD - 1), pc = f & 7;
                float sx[8], dx[8];
                unpack_h8(sv[it], sfac[it], sx);
                unpack_h8(dh[it], dfac[it], dx);
#pragma unroll
                for (int u = 0; u < 8; ++u) dot = fmaf(dx[u], sx[u], dot);
                put_piece_sw128(hb ? C1 : R4, j, pc, sx);
            }
        }
        // TF32 rounding of the copied K^ (U and dU arrive rounded by the state passes, S0^T as TF32
        // values), and zero rows of K^ past the chunk (the copy fills them from the next sequence)
#pragma unroll
        for (int it = 0; it < 32768 / 16 / kNTtc; ++it) {
            float4* v = reinterpret_cast<float4*>(R1) + tid + it * kNTtc;
            *v = tf32_round4(*v);
        }
        if (len < kC)
            for (int e = tid; e < (kC - len) * (kD / 4); e += kNTtc) {  // whole 128-byte row pieces
                const int r = len + e / (kD / 4), a = (e >> 3) & 3, u = e & 7;
                *reinterpret_cast<float4*>(R1 + 8192 * a + 128 * r + 16 * u) = z4;
            }
    }
    tc_sync();
    const uint32_t tmem = *slot;
    const uint32_t id64 = umma_idesc_tf32(kC, kC), id128 = umma_idesc_tf32(kD, kC), id64w = umma_idesc_tf32(kC, kD);
    uint32_t phase = 0;
    do {
        if (!ok) break;
        if (tid == 0) {
            const UmmaOp sK = op_sw(smem_u32(R1), kC), sU = op_sw(smem_u32(R3), kC);
            const UmmaOp sdU0 = op_sw(smem_u32(R5), kC), sdU1 = op_sw(smem_u32(R5) + 16384, kC);  // K-halves
            const UmmaOp sS0 = op_sw(smem_u32(R4), kD), sS1 = op_sw(smem_u32(C1), kD);
            const UmmaOp dO = op_k(smem_u32(R2), kSboD), dO1 = op_k(smem_u32(R2) + 2048, kSboD);
            umma_tf32_op(tmem + 0, dO, sU, id64, kD, false);        // dP
            umma_tf32_op(tmem + 64, sK, sK, id64, kD, false);       // K K^T
            umma_tf32_op(tmem + 128, sS0, dO, id128, kC, false);    // X_q
            umma_tf32_op(tmem + 128, sS1, dO1, id128, kC, true);
            umma_tf32_op(tmem + 256, sS0, sdU0, id128, kC, false);  // X_w
            umma_tf32_op(tmem + 256, sS1, sdU1, id128, kC, true);
            umma_tf32_op(tmem + 320, sdU0, sS0, id64w, kC, false);  // dU S0
            umma_tf32_op(tmem + 320, sdU1, sS1, id64w, kC, true);
            umma_commit(bar);
        }
        float qv[16];  // q^[r][j] for the dQ_S epilogue, in flight during the products
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int r = cg * 16 + m;
            qv[m] = r < len ? qb[(size_t)r * sk + jj] : 0.f;
        }
        if (!(ok = tc_wait(bar, phase))) break;
        // phase A2: the products above have read dO and both halves of S0^T.  D^T -> R2 (first K-half)
        // and C1|C2 (second), in the layout of the S0^T halves
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int f = tid + it * kNTtc, hb = f >> 10, j = (f >> 3) & (kD - 1), pc = f & 7;
            float dx[8];
            unpack_h8(dh[it], dfac[it], dx);
            put_piece_sw128(hb ? C1 : R2, j, pc, dx);
        }
        float kv[16];  // k^[r][j] for the U D epilogue
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int r = cg * 16 + m;
            kv[m] = r < len ? kb[(size_t)r * sk + jj] : 0.f;
        }
        {  // dW = -(dU S0) -> R4 (rows s, k = j): F1's A operand
            float y[16];
            tmem_ld16<4>(tmem + lane_base + 320 + cg * 32, y);
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<float2*>(R4 + umma_koff(ra + 8 * hr, cg * 32 + 8 * n + cp, kSboD)) =
                        make_float2(tf32_round(-y[4 * n + 2 * hr]), tf32_round(-y[4 * n + 2 * hr + 1]));
        }
        tc_sync();
        if (tid == 0) {
            const uint32_t u3 = smem_u32(R3);
            umma_tf32_op(tmem + 192, op_sw(smem_u32(R2), kD), op_sw(u3, kC), id128, kC, false);  // Y
            umma_tf32_op(tmem + 192, op_sw(smem_u32(C1), kD), op_sw(u3 + 16384, kC), id128, kC, true);
            umma_tf32_op(tmem + 320, op_k(smem_u32(R4), kSboD), op_sw(smem_u32(R1), kC), id64, kD, false);  // F1
            umma_commit(bar);
        }
        const float gl = sg[len - 1];
        {  // Gam_r X_q back into TMEM as dq^T's first term; q^_r . dQ_S,r
            float x[16];
            tmem_ld<2>(tmem + lane_base + 128 + cg * 16, x);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int r = cg * 16 + m;
                const float d = r < len ? sgE[r] * x[m] : 0.f;
                x[m] = d;
                qv[m] *= d;
            }
            tmem_st<2>(tmem + lane_base + 128 + cg * 16, x);
            const float part = warp_transpose_sum<16>(qv);
            if (lane < 16) part1[q * kC + cg * 16 + lane] = part;
        }
        if (!(ok = tc_wait(bar, phase))) break;
        // Y and F1 have read D^T, U and dW: by tensor copies (swizzled) Q K^T -> R4 (the first 16 KB) and
        // T -> R4 + 16 KB (64 rows x 64 each), Q^ -> R3 (64 rows x 128), and V (bf16) -> R2 + 16 KB, for
        // phases B and C
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_ld, 81920u);
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                tma_load_2d(R4 + 8192 * a, &tm_qk, bar_ld, 32 * a, (int)(ci * kC));
                tma_load_2d(R4 + 16384 + 8192 * a, &tm_t, bar_ld, 32 * a, (int)(ci * kC));
                tma_load_2d(R2 + 16384 + 8192 * a, &tm_v, bar_ld, h * kD + 64 * a, t0);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) tma_load_2d(R3 + 8192 * a, &tm_q, bar_ld, hk * kD + 32 * a, t0);
        }
        ld_pending = 1;
        {  // b_r Y back into TMEM as dk^T's first term; k^_r . Y_r
            float x[16];
            tmem_ld<2>(tmem + lane_base + 192 + cg * 16, x);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int r = cg * 16 + m;
                kv[m] *= x[m];
                x[m] = r < len ? sgL[r] * x[m] : 0.f;
            }
            tmem_st<2>(tmem + lane_base + 192 + cg * 16, x);
            const float part = warp_transpose_sum<16>(kv);
            if (lane < 16) part2[q * kC + cg * 16 + lane] = part;
        }
        const float dS = cta_sum(dot, rowp + kC);  // its barriers also publish part1 / part2
        for (int r = tid; r < kC; r += kNTtc) {
            float dg = 0.f, bd = 0.f;
            if (r < len) {
                dg = ((part1[r] + part1[kC + r]) + part1[2 * kC + r]) + part1[3 * kC + r];
                bd = sgL[r] * (((part2[r] + part2[kC + r]) + part2[2 * kC + r]) + part2[3 * kC + r]);
            }
            sdg[r] = dg - bd;
            rowp[r] = bd;
        }
        __syncthreads();
        if (tid == 0) {
            float tot = 0.f;
            for (int r = 0; r < len; ++r) tot += rowp[r];
            sdg[len - 1] += tot + __expf(gl) * dS;
        }
        if (!(ok = __syncthreads_and(mbar_wait_bounded(bar_ld, 1)))) break;
        ld_pending = -1;
        // phase B: dQK = lower(dP) E, dE = lower(dP) QK; dQK (C1) and its transpose (C2)
        {
            float y[8];
            tmem_ld16<2>(tmem + lane_base + 0 + cg * 16, y);
            // gam of this thread's two rows and four columns, read before any store
            const float gR[2] = {sg[ra], sg[ra + 8]};
            float gS[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) gS[c] = sg[cg * 16 + 8 * (c >> 1) + cp + (c & 1)];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = ra + 8 * hr;
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const int s = cg * 16 + 8 * n + cp;
                    const float2 qk = *reinterpret_cast<const float2*>(R4 + sw128_off(r, s, kC));
                    const float x0 = y[4 * n + 2 * hr], x1 = y[4 * n + 2 * hr + 1];
                    const bool in0 = s <= r && r < len, in1 = s + 1 <= r && r < len;
                    const float d0 = in0 ? x0 * __expf(gR[hr] - gS[2 * n]) : 0.f;
                    const float d1 = in1 ? x1 * __expf(gR[hr] - gS[2 * n + 1]) : 0.f;
                    *reinterpret_cast<float2*>(sE + r * kLdE + s) = make_float2(in0 ? x0 * qk.x : 0.f, in1 ? x1 * qk.y : 0.f);
                    *reinterpret_cast<float*>(C2 + umma_koff(s, r, kSboC)) = tf32_round(d0);
                    *reinterpret_cast<float*>(C2 + umma_koff(s + 1, r, kSboC)) = tf32_round(d1);
                    *reinterpret_cast<float2*>(C1 + umma_koff(r, s, kSboC)) = make_float2(tf32_round(d0), tf32_round(d1));
                }
            }
        }
        // V -> R2 (rows s, from its bf16 copy in R2 + 16 KB), K^T -> R3 (rows j, k = s) from the copy of K^
        // in R1, Q^T -> R1 (rows j, k = r) from the copy of Q^ in R3: every read before any write
        {
            using RV = RowsTc<kC, kD>;
            constexpr int kIt = kD * kC / 4 / kNTtc;
            float4 vv[RV::kItems], kt[kIt], qt[kIt];
#pragma unroll
            for (int it = 0; it < RV::kItems; ++it) {
                const int s = RV::row(it), k = RV::col(it);  // four bf16 of a 128-byte swizzled row
                const uint2 b = *reinterpret_cast<const uint2*>(
                    R2 + 16384 + (k >> 6) * 8192 + s * 128 + ((((k & 63) >> 3) ^ (s & 7)) << 4) + (k & 7) * 2);
                vv[it] = s < len ? make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                                               __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u))
                                 : z4;
            }
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, j = e % kD, s = (e / kD) * 4;
                float a[4], b[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    a[u] = *reinterpret_cast<const float*>(R1 + sw128_off(s + u, j, kC));  // zero past len
                    b[u] = s + u < len ? *reinterpret_cast<const float*>(R3 + sw128_off(s + u, j, kC)) : 0.f;
                }
                kt[it] = make_float4(a[0], a[1], a[2], a[3]);
                qt[it] = make_float4(b[0], b[1], b[2], b[3]);
            }
            __syncthreads();  // every read of R1, R2 + 16 KB and R3 is done
#pragma unroll
            for (int it = 0; it < RV::kItems; ++it)
                *reinterpret_cast<float4*>(R2 + umma_koff(RV::row(it), RV::col(it), kSboD)) = tf32_round4(vv[it]);
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kNTtc, j = e % kD, s = (e / kD) * 4;
                *reinterpret_cast<float4*>(R3 + umma_koff(j, s, kSboC)) = tf32_round4(kt[it]);
                *reinterpret_cast<float4*>(R1 + umma_koff(j, s, kSboC)) = tf32_round4(qt[it]);
            }
        }
        tc_sync();
        if (tid == 0) {
            umma_tf32_op(tmem + 384, op_sw(smem_u32(R5), kC), op_k(smem_u32(R2), kSboD), id64, kD, false);  // F2
            umma_tf32_k(tmem + 128, smem_u32(R3), kSboC, smem_u32(C1), kSboC, id128, kC, true);   // dq^T
            umma_tf32_k(tmem + 192, smem_u32(R1), kSboC, smem_u32(C2), kSboC, id128, kC, true);   // dk^T
            umma_commit(bar);
        }
        if (!(ok = tc_wait(bar, phase))) break;
        // phase C: column dots with T, dT (-> R4, rows s, k = r); dq update
        {
            float f1[8], f2[8];
            tmem_ld16_pair(tmem + lane_base + 320 + cg * 16, f1, tmem + lane_base + 384 + cg * 16, f2);
            // partial column sums over this thread's two rows: columns cg * 16 + 8 n + cp (+1) at [2 n (+1)]
            float c1[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
            float fbe[4], fge[4];  // beta_r and Gam_r of those four columns, read before any store
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = cg * 16 + 8 * (c >> 1) + cp + (c & 1);
                fbe[c] = sbe[r];
                fge[c] = sgE[r];
            }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int s = ra + 8 * hr;
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const int r = cg * 16 + 8 * n + cp, i = 4 * n + 2 * hr;
                    const float2 tv = *reinterpret_cast<const float2*>(R4 + 16384 + sw128_off(s, r, kC));
                    c1[2 * n] = fmaf(tv.x, f1[i], c1[2 * n]);
                    c1[2 * n + 1] = fmaf(tv.y, f1[i + 1], c1[2 * n + 1]);
                    c2[2 * n] = fmaf(tv.x, f2[i], c2[2 * n]);
                    c2[2 * n + 1] = fmaf(tv.y, f2[i + 1], c2[2 * n + 1]);
                    const float dt0 = fbe[2 * n] * fmaf(fge[2 * n], f1[i], f2[i]);
                    const float dt1 = fbe[2 * n + 1] * fmaf(fge[2 * n + 1], f1[i + 1], f2[i + 1]);
                    *reinterpret_cast<float2*>(R4 + umma_koff(s, r, kSboC)) = make_float2(tf32_round(dt0), tf32_round(dt1));
                }
            }
            // over the eight row groups of the warp (the lanes with this lane's lane % 4), fixed order
#pragma unroll
            for (int off = 4; off < 32; off <<= 1)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    c1[j] += __shfl_xor_sync(kFull, c1[j], off);
                    c2[j] += __shfl_xor_sync(kFull, c2[j], off);
                }
            if (lane < 4) {
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const int r = cg * 16 + 8 * n + cp;
                    part1[q * kC + r] = c1[2 * n];
                    part1[q * kC + r + 1] = c1[2 * n + 1];
                    part2[q * kC + r] = c2[2 * n];
                    part2[q * kC + r + 1] = c2[2 * n + 1];
                }
            }
            float x[16];
            float* dq = p.dqh + ((size_t)t0 * p.HV + h) * kD + jj;
            tmem_ld<2>(tmem + lane_base + 128 + cg * 16, x);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const int r = cg * 16 + t;
                if (r < len) dq[(size_t)r * p.HV * kD] = x[t];
            }
        }
        // dW^T = -X_w -> R2, dU^T -> R1 from the copy of dU in R5 (rows j / i, k = s); diag(beta Gam)-scaled
        // T^T -> C1, diag(beta)-scaled T^T -> C2 (rows r, k = s), from the copy of T in R4 + 16 KB, which
        // is then rounded in place as the B operand of Z
        {
            float x[16];
            tmem_ld<2>(tmem + lane_base + 256 + cg * 16, x);
#pragma unroll
            for (int t = 0; t < 16; t += 4)
                *reinterpret_cast<float4*>(R2 + umma_koff(jj, cg * 16 + t, kSboC)) =
                    tf32_round4(make_float4(-x[t], -x[t + 1], -x[t + 2], -x[t + 3]));
        }
        stage_cols_fn<kD, kC>(R1, [&](int s, int i) { return *reinterpret_cast<const float*>(R5 + sw128_off(s, i, kC)); });
        {
            const uint8_t* T4 = R4 + 16384;
            auto tv = [&](int s, int r) { return *reinterpret_cast<const float*>(T4 + sw128_off(s, r, kC)); };
            stage_cols_fn<kC, kC>(C1, [&](int s, int r) { return tv(s, r) * sbe[r] * sgE[r]; });
            stage_cols_fn<kC, kC>(C2, [&](int s, int r) { return tv(s, r) * sbe[r]; });
        }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < 16384 / 16 / kNTtc; ++it) {
            float4* v = reinterpret_cast<float4*>(R4 + 16384) + tid + it * kNTtc;
            *v = tf32_round4(*v);
        }
        for (int r = tid; r < kC; r += kNTtc) {
            const float a1 = ((part1[r] + part1[kC + r]) + part1[2 * kC + r]) + part1[3 * kC + r];
            const float a2 = ((part2[r] + part2[kC + r]) + part2[2 * kC + r]) + part2[3 * kC + r];
            const float Gr = sgE[r];
            sdb[r] += Gr * a1 + a2;
            sdg[r] += Gr * sbe[r] * a1;
        }
        tc_sync();
        if (tid == 0) {
            umma_tf32_k(tmem + 192, smem_u32(R2), kSboC, smem_u32(C1), kSboC, id128, kC, true);          // dk^T
            umma_tf32_k(tmem + 256, smem_u32(R1), kSboC, smem_u32(C2), kSboC, id128, kC, false);         // dv^T
            umma_tf32_op(tmem + 0, op_k(smem_u32(R4), kSboC), op_sw(smem_u32(R4) + 16384, kC), id64, kC, false);  // Z
            umma_commit(bar);
        }
        if (!(ok = tc_wait(bar, phase))) break;
        // phase D: dv out; Z^T -> R5 (rows s, k = a); T^T -> R5 + 16 KB (rows r, k = a)
        {
            float x[16];
            tmem_ld<2>(tmem + lane_base + 256 + cg * 16, x);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const int r = cg * 16 + t;
                if (r < len) st_any(p.dv_out, ((size_t)(t0 + r) * p.HV + h) * kD + jj, p.dtype, x[t]);
            }
            float z[8];
            tmem_ld16<2>(tmem + lane_base + 0 + cg * 16, z);
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        *reinterpret_cast<float*>(R5 + umma_koff(cg * 16 + 8 * n + cp + e, ra + 8 * hr, kSboC)) =
                            tf32_round(z[4 * n + 2 * hr + e]);
        }
        stage_cols_fn<kC, kC>(R5 + 16384, [&](int a, int r) {
            return *reinterpret_cast<const float*>(R4 + 16384 + sw128_off(a, r, kC));
        });
        tc_sync();
        if (tid == 0) {
            umma_tf32_k(tmem + 448, smem_u32(R5) + 16384, kSboC, smem_u32(R5), kSboC, id64, kC, false);  // T^T Z
            umma_commit(bar);
        }
        if (!(ok = tc_wait(bar, phase))) break;
        // phase E: dA = -strict_lower(T^T Z); dbeta_r += sum_s dA E KK; dKK = dA beta_r E, as TF32 operands
        // both ways round (C1: rows r, k = s; R2: its transpose), which the last dk product adds;
        // dE += dA beta_r KK, the last term of dE: each element's dE * E goes into this warp's partial
        // row sums (part1, per column group) and column sums (part2, per row quarter) for dgam
        {
            float a[8], kk[8];
            tmem_ld16_pair(tmem + lane_base + 448 + cg * 16, a, tmem + lane_base + 64 + cg * 16, kk);
            float cacc[4] = {0.f, 0.f, 0.f, 0.f};  // columns cg * 16 + 8 n + cp + e at [2 n + e]
            // gam and beta of this thread's two rows, gam of its four columns and its eight values of
            // dE so far, read before any store
            const float gR[2] = {sg[ra], sg[ra + 8]}, bR[2] = {sbe[ra], sbe[ra + 8]};
            float gS[4], e0[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) gS[c] = sg[cg * 16 + 8 * (c >> 1) + cp + (c & 1)];
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const float2 v = *reinterpret_cast<const float2*>(sE + (ra + 8 * ((i >> 1) & 1)) * kLdE + cg * 16 + 8 * (i >> 2) + cp);
                e0[i] = v.x;
                e0[i + 1] = v.y;
            }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = ra + 8 * hr;
                float acc = 0.f, racc = 0.f;
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    float dkk[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int s = cg * 16 + 8 * n + cp + e, i = 4 * n + 2 * hr + e;
                        // exp(gam_r - gam_s) only where s < r: above the diagonal it can overflow, and
                        // 0 * inf would be NaN
                        const float da = s < r ? -a[i] : 0.f, ex = s < r ? __expf(gR[hr] - gS[2 * n + e]) : 0.f;
                        acc = fmaf(da * ex, kk[i], acc);
                        dkk[e] = tf32_round(da * bR[hr] * ex);
                        *reinterpret_cast<float*>(R2 + umma_koff(s, r, kSboC)) = dkk[e];
                        const float de = fmaf(da * bR[hr], kk[i], e0[i]);  // dE[r][s], complete
                        const float pe = s < r ? de * ex : (s == r ? de : 0.f);     // dE * E on its support
                        racc += pe;
                        cacc[2 * n + e] += pe;
                    }
                    *reinterpret_cast<float2*>(C1 + umma_koff(r, cg * 16 + 8 * n + cp, kSboC)) = make_float2(dkk[0], dkk[1]);
                }
                // the row's 16 columns of this warp sit in the four lanes of its row group
                acc += __shfl_xor_sync(kFull, acc, 1);
                acc += __shfl_xor_sync(kFull, acc, 2);
                racc += __shfl_xor_sync(kFull, racc, 1);
                racc += __shfl_xor_sync(kFull, racc, 2);
                if ((lane & 3) == 0) {
                    rowp[cg * kC + r] = acc;
                    part1[cg * kC + r] = racc;
                }
            }
            // the warp's 16 rows of each column: the eight row groups, fixed order
#pragma unroll
            for (int off = 4; off < 32; off <<= 1)
#pragma unroll
                for (int j = 0; j < 4; ++j) cacc[j] += __shfl_xor_sync(kFull, cacc[j], off);
            if (lane < 4) {
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    part2[q * kC + cg * 16 + 8 * n + cp] = cacc[2 * n];
                    part2[q * kC + cg * 16 + 8 * n + cp + 1] = cacc[2 * n + 1];
                }
            }
        }
        __syncthreads();
        for (int r = tid; r < kC; r += kNTtc) sdb[r] += ((rowp[r] + rowp[kC + r]) + rowp[2 * kC + r]) + rowp[3 * kC + r];
        tc_sync();
        if (tid == 0) {  // dk^T += K^T (dKK + dKK^T)^T, one product per term
            umma_tf32_k(tmem + 192, smem_u32(R3), kSboC, smem_u32(C1), kSboC, id128, kC, true);
            umma_tf32_k(tmem + 192, smem_u32(R3), kSboC, smem_u32(R2), kSboC, id128, kC, true);
            umma_commit(bar);
        }
        if (!(ok = tc_wait(bar, phase))) break;
        // phase F: dk out (all four terms at once)
        {
            float x[16];
            float* dkk = p.dkh + ((size_t)t0 * p.HV + h) * kD + jj;
            tmem_ld<2>(tmem + lane_base + 192 + cg * 16, x);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const int r = cg * 16 + t;
                if (r < len) dkk[(size_t)r * p.HV * kD] = x[t];
            }
        }
    } while (false);
    if (ok) {
        // dgam from E (row sums minus column sums of dE * E, from phase E's partials), then
        // dg = reverse cumsum
        for (int r = tid; r < kC; r += kNTtc)
            sdg[r] += (((part1[r] + part1[kC + r]) + part1[2 * kC + r]) + part1[3 * kC + r]) -
                      (((part2[r] + part2[kC + r]) + part2[2 * kC + r]) + part2[3 * kC + r]);
        __syncthreads();
        if (warp == 0) {
            // dg = reverse cumsum of dgam: lane l takes rows len-1-2l and len-2-2l, a warp scan adds
            // the lanes below
            const int ra = len - 1 - 2 * lane, rb = ra - 1;
            const float a = ra >= 0 ? sdg[ra] : 0.f, b = rb >= 0 ? sdg[rb] : 0.f;
            float inc = a + b;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(kFull, inc, off);
                if (lane >= off) inc += y;
            }
            const float below = __shfl_up_sync(kFull, inc, 1);
            const float ea = (lane ? below : 0.f) + a, eb = ea + b;
            if (ra >= 0) {
                p.dg[(size_t)(t0 + ra) * p.HV + h] = ea;
                p.dbeta[(size_t)(t0 + ra) * p.HV + h] = sdb[ra];
            }
            if (rb >= 0) {
                p.dg[(size_t)(t0 + rb) * p.HV + h] = eb;
                p.dbeta[(size_t)(t0 + rb) * p.HV + h] = sdb[rb];
            }
        }
    }
    if (!ok && tid == 0) {
        atomicOr(p.err, GDN_DEVERR_TIMEOUT);
        if (ld_pending >= 0) mbar_wait_bounded(bar_ld, (uint32_t)ld_pending);  // copies in flight land first
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
    // The last of the G value-head CTAs of this (chunk, k-head) to arrive folds their dq^, dk^ rows
    // (fold_tokens: the heads in increasing order, whichever CTA folds).  No CTA waits for another.
    __threadfence();  // this CTA's rows are visible on the device before it is counted
    __syncthreads();
    if (tid == 0) {
        const unsigned prior = atomicAdd(p.fcnt + (size_t)c * p.HK + hk, 1u);
        __threadfence();  // and the other CTAs' rows before this one reads them
        *s_last = prior == (unsigned)(p.G - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (*s_last && ok) {  // rows warp + 16 u of the chunk, two at a time with their loads together
        for (int r = warp; r < len; r += 2 * (kNTtc / 32)) {
            const int r2 = r + kNTtc / 32;
            const long long ws[2] = {(long long)(t0 + r) * p.HK + hk, (long long)(t0 + min(r2, len - 1)) * p.HK + hk};
            const bool on[2] = {true, r2 < len};
            fold_tokens<2>(p, ws, on, lane);
        }
    }
}

// per (token, k-head), for the kernels that leave the fold to a pass of its own
__global__ void bwd_fold_kernel(BwdParams p) {
    const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (w >= (long long)p.T * p.HK) return;
    const long long ws[1] = {w};
    const bool on[1] = {true};
    fold_tokens<1>(p, ws, on, threadIdx.x & 31);
}

// ---------------------------------------------------------------------------
struct BwdLayout {
    size_t coff, qn, kn, qinv, kinv, gam, W, Ut, T, QK, P, BK, GQ, S, D, Ssc, Dsc, U, dU, dgA, dqh, dkh, fcnt, total;
    int nchm;
};

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

static BwdLayout bwd_layout(const gdn_shape* s) {
    BwdLayout L;
    const size_t T = s->T_total, HK = s->HK, HV = s->HV, dk = s->dk, dv = s->dv;
    L.nchm = s->N + (s->T_total + kC - 1) / kC;
    const size_t CH = (size_t)L.nchm * HV;
    size_t o = kWsHeader;
    auto take = [&](size_t bytes) { size_t at = o; o += al256(bytes); return at; };
    L.coff = take((s->N + 1) * 4);
    L.qn = take(T * HK * dk * 4);
    L.kn = take(T * HK * dk * 4);
    L.qinv = take(T * HK * 4);
    L.kinv = take(T * HK * 4);
    L.gam = take(T * HV * 4);
    L.W = take(CH * kC * dk * 4);
    L.Ut = take(CH * kC * dv * 4);
    L.T = take(CH * kC * kC * 4);
    L.QK = take(CH * kC * kC * 4);
    L.P = take(CH * kC * kC * 4);
    // diag(b) K and diag(Gam) Q (and the per-chunk dgam partials) only feed the mma.sync kernels; the
    // tcgen05 path at dk = dv = 128 (bf16) forms them on chip
    const bool tc128 = s->dtype == GDN_BF16 && dk == 128 && dv == 128;
    L.BK = take(tc128 ? 0 : CH * kC * dk * 4);
    L.GQ = take(tc128 ? 0 : CH * kC * dk * 4);
    // the chunk states: fp32, or at dk = dv = 128 (bf16) fp16 with a factor per 32 x 32 tile
    L.S = take(CH * dv * dk * (tc128 ? 2 : 4));
    L.D = take(CH * dv * dk * (tc128 ? 2 : 4));
    L.Ssc = take(tc128 ? CH * 16 * 4 : 0);
    L.Dsc = take(tc128 ? CH * 16 * 4 : 0);
    L.U = take(CH * kC * dv * 4);
    L.dU = take(CH * kC * dv * 4);
    L.dgA = take(tc128 ? 0 : CH * kC * 4);
    L.dqh = take(T * HV * dk * 4);
    L.dkh = take(T * HV * dk * 4);
    L.fcnt = take(tc128 ? (size_t)L.nchm * HK * 4 : 0);  // the on-chip fold's arrival counters
    L.total = o;
    return L;
}

size_t bwd_workspace_size(const gdn_shape* s) { return bwd_layout(s).total; }

template <typename K>
static bool set_smem(K kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
}

// The two state passes on tcgen05: one CTA of 512 threads per (sequence, head).
template <int DK>
static gdn_status launch_state_tc(const BwdParams& p, int N, int HV, cudaStream_t cs) {
    const dim3 grid(N, HV);
    const size_t tail = 64;  // mbarrier + TMEM address slot
    const size_t smem_f = (size_t)4 * (kC * DK + 128 * kC + DK * kC + kC) + tail;
    const size_t smem_b = (size_t)4 * (128 * kC + DK * kC + kC * kC + kC * DK + DK * kC + 128 * kC + 4 * kC) +
                          (size_t)2 * kC * (DK * 2 + 16) + tail;
    if (!set_smem(bwd_state_fwd_tc_kernel<DK>, smem_f)) return GDN_ERR_CUDA;
    bwd_state_fwd_tc_kernel<DK><<<grid, kNTtc, smem_f, cs>>>(p);
    if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
    if (!set_smem(bwd_state_bwd_tc_kernel<DK>, smem_b)) return GDN_ERR_CUDA;
    bwd_state_bwd_tc_kernel<DK><<<grid, kNTtc, smem_b, cs>>>(p);
    if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // namespace gdn

extern "C" gdn_status gdn_chunk_bwd(const gdn_shape* s, const void* q, const void* k, const void* v,
                                    const float* g, const float* beta, const float* init_state,
                                    const int32_t* cu_seqlens, const void* d_out, const float* d_final_state,
                                    void* dq, void* dk, void* dv, float* dg, float* dbeta, float* d_init_state,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    using namespace gdn;
    gdn_status st = check_shape(s);
    if (st != GDN_OK) return st;
    if (!cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (s->N == 0) return GDN_OK;
    if (s->T_total > 0 && (!q || !k || !v || !g || !beta || !d_out || !dq || !dk || !dv || !dg || !dbeta))
        return GDN_ERR_INVALID_ARG;
    const void* vec[] = {q, k, v, init_state, d_out, d_final_state, dq, dk, dv, d_init_state, workspace};
    for (const void* ptr : vec)
        if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
    const void* sca[] = {g, beta, cu_seqlens, dg, dbeta};
    for (const void* ptr : sca)
        if (ptr && !aligned4(ptr)) return GDN_ERR_INVALID_ARG;
    const void* outs[] = {dq, dk, dv, dg, dbeta, d_init_state};
    const void* ins[] = {q, k, v, g, beta, init_state, d_out, d_final_state};
    for (const void* o : outs)
        for (const void* i : ins)
            if (o && o == i) return GDN_ERR_INVALID_ARG;
    const BwdLayout L = bwd_layout(s);
    if (!workspace || workspace_bytes < L.total) return GDN_ERR_WORKSPACE;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);

    BwdParams p;
    p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.init_state = init_state; p.cu = cu_seqlens;
    p.dout = d_out; p.dfinal = d_final_state; p.dq_out = dq; p.dk_out = dk; p.dv_out = dv; p.dg = dg; p.dbeta = dbeta;
    p.dinit = d_init_state;
    p.err = reinterpret_cast<unsigned*>(ws);
    p.coff = reinterpret_cast<int32_t*>(ws + L.coff);
    p.qn = reinterpret_cast<float*>(ws + L.qn);
    p.kn = reinterpret_cast<float*>(ws + L.kn);
    p.qinv = reinterpret_cast<float*>(ws + L.qinv);
    p.kinv = reinterpret_cast<float*>(ws + L.kinv);
    p.gam = reinterpret_cast<float*>(ws + L.gam);
    p.Wb = reinterpret_cast<float*>(ws + L.W);
    p.Utb = reinterpret_cast<float*>(ws + L.Ut);
    p.Tb = reinterpret_cast<float*>(ws + L.T);
    p.QKb = reinterpret_cast<float*>(ws + L.QK);
    p.Pb = reinterpret_cast<float*>(ws + L.P);
    p.BKb = reinterpret_cast<float*>(ws + L.BK);
    p.GQb = reinterpret_cast<float*>(ws + L.GQ);
    p.Sb = reinterpret_cast<float*>(ws + L.S);
    p.Db = reinterpret_cast<float*>(ws + L.D);
    p.Sh = reinterpret_cast<__half*>(ws + L.S);
    p.Dh = reinterpret_cast<__half*>(ws + L.D);
    p.Ssc = reinterpret_cast<float*>(ws + L.Ssc);
    p.Dsc = reinterpret_cast<float*>(ws + L.Dsc);
    p.Ub = reinterpret_cast<float*>(ws + L.U);
    p.dUb = reinterpret_cast<float*>(ws + L.dU);
    p.dgamA = reinterpret_cast<float*>(ws + L.dgA);
    p.dqh = reinterpret_cast<float*>(ws + L.dqh);
    p.dkh = reinterpret_cast<float*>(ws + L.dkh);
    p.fcnt = reinterpret_cast<unsigned*>(ws + L.fcnt);
    p.N = s->N; p.T = s->T_total; p.HK = s->HK; p.HV = s->HV; p.G = s->HV / s->HK; p.dk = s->dk; p.dv = s->dv;
    p.use_norm = s->use_qk_l2norm ? 1 : 0;
    p.nchm = L.nchm;
    p.dtype = s->dtype;
    {
        int dev = 0, nsm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0)
            return GDN_ERR_CUDA;
        p.nsm = nsm;
        // the intra kernel's CTAs live about 50K SM cycles at dk = dv = 128; the first-wave spread
        // (two lifetimes) pays off only when the grid runs many waves
        const bool many = (long long)L.nchm * s->HV >= 8LL * nsm;
        p.stagger_intra = many ? STAGGER_INTRA_CYCLES : 0;
    }

    if (cudaMemsetAsync(ws, 0, sizeof(unsigned), cs) != cudaSuccess) return GDN_ERR_CUDA;
    if (L.fcnt != L.total && cudaMemsetAsync(ws + L.fcnt, 0, L.total - L.fcnt, cs) != cudaSuccess) return GDN_ERR_CUDA;
    bwd_offsets_kernel<<<1, 32, 0, cs>>>(p);
    if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
    if (s->T_total > 0) {
        const long long vec = (long long)s->T_total * s->HK;  // one warp each, 8 per CTA
        bwd_norm_kernel<<<(unsigned)((vec + 7) / 8), 256, 0, cs>>>(p);
        if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
    }
    const dim3 gch(L.nchm, s->HV);
    const bool tc_state = s->dtype == GDN_BF16 && s->dv == 128 && (s->dk == 32 || s->dk == 64 || s->dk == 128);
    // tensor maps of the normalised q and k ([T][HK * 128] fp32: a chunk's rows from token t0, columns
    // of head hk), copied by bwd_wy_tc_kernel and bwd_intra_tc_kernel
    CUtensorMap mk{}, mq{};
    const bool tc128 = tc_state && s->dk == 128;
    const uint64_t CH = (uint64_t)L.nchm * s->HV;
    if (tc128 && CH * 128 >= (1ull << 31)) return GDN_ERR_UNSUPPORTED;  // copy coordinates are 32-bit
    if (tc128 &&
        (encode_rows_sw128(&mk, p.kn, GDN_F32, (uint64_t)s->HK * 128, (uint64_t)std::max(s->T_total, 1),
                           (uint64_t)s->HK * 512, kC) != GDN_OK ||
         encode_rows_sw128(&mq, p.qn, GDN_F32, (uint64_t)s->HK * 128, (uint64_t)std::max(s->T_total, 1),
                           (uint64_t)s->HK * 512, kC) != GDN_OK))
        return GDN_ERR_CUDA;
    if (tc128) {
        CUtensorMap mvw{};  // V ([T][HV * 128] bf16), copied by bwd_wy_tc_kernel
        if (encode_rows_sw128(&mvw, v, GDN_BF16, (uint64_t)s->HV * 128, (uint64_t)std::max(s->T_total, 1),
                              (uint64_t)s->HV * 256, kC) != GDN_OK)
            return GDN_ERR_CUDA;
        if (!set_smem(bwd_wy_tc_kernel, kWyTcSmem)) return GDN_ERR_CUDA;
        bwd_wy_tc_kernel<<<(unsigned)CH, kNTtc, kWyTcSmem, cs>>>(mk, mq, mvw, p);
    } else {
        const size_t smem_wy = sizeof(float) * (2 * kC * kLdD + 2 * kC * kLdC + 3 * kC);
        if (!set_smem(bwd_wy_kernel, smem_wy)) return GDN_ERR_CUDA;
        bwd_wy_kernel<<<gch, kNTwy, smem_wy, cs>>>(p);
    }
    if (launch_status() != GDN_OK) return GDN_ERR_CUDA;

    if (tc_state) {
        gdn_status st = GDN_ERR_UNSUPPORTED;
        switch (s->dk) {
            case 32: st = launch_state_tc<32>(p, s->N, s->HV, cs); break;
            case 64: st = launch_state_tc<64>(p, s->N, s->HV, cs); break;
            case 128: st = launch_state_tc<128>(p, s->N, s->HV, cs); break;
        }
        if (st != GDN_OK) return st;
    } else {
        const int R = s->dv;  // one CTA per (sequence, head) holds every row of the state
        const dim3 gseq(s->N, s->HV, s->dv / R);
        const size_t smem_sf = sizeof(float) * (R * kLdD + 2 * kC * kLdD + 2 * kC * (R + 4));
        if (!set_smem(bwd_state_fwd_kernel, smem_sf)) return GDN_ERR_CUDA;
        bwd_state_fwd_kernel<<<gseq, kNTs, smem_sf, cs>>>(p, R);
        if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
        const size_t smem_sb = sizeof(float) * (R * kLdD + 2 * kC * kLdD + kC * kLdC + 2 * kC * (R + 4));
        if (!set_smem(bwd_state_bwd_kernel, smem_sb)) return GDN_ERR_CUDA;
        bwd_state_bwd_kernel<<<gseq, kNTs, smem_sb, cs>>>(p, R);
        if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
    }

    if (tc128) {
        // tensor maps of the other operands bwd_intra_tc_kernel copies: U and dU ([chunk-head * 64][128]),
        // S0^T ([chunk-head * 128][128] fp16), Q K^T and T ([chunk-head * 64][64]), V and dO ([T][HV * 128]
        // bf16)
        CUtensorMap mu{}, mdu{}, ms{}, mqk{}, mt{}, mv{}, mdo{};
        if (encode_rows_sw128(&mu, p.Ub, GDN_F32, 128, CH * kC, 512, kC) != GDN_OK ||
            encode_rows_sw128(&mdu, p.dUb, GDN_F32, 128, CH * kC, 512, kC) != GDN_OK ||
            encode_rows_sw128(&ms, p.Sh, GDN_BF16, 128, CH * 128, 256, 128) != GDN_OK ||  // 2-byte elements: fp16
            encode_rows_sw128(&mqk, p.QKb, GDN_F32, kC, CH * kC, 256, kC) != GDN_OK ||
            encode_rows_sw128(&mt, p.Tb, GDN_F32, kC, CH * kC, 256, kC) != GDN_OK ||
            encode_rows_sw128(&mv, v, GDN_BF16, (uint64_t)s->HV * 128, (uint64_t)std::max(s->T_total, 1),
                              (uint64_t)s->HV * 256, kC) != GDN_OK ||
            encode_rows_sw128(&mdo, d_out, GDN_BF16, (uint64_t)s->HV * 128, (uint64_t)std::max(s->T_total, 1),
                              (uint64_t)s->HV * 256, kC) != GDN_OK)
            return GDN_ERR_CUDA;
        if (!set_smem(bwd_intra_tc_kernel, kIntraCTcSmem)) return GDN_ERR_CUDA;
        // one-dimensional grid, value heads fastest: the G heads of a k-head fold on chip (no fold pass)
        bwd_intra_tc_kernel<<<(unsigned)CH, kNTtc, kIntraCTcSmem, cs>>>(mk, mu, mdu, ms, mqk, mt, mq, mv, mdo, p);
    } else {
        const size_t smem_is = sizeof(float) * (kMaxD * kLdD + 4 * kC * kLdD + 2 * kC + 32);
        if (!set_smem(bwd_intra_s_kernel, smem_is)) return GDN_ERR_CUDA;
        bwd_intra_s_kernel<<<gch, kNT, smem_is, cs>>>(p);
        if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
        const size_t smem_ic = sizeof(float) * (4 * kC * kLdD + 4 * kC * kLdC + 4 * kC);
        if (!set_smem(bwd_intra_c_kernel, smem_ic)) return GDN_ERR_CUDA;
        bwd_intra_c_kernel<<<gch, kNT, smem_ic, cs>>>(p);
    }
    if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
    if (!tc128 && s->T_total > 0) {
        const long long vec = (long long)s->T_total * s->HK;  // one warp each, 8 per CTA
        bwd_fold_kernel<<<(unsigned)((vec + 7) / 8), 256, 0, cs>>>(p);
        if (launch_status() != GDN_OK) return GDN_ERR_CUDA;
    }
    return GDN_OK;
}
