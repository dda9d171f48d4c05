// gdn_step.cuh -- the per-row token step shared by every forward-direction
// kernel (recurrent prefill/trainer forward and the decode step).
//
// Bit-invariance rests on this file: every kernel that advances a state row
// does it with exactly these IEEE operations in exactly this order, so the
// bits of a row depend only on that row's inputs.  Rows of S never interact
// in the gated delta rule (u_i = S_i . k^ and o_i = S_i . q^ involve row i
// only), so how rows are spread over threads, warps and CTAs is free; the
// lane->dk mapping, the in-lane summation order and the butterfly are not.
//
// Layout of one state row (dk fp32 values): row r lives in kLanesPerRow (L)
// consecutive lanes of a warp; lane e = lane % L holds the float4 chunks
// c = L*i + e, i = 0 .. dk/(4L)-1 (chunk c = elements 4c .. 4c+3).  A thread
// holds kRowsPerThread (R) consecutive rows.  A dk contraction is: per
// accumulator set j = i mod NS (NS = chunks/8 when a lane holds 16 or more
// chunks, else 1) two packed (x, y) / (z, w) fma chains over i in increasing
// order starting from +0; the sets summed in increasing j; then
// (x + y) + (z + w); then an xor butterfly over the L lanes of the row
// (commutative adds, so every lane ends with the same bits).
// The recurrence (gated delta rule, recurrent form as in "Defending Against
// the Training-Inference Numeric Mismatch in RL (Especially Linear
// Attention)", section 3.2):
//     u = S k^,  w = b (v - a u),  S <- a S + w k^T,  o = S q^
// which equals S <- a S (I - b k^ k^T) + b v k^T with o read after the update.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr float kNormEps = 1e-6f;
constexpr unsigned kFull = 0xffffffffu;

#ifndef GDN_LANES
#define GDN_LANES 4
#endif
#ifndef GDN_ROWS
#define GDN_ROWS 2
#endif
constexpr int kLanesPerRow = GDN_LANES;   // L
constexpr int kRowsPerThread = GDN_ROWS;  // R
static_assert(kLanesPerRow == 1 || kLanesPerRow == 2 || kLanesPerRow == 4 || kLanesPerRow == 8, "L");
static_assert(kRowsPerThread == 1 || kRowsPerThread == 2 || kRowsPerThread == 4, "R");
// threads that hold a 128-row state slice
constexpr int kThreadsPer128Rows = 128 * kLanesPerRow / kRowsPerThread;

// accumulator chain length: a lane's chunks are summed in kSets interleaved sets
#ifndef GDN_CHAIN
#define GDN_CHAIN 8
#endif
template <int DK>
struct RowFrag {
    static_assert(DK % (4 * kLanesPerRow) == 0, "dk must be a multiple of 4 L");
    static constexpr int kChunks = DK / (4 * kLanesPerRow);
    static constexpr int kSets = kChunks >= 2 * GDN_CHAIN ? kChunks / GDN_CHAIN : 1;
    // chunk i = elements (4c .. 4c+3), kept as the register pairs (x, y) = p[2i], (z, w) = p[2i+1]
    float2 p[2 * kChunks];
};

__device__ __forceinline__ int chunk_of(int i, int e) { return kLanesPerRow * i + e; }

__device__ __forceinline__ float ld_in(const float* p) { return *p; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Four consecutive input elements widened to fp32 (pointer 8-byte aligned for bf16,
// 16-byte aligned for fp32).
__device__ __forceinline__ float4 ld4_in(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4_in(const __nv_bfloat16* p) {
    uint2 raw = *reinterpret_cast<const uint2*>(p);
    __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
    __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
    float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}

// R adjacent values (a thread's rows) of v widened to fp32, and the R outputs
// stored rounded to nearest.
template <int R, typename T>
__device__ __forceinline__ void ld_rows_in(const T* p, float (&v)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = ld_in(p + r);
}
__device__ __forceinline__ void st_in(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_in(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
template <int R, typename T>
__device__ __forceinline__ void st_rows_out(T* p, const float (&o)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) st_in(p + r, o[r]);
}

// Two adjacent values (rows 2p, 2p+1) of v widened to fp32.
__device__ __forceinline__ float2 ld2_in(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld2_in(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// Store two adjacent outputs (rows 2p, 2p+1), rounding to nearest for bf16.
__device__ __forceinline__ void st2_out(float* p, float a, float b) {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
__device__ __forceinline__ void st2_out(__nv_bfloat16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

// L2-normalise one dk vector with one full warp: lane l owns elements
// 4l .. 4l+3 (lanes l >= dk/4 own nothing and contribute +0).  Sum of squares
// in-lane as ((x*x + y*y) + z*z) + w*w via fma, then an xor butterfly over
// offsets 16, 8, 4, 2, 1 (every lane ends with the same bits), then
// x * (1 / sqrt(ss + eps)) with a correctly rounded reciprocal square root.
// Writes the fp32 result to dst (16-byte aligned).  Must be called by all 32
// lanes of the warp.
template <int DK, typename Tin>
__device__ __forceinline__ void l2norm_warp(const Tin* __restrict__ src, float* __restrict__ dst,
                                            int lane, bool use_norm) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    const bool own = lane < DK / 4;
    if (own) x = ld4_in(src + 4 * lane);
    if (use_norm) {
        float ss = __fmul_rn(x.x, x.x);
        ss = __fmaf_rn(x.y, x.y, ss);
        ss = __fmaf_rn(x.z, x.z, ss);
        ss = __fmaf_rn(x.w, x.w, ss);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(kFull, ss, off));
        const float inv = __frsqrt_rn(__fadd_rn(ss, kNormEps));
        x.x = __fmul_rn(x.x, inv);
        x.y = __fmul_rn(x.y, inv);
        x.z = __fmul_rn(x.z, inv);
        x.w = __fmul_rn(x.w, inv);
    }
    if (own) *reinterpret_cast<float4*>(dst + 4 * lane) = x;
}

// NV vectors at once with exactly l2norm_warp's per-vector operations (the
// independent chains interleave); vectors v >= nvalid are skipped.
template <int DK, int NV, typename Tin>
__device__ __forceinline__ void l2norm_warp_multi(const Tin* const (&src)[NV], float* const (&dst)[NV], int nvalid,
                                                  int lane, bool use_norm) {
    float4 x[NV];
    const bool own = lane < DK / 4;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        x[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (own && v < nvalid) x[v] = ld4_in(src[v] + 4 * lane);
    }
    if (use_norm) {
        float ss[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            ss[v] = __fmul_rn(x[v].x, x[v].x);
            ss[v] = __fmaf_rn(x[v].y, x[v].y, ss[v]);
            ss[v] = __fmaf_rn(x[v].z, x[v].z, ss[v]);
            ss[v] = __fmaf_rn(x[v].w, x[v].w, ss[v]);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
            for (int v = 0; v < NV; ++v) ss[v] = __fadd_rn(ss[v], __shfl_xor_sync(kFull, ss[v], off));
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const float inv = __frsqrt_rn(__fadd_rn(ss[v], kNormEps));
            x[v].x = __fmul_rn(x[v].x, inv);
            x[v].y = __fmul_rn(x[v].y, inv);
            x[v].z = __fmul_rn(x[v].z, inv);
            x[v].w = __fmul_rn(x[v].w, inv);
        }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v)
        if (own && v < nvalid) *reinterpret_cast<float4*>(dst[v] + 4 * lane) = x[v];
}

// Gate values for one token: a = exp(g) (CUDA's expf, same call everywhere), b as given.
__device__ __forceinline__ float gate_alpha(float g) { return expf(g); }

// Finish of a dk contraction, in two parts that together are one fixed tree:
// lane_partial: the sets in increasing order, then (x + y) + (z + w);
// lanes_reduce: the xor butterfly over the L lanes of the row.  Splitting them
// only lets a caller overlap one contraction's butterfly with other work.
template <int NS>
__device__ __forceinline__ float lane_partial(const float2 (&xy)[NS], const float2 (&zw)[NS]) {
    float2 a = xy[0], b = zw[0];
#pragma unroll
    for (int j = 1; j < NS; ++j) {
        a.x = __fadd_rn(a.x, xy[j].x);
        a.y = __fadd_rn(a.y, xy[j].y);
        b.x = __fadd_rn(b.x, zw[j].x);
        b.y = __fadd_rn(b.y, zw[j].y);
    }
    return __fadd_rn(__fadd_rn(a.x, a.y), __fadd_rn(b.x, b.y));
}
__device__ __forceinline__ float lanes_reduce(float p) {
#pragma unroll
    for (int m = 1; m < kLanesPerRow; m <<= 1) p = __fadd_rn(p, __shfl_xor_sync(kFull, p, m));
    return p;
}
template <int NS>
__device__ __forceinline__ float finish_dot(const float2 (&xy)[NS], const float2 (&zw)[NS]) {
    return lanes_reduce(lane_partial<NS>(xy, zw));
}

// u[r] = S_r . x for the R rows a thread holds; x is a dk fp32 vector in shared memory.
// Must be called by all 32 lanes of the warp.
//
// Two instruction forms give the same bits: the packed form issues the (x, y)
// and (z, w) accumulator chains as one two-lane fma.rn.f32x2 each (sm_100+),
// which halves the issue slots the FP32 pipe work takes; every lane of it is
// the same IEEE round-to-nearest fma as the scalar form.  GDN_STEP_SCALAR
// selects the scalar form.
__device__ __forceinline__ float2 lo2(const float4& v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(const float4& v) { return make_float2(v.z, v.w); }

template <int DK, int R>
__device__ __forceinline__ void rows_dot_part(const RowFrag<DK> (&s)[R], const float* __restrict__ x,
                                              int e, float (&u)[R]) {
    constexpr int NC = RowFrag<DK>::kChunks, NS = RowFrag<DK>::kSets;
    float2 xy[R][NS], zw[R][NS];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < NS; ++j) xy[r][j] = zw[r][j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const float4 k4 = *reinterpret_cast<const float4*>(x + 4 * chunk_of(i, e));
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float2& A = xy[r][i % NS];
            float2& B = zw[r][i % NS];
#ifdef GDN_STEP_SCALAR
            A.x = __fmaf_rn(s[r].p[2 * i].x, k4.x, A.x);
            A.y = __fmaf_rn(s[r].p[2 * i].y, k4.y, A.y);
            B.x = __fmaf_rn(s[r].p[2 * i + 1].x, k4.z, B.x);
            B.y = __fmaf_rn(s[r].p[2 * i + 1].y, k4.w, B.y);
#else
            A = __ffma2_rn(s[r].p[2 * i], lo2(k4), A);
            B = __ffma2_rn(s[r].p[2 * i + 1], hi2(k4), B);
#endif
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) u[r] = lane_partial<NS>(xy[r], zw[r]);
}

template <int DK, int R>
__device__ __forceinline__ void rows_dot(const RowFrag<DK> (&s)[R], const float* __restrict__ x,
                                         int e, float (&u)[R]) {
    rows_dot_part<DK, R>(s, x, e, u);
#pragma unroll
    for (int r = 0; r < R; ++r) u[r] = lanes_reduce(u[r]);
}

// w = b (v - a u)
__device__ __forceinline__ float delta_w(float a, float b, float v, float u) {
    return __fmul_rn(b, __fsub_rn(v, __fmul_rn(a, u)));
}

// S_r <- a S_r + w_r k^T (per element fma(w, k_j, a * S_rj)), then o[r] = S_r . q.
// Must be called by all 32 lanes of the warp.  Same two forms as rows_dot.
template <int DK, int R>
__device__ __forceinline__ void rows_update_part(RowFrag<DK> (&s)[R], const float* __restrict__ k,
                                                 const float* __restrict__ q, int e, float a,
                                                 const float (&w)[R], float (&o)[R]) {
    constexpr int NC = RowFrag<DK>::kChunks, NS = RowFrag<DK>::kSets;
    float2 xy[R][NS], zw[R][NS];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < NS; ++j) xy[r][j] = zw[r][j] = make_float2(0.f, 0.f);
#ifndef GDN_STEP_SCALAR
    const float2 a2 = make_float2(a, a);
#endif
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const float4 k4 = *reinterpret_cast<const float4*>(k + 4 * chunk_of(i, e));
        const float4 q4 = *reinterpret_cast<const float4*>(q + 4 * chunk_of(i, e));
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float2& Sxy = s[r].p[2 * i];
            float2& Szw = s[r].p[2 * i + 1];
            float2& A = xy[r][i % NS];
            float2& B = zw[r][i % NS];
#ifdef GDN_STEP_SCALAR
            Sxy.x = __fmaf_rn(w[r], k4.x, __fmul_rn(a, Sxy.x));
            Sxy.y = __fmaf_rn(w[r], k4.y, __fmul_rn(a, Sxy.y));
            Szw.x = __fmaf_rn(w[r], k4.z, __fmul_rn(a, Szw.x));
            Szw.y = __fmaf_rn(w[r], k4.w, __fmul_rn(a, Szw.y));
            A.x = __fmaf_rn(Sxy.x, q4.x, A.x);
            A.y = __fmaf_rn(Sxy.y, q4.y, A.y);
            B.x = __fmaf_rn(Szw.x, q4.z, B.x);
            B.y = __fmaf_rn(Szw.y, q4.w, B.y);
#else
            const float2 w2 = make_float2(w[r], w[r]);
            Sxy = __ffma2_rn(w2, lo2(k4), __fmul2_rn(a2, Sxy));
            Szw = __ffma2_rn(w2, hi2(k4), __fmul2_rn(a2, Szw));
            A = __ffma2_rn(Sxy, lo2(q4), A);
            B = __ffma2_rn(Szw, hi2(q4), B);
#endif
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) o[r] = lane_partial<NS>(xy[r], zw[r]);
}

template <int DK, int R>
__device__ __forceinline__ void rows_update_out(RowFrag<DK> (&s)[R], const float* __restrict__ k,
                                                const float* __restrict__ q, int e, float a,
                                                const float (&w)[R], float (&o)[R]) {
    rows_update_part<DK, R>(s, k, q, e, a, w, o);
#pragma unroll
    for (int r = 0; r < R; ++r) o[r] = lanes_reduce(o[r]);
}

// One full token for the R rows of a thread: u, w, update, o.
template <int DK, int R>
__device__ __forceinline__ void token_step(RowFrag<DK> (&s)[R], const float* __restrict__ kn,
                                           const float* __restrict__ qn, int e, float a, float b,
                                           const float (&v)[R], float (&o)[R]) {
    float u[R], w[R];
    rows_dot<DK, R>(s, kn, e, u);
#pragma unroll
    for (int r = 0; r < R; ++r) w[r] = delta_w(a, b, v[r], u[r]);
    rows_update_out<DK, R>(s, kn, qn, e, a, w, o);
}

// Global <-> register transfer of the R rows a thread holds.  row0 points at
// the first row (row stride dk floats); rows r = 0..R-1 are consecutive.
template <int DK, int R>
__device__ __forceinline__ void load_rows(RowFrag<DK> (&s)[R], const float* __restrict__ row0, int e) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < RowFrag<DK>::kChunks; ++i) {
            const float4 v = __ldcs(reinterpret_cast<const float4*>(row0 + (size_t)r * DK + 4 * chunk_of(i, e)));
            s[r].p[2 * i] = make_float2(v.x, v.y);
            s[r].p[2 * i + 1] = make_float2(v.z, v.w);
        }
}

template <int DK, int R>
__device__ __forceinline__ void zero_rows(RowFrag<DK> (&s)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < 2 * RowFrag<DK>::kChunks; ++i) s[r].p[i] = make_float2(0.f, 0.f);
}

template <int DK, int R>
__device__ __forceinline__ void store_rows(const RowFrag<DK> (&s)[R], float* __restrict__ row0, int e) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int i = 0; i < RowFrag<DK>::kChunks; ++i)
            __stcs(reinterpret_cast<float4*>(row0 + (size_t)r * DK + 4 * chunk_of(i, e)),
                   make_float4(s[r].p[2 * i].x, s[r].p[2 * i].y, s[r].p[2 * i + 1].x, s[r].p[2 * i + 1].y));
}

}  // namespace gdn
