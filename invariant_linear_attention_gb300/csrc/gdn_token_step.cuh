// gdn_token_step.cuh -- the per-token state step of the recurrent prefill /
// trainer-forward kernel and of the decode-step kernel.
//
// Bit-invariance rests on this file: both kernels advance a state row with
// exactly these IEEE operations in exactly this order, so the bits of a row
// depend only on that row's own inputs.  Rows of S never interact in the
// gated delta rule (u_i = S_i . k^ and o_i = S_i . q^ involve row i only), so
// how rows are spread over warps and CTAs (the dv slice) and how a thread
// groups its rows for the cross-lane reduction are free; the lane -> dk
// mapping, the in-lane summation order and the cross-lane tree below are not.
//
// The recurrence (gated delta rule, recurrent form as in "Defending Against
// the Training-Inference Numeric Mismatch in RL (Especially Linear
// Attention)", section 3.2):
//     u = S k^,  w = b v - (a b) u,  S <- a S + w k^T,  o = S q^
// which equals S <- a S (I - b k^ k^T) + b v k^T with o read after the update.
//
// Layout.  A row group of L consecutive lanes holds R rows of S (4, or 2 or 1
// when a head is split over several CTAs): lane e of the group (e = lane % L)
// holds the float4 column chunks c = L*i + e, i = 0 .. NC-1 (NC = dk / (4 L)),
// of all R rows, so the k^/q^ chunks a group
// reads at one step are 16*L contiguous bytes of shared memory.  For the
// cross-lane reduction the rows form NG = R / RG slot groups of RG rows;
// within slot group g, slot j of lane e holds row g*RG + (j ^ own(e)),
// own(e) = e >> log2(L/RG).  With that order the reduction needs no selects:
// a reduce-scatter halves the slots at each level (keep slots [0, c/2), send
// [c/2, c) to the lane whose kept slots they are); after log2(RG) levels slot
// 0 holds row own(e) of the group, and the remaining levels are a butterfly
// over the lanes that own the same row (commutative adds: they end with the
// same bits).
//
// A dk contraction of a row is therefore, for any RG: one packed (even, odd)
// fma chain over the lane's columns 4c .. 4c+3 of chunks c in increasing i,
// as (x, y) then (z, w), starting from +0; then even + odd; then one add per
// lane stride L/2, L/4, ..., 1, each adding the partner lane's partial.  The
// owner lanes of a row compute w for it, and every lane gathers the RG values
// of w it needs with RG - 1 independent xor shuffles (one level of latency).  The
// prefill kernel uses RG = R (4, 2 or 1) and the decode kernel R = 4 in two
// groups of RG = 2; the per-row operations, and so the bits, are the same.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_step.cuh"

namespace gdn {
namespace ts {

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <int DK, int RG_ = 4, int R_ = 4>
struct Layout {
    static constexpr int L = DK >= 32 ? 8 : 4;  // lanes per row group
    static constexpr int R = R_;                // rows per thread (4, or 2 / 1 for a sliced head)
    static constexpr int RG = RG_;              // rows per slot group
    static constexpr int NG = R / RG;           // slot groups per thread
    static constexpr int NC = DK / (4 * L);     // float4 chunks per lane and row
    static constexpr int SH = ilog2(L / RG);    // own row = e >> SH
    static_assert(NC >= 1 && DK % (4 * L) == 0, "dk must be a multiple of 4 L");
    static_assert(RG <= L && R % RG == 0 && 32 % L == 0, "RG <= L, RG divides R, L divides the warp");
};

// Threads a CTA needs for `rows` rows of S at 4 rows per thread (at least one warp).
template <int DK>
__host__ __device__ constexpr int threads_for_rows(int rows) {
    return rows * Layout<DK>::L / 4 < 32 ? 32 : rows * Layout<DK>::L / 4;
}

// The rows a thread holds (room for 4; a thread with R rows uses slots 0 .. R-1):
// slot s = g * RG + j; chunk i of a slot is (x, y) = p[s][2i], (z, w) = p[s][2i + 1].
template <int DK>
struct Rows {
    float2 p[4][2 * Layout<DK>::NC];
};

// Where a thread sits: its lane in the row group, the row it owns within each
// slot group after a reduce-scatter, and its row group.
struct Place {
    int e, own, grp;
};

template <int DK, int RG>
__device__ __forceinline__ Place place_of(int tid) {
    using Y = Layout<DK, RG>;
    Place pl;
    pl.e = tid % Y::L;
    pl.own = pl.e >> Y::SH;
    pl.grp = tid / Y::L;
    return pl;
}

// Row (relative to the thread's first row) held in slot j of slot group g.
template <int DK, int RG>
__device__ __forceinline__ int row_of(int g, int j, int own) {
    return g * RG + (j ^ own);
}

__device__ __forceinline__ float2 lo2(const float4& v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(const float4& v) { return make_float2(v.z, v.w); }

// p[j] = lane partial of (row in slot j of group G) . x  (x: dk fp32 vector in shared memory).
template <int DK, int RG, int G>
__device__ __forceinline__ void dot_part(const Rows<DK>& s, const float* __restrict__ x, int e, float (&p)[RG]) {
    using Y = Layout<DK, RG>;
    float2 A[RG];
#pragma unroll
    for (int j = 0; j < RG; ++j) A[j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < Y::NC; ++i) {
        const float4 x4 = *reinterpret_cast<const float4*>(x + 4 * (Y::L * i + e));
#pragma unroll
        for (int j = 0; j < RG; ++j) {
            A[j] = __ffma2_rn(s.p[G * RG + j][2 * i], lo2(x4), A[j]);
            A[j] = __ffma2_rn(s.p[G * RG + j][2 * i + 1], hi2(x4), A[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < RG; ++j) p[j] = __fadd_rn(A[j].x, A[j].y);
}

// Cross-lane tree of the layout: returns the full contraction of the row the
// lane owns in this slot group (every owner lane ends with the same bits).
// All 32 lanes call it.
template <int DK, int RG>
__device__ __forceinline__ float reduce_scatter(float (&p)[RG]) {
    using Y = Layout<DK, RG>;
#pragma unroll
    for (int c = RG; c > 1; c >>= 1) {
        const int stride = (Y::L / RG) * (c / 2);
#pragma unroll
        for (int j = 0; j < c / 2; ++j) p[j] = __fadd_rn(p[j], __shfl_xor_sync(kFull, p[j + c / 2], stride));
    }
#pragma unroll
    for (int stride = Y::L / RG / 2; stride >= 1; stride >>= 1)
        p[0] = __fadd_rn(p[0], __shfl_xor_sync(kFull, p[0], stride));
    return p[0];
}

// w[j] for every slot j of a group, from the owner lanes' values, each as the
// pair (w, w) the packed update multiplies by: slot j holds row j ^ own(e),
// owned by lane e ^ (j << SH) of the same row group, so slot 0 is the lane's
// own value and the others take RG - 1 independent xor shuffles.
template <int DK, int RG>
__device__ __forceinline__ void gather_rows(float mine, float2 (&w)[RG]) {
    using Y = Layout<DK, RG>;
    w[0] = make_float2(mine, mine);
#pragma unroll
    for (int j = 1; j < RG; ++j) {
        const float x = __shfl_xor_sync(kFull, mine, j << Y::SH);
        w[j] = make_float2(x, x);
    }
}

// w = b (v - a u), evaluated as fma(-(a b), u, b v): ab = a * b is the token's
// and bv = b * v the row's, both known before u, so one rounding step is left
// on the recurrence's critical path.
__device__ __forceinline__ float delta_w(float ab, float bv, float u) { return __fmaf_rn(-ab, u, bv); }

// For every slot j of group G: S <- a S + w[j] k^T (per element fma(w, k_c, a * S_c)),
// and p[j] = lane partial of the updated row . q.
template <int DK, int RG, int G>
__device__ __forceinline__ void update_part(Rows<DK>& s, const float* __restrict__ k, const float* __restrict__ q,
                                            int e, float2 a2, const float2 (&w)[RG], float (&p)[RG]) {
    using Y = Layout<DK, RG>;
    float2 A[RG];
#pragma unroll
    for (int j = 0; j < RG; ++j) A[j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < Y::NC; ++i) {
        const float4 k4 = *reinterpret_cast<const float4*>(k + 4 * (Y::L * i + e));
        const float4 q4 = *reinterpret_cast<const float4*>(q + 4 * (Y::L * i + e));
#pragma unroll
        for (int j = 0; j < RG; ++j) {
            const float2 w2 = w[j];
            float2& Sxy = s.p[G * RG + j][2 * i];
            float2& Szw = s.p[G * RG + j][2 * i + 1];
            Sxy = __ffma2_rn(w2, lo2(k4), __fmul2_rn(a2, Sxy));
            Szw = __ffma2_rn(w2, hi2(k4), __fmul2_rn(a2, Szw));
            A[j] = __ffma2_rn(Sxy, lo2(q4), A[j]);
            A[j] = __ffma2_rn(Szw, hi2(q4), A[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < RG; ++j) p[j] = __fadd_rn(A[j].x, A[j].y);
}

// One whole token for the rows of a thread, grouped in slot groups of RG rows
// (the decode step): o[g] is the output of the row the lane owns in slot
// group g, v_own[g] its v.  All 32 lanes of the warp call it.
template <int DK, int RG>
__device__ __forceinline__ void token_step(Rows<DK>& s, const float* __restrict__ kn, const float* __restrict__ qn,
                                           const Place& pl, float a, float b,
                                           const float (&v_own)[Layout<DK, RG>::NG],
                                           float (&o)[Layout<DK, RG>::NG]) {
    static_assert(Layout<DK, RG>::NG == 2, "two slot groups");
    float p0[RG], p1[RG];
    float2 w0[RG], w1[RG];
    dot_part<DK, RG, 0>(s, kn, pl.e, p0);
    dot_part<DK, RG, 1>(s, kn, pl.e, p1);
    const float ab = __fmul_rn(a, b);
    const float u0 = reduce_scatter<DK, RG>(p0);
    const float u1 = reduce_scatter<DK, RG>(p1);
    gather_rows<DK, RG>(delta_w(ab, __fmul_rn(b, v_own[0]), u0), w0);
    gather_rows<DK, RG>(delta_w(ab, __fmul_rn(b, v_own[1]), u1), w1);
    update_part<DK, RG, 0>(s, kn, qn, pl.e, make_float2(a, a), w0, p0);
    update_part<DK, RG, 1>(s, kn, qn, pl.e, make_float2(a, a), w1, p1);
    o[0] = reduce_scatter<DK, RG>(p0);
    o[1] = reduce_scatter<DK, RG>(p1);
}

// Global <-> register transfer of a thread's rows.  rows points at the first
// row of the thread's group (row stride dk floats).  Every 32-byte sector is
// read or written whole by neighbouring lanes.
template <int DK, int RG, int R = 4>
__device__ __forceinline__ void load_rows(Rows<DK>& s, const float* __restrict__ rows, const Place& pl) {
    using Y = Layout<DK, RG, R>;
#pragma unroll
    for (int g = 0; g < Y::NG; ++g)
#pragma unroll
        for (int j = 0; j < RG; ++j)
#pragma unroll
            for (int i = 0; i < Y::NC; ++i) {
                const float4 v = __ldcs(reinterpret_cast<const float4*>(
                    rows + (size_t)row_of<DK, RG>(g, j, pl.own) * DK + 4 * (Y::L * i + pl.e)));
                s.p[g * RG + j][2 * i] = make_float2(v.x, v.y);
                s.p[g * RG + j][2 * i + 1] = make_float2(v.z, v.w);
            }
}

template <int DK>
__device__ __forceinline__ void zero_rows(Rows<DK>& s) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 2 * Layout<DK>::NC; ++i) s.p[j][i] = make_float2(0.f, 0.f);
}

template <int DK, int RG, int R = 4>
__device__ __forceinline__ void store_rows(const Rows<DK>& s, float* __restrict__ rows, const Place& pl) {
    using Y = Layout<DK, RG, R>;
#pragma unroll
    for (int g = 0; g < Y::NG; ++g)
#pragma unroll
        for (int j = 0; j < RG; ++j)
#pragma unroll
            for (int i = 0; i < Y::NC; ++i) {
                const float2 xy = s.p[g * RG + j][2 * i], zw = s.p[g * RG + j][2 * i + 1];
                __stcs(reinterpret_cast<float4*>(rows + (size_t)row_of<DK, RG>(g, j, pl.own) * DK +
                                                 4 * (Y::L * i + pl.e)),
                       make_float4(xy.x, xy.y, zw.x, zw.y));
            }
}

// True on the one lane per owned row that stores the row's output.
template <int DK, int RG>
__device__ __forceinline__ bool stores_row(const Place& pl) {
    return (pl.e & ((1 << Layout<DK, RG>::SH) - 1)) == 0;
}

}  // namespace ts
}  // namespace gdn
