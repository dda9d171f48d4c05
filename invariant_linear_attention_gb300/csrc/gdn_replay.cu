// gdn_replay.cu -- chunk-order-replaying prefill and decode for the gated
// delta rule (the alternative to running the recurrent kernel everywhere).
//
// Both kernels evaluate every term through the device functions in the first
// section below, with the same operands in the same order, which is what
// makes decode bit-identical to prefill.  The state S0 lives in registers in
// the row layout of gdn_step.cuh (its dk contractions are rows_dot); the
// chunk's rows, the coefficient rows and the per-row quantities live in
// shared memory.
//
// Prefill: one CTA per (sequence, head) walks its chunks.  Per chunk:
//   A  q^, k^ of the new rows (eight vectors per warp at a time), g, b, and v;
//   B  the cumulative log-decay gam (one thread, in order);
//   C  S0 k^_j and S0 q^_j (two rows at a time) -> x_j = v_j - Gam_j S0 k^_j,
//      o0_j = Gam_j S0 q^_j;
//   D  the coefficient rows c_j, p_j (one task per (row j, four columns i));
//   E  d_j by forward substitution in 16-row sub-blocks: the completed
//      sub-blocks' parts by all threads, then the in-block chains, rows in order;
//   F  o_j (four columns per thread);
//   G  at the chunk end, S0 <- Gam_last S0 + sum_i exp(gam_last - gam_i) d_i k^_i^T.
// Decode: one CTA per (sequence, head) does the same for its one new row j,
// reading S0 and rows 0 .. j-1 from the replay state (16-byte async copies).
#include <algorithm>

#include "../../include/gdn_replay.h"
#include "gdn_host.h"
#include "gdn_step.cuh"

namespace gdn {

gdn_status launch_unit_sched(const int32_t* cu, int N, int T, int HV, int nslices, int32_t* work, unsigned* err,
                             cudaStream_t stream);

namespace {

constexpr int kRC = GDN_REPLAY_CHUNK;
constexpr int kLdD = 128;  // row stride (floats) of the d / x / o0 tiles: dv <= 128

// ---------------------------------------------------------------- shared arithmetic
// <a, b> over dk: four interleaved fma chains over the float4s in increasing
// order, then (s0 + s1) + (s2 + s3).  a, b 16-byte aligned.
template <int DK>
__device__ __forceinline__ float vdot(const float* __restrict__ a, const float* __restrict__ b) {
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int c = 0; c < DK / 4; ++c) {
        const float4 x = *reinterpret_cast<const float4*>(a + 4 * c);
        const float4 y = *reinterpret_cast<const float4*>(b + 4 * c);
        s0 = __fmaf_rn(x.x, y.x, s0);
        s1 = __fmaf_rn(x.y, y.y, s1);
        s2 = __fmaf_rn(x.z, y.z, s2);
        s3 = __fmaf_rn(x.w, y.w, s3);
    }
    return __fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3));
}
// gam_j = g_0 + ... + g_j, accumulated in order from the chunk start
__device__ __forceinline__ float next_gamma(float prev, float g, int j) { return j == 0 ? g : __fadd_rn(prev, g); }
__device__ __forceinline__ float decay(float gj, float gi) { return expf(__fsub_rn(gj, gi)); }
__device__ __forceinline__ float coef(float gj, float gi, float dot) { return __fmul_rn(decay(gj, gi), dot); }
__device__ __forceinline__ float resid(float v, float Gam, float sk) { return __fsub_rn(v, __fmul_rn(Gam, sk)); }
__device__ __forceinline__ float out0(float Gam, float sq) { return __fmul_rn(Gam, sq); }
constexpr int kSub = 16;  // rows per sub-block of the forward substitution
#ifndef GDN_REPLAY_TI
#define GDN_REPLAY_TI 4
#endif
constexpr int kTI = GDN_REPLAY_TI;  // columns per coefficient task

// acc + sum_{i0<=i<i1} c_i D[i][r]: one fma chain in increasing i.  The operands
// are fetched eight at a time ahead of their fmas (shared-memory latency
// overlaps the chain); the chain itself is unchanged.
__device__ __forceinline__ float chain(float acc, const float* c, const float* D, int r, int i0, int i1) {
    int i = i0;
    for (; i + 8 <= i1; i += 8) {
        float cv[8], dv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            cv[u] = c[i + u];
            dv[u] = D[(i + u) * kLdD + r];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) acc = __fmaf_rn(cv[u], dv[u], acc);
    }
    for (; i < i1; ++i) acc = __fmaf_rn(c[i], D[i * kLdD + r], acc);
    return acc;
}
// The same chain for the four columns r .. r+3 at once (r a multiple of 4):
// four independent chains, each exactly chain()'s sequence of operations.
__device__ __forceinline__ float4 chain4(float4 acc, const float* c, const float* D, int r, int i0, int i1) {
    for (int i = i0; i < i1; ++i) {
        const float ci = c[i];
        const float4 d = *reinterpret_cast<const float4*>(D + i * kLdD + r);
        acc.x = __fmaf_rn(ci, d.x, acc.x);
        acc.y = __fmaf_rn(ci, d.y, acc.y);
        acc.z = __fmaf_rn(ci, d.z, acc.z);
        acc.w = __fmaf_rn(ci, d.w, acc.w);
    }
    return acc;
}
// T_j[r] = sum_{i<j} c_i d_i[r], as a left fold over the 16-row sub-blocks of
// per-block chains: ((P_0 + P_1) + P_2) + ..., P_b = chain over i in
// [16b, min(16b + 16, j)) from 0.  (Prefill computes the completed blocks'
// P_b in parallel; decode folds them in the same order.)
__device__ __forceinline__ float delta_sum(const float* c, const float* D, int r, int j) {
    float T = chain(0.f, c, D, r, 0, min(kSub, j));
    for (int b = 1; b <= j / kSub; ++b) T = __fadd_rn(T, chain(0.f, c, D, r, b * kSub, min(b * kSub + kSub, j)));
    return T;
}
// d_j[r] = b_j (x_j[r] - T_j[r])
__device__ __forceinline__ float delta_row(float b, float x, const float* c, const float* D, int r, int j) {
    return __fmul_rn(b, __fsub_rn(x, delta_sum(c, D, r, j)));
}
// o_j[r] = o0_j[r] + sum_{i<=j} p_i d_i[r]: one chain in increasing i
__device__ __forceinline__ float out_row(float o0, const float* p, const float* D, int r, int j) {
    return chain(o0, p, D, r, 0, j + 1);
}

// NV contractions S_r . x_v at once, each with exactly rows_dot's operations
// (gdn_step.cuh: per-lane packed chains over the lane's chunks in order, the
// sets in order, (x + y) + (z + w), the lane butterfly); interleaving only
// gives the scheduler independent work.  All 32 lanes of the warp call it.
template <int DK, int R, int NV>
__device__ __forceinline__ void rows_dot_multi(const RowFrag<DK> (&S)[R], const float* const (&x)[NV], int e,
                                               float (&u)[NV][R]) {
    constexpr int NC = RowFrag<DK>::kChunks, NS = RowFrag<DK>::kSets;
    float2 xy[NV][R][NS], zw[NV][R][NS];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < NS; ++j) xy[v][r][j] = zw[v][r][j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NC; ++i) {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const float4 k4 = *reinterpret_cast<const float4*>(x[v] + 4 * chunk_of(i, e));
#pragma unroll
            for (int r = 0; r < R; ++r) {
#ifdef GDN_STEP_SCALAR
                float2& A = xy[v][r][i % NS];
                float2& B = zw[v][r][i % NS];
                A.x = __fmaf_rn(S[r].p[2 * i].x, k4.x, A.x);
                A.y = __fmaf_rn(S[r].p[2 * i].y, k4.y, A.y);
                B.x = __fmaf_rn(S[r].p[2 * i + 1].x, k4.z, B.x);
                B.y = __fmaf_rn(S[r].p[2 * i + 1].y, k4.w, B.y);
#else
                xy[v][r][i % NS] = __ffma2_rn(S[r].p[2 * i], lo2(k4), xy[v][r][i % NS]);
                zw[v][r][i % NS] = __ffma2_rn(S[r].p[2 * i + 1], hi2(k4), zw[v][r][i % NS]);
#endif
            }
        }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) u[v][r] = lanes_reduce(lane_partial<NS>(xy[v][r], zw[v][r]));
}

// Four outputs (columns r .. r+3) rounded to the output type.
__device__ __forceinline__ void st4_out(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4_out(__nv_bfloat16* p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}
// 16 bytes of input widened to fp32 (8 bf16 or 4 fp32)
__device__ __forceinline__ int widen16(const __nv_bfloat16* p, float* out) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    return 8;
}
__device__ __forceinline__ int widen16(const float* p, float* out) {
    const float4 f = *reinterpret_cast<const float4*>(p);
    out[0] = f.x, out[1] = f.y, out[2] = f.z, out[3] = f.w;
    return 4;
}

// Chunk end, for the R rows a thread holds: every element is first scaled by
// Gam_last, then gets fma(w_i, k^_i, .) for i in increasing order with
// w_i = ew_i * d_i[row] (ew_i = exp(gam_last - gam_i)).  No shuffles.
template <int DK, int R>
__device__ __forceinline__ void rows_chunk_update(RowFrag<DK> (&S)[R], const float* kn, int ldk, const float* D,
                                                  const float* ew, float gam_last_exp, int row0, int e) {
    constexpr int NC = RowFrag<DK>::kChunks;
    const float2 g2 = make_float2(gam_last_exp, gam_last_exp);
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < 2 * NC; ++c) S[r].p[c] = __fmul2_rn(g2, S[r].p[c]);
    for (int i = 0; i < kRC; ++i) {
        float2 w2[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float w = __fmul_rn(ew[i], D[i * kLdD + row0 + r]);
            w2[r] = make_float2(w, w);
        }
        const float* ki = kn + i * ldk;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const float4 k4 = *reinterpret_cast<const float4*>(ki + 4 * chunk_of(c, e));
#pragma unroll
            for (int r = 0; r < R; ++r) {
                S[r].p[2 * c] = __ffma2_rn(w2[r], lo2(k4), S[r].p[2 * c]);
                S[r].p[2 * c + 1] = __ffma2_rn(w2[r], hi2(k4), S[r].p[2 * c + 1]);
            }
        }
    }
}

// ---------------------------------------------------------------- parameters
struct ReplayParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu;
    const int32_t* seq_pos;
    float* rs;
    const int32_t* idx;
    void* out;
    const int32_t* work;
    int num_slots, N, T, HK, HV, G, dv, use_norm;
    long long blk;  // floats per (slot, head)
};

__host__ __device__ inline long long block_floats(int dk, int dv) {
    return (long long)dv * dk + (long long)kRC * (dk + dv + 1);
}

// ---------------------------------------------------------------- prefill
template <int DK>
struct PrefillSmem {
    float kn[kRC][DK + 4];  // padded rows: float4 reads of different rows hit different banks
    float qn[kRC][DK + 4];
    float X[kRC][kLdD];
    float Q0[kRC][kLdD];
    float D[kRC][kLdD];
    float cm[kRC][kRC + 1];
    float pm[kRC][kRC + 1];
    float Tf[kSub][kLdD];  // the completed sub-blocks' folded parts of the current sub-block's rows
    float gam[kRC], Gam[kRC], beta[kRC], graw[kRC], ew[kRC];
};

template <typename Tin, int DK>
__global__ void __launch_bounds__(kThreadsPer128Rows, 1) replay_prefill_kernel(const ReplayParams p) {
    constexpr int R = kRowsPerThread;
    extern __shared__ unsigned char smem_raw[];
    PrefillSmem<DK>& sm =
        *reinterpret_cast<PrefillSmem<DK>*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5, nt = blockDim.x;
    const int e = tid % kLanesPerRow, grp = tid / kLanesPerRow;
    const int dv = p.dv;
    const int row = grp * R;
    const bool active = row < dv;
    const int unit = p.work[blockIdx.x];
    const int h = unit % p.HV, n = unit / p.HV, hk = h / p.G;
    const int bos = min(max(p.cu[n], 0), p.T), eos = min(max(p.cu[n + 1], bos), p.T);
    if (eos == bos) return;
    const int slot = p.idx ? p.idx[n] : n;
    if (slot < 0 || slot >= p.num_slots) return;
    float* gS = p.rs + ((long long)slot * p.HV + h) * p.blk;
    float* gK = gS + (size_t)dv * DK;
    float* gD = gK + (size_t)kRC * DK;
    float* gG = gD + (size_t)kRC * dv;
    const int pos0 = (p.seq_pos ? max(p.seq_pos[n], 0) : 0) % kRC;
    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    Tin* out = static_cast<Tin*>(p.out);

    RowFrag<DK> S[R];
    if (active) load_rows<DK, R>(S, gS + (size_t)row * DK, e);
    else zero_rows<DK, R>(S);
    // rows 0 .. pos0-1 of the open chunk
    for (int x = tid; x < pos0 * (DK / 4); x += nt) {
        const int i = x / (DK / 4), c = x % (DK / 4);
        *reinterpret_cast<float4*>(&sm.kn[i][4 * c]) = *reinterpret_cast<const float4*>(gK + (size_t)i * DK + 4 * c);
    }
    for (int x = tid; x < pos0 * dv; x += nt) sm.D[x / dv][x % dv] = gD[x];
    for (int i = tid; i < pos0; i += nt) sm.gam[i] = gG[i];

    int j0 = pos0;
    bool completed = false;
    for (int t = bos; t < eos;) {
        const int nj = min(kRC - j0, eos - t);
        __syncthreads();  // the previous chunk's readers are done; the cached rows are in
        // A: q^, k^, g, b and v of the new rows j0 .. j0+nj-1.  Eight vectors per
        // warp are normalised together (their loads are in flight at once); v
        // goes into the x tile with one coalesced pass.
        for (int w0 = warp; w0 < 2 * nj; w0 += 8 * nwarps) {
            const Tin* src[8];
            float* dst[8];
            int nv = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int w = w0 + u * nwarps, jj = w >> 1;
                const bool ok = w < 2 * nj;
                nv += ok;
                const size_t off = ((size_t)(t + (ok ? jj : 0)) * p.HK + hk) * DK;
                src[u] = (w & 1) ? k + off : q + off;
                dst[u] = ok ? ((w & 1) ? &sm.kn[j0 + jj][0] : &sm.qn[j0 + jj][0]) : &sm.qn[j0][0];
            }
            l2norm_warp_multi<DK, 8>(src, dst, nv, lane, p.use_norm != 0);
        }
        {
            constexpr int VN = 16 / sizeof(Tin);
            const int nvec = dv / VN;
            for (int x0 = tid; x0 < nj * nvec; x0 += 4 * nt) {
                float buf[4][8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int x = x0 + u * nt;
                    if (x < nj * nvec)
                        widen16(v + ((size_t)(t + x / nvec) * p.HV + h) * dv + (x % nvec) * VN, buf[u]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int x = x0 + u * nt;
                    if (x < nj * nvec) {
#pragma unroll
                        for (int m = 0; m < VN; ++m) sm.X[j0 + x / nvec][(x % nvec) * VN + m] = buf[u][m];
                    }
                }
            }
        }
        for (int i = tid; i < nj; i += nt) {  // nt can be 32 (dv = 16)
            const size_t gi = (size_t)(t + i) * p.HV + h;
            sm.graw[j0 + i] = p.g[gi];
            sm.beta[j0 + i] = p.beta[gi];
        }
        __syncthreads();
        // B
        if (tid == 0) {
            float gm = j0 > 0 ? sm.gam[j0 - 1] : 0.f;
            for (int j = j0; j < j0 + nj; ++j) {
                gm = next_gamma(gm, sm.graw[j], j);
                sm.gam[j] = gm;
                sm.Gam[j] = expf(gm);
            }
        }
        __syncthreads();
        // C: two rows j at a time (four contractions interleaved)
        for (int j = j0; j < j0 + nj; j += 2) {
            const int j2 = min(j + 1, j0 + nj - 1);
            const float* xs[4] = {&sm.kn[j][0], &sm.qn[j][0], &sm.kn[j2][0], &sm.qn[j2][0]};
            float u[4][R];
            rows_dot_multi<DK, R, 4>(S, xs, e, u);
            if (active && e == 0) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int jj = h2 ? j2 : j;
                    if (h2 && j2 == j) break;
                    const float Gj = sm.Gam[jj];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        sm.X[jj][row + r] = resid(sm.X[jj][row + r], Gj, u[2 * h2][r]);
                        sm.Q0[jj][row + r] = out0(Gj, u[2 * h2 + 1][r]);
                    }
                }
            }
        }
        // D: coefficient rows, one task per (new row j, group of kTI columns i):
        // the dots of k^_j and q^_j with k^_i .. k^_{i+kTI-1}, each element with
        // vdot's chains and final sum
        for (int x = tid; x < nj * (kRC / kTI); x += nt) {
            const int j = j0 + x % nj, i0 = kTI * (x / nj);
            if (i0 > j) continue;
            float sk[kTI][4], sq[kTI][4];
#pragma unroll
            for (int m = 0; m < kTI; ++m)
#pragma unroll
                for (int c = 0; c < 4; ++c) sk[m][c] = sq[m][c] = 0.f;
#pragma unroll 4
            for (int c = 0; c < DK / 4; ++c) {
                const float4 a = *reinterpret_cast<const float4*>(&sm.kn[j][4 * c]);
                const float4 b = *reinterpret_cast<const float4*>(&sm.qn[j][4 * c]);
#pragma unroll
                for (int m = 0; m < kTI; ++m) {
                    const float4 y = *reinterpret_cast<const float4*>(&sm.kn[i0 + m][4 * c]);
                    sk[m][0] = __fmaf_rn(a.x, y.x, sk[m][0]);
                    sk[m][1] = __fmaf_rn(a.y, y.y, sk[m][1]);
                    sk[m][2] = __fmaf_rn(a.z, y.z, sk[m][2]);
                    sk[m][3] = __fmaf_rn(a.w, y.w, sk[m][3]);
                    sq[m][0] = __fmaf_rn(b.x, y.x, sq[m][0]);
                    sq[m][1] = __fmaf_rn(b.y, y.y, sq[m][1]);
                    sq[m][2] = __fmaf_rn(b.z, y.z, sq[m][2]);
                    sq[m][3] = __fmaf_rn(b.w, y.w, sq[m][3]);
                }
            }
            const float gj = sm.gam[j];
#pragma unroll
            for (int m = 0; m < kTI; ++m) {
                const int i = i0 + m;
                if (i <= j) {
                    const float gi = sm.gam[i];
                    if (i < j)
                        sm.cm[j][i] = coef(gj, gi, __fadd_rn(__fadd_rn(sk[m][0], sk[m][1]), __fadd_rn(sk[m][2], sk[m][3])));
                    sm.pm[j][i] = coef(gj, gi, __fadd_rn(__fadd_rn(sq[m][0], sq[m][1]), __fadd_rn(sq[m][2], sq[m][3])));
                }
            }
        }
        __syncthreads();
        // E: d by sub-blocks of 16 rows.  E1: the completed sub-blocks' parts of
        // the block's new rows, folded in order (4 columns per thread, all
        // threads); E2: the in-block chains, one thread per column, rows in order.
        for (int B = j0 / kSub; B * kSub < j0 + nj; ++B) {
            const int jb = max(j0, B * kSub), je = min(j0 + nj, B * kSub + kSub);
            if (B > 0) {
                const int nq = dv / 4;
                for (int x = tid; x < (je - jb) * nq; x += nt) {
                    const int j = jb + x / nq, r = 4 * (x % nq);
                    float4 T = chain4(make_float4(0.f, 0.f, 0.f, 0.f), &sm.cm[j][0], &sm.D[0][0], r, 0, kSub);
                    for (int b = 1; b < B; ++b) {
                        const float4 P =
                            chain4(make_float4(0.f, 0.f, 0.f, 0.f), &sm.cm[j][0], &sm.D[0][0], r, b * kSub, b * kSub + kSub);
                        T.x = __fadd_rn(T.x, P.x);
                        T.y = __fadd_rn(T.y, P.y);
                        T.z = __fadd_rn(T.z, P.z);
                        T.w = __fadd_rn(T.w, P.w);
                    }
                    *reinterpret_cast<float4*>(&sm.Tf[j - B * kSub][r]) = T;
                }
                __syncthreads();
            }
            if (tid < dv) {
                for (int j = jb; j < je; ++j) {
                    float T = chain(0.f, &sm.cm[j][0], &sm.D[0][0], tid, B * kSub, j);
                    if (B > 0) T = __fadd_rn(sm.Tf[j - B * kSub][tid], T);
                    sm.D[j][tid] = __fmul_rn(sm.beta[j], __fsub_rn(sm.X[j][tid], T));
                }
            }
            __syncthreads();
        }
        // F: outputs, four columns per thread
        {
            const int nq = dv / 4;
            for (int x = tid; x < nj * nq; x += nt) {
                const int jj = x / nq, r = 4 * (x % nq), j = j0 + jj;
                const float4 o = chain4(*reinterpret_cast<const float4*>(&sm.Q0[j][r]), &sm.pm[j][0], &sm.D[0][0], r, 0,
                                        j + 1);
                st4_out(out + ((size_t)(t + jj) * p.HV + h) * dv + r, o);
            }
        }
        t += nj;
        if (j0 + nj == kRC) {
            // G
            for (int i = tid; i < kRC; i += nt) sm.ew[i] = decay(sm.gam[kRC - 1], sm.gam[i]);
            __syncthreads();
            if (active) rows_chunk_update<DK, R>(S, &sm.kn[0][0], DK + 4, &sm.D[0][0], sm.ew, sm.Gam[kRC - 1], row, e);
            j0 = 0;
            completed = true;
        } else {
            j0 += nj;
        }
    }
    __syncthreads();
    // write back the chunk-start state (when a chunk ended) and the open chunk's new rows
    if (completed && active) store_rows<DK, R>(S, gS + (size_t)row * DK, e);
    const int r0 = completed ? 0 : pos0;
    for (int x = tid; x < (j0 - r0) * (DK / 4); x += nt) {
        const int i = r0 + x / (DK / 4), c = x % (DK / 4);
        *reinterpret_cast<float4*>(gK + (size_t)i * DK + 4 * c) = *reinterpret_cast<const float4*>(&sm.kn[i][4 * c]);
    }
    for (int x = tid; x < (j0 - r0) * dv; x += nt) {
        const int i = r0 + x / dv, r = x % dv;
        gD[(size_t)i * dv + r] = sm.D[i][r];
    }
    for (int i = r0 + tid; i < j0; i += nt) gG[i] = sm.gam[i];
}

// ---------------------------------------------------------------- decode
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <int DK>
struct DecodeSmem {
    float kn[kRC][DK + 4];
    float D[kRC][kLdD];
    float qn[DK];
    float c[kRC], pp[kRC], gam[kRC], ew[kRC];
    float X[kLdD], Q0[kLdD];
    float Gj, bj;
};

template <typename Tin, int DK>
__global__ void __launch_bounds__(kThreadsPer128Rows, 2) replay_decode_kernel(const ReplayParams p) {
    constexpr int R = kRowsPerThread;
    extern __shared__ unsigned char smem_raw[];
    DecodeSmem<DK>& sm =
        *reinterpret_cast<DecodeSmem<DK>*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5, nt = blockDim.x;
    const int e = tid % kLanesPerRow, grp = tid / kLanesPerRow;
    const int dv = p.dv;
    const int row = grp * R;
    const bool active = row < dv;
    const int b = blockIdx.x / p.HV, h = blockIdx.x % p.HV, hk = h / p.G;
    const int slot = p.idx ? p.idx[b] : b;
    if (slot < 0 || slot >= p.num_slots) return;
    float* gS = p.rs + ((long long)slot * p.HV + h) * p.blk;
    float* gK = gS + (size_t)dv * DK;
    float* gD = gK + (size_t)kRC * DK;
    float* gG = gD + (size_t)kRC * dv;
    const int j = max(p.seq_pos[b], 0) % kRC;
    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);

    // the open chunk's cached rows: 16-byte asynchronous copies, all in flight at once
    for (int x = tid; x < j * (DK / 4); x += nt) {
        const int i = x / (DK / 4), c = x % (DK / 4);
        cp_async16(&sm.kn[i][4 * c], gK + (size_t)i * DK + 4 * c);
    }
    for (int x = tid; x < j * (dv / 4); x += nt) {
        const int i = x / (dv / 4), c = x % (dv / 4);
        cp_async16(&sm.D[i][4 * c], gD + (size_t)i * dv + 4 * c);
    }
    for (int x = tid; x < (j + 3) / 4; x += nt) cp_async16(&sm.gam[4 * x], gG + 4 * x);
    cp_async_commit();
    const size_t off = ((size_t)b * p.HK + hk) * DK;
    if (warp == 0) l2norm_warp<DK>(q + off, sm.qn, lane, p.use_norm != 0);
    if (warp == (nwarps > 1 ? 1 : 0)) l2norm_warp<DK>(k + off, &sm.kn[j][0], lane, p.use_norm != 0);
    float sk[R], sq[R];
    {
        // S0 is needed twice: here for S0 k^ and S0 q^, and at a chunk end (one
        // step in 64), where it is read again rather than kept live throughout
        RowFrag<DK> S[R];
        if (active) load_rows<DK, R>(S, gS + (size_t)row * DK, e);
        else zero_rows<DK, R>(S);
        cp_async_wait_all();
        __syncthreads();
        rows_dot<DK, R>(S, &sm.kn[j][0], e, sk);
        rows_dot<DK, R>(S, sm.qn, e, sq);
    }
    if (tid == 0) {
        const size_t gi = (size_t)b * p.HV + h;
        const float gm = next_gamma(j > 0 ? sm.gam[j - 1] : 0.f, p.g[gi], j);
        sm.gam[j] = gm;
        sm.Gj = expf(gm);
        sm.bj = p.beta[gi];
    }
    __syncthreads();
    if (active && e == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float vv = ld_in(v + ((size_t)b * p.HV + h) * dv + row + r);
            sm.X[row + r] = resid(vv, sm.Gj, sk[r]);
            sm.Q0[row + r] = out0(sm.Gj, sq[r]);
        }
    }
    const float gj = sm.gam[j];
    for (int i = tid; i <= j; i += nt) {
        const float gi = sm.gam[i];
        if (i < j) sm.c[i] = coef(gj, gi, vdot<DK>(&sm.kn[j][0], &sm.kn[i][0]));
        sm.pp[i] = coef(gj, gi, vdot<DK>(sm.qn, &sm.kn[i][0]));
    }
    __syncthreads();
    if (tid < dv) sm.D[j][tid] = delta_row(sm.bj, sm.X[tid], sm.c, &sm.D[0][0], tid, j);
    __syncthreads();
    if (tid < dv)
        st_in(static_cast<Tin*>(p.out) + ((size_t)b * p.HV + h) * dv + tid,
              out_row(sm.Q0[tid], sm.pp, &sm.D[0][0], tid, j));
    // the new row of the open chunk
    for (int c = tid; c < DK / 4; c += nt)
        *reinterpret_cast<float4*>(gK + (size_t)j * DK + 4 * c) = *reinterpret_cast<const float4*>(&sm.kn[j][4 * c]);
    if (tid < dv) gD[(size_t)j * dv + tid] = sm.D[j][tid];
    if (tid == 0) gG[j] = gj;
    if (j == kRC - 1) {
        for (int i = tid; i < kRC; i += nt) sm.ew[i] = decay(gj, sm.gam[i]);
        __syncthreads();
        if (active) {
            RowFrag<DK> S[R];
            load_rows<DK, R>(S, gS + (size_t)row * DK, e);
            rows_chunk_update<DK, R>(S, &sm.kn[0][0], DK + 4, &sm.D[0][0], sm.ew, sm.Gj, row, e);
            store_rows<DK, R>(S, gS + (size_t)row * DK, e);
        }
    }
}

// ---------------------------------------------------------------- launch
template <typename Tin, int DK>
gdn_status launch_prefill_t(const ReplayParams& p, int units, int nt, cudaStream_t s) {
    const size_t smem = sizeof(PrefillSmem<DK>) + 16;
    auto kern = replay_prefill_kernel<Tin, DK>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    kern<<<units, nt, smem, s>>>(p);
    return launch_status();
}

template <typename Tin, int DK>
gdn_status launch_decode_t(const ReplayParams& p, int units, int nt, cudaStream_t s) {
    const size_t smem = sizeof(DecodeSmem<DK>) + 16;
    auto kern = replay_decode_kernel<Tin, DK>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    kern<<<units, nt, smem, s>>>(p);
    return launch_status();
}

template <bool kPrefill, typename Tin>
gdn_status launch_dk(int dk, const ReplayParams& p, int units, int nt, cudaStream_t s) {
    switch (dk) {
        case 16: return kPrefill ? launch_prefill_t<Tin, 16>(p, units, nt, s) : launch_decode_t<Tin, 16>(p, units, nt, s);
        case 32: return kPrefill ? launch_prefill_t<Tin, 32>(p, units, nt, s) : launch_decode_t<Tin, 32>(p, units, nt, s);
        case 64: return kPrefill ? launch_prefill_t<Tin, 64>(p, units, nt, s) : launch_decode_t<Tin, 64>(p, units, nt, s);
        case 128:
            return kPrefill ? launch_prefill_t<Tin, 128>(p, units, nt, s) : launch_decode_t<Tin, 128>(p, units, nt, s);
    }
    return GDN_ERR_UNSUPPORTED;
}

gdn_status check_replay(const gdn_shape* s, const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const float* rs, const int32_t* idx, int num_slots, const void* out) {
    gdn_status st = check_shape(s);
    if (st != GDN_OK) return st;
    if (!rs || num_slots < 0) return GDN_ERR_INVALID_ARG;
    if (!idx && num_slots < s->N) return GDN_ERR_INVALID_ARG;
    if (s->T_total > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
    if ((q && !aligned16(q)) || (k && !aligned16(k)) || (v && !aligned16(v)) || (out && !aligned16(out)) ||
        !aligned16(rs) || (g && !aligned4(g)) || (beta && !aligned4(beta)) || (idx && !aligned4(idx)))
        return GDN_ERR_INVALID_ARG;
    if (out && (out == q || out == k || out == v || out == rs)) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

ReplayParams make_params(const gdn_shape* s, const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const int32_t* cu, const int32_t* seq_pos, float* rs,
                         const int32_t* idx, int num_slots, void* out, const int32_t* work) {
    ReplayParams p;
    p.q = q, p.k = k, p.v = v, p.g = g, p.beta = beta, p.cu = cu, p.seq_pos = seq_pos, p.rs = rs, p.idx = idx;
    p.out = out, p.work = work, p.num_slots = num_slots, p.N = s->N, p.T = s->T_total, p.HK = s->HK;
    p.HV = s->HV, p.G = s->HV / s->HK, p.dv = s->dv, p.use_norm = s->use_qk_l2norm ? 1 : 0;
    p.blk = block_floats(s->dk, s->dv);
    return p;
}

}  // namespace
}  // namespace gdn

extern "C" size_t gdn_replay_block_floats(int dk, int dv) {
    using namespace gdn;
    if (!dim_ok(dk) || !dim_ok(dv)) return 0;
    return (size_t)block_floats(dk, dv);
}

extern "C" size_t gdn_replay_workspace_size(const gdn_shape* s) {
    using namespace gdn;
    if (check_shape(s) != GDN_OK) return 0;
    return kWsHeader + (((size_t)s->N * s->HV * sizeof(int32_t) + 255) & ~size_t(255));
}

extern "C" gdn_status gdn_replay_prefill(const gdn_shape* shape, const void* q, const void* k, const void* v,
                                         const float* g, const float* beta, const int32_t* cu_seqlens,
                                         const int32_t* seq_pos, float* replay_state, const int32_t* state_indices,
                                         int num_slots, void* out, void* workspace, size_t workspace_bytes,
                                         void* stream) {
    using namespace gdn;
    gdn_status st = check_replay(shape, q, k, v, g, beta, replay_state, state_indices, num_slots, out);
    if (st != GDN_OK) return st;
    if (!cu_seqlens || !aligned4(cu_seqlens) || (seq_pos && !aligned4(seq_pos))) return GDN_ERR_INVALID_ARG;
    if (shape->N == 0) return GDN_OK;
    if (!workspace || !aligned16(workspace) || workspace_bytes < gdn_replay_workspace_size(shape))
        return GDN_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    int32_t* work = reinterpret_cast<int32_t*>(ws + kWsHeader);
    st = launch_unit_sched(cu_seqlens, shape->N, shape->T_total, shape->HV, 1, work, reinterpret_cast<unsigned*>(ws),
                           s);
    if (st != GDN_OK) return st;
    const ReplayParams p = make_params(shape, q, k, v, g, beta, cu_seqlens, seq_pos, replay_state, state_indices,
                                       num_slots, out, work);
    const int nt = std::max(32, shape->dv * kLanesPerRow / kRowsPerThread);
    const int units = shape->N * shape->HV;
    return shape->dtype == GDN_BF16 ? launch_dk<true, __nv_bfloat16>(shape->dk, p, units, nt, s)
                                    : launch_dk<true, float>(shape->dk, p, units, nt, s);
}

extern "C" gdn_status gdn_replay_decode(const gdn_shape* shape, const void* q, const void* k, const void* v,
                                        const float* g, const float* beta, const int32_t* seq_pos,
                                        float* replay_state, const int32_t* state_indices, int num_slots, void* out,
                                        void* stream) {
    using namespace gdn;
    gdn_status st = check_replay(shape, q, k, v, g, beta, replay_state, state_indices, num_slots, out);
    if (st != GDN_OK) return st;
    if (shape->T_total != shape->N) return GDN_ERR_INVALID_ARG;
    if (!seq_pos || !aligned4(seq_pos)) return GDN_ERR_INVALID_ARG;
    if (shape->N == 0) return GDN_OK;
    const ReplayParams p = make_params(shape, q, k, v, g, beta, nullptr, seq_pos, replay_state, state_indices,
                                       num_slots, out, nullptr);
    const int nt = std::max(32, shape->dv * kLanesPerRow / kRowsPerThread);
    const long long units = (long long)shape->N * shape->HV;
    if (units >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return shape->dtype == GDN_BF16 ? launch_dk<false, __nv_bfloat16>(shape->dk, p, (int)units, nt, s)
                                    : launch_dk<false, float>(shape->dk, p, (int)units, nt, s);
}
