// gdn_layer.cu -- the ops either side of the Gated DeltaNet recurrence: gate
// activations, short causal depthwise conv (prefill and decode update over a
// conv state cache), gated RMSNorm.  All of them stream from and to HBM with a
// handful of flops per byte, so the design is about access shape, not math:
// 16-byte vector loads and stores coalesced along the contiguous axis, enough
// independent loads per thread in flight, grids in multiples of the SM count.
//
// Invariance: each output element is produced by one thread with one fixed
// sequence of fp32 operations (explicit _rn intrinsics, no contraction left to
// the compiler) that depends only on its own row; the conv's per-element
// arithmetic is one function shared by the prefill and the decode kernels.
#include <cuda_bf16.h>

#include "../../include/gdn_layer.h"
#include "gdn_host.h"

namespace gdn {
namespace {

constexpr int kSMs = 152;

// ---------------------------------------------------------------- 16-byte vectors
template <typename T>
struct V16;
template <>
struct V16<float> {
    static constexpr int n = 4;
};
template <>
struct V16<__nv_bfloat16> {
    static constexpr int n = 8;
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t bf_pack(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void unpack(const uint4& u, float (&f)[8]) {
    f[0] = bf_lo(u.x), f[1] = bf_hi(u.x), f[2] = bf_lo(u.y), f[3] = bf_hi(u.y);
    f[4] = bf_lo(u.z), f[5] = bf_hi(u.z), f[6] = bf_lo(u.w), f[7] = bf_hi(u.w);
}
__device__ __forceinline__ void unpack(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x), f[1] = __uint_as_float(u.y), f[2] = __uint_as_float(u.z),
    f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 pack(const float (&f)[8]) {
    return make_uint4(bf_pack(f[0], f[1]), bf_pack(f[2], f[3]), bf_pack(f[4], f[5]), bf_pack(f[6], f[7]));
}
__device__ __forceinline__ uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}

__device__ __forceinline__ uint4 ld16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ uint4 ld16_stream(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void st16(void* p, const uint4& v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ void st16_stream(void* p, const uint4& v) { __stcs(reinterpret_cast<uint4*>(p), v); }

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------- activations
// The gates feed the recurrence's decay and mixing weights: accurate library
// exp / log1p and a correctly rounded divide.
__device__ __forceinline__ float sigmoid_f(float x) { return __fdiv_rn(1.f, __fadd_rn(1.f, expf(-x))); }
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }
// SiLU on the streaming paths (conv output, RMSNorm gate): x * (1 / (1 + e^-x))
// with the hardware exponential and the hardware approximate reciprocal, a
// few ulp (far below the bf16 rounding of the outputs) at a fraction of the
// instruction count, which these HBM-bound kernels would otherwise be limited
// by.  The reciprocal is the bare rcp.approx.ftz instruction: for x < -87 the
// exponential overflows to +inf and 1 / inf = 0, the limit SiLU has there.
// Deterministic, and one function for every kernel, so prefill and decode
// agree bit for bit.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float silu_fast(float x) { return __fmul_rn(x, rcp_approx(__fadd_rn(1.f, __expf(-x)))); }

// ---------------------------------------------------------------- gates
__device__ __forceinline__ void gate_one(float av, float bv, int h, const float* __restrict__ A_log,
                                         const float* __restrict__ dt_bias, float& g, float& beta) {
    const float x = dt_bias ? __fadd_rn(av, __ldg(dt_bias + h)) : av;
    g = __fmul_rn(-expf(__ldg(A_log + h)), softplus_f(x));
    beta = sigmoid_f(bv);
}

// Scalar form: any T * HV.
template <typename Tin>
__global__ void __launch_bounds__(256) gates_kernel(int64_t n, int HV, const Tin* __restrict__ a,
                                                    const Tin* __restrict__ b, const float* __restrict__ A_log,
                                                    const float* __restrict__ dt_bias, float* __restrict__ g,
                                                    float* __restrict__ beta) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        gate_one(to_f(a[i]), to_f(b[i]), (int)(i % HV), A_log, dt_bias, g[i], beta[i]);
}

// Vector form (HV % 8 == 0): a thread takes 8 consecutive elements of one
// token, 16-byte (bf16) or 2 x 16-byte (fp32) loads and 2 x 16-byte stores.
// The grid stride (in elements) is a multiple of HV, so a thread keeps the
// same 8 heads on every iteration: their -exp(A_log) and dt_bias are taken
// once, before the token loop.
template <typename Tin>
__global__ void __launch_bounds__(256) gates_kernel_v8(int64_t n8, int HV, const Tin* __restrict__ a,
                                                       const Tin* __restrict__ b, const float* __restrict__ A_log,
                                                       const float* __restrict__ dt_bias, float* __restrict__ g,
                                                       float* __restrict__ beta) {
    constexpr int VN = V16<Tin>::n;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t v0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (v0 >= n8) return;
    const int h0 = (int)((v0 * 8) % HV);
    float nA[8], dtb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        nA[e] = -expf(__ldg(A_log + h0 + e));
        dtb[e] = dt_bias ? __ldg(dt_bias + h0 + e) : 0.f;
    }
    for (int64_t v = v0; v < n8; v += stride) {
        const int64_t i = v * 8;
        float av[8], bv[8], go[8], bo[8];
#pragma unroll
        for (int j = 0; j < 8; j += VN) {
            float t[VN];
            unpack(ld16_stream(a + i + j), t);
#pragma unroll
            for (int e = 0; e < VN; ++e) av[j + e] = t[e];
            unpack(ld16_stream(b + i + j), t);
#pragma unroll
            for (int e = 0; e < VN; ++e) bv[j + e] = t[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float xg = dt_bias ? __fadd_rn(av[e], dtb[e]) : av[e];
            go[e] = __fmul_rn(nA[e], softplus_f(xg));
            bo[e] = sigmoid_f(bv[e]);
        }
#pragma unroll
        for (int j = 0; j < 8; j += 4) {
            const float ga[4] = {go[j], go[j + 1], go[j + 2], go[j + 3]};
            const float ba[4] = {bo[j], bo[j + 1], bo[j + 2], bo[j + 3]};
            st16_stream(g + i + j, pack(ga));
            st16_stream(beta + i + j, pack(ba));
        }
    }
}

// ---------------------------------------------------------------- gated RMSNorm
// A group of LPR lanes (a power of two, <= 32) owns one row; lane li of the
// group holds the row's 16-byte chunks li, li + LPR, ... (NC of them at most).
// A warp handles UR row groups per iteration and issues all their o and z
// loads before any arithmetic, so 2 * UR * NC 16-byte loads per lane are in
// flight at once.  y may alias o: every element of a row is loaded before the
// row's first store, by the same lane.
template <typename T, int NC, int UR>
__global__ void __launch_bounds__(256) rmsnorm_kernel(int64_t rows, int d, int lpr, const T* o,
                                                      const T* __restrict__ z, const float* __restrict__ w,
                                                      float eps, T* y) {
    constexpr int VN = V16<T>::n;
    const int lane = threadIdx.x & 31;
    const int li = lane & (lpr - 1);
    const int rpw = 32 / lpr;  // rows per warp and row group
    const int chunks = d / VN;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const bool gate = z != nullptr;
    for (int64_t base = warp * rpw * UR; base < rows; base += nwarps * rpw * UR) {
        uint4 xo[UR][NC], xz[UR][NC];
#pragma unroll
        for (int u = 0; u < UR; ++u) {
            const int64_t row = base + (int64_t)u * rpw + lane / lpr;
#pragma unroll
            for (int j = 0; j < NC; ++j) {
                const int c = li + j * lpr;
                const bool ok = row < rows && c < chunks;
                xo[u][j] = ok ? ld16_stream(o + row * d + (int64_t)c * VN) : make_uint4(0u, 0u, 0u, 0u);
                xz[u][j] = ok && gate ? ld16_stream(z + row * d + (int64_t)c * VN) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < UR; ++u) {
            const int64_t row = base + (int64_t)u * rpw + lane / lpr;
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < NC; ++j) {
                float x[VN];
                unpack(xo[u][j], x);
#pragma unroll
                for (int e = 0; e < VN; ++e) ss = __fmaf_rn(x[e], x[e], ss);
            }
            for (int off = 1; off < lpr; off <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
            const float r = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)d), eps));
#pragma unroll
            for (int j = 0; j < NC; ++j) {
                const int c = li + j * lpr;
                if (row < rows && c < chunks) {
                    float x[VN], gz[VN], wv[VN], out[VN];
                    unpack(xo[u][j], x);
                    unpack(xz[u][j], gz);
                    const float4* wp = reinterpret_cast<const float4*>(w + (int64_t)c * VN);
#pragma unroll
                    for (int e = 0; e < VN; e += 4) {
                        const float4 t = __ldg(wp + e / 4);
                        wv[e] = t.x, wv[e + 1] = t.y, wv[e + 2] = t.z, wv[e + 3] = t.w;
                    }
#pragma unroll
                    for (int e = 0; e < VN; ++e) {
                        const float s = gate ? silu_fast(gz[e]) : 1.f;
                        out[e] = __fmul_rn(__fmul_rn(__fmul_rn(x[e], r), wv[e]), s);
                    }
                    st16_stream(y + row * d + (int64_t)c * VN, pack(out));
                }
            }
        }
    }
}

// ---------------------------------------------------------------- causal conv
// One thread owns VN consecutive channels.  The per-element arithmetic, shared
// by the prefill and the decode kernels: acc = bias, then one fused
// multiply-add per tap from the oldest row to the current one, then the
// activation.
template <int W, int VN>
struct ConvTaps {
    float w[W][VN];
    float b[VN];
};

// The CTA's taps (blockDim.x * VN channels x W, contiguous in the [C, W]
// weight) are staged through shared memory: coalesced 16-byte loads in, then
// each thread reads its own PT = VN*W/4 float4s at an odd float4 stride, which
// is free of bank conflicts.  (Read straight from global memory, each warp
// instruction would touch 32 different cache lines.)  Must be called by every
// thread of the CTA; the weight pointer is 16-byte aligned.
template <int W, int VN>
struct TapStage {
    static constexpr int PT = VN * W / 4;                  // float4s per thread
    static constexpr int ST = (PT & 1) ? PT : PT + 1;      // odd stride in float4s
    static constexpr int kFloat4s = 128 * ST;              // for a 128-thread CTA
};

template <int W, int VN>
__device__ __forceinline__ void load_taps(ConvTaps<W, VN>& t, float4* stage, const float* __restrict__ w,
                                          const float* __restrict__ bias, int cblk0, int C) {
    constexpr int PT = TapStage<W, VN>::PT, ST = TapStage<W, VN>::ST;
    const int nch = min(C - cblk0, (int)blockDim.x * VN);
    const int nf4 = nch * W / 4;
    const float4* src = reinterpret_cast<const float4*>(w + (int64_t)cblk0 * W);
    for (int f = threadIdx.x; f < nf4; f += blockDim.x) stage[(f / PT) * ST + f % PT] = __ldg(src + f);
    __syncthreads();
    const int c0 = cblk0 + threadIdx.x * VN;
    if (c0 >= C) return;
    float flat[VN * W];  // channel-major: flat[e * W + i] = w[c0 + e][i]
#pragma unroll
    for (int j = 0; j < PT; ++j) {
        const float4 v = stage[threadIdx.x * ST + j];
        flat[4 * j] = v.x, flat[4 * j + 1] = v.y, flat[4 * j + 2] = v.z, flat[4 * j + 3] = v.w;
    }
#pragma unroll
    for (int e = 0; e < VN; ++e) {
#pragma unroll
        for (int i = 0; i < W; ++i) t.w[i][e] = flat[e * W + i];
        t.b[e] = bias ? __ldg(bias + c0 + e) : 0.f;
    }
}

template <int W, int VN>
__device__ __forceinline__ void conv_point(const ConvTaps<W, VN>& t, const float (&win)[W - 1][VN],
                                           const float (&xc)[VN], bool act, float (&out)[VN]) {
#pragma unroll
    for (int e = 0; e < VN; ++e) {
        float acc = t.b[e];
#pragma unroll
        for (int i = 0; i < W - 1; ++i) acc = __fmaf_rn(t.w[i][e], win[i][e], acc);
        acc = __fmaf_rn(t.w[W - 1][e], xc[e], acc);
        out[e] = act ? silu_fast(acc) : acc;
    }
}

struct ConvParams {
    int N, T_total, C, TT;
    const void* x;
    const float* w;
    const float* bias;
    const int32_t* cu;
    void* state;
    const int32_t* idx;
    int num_slots;
    const int32_t* has_init;
    void* y;
    int act;
};

// Token tiles: sequence n owns the virtual tiles [f(n), f(n+1)) with
// f(n) = floor(cu[n] / TT) + n, which is always at least ceil(len_n / TT) of
// them; its k-th tile covers tokens bos + k*TT .. bos + (k+1)*TT - 1 and the
// surplus tiles exit.  A tile never spans two sequences, so the first tile of
// a sequence is the only reader of its initial conv state and can also write
// the final state afterwards: in-place slots are safe.
template <typename T, int W>
__global__ void __launch_bounds__(128, (W <= 4 ? 4 : 2)) conv_fwd_kernel(const ConvParams p) {
    constexpr int VN = V16<T>::n;
    constexpr int WM = W - 1;
    constexpr int U = 4;  // rows per register buffer (two buffers)
    __shared__ float4 stage[TapStage<W, VN>::kFloat4s];
    const int cblk0 = blockIdx.y * blockDim.x * VN;
    const int c0 = cblk0 + threadIdx.x * VN;
    const int j = blockIdx.x;
    // largest n in [0, N) with f(n) <= j
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.cu + mid) / p.TT + mid <= j) lo = mid; else hi = mid - 1;
    }
    const int n = lo;
    const int cu0 = __ldg(p.cu + n), cu1 = __ldg(p.cu + n + 1);
    const int bos = max(0, min(cu0, p.T_total)), eos = max(bos, min(cu1, p.T_total));
    const int k = j - (cu0 / p.TT + n);
    const int t0 = bos + k * p.TT;
    if (k < 0 || (k > 0 && t0 >= eos)) return;
    const int t1 = min(eos, t0 + p.TT);
    const T* x = static_cast<const T*>(p.x);
    T* y = static_cast<T*>(p.y);
    const int slot = !p.state ? -1 : (p.idx ? __ldg(p.idx + n) : n);
    const bool has_slot = slot >= 0 && slot < p.num_slots;
    T* st = has_slot && c0 < p.C ? static_cast<T*>(p.state) + (int64_t)slot * WM * p.C + c0 : nullptr;
    const bool use_init = has_slot && (!p.has_init || __ldg(p.has_init + n) != 0);

    ConvTaps<W, VN> taps;
    load_taps<W, VN>(taps, stage, p.w, p.bias, cblk0, p.C);  // CTA-uniform up to here
    if (c0 >= p.C) return;
    float win[WM][VN];
#pragma unroll
    for (int i = 0; i < WM; ++i) {
        const int r = t0 - WM + i;
        if (r >= bos) {
            unpack(ld16(x + (int64_t)r * p.C + c0), win[i]);
        } else if (use_init) {
            unpack(ld16(st + (int64_t)(r - bos + WM) * p.C), win[i]);
        } else {
#pragma unroll
            for (int e = 0; e < VN; ++e) win[i][e] = 0.f;
        }
    }
    const bool act = p.act != 0;
    // two register buffers of U rows: the loads of the next U rows are in
    // flight while the current ones are computed and stored.  Whole blocks of
    // rows run without per-row conditions, so the window slides by register
    // renaming inside a block; only the tail block checks each row.
    uint4 ra[U], rb[U];
    auto load = [&](uint4(&r)[U], int b0) {
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (b0 + u < t1) r[u] = ld16_stream(x + (int64_t)(b0 + u) * p.C + c0);
    };
    auto row = [&](const uint4& r, int t) {
        float xc[VN], out[VN];
        unpack(r, xc);
        conv_point<W, VN>(taps, win, xc, act, out);
        st16_stream(y + (int64_t)t * p.C + c0, pack(out));
#pragma unroll
        for (int i = 0; i + 1 < WM; ++i)
#pragma unroll
            for (int e = 0; e < VN; ++e) win[i][e] = win[i + 1][e];
#pragma unroll
        for (int e = 0; e < VN; ++e) win[WM - 1][e] = xc[e];
    };
    auto consume_full = [&](const uint4(&r)[U], int b0) {
#pragma unroll
        for (int u = 0; u < U; ++u) row(r[u], b0 + u);
    };
    auto consume_tail = [&](const uint4(&r)[U], int b0) {
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (b0 + u < t1) row(r[u], b0 + u);
    };
    load(ra, t0);
    int base = t0;
    for (; base + 2 * U <= t1; base += 2 * U) {
        load(rb, base + U);
        consume_full(ra, base);
        load(ra, base + 2 * U);
        consume_full(rb, base + U);
    }
    if (base < t1) {
        load(rb, base + U);
        consume_tail(ra, base);
        consume_tail(rb, base + U);
    }
    if (k == 0 && has_slot) {
        // final state: the last W-1 rows of (initial state ++ the sequence)
        if (t1 == eos) {
#pragma unroll
            for (int i = 0; i < WM; ++i) st16(st + (int64_t)i * p.C, pack(win[i]));
        } else {
#pragma unroll
            for (int i = 0; i < WM; ++i) st16(st + (int64_t)i * p.C, ld16(x + (int64_t)(eos - WM + i) * p.C + c0));
        }
    }
}

// Decode update: a CTA takes kUpdRows consecutive batch rows of one channel
// block, so the staged taps serve all of them, and a thread's rows are
// independent (all their loads in flight together).
constexpr int kUpdRows = 8;

template <typename T, int W>
__global__ void __launch_bounds__(128) conv_update_kernel(const ConvParams p) {
    constexpr int VN = V16<T>::n;
    constexpr int WM = W - 1;
    __shared__ float4 stage[TapStage<W, VN>::kFloat4s];
    const int cblk0 = blockIdx.y * blockDim.x * VN;
    const int c0 = cblk0 + threadIdx.x * VN;
    const int b0 = blockIdx.x * kUpdRows;
    ConvTaps<W, VN> taps;
    load_taps<W, VN>(taps, stage, p.w, p.bias, cblk0, p.C);  // CTA-uniform up to here
    if (c0 >= p.C) return;
    const T* x = static_cast<const T*>(p.x);
    T* y = static_cast<T*>(p.y);
    const bool act = p.act != 0;
#pragma unroll 2
    for (int r = 0; r < kUpdRows; ++r) {
        const int b = b0 + r;
        if (b >= p.N) break;
        const int slot = p.idx ? __ldg(p.idx + b) : b;
        if (slot < 0 || slot >= p.num_slots) continue;
        T* st = static_cast<T*>(p.state) + (int64_t)slot * WM * p.C + c0;
        float win[WM][VN], xc[VN], out[VN];
#pragma unroll
        for (int i = 0; i < WM; ++i) unpack(ld16(st + (int64_t)i * p.C), win[i]);
        unpack(ld16(x + (int64_t)b * p.C + c0), xc);
        conv_point<W, VN>(taps, win, xc, act, out);
        st16(y + (int64_t)b * p.C + c0, pack(out));
#pragma unroll
        for (int i = 0; i + 1 < WM; ++i) st16(st + (int64_t)i * p.C, pack(win[i + 1]));
        st16(st + (int64_t)(WM - 1) * p.C, pack(xc));
    }
}

gdn_status check_conv(const gdn_conv_shape* s) {
    if (!s) return GDN_ERR_INVALID_ARG;
    if (s->N < 0 || s->T_total < 0 || s->C <= 0) return GDN_ERR_INVALID_ARG;
    if (s->dtype != GDN_F32 && s->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (s->W < 2 || s->W > 8) return GDN_ERR_UNSUPPORTED;
    if (s->C % (s->dtype == GDN_BF16 ? 8 : 4)) return GDN_ERR_UNSUPPORTED;
    if ((long long)s->T_total * s->C >= (1LL << 40)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// Tokens per conv tile: the halo of W-1 rows re-read per tile is <= 7/256 of the input.
constexpr int kConvTile = 256;

// One launcher per kernel so that the tap count can be dispatched generically.
template <typename T, int W>
struct FwdK {
    static void go(dim3 g, cudaStream_t s, const ConvParams& p) { conv_fwd_kernel<T, W><<<g, 128, 0, s>>>(p); }
};
template <typename T, int W>
struct UpdK {
    static void go(dim3 g, cudaStream_t s, const ConvParams& p) { conv_update_kernel<T, W><<<g, 128, 0, s>>>(p); }
};
template <template <typename, int> class K, typename T>
gdn_status dispatch_w(int W, dim3 grid, cudaStream_t s, const ConvParams& p) {
    switch (W) {
        case 2: K<T, 2>::go(grid, s, p); break;
        case 3: K<T, 3>::go(grid, s, p); break;
        case 4: K<T, 4>::go(grid, s, p); break;
        case 5: K<T, 5>::go(grid, s, p); break;
        case 6: K<T, 6>::go(grid, s, p); break;
        case 7: K<T, 7>::go(grid, s, p); break;
        case 8: K<T, 8>::go(grid, s, p); break;
        default: return GDN_ERR_UNSUPPORTED;
    }
    return launch_status();
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_gates(int64_t T, int HV, gdn_dtype in_dtype, const void* a, const void* b,
                                const float* A_log, const float* dt_bias, float* g, float* beta, void* stream) {
    using namespace gdn;
    if (T < 0 || HV <= 0) return GDN_ERR_INVALID_ARG;
    if (in_dtype != GDN_F32 && in_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    const int64_t n = T * HV;
    if (n == 0) return GDN_OK;
    const uintptr_t ia = in_dtype == GDN_BF16 ? 2 : 4;
    auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
    if (!a || !b || !A_log || !g || !beta) return GDN_ERR_INVALID_ARG;
    if (!al(a, ia) || !al(b, ia) || !aligned4(A_log) || !aligned4(g) || !aligned4(beta) ||
        (dt_bias && !aligned4(dt_bias)))
        return GDN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool vec = HV % 8 == 0 && aligned16(a) && aligned16(b) && aligned16(g) && aligned16(beta);
    // The vector form runs a few tokens per thread and keeps each thread on the same heads:
    // when the grid does not cover every item at once, its stride of 2048 * grid elements must
    // be a multiple of HV (true for any grid when HV divides 2048).  If no grid up to the cap
    // qualifies, the scalar form runs instead.
    int grid = 0;
    if (vec) {
        const int64_t want = (n / 8 + 255) / 256;
        grid = (int)(want < kSMs * 4 ? want : kSMs * 4);
        if (grid < want) {
            while (grid > 1 && (2048LL * grid) % HV) --grid;
            if ((2048LL * grid) % HV) vec = false;
        }
    }
    const int64_t items = vec ? n / 8 : n;
    if (!vec) {
        const int64_t want = (n + 255) / 256;
        grid = (int)(want < kSMs * 16 ? want : kSMs * 16);
    }
    if (in_dtype == GDN_BF16) {
        auto a_ = static_cast<const __nv_bfloat16*>(a);
        auto b_ = static_cast<const __nv_bfloat16*>(b);
        if (vec) gates_kernel_v8<<<grid, 256, 0, s>>>(items, HV, a_, b_, A_log, dt_bias, g, beta);
        else gates_kernel<<<grid, 256, 0, s>>>(n, HV, a_, b_, A_log, dt_bias, g, beta);
    } else {
        auto a_ = static_cast<const float*>(a);
        auto b_ = static_cast<const float*>(b);
        if (vec) gates_kernel_v8<<<grid, 256, 0, s>>>(items, HV, a_, b_, A_log, dt_bias, g, beta);
        else gates_kernel<<<grid, 256, 0, s>>>(n, HV, a_, b_, A_log, dt_bias, g, beta);
    }
    return launch_status();
}

extern "C" gdn_status gdn_gated_rmsnorm(int64_t rows, int d, gdn_dtype dtype, const void* o, const void* z,
                                        const float* weight, float eps, void* y, void* stream) {
    using namespace gdn;
    if (rows < 0 || d <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    const int vn = dtype == GDN_BF16 ? 8 : 4;
    if (d % vn || d > 2048) return GDN_ERR_UNSUPPORTED;
    if (!(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    if (rows == 0) return GDN_OK;
    if (!o || !weight || !y) return GDN_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(y) || (z && !aligned16(z)) || !aligned16(weight)) return GDN_ERR_INVALID_ARG;
    const int chunks = d / vn;
    int lpr = 1;
    while (lpr * 2 <= chunks && lpr < 32) lpr *= 2;
    const int nc = (chunks + lpr - 1) / lpr;          // <= 8 (d <= 2048)
    const int ur = nc == 1 ? 4 : (nc == 2 ? 2 : 1);   // row groups per warp iteration
    const int64_t per_warp = (int64_t)(32 / lpr) * ur;
    const int64_t warps = (rows + per_warp - 1) / per_warp;
    const int64_t want = (warps + 7) / 8;
    const int grid = (int)(want < kSMs * 16 ? want : kSMs * 16);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
#define GDN_RMS_LAUNCH(T, NC, UR)                                                                        \
    rmsnorm_kernel<T, NC, UR><<<grid, 256, 0, s>>>(rows, d, lpr, static_cast<const T*>(o),                 \
                                                   static_cast<const T*>(z), weight, eps, static_cast<T*>(y))
    if (dtype == GDN_BF16) {
        if (nc == 1) GDN_RMS_LAUNCH(__nv_bfloat16, 1, 4);
        else if (nc == 2) GDN_RMS_LAUNCH(__nv_bfloat16, 2, 2);
        else if (nc <= 4) GDN_RMS_LAUNCH(__nv_bfloat16, 4, 1);
        else GDN_RMS_LAUNCH(__nv_bfloat16, 8, 1);
    } else {
        if (nc == 1) GDN_RMS_LAUNCH(float, 1, 4);
        else if (nc == 2) GDN_RMS_LAUNCH(float, 2, 2);
        else if (nc <= 4) GDN_RMS_LAUNCH(float, 4, 1);
        else GDN_RMS_LAUNCH(float, 8, 1);
    }
#undef GDN_RMS_LAUNCH
    return launch_status();
}

extern "C" gdn_status gdn_causal_conv1d_fwd(const gdn_conv_shape* shape, const void* x, const float* weight,
                                            const float* bias, const int32_t* cu_seqlens, void* conv_state,
                                            const int32_t* state_indices, int num_slots,
                                            const int32_t* has_initial_state, void* y, void* stream) {
    using namespace gdn;
    gdn_status st = check_conv(shape);
    if (st != GDN_OK) return st;
    if (shape->N == 0) return shape->T_total == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!weight || !cu_seqlens || (shape->T_total > 0 && (!x || !y))) return GDN_ERR_INVALID_ARG;
    if (x && x == y) return GDN_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (y && !aligned16(y)) || (conv_state && !aligned16(conv_state)) ||
        !aligned16(weight) || (bias && !aligned4(bias)) || !aligned4(cu_seqlens) ||
        (state_indices && !aligned4(state_indices)) || (has_initial_state && !aligned4(has_initial_state)))
        return GDN_ERR_INVALID_ARG;
    if (conv_state && num_slots < 0) return GDN_ERR_INVALID_ARG;
    if (conv_state && !state_indices && num_slots < shape->N) return GDN_ERR_INVALID_ARG;
    const int vn = shape->dtype == GDN_BF16 ? 8 : 4;
    const long long tiles = (long long)shape->T_total / kConvTile + shape->N;
    if (tiles >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    ConvParams p{shape->N, shape->T_total, shape->C, kConvTile, x, weight, bias, cu_seqlens, conv_state,
                 state_indices, conv_state ? num_slots : 0, has_initial_state, y, shape->activation};
    const dim3 grid((unsigned)tiles, (unsigned)((shape->C / vn + 127) / 128));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return shape->dtype == GDN_BF16 ? dispatch_w<FwdK, __nv_bfloat16>(shape->W, grid, s, p)
                                    : dispatch_w<FwdK, float>(shape->W, grid, s, p);
}

extern "C" gdn_status gdn_causal_conv1d_update(const gdn_conv_shape* shape, const void* x, const float* weight,
                                               const float* bias, void* conv_state, const int32_t* state_indices,
                                               int num_slots, void* y, void* stream) {
    using namespace gdn;
    gdn_status st = check_conv(shape);
    if (st != GDN_OK) return st;
    if (shape->T_total != shape->N) return GDN_ERR_INVALID_ARG;
    if (shape->N == 0) return GDN_OK;
    if (!x || !y || !weight || !conv_state || num_slots < 0) return GDN_ERR_INVALID_ARG;
    if (!state_indices && num_slots < shape->N) return GDN_ERR_INVALID_ARG;
    if (x == y) return GDN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || !aligned16(conv_state) || !aligned16(weight) || (bias && !aligned4(bias)) ||
        (state_indices && !aligned4(state_indices)))
        return GDN_ERR_INVALID_ARG;
    const int vn = shape->dtype == GDN_BF16 ? 8 : 4;
    ConvParams p{shape->N, shape->T_total, shape->C, 1, x, weight, bias, nullptr, conv_state, state_indices,
                 num_slots, nullptr, y, shape->activation};
    const dim3 grid((unsigned)((shape->N + kUpdRows - 1) / kUpdRows), (unsigned)((shape->C / vn + 127) / 128));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return shape->dtype == GDN_BF16 ? dispatch_w<UpdK, __nv_bfloat16>(shape->W, grid, s, p)
                                    : dispatch_w<UpdK, float>(shape->W, grid, s, p);
}
