// gdn_fwd.cu -- varlen scheduler + batch-invariant recurrent forward.
//
// One CTA owns one unit (sequence n, value head h, slice of dv rows) for the
// whole sequence: its rows of the fp32 state S stay in registers from the
// first token to the last, so there is no state hand-off between CTAs and
// nothing is reduced across sequences or split over dk ("the recurrent kernel
// reads only that sequence's own state and walks that sequence's tokens in a
// fixed order": "Defending Against the Training-Inference Numeric Mismatch in
// RL (Especially Linear Attention)", section 3.2).
//
// Per chunk of TC tokens, thread 0 streams q/k (k-head hk) and the v slice
// with three TMA tensor copies into a double-buffered shared-memory stage.
// The CTA then L2-normalises q and k (one warp per vector, fixed butterfly),
// computes a = exp(g), and every thread walks the chunk's tokens over its
// rows with the shared step of gdn_step.cuh (row layout over lanes and rows
// per thread as defined there).  Outputs go straight from registers to
// global memory.  Two units share an SM.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "gdn_async.cuh"
#include "gdn_host.h"
#include "gdn_step.cuh"
#include "gdn_token_step.cuh"

namespace gdn {

#ifndef GDN_TC
#define GDN_TC 32
#endif
constexpr int kTC = GDN_TC;  // tokens per chunk (one TMA stage)
constexpr int kStages = 2;   // TMA stages
constexpr int kMaxSlice = 128;

struct FwdParams {
    const float* g;
    const float* beta;
    const float* init_state;
    const int32_t* cu;
    void* out;
    float* final_state;
    const int32_t* work;
    unsigned* err;
    int N, T, HV, G, dv, dvs, nslices, use_norm;
    int tb;  // tokens per TMA box: min(kTC, T)
};

// Parameters of the snapshot-taking forward: the plain forward's, plus where
// to put a copy of the state after every snap_every-th token of a sequence.
// A separate type keeps the plain kernel's parameters (and code) untouched.
struct SnapParams : FwdParams {
    float* snap;
    const int32_t* snap_cu;
    int snap_every, snap_slots;
};

template <typename Tin, int DK>
struct alignas(128) FwdSmem {
    Tin q[kStages][kTC * DK];
    Tin k[kStages][kTC * DK];
    Tin v[kStages][kTC * kMaxSlice];
    float qn[kTC * DK];
    float kn[kTC * DK];
    float2 ab[kTC];
    uint64_t bar[kStages];
    int abort_flag;
};

// ---------------------------------------------------------------------------
// Varlen scheduler: rank every sequence by length (longest first, ties by
// index: a stable order), then emit its units (n, h, slice) in that order.
// Launch order only decides which SM runs a unit when; it never changes a bit.
// Also validates cu_seqlens and flags GDN_DEVERR_CU_SEQLENS in the error word.
__global__ void gdn_sched_kernel(const int32_t* __restrict__ cu, int N, int T, int HV, int nslices,
                                 int32_t* __restrict__ work, unsigned* __restrict__ err) {
    constexpr int kTile = 1024;
    __shared__ int lens[kTile];
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    int my_len = 0;
    if (n < N) {
        const int a = cu[n], b = cu[n + 1];
        if ((n == 0 && a != 0) || b < a || (n == N - 1 && b != T)) atomicOr(err, GDN_DEVERR_CU_SEQLENS);
        const int lo = min(max(a, 0), T), hi = min(max(b, lo), T);
        my_len = hi - lo;
    }
    int rank = 0;
    for (int base = 0; base < N; base += kTile) {
        __syncthreads();
        for (int i = threadIdx.x; i < kTile && base + i < N; i += blockDim.x) {
            const int a = cu[base + i], b = cu[base + i + 1];
            const int lo = min(max(a, 0), T), hi = min(max(b, lo), T);
            lens[i] = hi - lo;
        }
        __syncthreads();
        if (n < N) {
            const int cnt = min(kTile, N - base);
            for (int i = 0; i < cnt; ++i) {
                const int lm = lens[i], m = base + i;
                rank += (lm > my_len) || (lm == my_len && m < n);
            }
        }
    }
    if (n < N) {
        for (int h = 0; h < HV; ++h)
            for (int s = 0; s < nslices; ++s)
                work[((size_t)rank * HV + h) * nslices + s] = (n * HV + h) * nslices + s;
    }
}

// Thread 0: start the three TMA copies of chunk c into stage c % kStages.
template <typename Tin, int DK>
__device__ __forceinline__ void issue_chunk(FwdSmem<Tin, DK>& sm, const CUtensorMap* tq, const CUtensorMap* tk,
                                            const CUtensorMap* tv, int c, int bos, int hk, int h, int col,
                                            uint32_t bytes) {
    const int st = c % kStages, t0 = bos + c * kTC;
    mbar_arrive_expect_tx(&sm.bar[st], bytes);
    tma_load_3d(sm.q[st], tq, &sm.bar[st], 0, hk, t0);
    tma_load_3d(sm.k[st], tk, &sm.bar[st], 0, hk, t0);
    tma_load_3d(sm.v[st], tv, &sm.bar[st], col, h, t0);
}

// ---------------------------------------------------------------------------
template <typename Tin, int DK, typename Prm>
__global__ void __launch_bounds__(ts::threads_for_rows<DK>(kMaxSlice), 2)
    gdn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Prm p) {
    constexpr int RG = 4;  // one slot group: one reduce-scatter over all four rows of a thread
    using Y = ts::Layout<DK, RG>;
    extern __shared__ unsigned char smem_raw[];
    FwdSmem<Tin, DK>& sm =
        *reinterpret_cast<FwdSmem<Tin, DK>*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const ts::Place pl = ts::place_of<DK, RG>(tid);
    const int dvs = p.dvs;
    const bool active = pl.grp * Y::R < dvs;
    const bool storer = active && ts::stores_row<DK, RG>(pl);

    const int unit = p.work[blockIdx.x];
    const int slice = unit % p.nslices;
    const int h = (unit / p.nslices) % p.HV;
    const int n = unit / (p.nslices * p.HV);
    const int hk = h / p.G;
    int bos = p.cu[n], eos = p.cu[n + 1];
    bos = min(max(bos, 0), p.T);
    eos = min(max(eos, bos), p.T);
    const int L = eos - bos;
    const int row = slice * dvs + pl.grp * Y::R;  // first row of this thread's group
    const int orow = row + pl.own;                 // the row whose output this thread may store
    const size_t soff = (((size_t)n * p.HV + h) * p.dv + row) * DK;

    ts::Rows<DK> S;
    if (active && p.init_state) ts::load_rows<DK, RG>(S, p.init_state + soff, pl);
    else ts::zero_rows<DK>(S);

    if (L > 0) {
        const int nchunks = (L + kTC - 1) / kTC;
        const uint32_t bytes = (uint32_t)((2 * p.tb * DK + p.tb * dvs) * sizeof(Tin));
        if (tid == 0) {
            for (int s = 0; s < kStages; ++s) mbar_init(&sm.bar[s], 1);
            sm.abort_flag = 0;
            fence_barrier_init();
        }
        __syncthreads();
        if (tid == 0)
            for (int c = 0; c < min(kStages, nchunks); ++c)
                issue_chunk(sm, &tm_q, &tm_k, &tm_v, c, bos, hk, h, slice * dvs, bytes);

        // gate inputs of the next chunk, prefetched into registers one chunk ahead
        float2 gb = make_float2(0.f, 0.f);
        if (tid < min(kTC, L)) {
            const size_t gi = (size_t)(bos + tid) * p.HV + h;
            gb = make_float2(p.g[gi], p.beta[gi]);
        }
        Tin* __restrict__ out = reinterpret_cast<Tin*>(p.out);

        for (int c = 0; c < nchunks; ++c) {
            const int st = c % kStages;
            const int t0 = bos + c * kTC;
            const int tc = min(kTC, eos - t0);
            if (!mbar_wait_bounded(&sm.bar[st], (uint32_t)((c / kStages) & 1))) sm.abort_flag = 1;
            // normalise the chunk's 2*tc q/k vectors, four per warp at a time
            for (int j0 = warp; j0 < 2 * tc; j0 += 4 * nwarps) {
                const Tin* src[4];
                float* dst[4];
                int nv = 0;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int j = j0 + v * nwarps, t = j >> 1;
                    const bool ok = j < 2 * tc;
                    nv += ok;
                    src[v] = ok ? ((j & 1) ? sm.k[st] + t * DK : sm.q[st] + t * DK) : sm.q[st];
                    dst[v] = ok ? ((j & 1) ? sm.kn + t * DK : sm.qn + t * DK) : sm.qn;
                }
                l2norm_warp_multi<DK, 4>(src, dst, nv, lane, p.use_norm);
            }
            if (tid < tc) sm.ab[tid] = make_float2(gate_alpha(gb.x), gb.y);
            __syncthreads();
            if (sm.abort_flag) {
                if (tid == 0) {
                    atomicOr(p.err, GDN_DEVERR_TIMEOUT);
                    // leave no bulk copy of this CTA in flight into shared memory that a later
                    // CTA may own: wait (bounded again) for this chunk's stage and the next one's
                    mbar_wait_bounded(&sm.bar[st], (uint32_t)((c / kStages) & 1));
                    if (c + 1 < nchunks)
                        mbar_wait_bounded(&sm.bar[(c + 1) % kStages], (uint32_t)(((c + 1) / kStages) & 1));
                }
                return;
            }
            if (c + 1 < nchunks && tid < min(kTC, eos - (t0 + kTC))) {
                const size_t gi = (size_t)(t0 + kTC + tid) * p.HV + h;
                gb = make_float2(p.g[gi], p.beta[gi]);
            }
            const Tin* __restrict__ vs = sm.v[st] + pl.grp * Y::R + pl.own;
            // Token loop, software-pipelined by one token: the reduce-scatter of
            // token t's output runs next to token t+1's u reduction (it is off
            // the recurrence's critical path); every operation is unchanged.
            float op[RG];
            for (int t = 0; t < tc; ++t) {
                const float2 ab = sm.ab[t];
                const float vown = active ? ld_in(vs + t * dvs) : 0.f;
                float up[RG], w[RG];
                ts::dot_part<DK, RG, 0>(S, sm.kn + t * DK, pl.e, up);
                float oprev = 0.f;
                if (t > 0) oprev = ts::reduce_scatter<DK, RG>(op);
                const float u = ts::reduce_scatter<DK, RG>(up);
                if (t > 0 && storer) st_in(out + ((size_t)(t0 + t - 1) * p.HV + h) * p.dv + orow, oprev);
                ts::gather_rows<DK, RG>(ts::delta_w(ab.x, ab.y, vown, u), lane, pl.own, w);
                ts::update_part<DK, RG, 0>(S, sm.kn + t * DK, sm.qn + t * DK, pl.e, ab.x, w, op);
            }
            const float olast = ts::reduce_scatter<DK, RG>(op);
            if (storer) st_in(out + ((size_t)(t0 + tc - 1) * p.HV + h) * p.dv + orow, olast);
            if constexpr (std::is_same<Prm, SnapParams>::value) {
                // the state after `done` tokens of this sequence, at every snap_every-th token
                const int done = t0 + tc - bos;
                if (done % p.snap_every == 0) {
                    const int slot = p.snap_cu[n] + done / p.snap_every - 1;
                    if (active && slot >= 0 && slot < p.snap_cu[n + 1] && slot < p.snap_slots)
                        ts::store_rows<DK, RG>(S, p.snap + (((size_t)slot * p.HV + h) * p.dv + row) * DK, pl);
                }
            }
            __syncthreads();
            if (tid == 0 && c + kStages < nchunks)
                issue_chunk(sm, &tm_q, &tm_k, &tm_v, c + kStages, bos, hk, h, slice * dvs, bytes);
        }
    }
    if (active && p.final_state) ts::store_rows<DK, RG>(S, p.final_state + soff, pl);
}

template <typename Tin, int DK, typename Prm>
static gdn_status launch_fwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                               const Prm& p, int units, cudaStream_t stream) {
    const size_t smem = sizeof(FwdSmem<Tin, DK>) + 128;
    auto kern = gdn_fwd_kernel<Tin, DK, Prm>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    const int nt = ts::threads_for_rows<DK>(p.dvs);
    kern<<<units, nt, smem, stream>>>(mq, mk, mv, p);
    return launch_status();
}

template <typename Tin, typename Prm>
static gdn_status launch_fwd_dk(int dk, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                const Prm& p, int units, cudaStream_t stream) {
    switch (dk) {
        case 16: return launch_fwd_t<Tin, 16, Prm>(mq, mk, mv, p, units, stream);
        case 32: return launch_fwd_t<Tin, 32, Prm>(mq, mk, mv, p, units, stream);
        case 64: return launch_fwd_t<Tin, 64, Prm>(mq, mk, mv, p, units, stream);
        case 128: return launch_fwd_t<Tin, 128, Prm>(mq, mk, mv, p, units, stream);
    }
    return GDN_ERR_UNSUPPORTED;
}

// Host launcher of the varlen scheduler for the other kernels that run one
// CTA per (sequence, head) unit (the chunk-replay prefill).
gdn_status launch_unit_sched(const int32_t* cu, int N, int T, int HV, int nslices, int32_t* work, unsigned* err,
                             cudaStream_t stream) {
    if (cudaMemsetAsync(err, 0, sizeof(unsigned), stream) != cudaSuccess) return GDN_ERR_CUDA;
    gdn_sched_kernel<<<(N + 255) / 256, 256, 0, stream>>>(cu, N, T, HV, nslices, work, err);
    return launch_status();
}

size_t fwd_workspace_size(const gdn_shape* s) {
    const int dvs = pick_dv_slice(s);
    return kWsHeader + (((size_t)s->N * s->HV * (s->dv / dvs) * sizeof(int32_t) + 255) & ~size_t(255));
}

// Shared by the allocating entry point and any caller that supplies the
// work-list and error-word buffers itself.
gdn_status run_recurrent_fwd(const gdn_shape* s, const void* q, const void* k, const void* v, const float* g,
                             const float* beta, const float* init_state, const int32_t* cu, void* out,
                             float* final_state, int32_t* work, unsigned* err, cudaStream_t stream,
                             float* snap = nullptr, const int32_t* snap_cu = nullptr, int snap_every = 0,
                             int snap_slots = 0) {
    const int dvs = pick_dv_slice(s);
    const int nslices = s->dv / dvs;
    const int units = s->N * s->HV * nslices;
    if (s->N == 0) return GDN_OK;

    CUtensorMap mq{}, mk{}, mv{};
    if (s->T_total > 0) {
        gdn_status st;
        // box height min(kTC, T): a sequence shorter than kTC never needs more rows than T
        const uint32_t tb = (uint32_t)std::min(kTC, s->T_total);
        if ((st = encode_map_3d(&mq, q, s->dtype, s->dk, s->HK, s->T_total, s->dk, tb)) != GDN_OK) return st;
        if ((st = encode_map_3d(&mk, k, s->dtype, s->dk, s->HK, s->T_total, s->dk, tb)) != GDN_OK) return st;
        if ((st = encode_map_3d(&mv, v, s->dtype, s->dv, s->HV, s->T_total, dvs, tb)) != GDN_OK) return st;
    }
    if (cudaMemsetAsync(err, 0, sizeof(unsigned), stream) != cudaSuccess) return GDN_ERR_CUDA;
    gdn_sched_kernel<<<(s->N + 255) / 256, 256, 0, stream>>>(cu, s->N, s->T_total, s->HV, nslices, work, err);
    if (launch_status() != GDN_OK) return GDN_ERR_CUDA;

    FwdParams p;
    p.g = g;
    p.beta = beta;
    p.init_state = init_state;
    p.cu = cu;
    p.out = out;
    p.final_state = final_state;
    p.work = work;
    p.err = err;
    p.N = s->N;
    p.T = s->T_total;
    p.HV = s->HV;
    p.G = s->HV / s->HK;
    p.dv = s->dv;
    p.dvs = dvs;
    p.nslices = nslices;
    p.use_norm = s->use_qk_l2norm ? 1 : 0;
    p.tb = std::min(kTC, s->T_total);
    if (snap && snap_cu && snap_slots > 0 && snap_every > 0) {
        SnapParams sp;
        static_cast<FwdParams&>(sp) = p;
        sp.snap = snap;
        sp.snap_cu = snap_cu;
        sp.snap_every = snap_every;
        sp.snap_slots = snap_slots;
        if (s->dtype == GDN_BF16) return launch_fwd_dk<__nv_bfloat16>(s->dk, mq, mk, mv, sp, units, stream);
        return launch_fwd_dk<float>(s->dk, mq, mk, mv, sp, units, stream);
    }
    if (s->dtype == GDN_BF16) return launch_fwd_dk<__nv_bfloat16>(s->dk, mq, mk, mv, p, units, stream);
    return launch_fwd_dk<float>(s->dk, mq, mk, mv, p, units, stream);
}

gdn_status check_fwd_args(const gdn_shape* s, const void* q, const void* k, const void* v, const float* g,
                          const float* beta, const float* init_state, const int32_t* cu, const void* out,
                          const float* final_state) {
    gdn_status st = check_shape(s);
    if (st != GDN_OK) return st;
    if (!cu) return GDN_ERR_INVALID_ARG;
    if (s->T_total > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
    // vector / TMA operands need 16 bytes, scalar-loaded ones 4
    const void* vec[] = {q, k, v, init_state, out, final_state};
    for (const void* ptr : vec)
        if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
    const void* sca[] = {g, beta, cu};
    for (const void* ptr : sca)
        if (ptr && !aligned4(ptr)) return GDN_ERR_INVALID_ARG;
    // out must not alias an input it is computed from
    if (out && (out == q || out == k || out == v)) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

}  // namespace gdn

extern "C" gdn_status gdn_recurrent_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
                                        const float* g, const float* beta, const float* init_state,
                                        const int32_t* cu_seqlens, void* out, float* final_state,
                                        void* workspace, size_t workspace_bytes, void* stream) {
    using namespace gdn;
    gdn_status st = check_fwd_args(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state);
    if (st != GDN_OK) return st;
    if (shape->N == 0) return GDN_OK;
    if (!workspace || !aligned16(workspace) || workspace_bytes < fwd_workspace_size(shape)) return GDN_ERR_WORKSPACE;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    return run_recurrent_fwd(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state,
                             reinterpret_cast<int32_t*>(ws + kWsHeader), reinterpret_cast<unsigned*>(ws),
                             static_cast<cudaStream_t>(stream));
}

extern "C" gdn_status gdn_recurrent_fwd_snapshots(const gdn_shape* shape, const void* q, const void* k,
                                                  const void* v, const float* g, const float* beta,
                                                  const float* init_state, const int32_t* cu_seqlens, void* out,
                                                  float* final_state, int snap_every, const int32_t* snap_cu,
                                                  int num_snap_slots, float* snap_states, void* workspace,
                                                  size_t workspace_bytes, void* stream) {
    using namespace gdn;
    gdn_status st = check_fwd_args(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state);
    if (st != GDN_OK) return st;
    if (snap_every <= 0 || snap_every % kTC) return GDN_ERR_UNSUPPORTED;
    if (num_snap_slots < 0 || (num_snap_slots > 0 && (!snap_states || !snap_cu))) return GDN_ERR_INVALID_ARG;
    if ((snap_states && !aligned16(snap_states)) || (snap_cu && !aligned4(snap_cu))) return GDN_ERR_INVALID_ARG;
    if (snap_states && (snap_states == init_state || snap_states == final_state)) return GDN_ERR_INVALID_ARG;
    if (shape->N == 0) return GDN_OK;
    if (!workspace || !aligned16(workspace) || workspace_bytes < fwd_workspace_size(shape)) return GDN_ERR_WORKSPACE;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    return run_recurrent_fwd(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state,
                             reinterpret_cast<int32_t*>(ws + kWsHeader), reinterpret_cast<unsigned*>(ws),
                             static_cast<cudaStream_t>(stream), snap_states, snap_cu, snap_every, num_snap_slots);
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  Its scratch (device error word + work list) is a
// fixed array in the library's own device memory instead of a caller-supplied
// workspace.  Every device that loads the library holds this array (about
// 256 KB) until the process exits.  All calls share it, so two calls whose
// work overlaps on the GPU race on it; the error word is cleared by each call
// and the work list is rewritten in full by each call.
namespace gdn {

constexpr int kStaticUnits = 1 << 16;    // max N * HV * (dv / dv_slice)
constexpr int kStaticHeaderWords = 64;   // 256 bytes: word 0 is the error word
static __device__ __align__(256) int32_t g_fwd_static_scratch[kStaticHeaderWords + kStaticUnits];

// Device address of the array on the current device, looked up once per device
// (with that device current) and cached for the life of the process; a
// cudaDeviceReset of that device invalidates it (the header says so).
// nullptr if the lookup fails.
static int32_t* static_scratch_on_current_device() {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static int32_t* addr[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fwd_static_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = static_cast<int32_t*>(p);
    }
    return addr[dev];
}

}  // namespace gdn

extern "C" gdn_status gdn_recurrent_fwd_noalloc(const gdn_shape* shape, const void* q, const void* k,
                                                const void* v, const float* g, const float* beta,
                                                const float* init_state, const int32_t* cu_seqlens, void* out,
                                                float* final_state, void* stream) {
    using namespace gdn;
    gdn_status st = check_fwd_args(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state);
    if (st != GDN_OK) return st;
    if (shape->N == 0) return GDN_OK;
    const long long units = (long long)shape->N * shape->HV * (shape->dv / pick_dv_slice(shape));
    if (units > kStaticUnits) return GDN_ERR_WORKSPACE;
    int32_t* base = static_scratch_on_current_device();
    if (!base) return GDN_ERR_CUDA;
    return run_recurrent_fwd(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state,
                             base + kStaticHeaderWords, reinterpret_cast<unsigned*>(base),
                             static_cast<cudaStream_t>(stream));
}
