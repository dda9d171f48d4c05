// gdn_fwd.cu -- varlen scheduler + batch-invariant recurrent forward.
//
// One CTA owns one unit (sequence n, value head h, a slice of the dv rows of
// S) for the whole sequence: its rows of the fp32 state stay in registers from
// the first token to the last, so no state passes between CTAs and nothing is
// reduced across sequences or split over dk.  This is the property the
// recurrent kernel of "Defending Against the Training-Inference Numeric
// Mismatch in RL (Especially Linear Attention)", section 3.2, relies on for
// batch invariance: each sequence's state sees only its own tokens, in order.
//
// Per chunk of TC tokens, thread 0 streams q/k (k-head hk) and the v rows
// with three TMA tensor copies into a double-buffered shared-memory stage.
// The CTA then L2-normalises q and k (one warp per vector, fixed butterfly),
// computes a = exp(g), and every thread walks the chunk's tokens over its
// rows with the shared step of gdn_token_step.cuh.  Outputs go straight from
// registers to global memory.  Two CTAs share an SM.
//
// Slices.  By default a unit is a whole head (dv rows, 4 rows per thread).
// The scheduler gives a long sequence's heads 2 or 4 slices of dv/2 or dv/4
// rows (2 or 1 rows per thread, same CTA size) when the sequence is more than
// 1.5 or 3 times the average work per CTA slot: its chains then run on more
// SMs at once, with fewer rows each.  A row's operations do not depend on the rows
// per thread (the tree of gdn_token_step.cuh is the same for every slot
// grouping), so slicing never changes a bit.  A caller-forced dv_slice gives
// every head that many uniform slices instead.
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
    const int32_t* work;   // work items, longest sequence first (fwd_sched_kernel)
    const int32_t* nwork;  // how many there are
    unsigned* err;
    int N, T, HV, G, dv, use_norm;
    int rows4;   // rows of a unit at 4 rows per thread: dv, or the forced dv_slice
    int forced;  // 1: the caller fixed dv_slice (uniform slices), 0: automatic slices
    int vw;      // v columns per TMA box: dv (automatic) or dv_slice (forced)
    int tb;      // tokens per TMA box: min(kTC, T)
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
    float4 ab[kTC];  // per token: (a, a, b, a * b)
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

// Work item of the forward: (n * HV + h) << 5 | (first row / 16) << 2 | log2(rows per thread).
__host__ __device__ constexpr int32_t fwd_item(int nh, int row0, int rlog) {
    return (int32_t)((nh << 5) | ((row0 >> 4) << 2) | rlog);
}

// Slices of each head of a sequence of length len: forced_ns when the caller
// fixed dv_slice; otherwise, when splitting is allowed, 2 if the sequence is
// longer than 1.5 times the average work per CTA slot (T * HV / slots) and 4
// if longer than 3 times it, else 1.  Below 1.5 the whole heads already
// balance: a sliced head does the same work with more shared-memory traffic
// per FMA (fewer rows per thread), which only pays when it frees idle SMs.
__device__ __forceinline__ int fwd_slices(int len, int forced_ns, int split, int slots, long long work) {
    if (forced_ns > 0) return forced_ns;
    if (!split) return 1;
    const long long l = (long long)len * slots;
    return l > 3 * work ? 4 : (2 * l > 3 * work ? 2 : 1);
}

// The forward's varlen scheduler: ranks sequences by length (longest first,
// ties by index: a stable order), gives each the slice count above, and writes
// every (sequence, head, slice) work item in rank order, so the hardware's
// in-order CTA dispatch runs the longest chains first (LPT).  *nwork gets the
// item count.  Validates cu_seqlens into the error word.  Neither the order
// nor the slicing changes a bit.  With valid cu_seqlens the items fit the
// host's bound `cap`; items past it (possible only for malformed cu_seqlens,
// whose clamped lengths may add up to more than T) are not written.
__global__ void fwd_sched_kernel(const int32_t* __restrict__ cu, int N, int T, int HV, int dv, int forced_ns,
                                 int split, int slots, long long cap, int32_t* __restrict__ work,
                                 int32_t* __restrict__ nwork, unsigned* __restrict__ err) {
    constexpr int kTile = 1024;
    __shared__ int lens[kTile];
    const long long total = (long long)T * HV;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    int my_len = 0;
    if (n < N) {
        const int a = cu[n], b = cu[n + 1];
        if ((n == 0 && a != 0) || b < a || (n == N - 1 && b != T)) atomicOr(err, GDN_DEVERR_CU_SEQLENS);
        const int lo = min(max(a, 0), T), hi = min(max(b, lo), T);
        my_len = hi - lo;
    }
    long long offset = 0;
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
                if ((lm > my_len) || (lm == my_len && m < n))
                    offset += (long long)HV * fwd_slices(lm, forced_ns, split, slots, total);
            }
        }
    }
    if (n < N) {
        const int ns = fwd_slices(my_len, forced_ns, split, slots, total);
        const int rows = dv / ns, rlog = forced_ns > 0 ? 2 : (ns == 4 ? 0 : (ns == 2 ? 1 : 2));
        for (int h = 0; h < HV; ++h)
            for (int sl = 0; sl < ns; ++sl) {
                const long long idx = offset + (long long)h * ns + sl;
                if (idx < cap) work[idx] = fwd_item(n * HV + h, sl * rows, rlog);
            }
        atomicAdd(nwork, HV * ns);
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
// One unit (sequence n, head h, rows row0 .. row0 + rows - 1) with R rows per
// thread, all of them in one slot group of gdn_token_step.cuh.
template <typename Tin, int DK, typename Prm, int R>
__device__ __forceinline__ void fwd_unit(FwdSmem<Tin, DK>& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                         const CUtensorMap* tm_v, const Prm& p, int n, int h, int row0) {
    using Y = ts::Layout<DK, R, R>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const ts::Place pl = ts::place_of<DK, R>(tid);
    const int rows = p.rows4 * R / 4;
    // every thread holds rows unless a warp spans more rows than the smallest unit (16 rows)
    constexpr bool kAllActive = 32 * R / Y::L <= 16;
    const bool active = kAllActive || pl.grp * R < rows;
    const bool storer = active && ts::stores_row<DK, R>(pl);
    const int hk = h / p.G;
    const int vcol = p.forced ? row0 : 0;  // first v column of the TMA box
    int bos = p.cu[n], eos = p.cu[n + 1];
    bos = min(max(bos, 0), p.T);
    eos = min(max(eos, bos), p.T);
    const int L = eos - bos;
    const int row = row0 + pl.grp * R;  // first row of this thread's group
    const int orow = row + pl.own;      // the row whose output this thread may store
    const size_t soff = (((size_t)n * p.HV + h) * p.dv + row) * DK;

    ts::Rows<DK> S;
    if (active && p.init_state) ts::load_rows<DK, R, R>(S, p.init_state + soff, pl);
    else ts::zero_rows<DK>(S);

    if (L > 0) {
        const int nchunks = (L + kTC - 1) / kTC;
        const uint32_t bytes = (uint32_t)((2 * p.tb * DK + p.tb * p.vw) * sizeof(Tin));
        if (tid == 0) {
            for (int s = 0; s < kStages; ++s) mbar_init(&sm.bar[s], 1);
            sm.abort_flag = 0;
            fence_barrier_init();
        }
        __syncthreads();
        if (tid == 0)
            for (int c = 0; c < min(kStages, nchunks); ++c)
                issue_chunk(sm, tm_q, tm_k, tm_v, c, bos, hk, h, vcol, bytes);

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
            if (tid < tc) {
                const float a = gate_alpha(gb.x);
                sm.ab[tid] = make_float4(a, a, gb.y, __fmul_rn(a, gb.y));
            }
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
            const Tin* __restrict__ vt = sm.v[st] + (orow - vcol);  // this thread's v, token by token
            // Token loop, software-pipelined by one token: the reduce-scatter of
            // token t's output runs next to token t+1's u reduction (it is off
            // the recurrence's critical path); every operation is unchanged.
            float op[R];
#pragma unroll
            for (int j = 0; j < R; ++j) op[j] = 0.f;
            const size_t ostride = (size_t)p.HV * p.dv;
            Tin* __restrict__ optr = out + ((size_t)t0 * p.HV + h) * p.dv + orow - ostride;  // token t - 1's row
            const float* kt = sm.kn;
            const float* qt = sm.qn;
            for (int t = 0; t < tc; ++t) {
                const float4 ab = sm.ab[t];
                const float bv = __fmul_rn(ab.z, active ? ld_in(vt) : 0.f);
                float up[R];
                float2 w[R];
                ts::dot_part<DK, R, 0>(S, kt, pl.e, up);
                const float oprev = ts::reduce_scatter<DK, R>(op);  // token t - 1's output (t > 0)
                const float u = ts::reduce_scatter<DK, R>(up);
                if (t > 0 && storer) st_in(optr, oprev);
                ts::gather_rows<DK, R>(ts::delta_w(ab.w, bv, u), w);
                ts::update_part<DK, R, 0>(S, kt, qt, pl.e, make_float2(ab.x, ab.y), w, op);
                vt += p.vw;
                optr += ostride;
                kt += DK;
                qt += DK;
            }
            const float olast = ts::reduce_scatter<DK, R>(op);
            if (storer) st_in(optr, olast);
            if constexpr (std::is_same<Prm, SnapParams>::value) {
                // the state after `done` tokens of this sequence, at every snap_every-th token
                const int done = t0 + tc - bos;
                if (done % p.snap_every == 0) {
                    const int slot = p.snap_cu[n] + done / p.snap_every - 1;
                    if (active && slot >= 0 && slot < p.snap_cu[n + 1] && slot < p.snap_slots)
                        ts::store_rows<DK, R, R>(S, p.snap + (((size_t)slot * p.HV + h) * p.dv + row) * DK, pl);
                }
            }
            __syncthreads();
            if (tid == 0 && c + kStages < nchunks)
                issue_chunk(sm, tm_q, tm_k, tm_v, c + kStages, bos, hk, h, vcol, bytes);
        }
    }
    if (active && p.final_state) ts::store_rows<DK, R, R>(S, p.final_state + soff, pl);
}

// The grid is an upper bound on the number of work items; the CTAs past it exit.
template <typename Tin, int DK, typename Prm>
__global__ void __launch_bounds__(ts::threads_for_rows<DK>(kMaxSlice), 2)
    gdn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Prm p) {
    if ((int)blockIdx.x >= *p.nwork) return;
    extern __shared__ unsigned char smem_raw[];
    FwdSmem<Tin, DK>& sm =
        *reinterpret_cast<FwdSmem<Tin, DK>*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int item = p.work[blockIdx.x];
    const int nh = item >> 5, row0 = ((item >> 2) & 7) << 4, rlog = item & 3;
    const int h = nh % p.HV, n = nh / p.HV;
    if (rlog == 2) fwd_unit<Tin, DK, Prm, 4>(sm, &tm_q, &tm_k, &tm_v, p, n, h, row0);
    else if (rlog == 1) fwd_unit<Tin, DK, Prm, 2>(sm, &tm_q, &tm_k, &tm_v, p, n, h, row0);
    else fwd_unit<Tin, DK, Prm, 1>(sm, &tm_q, &tm_k, &tm_v, p, n, h, row0);
}

template <typename Tin, int DK, typename Prm>
static gdn_status launch_fwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                               const Prm& p, long long grid, cudaStream_t stream) {
    const size_t smem = sizeof(FwdSmem<Tin, DK>) + 128;
    auto kern = gdn_fwd_kernel<Tin, DK, Prm>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    kern<<<(unsigned)grid, ts::threads_for_rows<DK>(p.rows4), smem, stream>>>(mq, mk, mv, p);
    return launch_status();
}

template <typename Tin, typename Prm>
static gdn_status launch_fwd_dk(int dk, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                const Prm& p, long long grid, cudaStream_t stream) {
    switch (dk) {
        case 16: return launch_fwd_t<Tin, 16, Prm>(mq, mk, mv, p, grid, stream);
        case 32: return launch_fwd_t<Tin, 32, Prm>(mq, mk, mv, p, grid, stream);
        case 64: return launch_fwd_t<Tin, 64, Prm>(mq, mk, mv, p, grid, stream);
        case 128: return launch_fwd_t<Tin, 128, Prm>(mq, mk, mv, p, grid, stream);
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

// Slicing plan of a forward call.  Automatic slices (dv_slice == 0) may split
// the heads of long sequences in 2 or 4 when dk >= 32 and dv >= 64 (units of
// at least 16 rows); a forced dv_slice gives every head dv / dv_slice slices.
struct FwdPlan {
    int forced_ns;  // slices per head when forced, else 0
    int split;      // automatic splitting allowed
    int rows4;      // rows of a unit at 4 rows per thread
};

static FwdPlan fwd_plan(const gdn_shape* s) {
    FwdPlan pl;
    const int dvs = pick_dv_slice(s);
    pl.forced_ns = s->dv_slice ? s->dv / dvs : 0;
    pl.split = !s->dv_slice && s->dk >= 32 && s->dv >= 64;
    pl.rows4 = dvs;
    return pl;
}

// Work items a call can produce on a device with `slots` CTA slots: forced,
// N * HV * forced_ns; automatic, N * HV plus up to 3 * HV more for each
// sequence longer than 1.5 T * HV / slots, of which there are fewer than slots / HV.
// slots = 0 gives the bound for any device (every head split in 4).
long long fwd_max_items(const gdn_shape* s, int slots) {
    const FwdPlan pl = fwd_plan(s);
    const long long nh = (long long)s->N * s->HV;
    if (pl.forced_ns) return nh * pl.forced_ns;
    if (!pl.split) return nh;
    if (slots <= 0) return 4 * nh;
    return nh + 3LL * s->HV * std::min<long long>(s->N, slots / s->HV + 1);
}

// Workspace: the 256-byte header (word 0: device error bits, word 1: the
// number of work items) and the work list.
size_t fwd_workspace_size(const gdn_shape* s) {
    return kWsHeader + (((size_t)fwd_max_items(s, 0) * sizeof(int32_t) + 255) & ~size_t(255));
}

// CTA slots of the current device: two forward CTAs per SM.
static int fwd_slots() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 0;
    return 2 * sms;
}

// Shared by the allocating entry points and the allocation-free one: `header`
// is the workspace header (error word, item count) and `work` the list, room
// for fwd_max_items(s, slots) items.
gdn_status run_recurrent_fwd(const gdn_shape* s, const void* q, const void* k, const void* v, const float* g,
                             const float* beta, const float* init_state, const int32_t* cu, void* out,
                             float* final_state, int32_t* work, unsigned* header, int slots, cudaStream_t stream,
                             float* snap = nullptr, const int32_t* snap_cu = nullptr, int snap_every = 0,
                             int snap_slots = 0) {
    if (s->N == 0) return GDN_OK;
    const FwdPlan plan = fwd_plan(s);
    const int split = plan.split && slots > 0;
    const long long grid = split ? fwd_max_items(s, slots) : fwd_max_items(s, 0) / (plan.split ? 4 : 1);
    const int vw = plan.forced_ns ? plan.rows4 : s->dv;

    CUtensorMap mq{}, mk{}, mv{};
    if (s->T_total > 0) {
        gdn_status st;
        // box height min(kTC, T): a sequence shorter than kTC never needs more rows than T
        const uint32_t tb = (uint32_t)std::min(kTC, s->T_total);
        if ((st = encode_map_3d(&mq, q, s->dtype, s->dk, s->HK, s->T_total, s->dk, tb)) != GDN_OK) return st;
        if ((st = encode_map_3d(&mk, k, s->dtype, s->dk, s->HK, s->T_total, s->dk, tb)) != GDN_OK) return st;
        if ((st = encode_map_3d(&mv, v, s->dtype, s->dv, s->HV, s->T_total, vw, tb)) != GDN_OK) return st;
    }
    unsigned* err = header;
    int32_t* nwork = reinterpret_cast<int32_t*>(header + 1);
    if (cudaMemsetAsync(header, 0, 2 * sizeof(unsigned), stream) != cudaSuccess) return GDN_ERR_CUDA;
    fwd_sched_kernel<<<(s->N + 255) / 256, 256, 0, stream>>>(cu, s->N, s->T_total, s->HV, s->dv, plan.forced_ns,
                                                           split, slots, grid, work, nwork, err);
    if (launch_status() != GDN_OK) return GDN_ERR_CUDA;

    FwdParams p;
    p.g = g;
    p.beta = beta;
    p.init_state = init_state;
    p.cu = cu;
    p.out = out;
    p.final_state = final_state;
    p.work = work;
    p.nwork = nwork;
    p.err = err;
    p.N = s->N;
    p.T = s->T_total;
    p.HV = s->HV;
    p.G = s->HV / s->HK;
    p.dv = s->dv;
    p.use_norm = s->use_qk_l2norm ? 1 : 0;
    p.rows4 = plan.rows4;
    p.forced = plan.forced_ns ? 1 : 0;
    p.vw = vw;
    p.tb = std::min(kTC, s->T_total);
    if (snap && snap_cu && snap_slots > 0 && snap_every > 0) {
        SnapParams sp;
        static_cast<FwdParams&>(sp) = p;
        sp.snap = snap;
        sp.snap_cu = snap_cu;
        sp.snap_every = snap_every;
        sp.snap_slots = snap_slots;
        if (s->dtype == GDN_BF16) return launch_fwd_dk<__nv_bfloat16>(s->dk, mq, mk, mv, sp, grid, stream);
        return launch_fwd_dk<float>(s->dk, mq, mk, mv, sp, grid, stream);
    }
    if (s->dtype == GDN_BF16) return launch_fwd_dk<__nv_bfloat16>(s->dk, mq, mk, mv, p, grid, stream);
    return launch_fwd_dk<float>(s->dk, mq, mk, mv, p, grid, stream);
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
                             fwd_slots(), static_cast<cudaStream_t>(stream));
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
                             fwd_slots(), static_cast<cudaStream_t>(stream), snap_states, snap_cu, snap_every,
                             num_snap_slots);
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  Its scratch (device error word, item count and work list) is a
// fixed array in the library's own device memory instead of a caller-supplied
// workspace.  Every device that loads the library holds this array (about
// 256 KB) until the process exits.  All calls share it, so two calls whose
// work overlaps on the GPU race on it; the error word is cleared by each call
// and the work list is rewritten in full by each call.
namespace gdn {

constexpr int kStaticUnits = 1 << 16;    // max work items (fwd_max_items)
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
    const int slots = fwd_slots();
    if (fwd_max_items(shape, slots) > kStaticUnits) return GDN_ERR_WORKSPACE;
    int32_t* base = static_scratch_on_current_device();
    if (!base) return GDN_ERR_CUDA;
    return run_recurrent_fwd(shape, q, k, v, g, beta, init_state, cu_seqlens, out, final_state,
                             base + kStaticHeaderWords, reinterpret_cast<unsigned*>(base), slots,
                             static_cast<cudaStream_t>(stream));
}
