// gdn_decode.cu -- one decode token per sequence on a cached fp32 state.
//
// The same recurrent step as the prefill kernel (gdn_token_step.cuh), applied
// once to the state the cache holds, so a prompt run by gdn_recurrent_fwd and
// continued token by token here yields exactly the bits of one pass over the
// whole sequence: the page "Defending Against the Training-Inference Numeric
// Mismatch in RL (Especially Linear Attention)", section 3.2, gets its
// prefill/decode parity by running one recurrent kernel for both.  The state round trip
// (dv x dk fp32 read and written per (sequence, head)) makes this HBM-bound:
// each thread issues all of its row loads up front, the q/k normalisation
// runs while they are in flight, and the new rows are streamed back.
#include <algorithm>

#include "gdn_host.h"
#include "gdn_step.cuh"
#include "gdn_token_step.cuh"

namespace gdn {

struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    float* state;
    const int32_t* idx;
    void* out;
    int N, HK, HV, G, dv, dvs, nslices, num_slots, use_norm;
};

template <typename Tin, int DK>
__global__ void __launch_bounds__(ts::threads_for_rows<DK>(128)) gdn_decode_kernel(const DecodeParams p) {
    constexpr int RG = 2;  // two slot groups: their reduce-scatters interleave (a decode step has one token)
    using Y = ts::Layout<DK, RG>;
    __shared__ __align__(16) float qn[DK];
    __shared__ __align__(16) float kn[DK];
    __shared__ float2 ab;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const ts::Place pl = ts::place_of<DK, RG>(tid);
    const int dvs = p.dvs;
    const bool active = pl.grp * Y::R < dvs;
    const int unit = blockIdx.x;
    const int slice = unit % p.nslices;
    const int h = (unit / p.nslices) % p.HV;
    const int b = unit / (p.nslices * p.HV);
    const int hk = h / p.G;
    const int slot = p.idx ? p.idx[b] : b;
    if (slot < 0 || slot >= p.num_slots) return;  // uniform over the CTA

    const int row = slice * dvs + pl.grp * Y::R;
    float* srow = p.state + (((size_t)slot * p.HV + h) * p.dv + row) * DK;
    ts::Rows<DK> S;
    if (active) ts::load_rows<DK, RG>(S, srow, pl);
    else ts::zero_rows<DK>(S);

    const Tin* q = reinterpret_cast<const Tin*>(p.q) + ((size_t)b * p.HK + hk) * DK;
    const Tin* k = reinterpret_cast<const Tin*>(p.k) + ((size_t)b * p.HK + hk) * DK;
    for (int j = warp; j < 2; j += nwarps) {
        if (j) l2norm_warp<DK>(k, kn, lane, p.use_norm);
        else l2norm_warp<DK>(q, qn, lane, p.use_norm);
    }
    if (tid == 0) {
        const size_t gi = (size_t)b * p.HV + h;
        ab = make_float2(gate_alpha(p.g[gi]), p.beta[gi]);
    }
    const size_t vo = ((size_t)b * p.HV + h) * p.dv + row;
    const int lr0 = ts::row_of<DK, RG>(0, 0, pl.own), lr1 = ts::row_of<DK, RG>(1, 0, pl.own);
    const Tin* v = reinterpret_cast<const Tin*>(p.v) + vo;
    const float vown[2] = {active ? ld_in(v + lr0) : 0.f, active ? ld_in(v + lr1) : 0.f};
    __syncthreads();
    const float2 gab = ab;
    float o[2];
    ts::token_step<DK, RG>(S, kn, qn, pl, gab.x, gab.y, vown, o);
    if (active) {
        if (ts::stores_row<DK, RG>(pl)) {
            Tin* out = reinterpret_cast<Tin*>(p.out) + vo;
            st_in(out + lr0, o[0]);
            st_in(out + lr1, o[1]);
        }
        ts::store_rows<DK, RG>(S, srow, pl);
    }
}

template <typename Tin, int DK>
static gdn_status launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
    const int units = p.N * p.HV * p.nslices;
    gdn_decode_kernel<Tin, DK><<<units, ts::threads_for_rows<DK>(p.dvs), 0, stream>>>(p);
    return launch_status();
}

template <typename Tin>
static gdn_status launch_decode_dk(int dk, const DecodeParams& p, cudaStream_t stream) {
    switch (dk) {
        case 16: return launch_decode_t<Tin, 16>(p, stream);
        case 32: return launch_decode_t<Tin, 32>(p, stream);
        case 64: return launch_decode_t<Tin, 64>(p, stream);
        case 128: return launch_decode_t<Tin, 128>(p, stream);
    }
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn

extern "C" gdn_status gdn_decode_step(const gdn_shape* s, const void* q, const void* k, const void* v,
                                      const float* g, const float* beta, float* state,
                                      const int32_t* state_indices, int num_slots, void* out, void* stream) {
    using namespace gdn;
    gdn_status st = check_shape(s);
    if (st != GDN_OK) return st;
    if (s->T_total != s->N) return GDN_ERR_INVALID_ARG;
    if (s->N == 0) return GDN_OK;
    if (!q || !k || !v || !g || !beta || !state || !out || num_slots <= 0) return GDN_ERR_INVALID_ARG;
    if (!state_indices && num_slots < s->N) return GDN_ERR_INVALID_ARG;
    const void* vec[] = {q, k, v, state, out};
    for (const void* ptr : vec)
        if (ptr && !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
    const void* sca[] = {g, beta, state_indices};
    for (const void* ptr : sca)
        if (ptr && !aligned4(ptr)) return GDN_ERR_INVALID_ARG;
    if (out == q || out == k || out == v || out == state) return GDN_ERR_INVALID_ARG;

    DecodeParams p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.g = g;
    p.beta = beta;
    p.state = state;
    p.idx = state_indices;
    p.out = out;
    p.N = s->N;
    p.HK = s->HK;
    p.HV = s->HV;
    p.G = s->HV / s->HK;
    p.dv = s->dv;
    // automatic slice for decode: 64 rows (smaller CTAs keep more state bytes in
    // flight per SM; measured 157 us vs 164 us for 128 rows at batch 256)
    p.dvs = s->dv_slice ? s->dv_slice : std::min(s->dv, 64);
    p.nslices = s->dv / p.dvs;
    p.num_slots = num_slots;
    p.use_norm = s->use_qk_l2norm ? 1 : 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (s->dtype == GDN_BF16) return launch_decode_dk<__nv_bfloat16>(s->dk, p, cs);
    return launch_decode_dk<float>(s->dk, p, cs);
}
