// gdn_host.h -- host-side helpers shared by the entry points: argument
// validation, tensor-map encoding, device error word.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

// Workspace header: one 32-bit device error word, padded to 256 bytes.
constexpr size_t kWsHeader = 256;

inline bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline size_t elem_size(gdn_dtype t) { return t == GDN_BF16 ? 2 : 4; }

// Basic shape check common to every op.
inline gdn_status check_shape(const gdn_shape* s) {
    if (!s) return GDN_ERR_INVALID_ARG;
    if (s->N < 0 || s->T_total < 0 || s->HK <= 0 || s->HV <= 0 || s->HV % s->HK) return GDN_ERR_INVALID_ARG;
    if (s->dtype != GDN_F32 && s->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (!dim_ok(s->dk) || !dim_ok(s->dv)) return GDN_ERR_UNSUPPORTED;
    if (s->dv_slice != 0 && (!dim_ok(s->dv_slice) || s->dv_slice > s->dv)) return GDN_ERR_UNSUPPORTED;
    // The kernels index (token, head) pairs and work units with 32-bit integers and
    // elements with 64-bit offsets: T_total * HV (>= T_total * HK) and the unit count
    // N * HV * (dv / 16) must stay below 2^31, and a forward work item packs
    // n * HV + h into 26 bits.
    if ((long long)s->T_total * s->HV >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    if ((long long)s->N * s->HV * (s->dv / 16) >= (1LL << 31)) return GDN_ERR_UNSUPPORTED;
    if ((long long)s->N * s->HV >= (1LL << 26)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

// Rows of S per CTA.  Automatic choice: the whole head (dv <= 128).
inline int pick_dv_slice(const gdn_shape* s) { return s->dv_slice ? s->dv_slice : s->dv; }

// Encode a rank-3 tiled tensor map over a [d2][d1][d0] row-major tensor with box {b0, 1, b2}.
gdn_status encode_map_3d(CUtensorMap* map, const void* base, gdn_dtype dt, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint32_t b0, uint32_t b2);

// Encode a rank-2 tiled tensor map over rows of d0 elements of dt (row stride `stride` bytes, d1
// rows) with box {128 bytes of a row, box_rows} and the 128-byte swizzle: one copy lands box_rows
// rows of 128 bytes in the K-major swizzled operand layout of the tensor cores.
gdn_status encode_rows_sw128(CUtensorMap* map, const void* base, gdn_dtype dt, uint64_t d0, uint64_t d1, uint64_t stride,
                             uint32_t box_rows);

inline gdn_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
