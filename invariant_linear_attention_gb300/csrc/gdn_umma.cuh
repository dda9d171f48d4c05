// gdn_umma.cuh -- fifth-generation tensor core (tcgen05) building blocks for the
// chunked backward: TF32 products with operands in shared memory, fp32
// accumulators in tensor memory (TMEM), completion on an mbarrier, and the 2-D
// tensor copies that bring operands into the 128-byte-swizzled layout.
//
// Operand layout ("K-major, no swizzle"): a matrix X with rows n and reduction
// index k is stored as 8-row x 16-byte core matrices (8 rows of 4 fp32 each,
// 128 contiguous bytes).  Core matrices that follow each other along k are 128
// bytes apart (the descriptor's leading byte offset); groups of 8 rows are
// `sbo` bytes apart (its stride byte offset).  With every k of a row group
// stored together, sbo = 8 rows x K x 4 bytes, and element (n, k) sits at
//     (n / 8) * sbo + (k / 4) * 128 + (n % 8) * 16 + (k % 4) * 4.
// One MMA instruction of kind::tf32 consumes 8 values of k (two core matrices),
// so the descriptor of step s starts 256 * s bytes into the operand.
//
// Accumulator layout for M = 128 with one CTA: row m of D is TMEM lane m, column
// n is TMEM column (base + n).  A warp reads only the 32 lanes of its quarter
// (warp index mod 4).
//
// Values enter the tensor core as TF32: the producers round each operand to
// TF32 (round to nearest, ties away) when they write it, as the mma.sync
// path does for bf16 inputs.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_async.cuh"

namespace gdn {

__host__ __device__ constexpr uint32_t umma_koff(int n, int k, uint32_t sbo) {
    return (uint32_t)(n >> 3) * sbo + (uint32_t)(k >> 2) * 128u + (uint32_t)(n & 7) * 16u + (uint32_t)(k & 3) * 4u;
}

// Shared-memory matrix descriptor: start address, leading byte offset 128, stride byte offset
// sbo (all >> 4), descriptor version 1 (bits 46-48 = 0b001), no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
           ((uint64_t)1 << 46);
}

// Instruction descriptor for kind::tf32: D fp32 (bits 4-5 = 1), A and B TF32 (bits 7-9 and
// 10-12 = 2), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ float tf32_round(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
__device__ __forceinline__ float4 tf32_round4(float4 v) {
    return make_float4(tf32_round(v.x), tf32_round(v.y), tf32_round(v.z), tf32_round(v.w));
}

// TMEM allocation by one whole warp; the address lands in *slot (shared memory).  An allocation
// waits while the SM's 512 columns are taken.  The kernels here hold 512 columns with one CTA per
// SM (512 threads at up to 128 registers fill the register file) or 256 columns with at most two
// CTAs per SM (512 threads at 64 registers), so the allocation never waits.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D (+)= A B^T over one K = 8 step; issued by a single thread.
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D (+)= A B^T for A (M x K) and B (N x K) in the layout above, K a multiple of 8.
__device__ __forceinline__ void umma_tf32_k(uint32_t d_tmem, uint32_t a_saddr, uint32_t a_sbo, uint32_t b_saddr,
                                            uint32_t b_sbo, uint32_t idesc, int K, bool accumulate) {
    for (int s = 0; s < K / 8; ++s)
        umma_tf32(d_tmem, umma_desc(a_saddr + 256u * s, a_sbo), umma_desc(b_saddr + 256u * s, b_sbo), idesc,
                  accumulate || s > 0);
}

// D (+)= A B^T over one K = 8 step with A in TMEM (row m in lane m, its 8 values of k in the columns
// from a_tmem on, read as TF32) and B in shared memory; issued by a single thread.
__device__ __forceinline__ void umma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// An MMA operand in shared memory, in one of two layouts:
//   rows == 0: the layout above, row groups sbo apart;
//   rows != 0: K-major with the 128-byte swizzle: rows of 32 values (128 bytes) whose 16-byte chunks
//     sit at position chunk ^ (row % 8), 8-row atoms of 1 KB (sbo = 1024), and atom columns of
//     rows x 128 bytes along k -- what a tensor copy with the 128-byte swizzle writes for a box of 32
//     values x rows.  The atoms must start on 1 KB boundaries.  A K = 8 step inside an atom column
//     moves the start address by 32 bytes; the swizzle applies to the address bits.
struct UmmaOp {
    uint32_t base, sbo, rows;
};
__device__ __forceinline__ UmmaOp op_k(uint32_t base, uint32_t sbo) { return UmmaOp{base, sbo, 0u}; }
__device__ __forceinline__ UmmaOp op_sw(uint32_t base, uint32_t rows) { return UmmaOp{base, 1024u, rows}; }

// Descriptor of the swizzled layout: leading byte offset unused (16), stride byte offset 1024,
// version 1, base offset 0, layout type 2 (128-byte swizzle) at bits 61-63.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024u >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint64_t umma_op_desc(const UmmaOp& o, int s) {
    return o.rows ? umma_desc_sw128(o.base + (uint32_t)(s >> 2) * o.rows * 128u + (uint32_t)(s & 3) * 32u)
                  : umma_desc(o.base + 256u * s, o.sbo);
}
// Byte offset of element (n, k) in the swizzled layout with `rows` rows.
__host__ __device__ constexpr uint32_t sw128_off(int n, int k, int rows) {
    return (uint32_t)(k >> 5) * (uint32_t)rows * 128u + (uint32_t)n * 128u +
           ((uint32_t)(((k & 31) >> 2) ^ (n & 7)) << 4) + (uint32_t)(k & 3) * 4u;
}

// D (+)= A B^T for operands in either layout, K a multiple of 8.
__device__ __forceinline__ void umma_tf32_op(uint32_t d_tmem, const UmmaOp& a, const UmmaOp& b, uint32_t idesc, int K,
                                             bool accumulate) {
    for (int s = 0; s < K / 8; ++s) umma_tf32(d_tmem, umma_op_desc(a, s), umma_op_desc(b, s), idesc, accumulate || s > 0);
}

// 2-D tiled tensor copy of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Arrive on bar once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Columns [col, col + 8 * NX) of this warp's 32 lanes, one lane per thread, into v: one load of shape
// 32x32b.x8, .x16 or .x32 (NX = 1, 2 or 4) and its wait in one asm statement, so no use of the
// registers can move ahead of the wait.
template <int NX>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[8 * NX]) {
    static_assert(NX == 1 || NX == 2 || NX == 4, "8, 16 or 32 columns");
    uint32_t r[8 * NX];
    if constexpr (NX == 1) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr)
                     : "memory");
    } else if constexpr (NX == 2) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                     "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                       "=r"(r[14]), "=r"(r[15])
                     : "r"(taddr)
                     : "memory");
    } else {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                     "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                     "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                       "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
                       "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
                       "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                     : "r"(taddr)
                     : "memory");
    }
#pragma unroll
    for (int j = 0; j < 8 * NX; ++j) v[j] = __uint_as_float(r[j]);
}

// Two loads of 16 columns (at ta into va, at tb into vb) and one wait for both.
__device__ __forceinline__ void tmem_ld_pair(uint32_t ta, float (&va)[16], uint32_t tb, float (&vb)[16]) {
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(ta), "r"(tb)
                 : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        va[j] = __uint_as_float(r[j]);
        vb[j] = __uint_as_float(r[16 + j]);
    }
}

// Rows 16 lanes x 8 * NX columns of TMEM from taddr on (an M = 64 accumulator keeps 16 rows in
// lanes 0..15 of each warp quarter) over all 32 threads, shape 16x256b (NX = 2 or 4): in column
// block n (columns 8 n ..) thread t holds v[4 n] = (row t / 4, column 8 n + 2 (t % 4)), v[4 n + 1]
// the next column, v[4 n + 2], v[4 n + 3] the same two columns of row t / 4 + 8.  One load and its
// wait in one asm statement.
template <int NX>
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[4 * NX]) {
    static_assert(NX == 2 || NX == 4, "16 or 32 columns");
    uint32_t r[4 * NX];
    if constexpr (NX == 2) {
        asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr)
                     : "memory");
    } else {
        asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 "
                     "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                       "=r"(r[14]), "=r"(r[15])
                     : "r"(taddr)
                     : "memory");
    }
#pragma unroll
    for (int j = 0; j < 4 * NX; ++j) v[j] = __uint_as_float(r[j]);
}

// Two 16x256b loads of 16 columns (at ta into va, at tb into vb) and one wait for both.
__device__ __forceinline__ void tmem_ld16_pair(uint32_t ta, float (&va)[8], uint32_t tb, float (&vb)[8]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n\t"
                 "tcgen05.ld.sync.aligned.16x256b.x2.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(ta), "r"(tb)
                 : "memory");
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        va[j] = __uint_as_float(r[j]);
        vb[j] = __uint_as_float(r[8 + j]);
    }
}

// The reverse of tmem_ld (NX = 1 or 2): v into columns [col, col + 8 * NX) of this warp's 32 lanes,
// then a wait for the stores, so that a barrier after it orders them before the next MMA on those
// columns.
template <int NX>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float (&v)[8 * NX]) {
    static_assert(NX == 1 || NX == 2, "8 or 16 columns");
    uint32_t r[8 * NX];
#pragma unroll
    for (int j = 0; j < 8 * NX; ++j) r[j] = __float_as_uint(v[j]);
    if constexpr (NX == 1) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n\t"
                     "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
    } else {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                     "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
                     "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                     "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                     : "memory");
    }
}

}  // namespace gdn
