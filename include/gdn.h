/*
 * gdn.h -- C ABI of the batch-invariant Gated DeltaNet library (sm_103a).
 *
 * The operation.  For every sequence n (tokens cu_seqlens[n] .. cu_seqlens[n+1]-1
 * of a packed batch) and every value head h, with k-head hk = h / (HV/HK):
 *
 *     q^_t = q_t / sqrt(|q_t|^2 + 1e-6),  k^_t likewise       (use_qk_l2norm != 0)
 *     a_t  = exp(g_t)                                           (g: log-decay)
 *     S_t  = a_t S_{t-1} (I - b_t k^_t k^_t^T) + b_t v_t k^_t^T (S: dv x dk, fp32)
 *     o_t  = S_t q^_t                                           (read after the update)
 *
 * This is the gated delta rule of "Defending Against the Training-Inference
 * Numeric Mismatch in RL (Especially Linear Attention)" (section 3.2): one
 * recurrent kernel serves the RL trainer's forward pass and the rollout
 * engine's prefill and decode alike, the state cache is fp32 (section 4.2
 * setup tables), and the chunked form is kept for gradients only.
 *
 * Invariance contract.  The bits of o and of the final state of a sequence
 * depend only on that sequence's own inputs: not on which other sequences
 * share the batch, not on N or the packing order, not on dv_slice, and not on
 * whether its tokens arrive in one gdn_recurrent_fwd call or as one call
 * followed by any number of gdn_decode_step calls (or any split into several
 * gdn_recurrent_fwd calls chained through final_state -> init_state).
 * Every dk contraction uses one fixed reduction tree; nothing is reduced
 * across sequences or split over dk.
 *
 * Memory and ownership.  Every tensor pointer is a caller-owned DEVICE
 * pointer to dense row-major data: q, k, v, out, d_out, dq, dk, dv, every
 * state and the workspace 16-byte aligned; g, beta, dg, dbeta, cu_seqlens and
 * state_indices 4-byte aligned.  The library allocates
 * no device memory; scratch comes from the caller's workspace, sized by
 * gdn_workspace_size, except for gdn_recurrent_fwd_noalloc, whose scratch is
 * a fixed array inside the library (described at that entry point).  All calls are asynchronous on `stream` (a
 * cudaStream_t; NULL = legacy default stream).  The return value reports
 * host-side validation and launch errors only; device faults surface at the
 * caller's next synchronisation.  No call throws.  Layouts:
 *
 *     q, k        [T_total, HK, dk]        dtype            (bf16 or fp32)
 *     v, out      [T_total, HV, dv]        dtype
 *     g, beta     [T_total, HV]            fp32  (beta already in (0,1): sigmoid applied by caller)
 *     states      [N, HV, dv, dk]          fp32, dk fastest
 *     cu_seqlens  [N + 1]                  int32, cu[0] = 0, non-decreasing, cu[N] = T_total
 *
 * Supported: dk, dv in {16, 32, 64, 128}; HV % HK == 0; dv_slice in
 * {0 (auto), 16, 32, 64, 128} dividing dv.  Anything else returns
 * GDN_ERR_UNSUPPORTED or GDN_ERR_INVALID_ARG.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad shape, aliasing not allowed */
    GDN_ERR_UNSUPPORTED = -2, /* dk/dv/dtype/dv_slice outside the supported set */
    GDN_ERR_WORKSPACE = -3,   /* workspace missing or smaller than gdn_workspace_size */
    GDN_ERR_CUDA = -4         /* a CUDA runtime call or kernel launch failed */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype; /* dtype of q, k, v, out, d_out, dq, dk, dv */

typedef enum { GDN_OP_FWD = 0, GDN_OP_DECODE = 1, GDN_OP_BWD = 2 } gdn_op;

typedef struct {
    int N;             /* sequences (decode: batch size) */
    int T_total;       /* packed tokens (decode: must equal N) */
    int HK, HV;        /* k-heads (q has HK heads too) and value heads, HV % HK == 0 */
    int dk, dv;        /* key and value head dims */
    gdn_dtype dtype;
    int use_qk_l2norm; /* 1: normalise q and k inside the kernel (eps 1e-6); 0: use as given */
    int dv_slice;      /* rows of S per CTA; 0 = automatic.  Never changes any output bit. */
} gdn_shape;

/* Device-side error bits, readable with gdn_read_device_error. */
#define GDN_DEVERR_CU_SEQLENS 1u /* cu_seqlens not 0-based, decreasing, or cu[N] != T_total */
#define GDN_DEVERR_TIMEOUT 2u    /* a bounded wait on an asynchronous copy gave up */
#define GDN_DEVERR_SMEM_ALIGN 4u /* shared memory not 1 KB aligned for a swizzled tensor-core operand */

/* Bytes of device workspace `op` needs for `shape` (0 if it needs none or the
 * shape is invalid).  FWD: the varlen work list; BWD: chunk states and
 * per-chunk factors.  DECODE needs none. */
size_t gdn_workspace_size(const gdn_shape* shape, int op);

/*
 * Recurrent forward over a packed varlen batch (prefill and trainer forward).
 * init_state may be NULL (zero state); final_state may be NULL (not written)
 * and may alias init_state (each (sequence, head) reads its state before
 * writing it).  out must not alias any input.  A sequence of length 0 copies
 * its init_state (or zeros) to final_state.  Two launches on `stream`: the
 * varlen scheduler (work list sorted by length, longest first, into the
 * workspace) and the recurrent kernel.  No host synchronisation.
 */
gdn_status gdn_recurrent_fwd(const gdn_shape* shape, const void* q, const void* k,
                             const void* v, const float* g, const float* beta,
                             const float* init_state, const int32_t* cu_seqlens, void* out,
                             float* final_state, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * gdn_recurrent_fwd that also keeps state snapshots for prefix caching (on
 * the pages, vLLM's --mamba-cache-mode align snapshots keep prefix caching
 * working once every path runs the recurrent kernel: "Defending Against the
 * Training-Inference Numeric Mismatch in RL (Especially Linear Attention)",
 * section 3.2).  For every sequence n, after each snap_every-th
 * token of that sequence (token counts snap_every, 2*snap_every, ...), the
 * fp32 state is written to snap_states[snap_cu[n] + m - 1] for the m-th
 * snapshot, as long as that slot is below snap_cu[n + 1] and num_snap_slots;
 * snap_states is [num_snap_slots, HV, dv, dk], snap_cu int32 [N + 1] on the
 * device (the caller sizes it, e.g. with floor(len_n / snap_every) slots per
 * sequence).  snap_every must be a positive multiple of 32 (snapshots are
 * taken at the kernel's 32-token chunk boundaries), else GDN_ERR_UNSUPPORTED;
 * snap_states must not alias init_state or final_state.  Each snapshot is bit
 * for bit the final_state of gdn_recurrent_fwd over that prefix, so resuming
 * from it reproduces the rest of the sequence exactly.  Same workspace, launches
 * and outputs as gdn_recurrent_fwd.
 */
gdn_status gdn_recurrent_fwd_snapshots(const gdn_shape* shape, const void* q, const void* k,
                                       const void* v, const float* g, const float* beta,
                                       const float* init_state, const int32_t* cu_seqlens,
                                       void* out, float* final_state, int snap_every,
                                       const int32_t* snap_cu, int num_snap_slots,
                                       float* snap_states, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * One decode token per sequence on a cached fp32 state, updated in place.
 * shape->T_total must equal shape->N; q, k, v, g, beta, out hold one token
 * per sequence.  state is a pool [num_slots, HV, dv, dk]; sequence b uses
 * slot state_indices[b] (state_indices NULL: slot b, needs num_slots >= N).
 * A negative or out-of-range slot skips sequence b (its out row is left
 * untouched).  The non-negative entries of state_indices must be distinct:
 * the library does not check this, and two batch rows on one slot would read
 * and write that slot at the same time (a race with an undefined result).
 * Bit-identical to continuing gdn_recurrent_fwd by one token.
 * One launch, no workspace, no host synchronisation: capturable as-is.
 */
gdn_status gdn_decode_step(const gdn_shape* shape, const void* q, const void* k, const void* v,
                           const float* g, const float* beta, float* state,
                           const int32_t* state_indices, int num_slots, void* out,
                           void* stream);

/*
 * Chunked (WY-form) backward of gdn_recurrent_fwd for the loss
 * L = sum <d_out, out> + <d_final_state, final_state>, chunk size 64,
 * chunks restarting at every sequence start.  Produces dq, dk (dtype, [T,HK,dk],
 * summed over the value heads that share a k-head), dv (dtype), dg and dbeta
 * (fp32, [T,HV]) and d_init_state (fp32, may be NULL).  init_state and
 * d_final_state may be NULL (zero).  Gradients are not bit-invariant (the
 * pages need invariance only for the forward); they are deterministic.  Dense
 * products run on the tensor cores: TF32 operands with fp32 accumulation for
 * bf16 inputs, a 3xTF32 split (about fp32 accuracy) for fp32 inputs.  At
 * dk = dv = 128 with bf16 inputs, the per-chunk states and state gradients
 * pass between the kernels (in the workspace) as fp16 of their TF32 values,
 * with a power-of-two factor per 32 x 32 tile: the products read the same
 * TF32 operands as from fp32 copies, except for values below 2^-29 of their
 * tile's largest.
 */
gdn_status gdn_chunk_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* init_state,
                         const int32_t* cu_seqlens, const void* d_out,
                         const float* d_final_state, void* dq, void* dk, void* dv, float* dg,
                         float* dbeta, float* d_init_state, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * gdn_recurrent_fwd without a caller workspace.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc: a host program whose device memory is owned by another
 * allocator (a framework's caching allocator or a serving engine that
 * reserves the whole device at start-up) and that has no buffer to lend, or
 * a path where allocating is not allowed because cudaMalloc / cudaFree may
 * synchronise the device.  Same arguments, results and bits as
 * gdn_recurrent_fwd minus the workspace; it allocates nothing.
 *
 * Its scratch is a fixed array inside the library's device memory, sized for
 * N * HV * (dv / dv_slice) <= 65536 work units (about 256 KB, held on every
 * device that loads the library until the process exits).  Larger shapes
 * return GDN_ERR_WORKSPACE.  The first call on a device looks the array's
 * address up (cudaGetSymbolAddress, with that device current); make that
 * first call before any stream capture.  The address is kept for the life of
 * the process: after cudaDeviceReset on a device, do not call this entry
 * point on that device again (the kept address may be stale).  All calls
 * share the array: calls
 * that overlap on the GPU (on different streams, or from several threads)
 * race on it and must be serialised by the caller.  Its device error bits are
 * not readable through gdn_read_device_error.
 */
gdn_status gdn_recurrent_fwd_noalloc(const gdn_shape* shape, const void* q, const void* k,
                                     const void* v, const float* g, const float* beta,
                                     const float* init_state, const int32_t* cu_seqlens,
                                     void* out, float* final_state, void* stream);

/* Read (and clear) the device error bits a FWD or BWD call left in its
 * workspace.  Synchronises `stream`.  *bits = 0 means no device error. */
gdn_status gdn_read_device_error(void* workspace, unsigned int* bits, void* stream);

/* Static text for a status code. */
const char* gdn_status_string(gdn_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
