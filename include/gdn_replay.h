/*
 * gdn_replay.h -- C ABI of the chunk-order-replaying variant of the Gated
 * DeltaNet forward (sm_103a).
 *
 * The main library makes prefill and decode agree by running ONE recurrent
 * kernel for both ("Defending Against the Training-Inference Numeric
 * Mismatch in RL (Especially Linear Attention)", section 3.2).  The other way
 * to the same guarantee is the one the Nemotron experiment takes for its
 * Mamba-2 layers: keep the chunked computation for prefill and make decode
 * replay the chunked order ("Finish RL Training Faster: Bitwise-Consistent,
 * High-Performance, Agent-Driven", the transfer experiment).  This header is
 * that variant for the gated delta rule, so the two designs can be compared
 * on the same hardware.
 *
 * The computation.  Chunks of GDN_REPLAY_CHUNK tokens start at every
 * sequence start.  Inside a chunk with start state S0, for its tokens
 * j = 0, 1, ... (k^, q^ L2-normalised as in gdn.h, gam_j the chunk's
 * cumulative log-decay g_0 + ... + g_j, Gam_j = exp(gam_j)):
 *
 *     c_ji = exp(gam_j - gam_i) <k^_j, k^_i>        (i < j)
 *     p_ji = exp(gam_j - gam_i) <q^_j, k^_i>        (i <= j)
 *     d_j  = b_j ( v_j - Gam_j S0 k^_j - sum_{i<j} c_ji d_i )
 *     o_j  = Gam_j S0 q^_j + sum_{i<=j} p_ji d_i
 *     S0  <- Gam_last S0 + sum_i exp(gam_last - gam_i) d_i k^_i^T   (chunk end)
 *
 * which is the delta rule S_t = a_t S_{t-1} (I - b_t k^ k^T) + b_t v k^T,
 * o_t = S_t q^_t, unrolled over the chunk (d_t = b_t (v_t - a_t S_{t-1} k^_t)).
 * Every sum above is one fixed order (increasing i; the dk dots as four
 * interleaved fma chains then (s0 + s1) + (s2 + s3); S0 k and S0 q through the
 * row layout of the recurrent kernel), and gdn_replay_prefill and
 * gdn_replay_decode evaluate each term with the same code.  So a sequence's
 * outputs and replay state have the same bits however its tokens are split
 * between prefill calls and decode steps, and whatever else is in the batch.
 * They are not bit-equal to gdn_recurrent_fwd (another rounding order of the
 * same function).
 *
 * The replay state.  A pool [num_slots, HV, B] fp32, B =
 * gdn_replay_block_floats(dk, dv); per (slot, head) it holds S0 [dv, dk]
 * (offset 0), then the open chunk's rows k^ [C, dk], d [C, dv] and gam [C]
 * (C = GDN_REPLAY_CHUNK).  A sequence that has processed P tokens uses rows
 * 0 .. (P mod C) - 1.  To start a sequence, set its S0 to the initial state
 * (zeros for none); the rows need no initialisation.  The memory per head is
 * about twice the plain fp32 state's.
 *
 * seq_pos[n] is the number of tokens sequence n has processed before the call
 * (negative values are taken as 0); prefill may pass NULL (all 0).  Shapes,
 * dtypes, alignment and the error convention are those of gdn.h (dv_slice is
 * ignored); replay_state is 16-byte aligned.  Slots: state_indices[n]
 * (NULL: slot n, needs num_slots >= N); a negative or out-of-range slot skips
 * the sequence (its outputs are left untouched).  Slots of different
 * sequences must differ.
 */
#ifndef GDN_REPLAY_H_
#define GDN_REPLAY_H_

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_REPLAY_CHUNK 64

/* Floats per (slot, head) block of the replay-state pool (0 for unsupported dk, dv). */
size_t gdn_replay_block_floats(int dk, int dv);

/* Bytes of workspace gdn_replay_prefill needs (error word + work list), 0 if the shape is invalid. */
size_t gdn_replay_workspace_size(const gdn_shape* shape);

/*
 * Chunked prefill over a packed varlen batch that continues each sequence
 * from its replay state (position seq_pos[n]) and leaves the state after its
 * last token.  out [T_total, HV, dv] in dtype.  One CTA per (sequence, head),
 * ordered longest first by the varlen scheduler (two launches).
 */
gdn_status gdn_replay_prefill(const gdn_shape* shape, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const int32_t* cu_seqlens,
                              const int32_t* seq_pos, float* replay_state,
                              const int32_t* state_indices, int num_slots, void* out,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * One decode token per sequence (shape->T_total == shape->N), replaying the
 * chunked order: bit-identical to gdn_replay_prefill run one token further.
 * seq_pos is required.  One launch, no workspace.
 */
gdn_status gdn_replay_decode(const gdn_shape* shape, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const int32_t* seq_pos,
                             float* replay_state, const int32_t* state_indices, int num_slots,
                             void* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_REPLAY_H_ */
