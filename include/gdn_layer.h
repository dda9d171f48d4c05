/*
 * gdn_layer.h -- C ABI of the Gated DeltaNet layer's ops either side of the
 * recurrence (sm_103a): the gate activations that turn the layer's raw
 * projections into (g, beta), the short causal depthwise convolution over the
 * q/k/v projections with its per-sequence conv state cache (prefill and
 * decode), and the gated RMSNorm applied to the recurrence's output.
 *
 * "Defending Against the Training-Inference Numeric Mismatch in RL
 * (Especially Linear Attention)" keeps these ops identical on the trainer and
 * the generator (section 3.1: one model definition, with A_log kept in fp32
 * through the trainer's bf16 wrapping) and reuses the serving engine's conv
 * state cache unchanged (section 3.2).  Their formulas are the standard GDN
 * layer's:
 *
 *     g    = -exp(A_log[h]) * softplus(a + dt_bias[h]),   beta = sigmoid(b)
 *     conv y[t, c] = act( bias[c] + sum_{i<W} w[c, i] * xw[t + i, c] ),
 *          xw = (the W-1 rows before the sequence: its conv state) ++ (its rows)
 *     norm y = o / sqrt(mean(o^2) + eps) * weight * silu(z)   (per row of d)
 *
 * Invariance.  Every output element is computed by one thread with one fixed
 * order of operations that depends on nothing but its own row (conv: its own
 * sequence's rows): results do not depend on the batch, on how a batch is
 * tiled, or on whether a token goes through the prefill or the decode entry
 * point (gdn_causal_conv1d_fwd and gdn_causal_conv1d_update share the
 * per-element arithmetic, so prefill-then-update is bit-identical to one
 * prefill over the whole sequence).
 *
 * Memory and ownership as in gdn.h: caller-owned, dense row-major DEVICE
 * pointers; x, y, o, z, the conv state, the conv weight and the RMSNorm
 * weight 16-byte aligned; g, beta, A_log, dt_bias, the conv bias, cu_seqlens,
 * state_indices and has_initial_state 4-byte aligned (a and b: their element
 * size).  Misalignment returns GDN_ERR_INVALID_ARG.  Nothing is allocated;
 * every call is one asynchronous launch on `stream` (a cudaStream_t; NULL =
 * legacy default stream) and returns host-side validation or launch errors
 * only.
 */
#ifndef GDN_LAYER_H_
#define GDN_LAYER_H_

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Gate activations.  a, b: [T, HV] in in_dtype (bf16 or fp32, the projection
 * outputs); A_log, dt_bias: [HV] fp32 (dt_bias may be NULL: zero).  Writes
 * g = -exp(A_log) * softplus(a + dt_bias) and beta = sigmoid(b), both [T, HV]
 * fp32, the inputs gdn_recurrent_fwd / gdn_decode_step take.  softplus(x) is
 * log(1 + exp(x)), taken as x itself above x = 20.
 */
gdn_status gdn_gates(int64_t T, int HV, gdn_dtype in_dtype, const void* a, const void* b,
                     const float* A_log, const float* dt_bias, float* g, float* beta,
                     void* stream);

/*
 * Gated RMSNorm over the last axis: o, z, y are [rows, d] in dtype (for the
 * recurrence's output rows = T * HV and d = dv); weight [d] fp32.  z may be
 * NULL (no gate: plain RMSNorm).  y may alias o.  d must be a multiple of 8
 * (bf16) or 4 (fp32) and at most 2048; eps >= 0.  The sum of squares of a row
 * is taken in fp32 in one fixed order (each lane of a fixed lane group sums
 * its own 16-byte chunks in ascending order, then a fixed xor butterfly).
 */
gdn_status gdn_gated_rmsnorm(int64_t rows, int d, gdn_dtype dtype, const void* o, const void* z,
                             const float* weight, float eps, void* y, void* stream);

typedef struct {
    int N;           /* sequences (update: batch size) */
    int T_total;     /* packed tokens (update: must equal N) */
    int C;           /* channels, e.g. q, k and v projections side by side */
    int W;           /* taps, 2..8 */
    gdn_dtype dtype; /* x, y and the conv state */
    int activation;  /* 1: SiLU on the output; 0: none */
} gdn_conv_shape;

/*
 * Causal depthwise conv over a packed varlen batch (prefill, trainer forward).
 * x, y [T_total, C]; weight [C, W] fp32 (tap W-1 multiplies the current row);
 * bias [C] fp32 or NULL; cu_seqlens int32 [N + 1] as in gdn.h.  conv_state is
 * a pool [num_slots, W-1, C] in dtype (NULL: every sequence starts from zeros
 * and no state is written); sequence n uses slot state_indices[n]
 * (state_indices NULL: slot n, and num_slots must be >= N).  The slot's rows
 * are read as the sequence's initial state when has_initial_state is NULL or
 * has_initial_state[n] != 0 (else zeros), and are then overwritten with the
 * sequence's final state, the last W-1 rows of (initial state ++ its rows); a
 * sequence of length 0 leaves its slot as it was (or zeroes it when its
 * initial state is off).  A negative or out-of-range slot: zero initial
 * state, nothing written.  Slots of different sequences must differ; y must
 * not alias x.  C must be a multiple of 8 (bf16) or 4 (fp32).
 */
gdn_status gdn_causal_conv1d_fwd(const gdn_conv_shape* shape, const void* x, const float* weight,
                                 const float* bias, const int32_t* cu_seqlens, void* conv_state,
                                 const int32_t* state_indices, int num_slots,
                                 const int32_t* has_initial_state, void* y, void* stream);

/*
 * One decode token per sequence: x, y [N, C] (shape->T_total == N); the
 * pool conv_state [num_slots, W-1, C] is updated in place (rows shift up by
 * one, x enters as the newest row).  Sequence b uses slot state_indices[b]
 * (NULL: slot b, and num_slots must be >= N); a negative or out-of-range slot
 * skips it (y row untouched).  Slots of different sequences must differ; y
 * must not alias x.  Bit-identical to running gdn_causal_conv1d_fwd one
 * token further.
 */
gdn_status gdn_causal_conv1d_update(const gdn_conv_shape* shape, const void* x, const float* weight,
                                    const float* bias, void* conv_state,
                                    const int32_t* state_indices, int num_slots, void* y,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_LAYER_H_ */
