/*
 * gdn_layer.h -- C ABI of the Gated DeltaNet layer steps on either side of
 * the recurrence (gdn.h), on NVIDIA B300 (sm_103a).
 *
 * The Qwen3.8-Next reading notes (jianyuh.github.io, section 2.1 "Gated
 * DeltaNet") parameterise the recurrence's inputs from the layer input x_t
 * ("Feature parameterization", "Gating dynamics"):
 *
 *   q_t = L2Norm(SiLU(ShortConv(W_q x_t)))      k_t likewise with W_k
 *   v_t = SiLU(ShortConv(W_v x_t))
 *   beta_t  = sigma(W_beta x_t)
 *   alpha_t = exp(-exp(A) * softplus(W_alpha x_t + b_alpha))   (per-head A, b_alpha)
 *
 * and its output through a sigmoid gate and a zero-centred RMSNorm:
 *
 *   o_t = W_o [ sigma(W_z x_t) * RMSNorm(y_t) ].
 *
 * The projections W_* x_t and W_o are plain GEMMs and stay outside: the
 * prologue below starts from the projected features and ends with q, k, v,
 * alpha, beta in the layouts gdn_prefill / gdn_decode_step take; the epilogue
 * starts from y and z and ends before W_o.  Both are single fused passes over
 * HBM.
 *
 * Definitions of the steps the pages name without spelling out:
 *   ShortConv: causal depthwise convolution along time with kconv taps per
 *     channel, no bias; for channel c of token t,
 *       u[t][c] = sum_{i < kconv} w[c][i] * x[t - kconv + 1 + i][c],
 *     tap kconv-1 multiplying the current token.  The kconv-1 inputs before
 *     token 0 come from a convolution state (zeros when none is given) and
 *     the last kconv-1 inputs can be written out as the next state, so a
 *     sequence can be continued by a later call (prefill then decode).
 *   L2Norm(u) = u / sqrt(sum_e u_e^2 + 1e-6) over the head dimension d.
 *   RMSNorm(y) = y / sqrt(mean_e y_e^2 + eps) * (1 + w) over dv: the learned
 *     weight is stored as its offset from 1 ("zero-centred"), one vector of
 *     dv values shared by every head.
 *   softplus(u) = log(1 + e^u); sigma(u) = 1 / (1 + e^-u).
 * All arithmetic is fp32; bf16 outputs are rounded to nearest even.
 *
 * Layouts (dense, row-major, no padding; C_q = Hqk*d, C_v = Hv*d channels):
 *   xq, xk, q, k      [B, T, Hqk, d]  bf16
 *   xv, v, y, z, o    [B, T, Hv, d]   bf16
 *   wq, wk            [C_q, kconv]    fp32      wv [C_v, kconv] fp32
 *   conv states       [B, kconv-1, C] bf16      (the raw projected inputs)
 *   a_raw, b_raw,
 *   alpha, beta       [B, T, Hv]      fp32
 *   A, b_alpha        [Hv]            fp32
 *   norm_w            [d]             fp32
 * Supported: d in {64, 128}; Hv a multiple of Hqk; 1 <= kconv <= 4; every
 * bf16 tensor 16-byte aligned, every fp32 tensor 4-byte aligned.
 *
 * Ownership, execution and errors as in gdn.h: the caller owns every buffer;
 * calls validate on the host, enqueue on `stream` and return without
 * synchronising; argument errors come back before anything is launched.
 * Outputs must not overlap inputs (GDN_ERR_ALIASING); a state-out buffer may
 * not be the state-in buffer of the same tensor.
 */
#ifndef GDN_LAYER_H
#define GDN_LAYER_H

#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int64_t B, T;
    int32_t Hqk, Hv, d;
    int32_t kconv;          /* taps of the short convolution, 1..4 */
} gdn_layer_shape;

/* Buffers of gdn_layer_prologue (device pointers; NULL where marked optional). */
typedef struct {
    const void *xq, *xk, *xv;            /* projected features W_q x, W_k x, W_v x */
    const float *wq, *wk, *wv;           /* convolution taps */
    const void *state_q_in, *state_k_in, *state_v_in;   /* optional: NULL = zeros */
    void *state_q_out, *state_k_out, *state_v_out;      /* optional: NULL = not written */
    const float *a_raw, *b_raw;          /* W_alpha x, W_beta x */
    const float *A, *b_alpha;            /* per value head */
    void *q, *k, *v;                     /* outputs for the recurrence */
    float *alpha, *beta;
} gdn_prologue_io;

/*
 * Prologue: q, k, v, alpha and beta of T tokens from the projected features.
 * One pass: each input element is read once (plus kconv-1 tokens of overlap
 * per 64-token tile) and each output written once.  T == 0 only copies the
 * incoming convolution states (or zeros) to the outgoing ones; the token
 * tensors, taps and gate parameters may then be NULL.
 */
gdn_status gdn_layer_prologue(const gdn_layer_shape *shape, const gdn_prologue_io *io, void *stream);

/*
 * Epilogue: o = sigma(z) * RMSNorm(y) for every (token, value head), with eps
 * > 0 (the pages give none; 1e-6 is the usual choice).  y, z, o bf16
 * [B, T, Hv, d]; norm_w fp32 [d].  o must not overlap y or z.  With B*T == 0
 * nothing is read or written and the pointers may be NULL.
 */
gdn_status gdn_layer_epilogue(const gdn_layer_shape *shape, const void *y, const void *z, const float *norm_w,
                              float eps, void *o, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_LAYER_H */
