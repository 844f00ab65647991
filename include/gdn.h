/*
 * gdn.h -- C ABI of the Gated DeltaNet (GDN) token-mixing core on NVIDIA B300
 * (sm_103a).
 *
 * The operation (Qwen3.8-Next reading notes, jianyuh.github.io, section 2.1
 * "Gated DeltaNet", the four-line gated delta recurrence): per head, with a
 * matrix state S in R^{dk x dv} stored key-dimension-major ("transposed
 * convention", dv contiguous), for each token t in order
 *
 *     S~  = alpha_t * S_{t-1}
 *     e_t = v_t - S~^T k_t
 *     S_t = S~ + beta_t * k_t e_t^T
 *     y_t = S_t^T q_t
 *
 * alpha_t in (0,1] is the decay gate and beta_t in [0,1] the write strength
 * (same section, "where alpha_t ... beta_t ..."; alpha = 1 and beta in {0,1}
 * are accepted as boundary values).  q and k are expected L2-normalised per
 * token (same section, "Feature parameterization": the normalisation keeps the
 * rank-one transition I - beta k k^T well conditioned); the core does not
 * re-normalise.
 *
 * Tensor layouts (dense, row-major, no padding):
 *   q, k          [B, T, Hqk, dk]   dtype of gdn_shape.dtype
 *   v, y          [B, T, Hv,  dv]   dtype of gdn_shape.dtype
 *   alpha, beta   [B, T, Hv]        fp32
 *   S0, S_T,
 *   S_inout       [B, Hv, dk, dv]   fp32, dv contiguous
 * Value head h reads query/key head h / (Hv / Hqk) (contiguous grouping);
 * alpha, beta and the state are per value head.
 *
 * Supported: dk == dv in {64, 128}; Hv a multiple of Hqk; q, k, v, y, S0,
 * S_T, S_inout 16-byte aligned; alpha, beta 4-byte aligned.  bf16 prefill runs
 * the chunked tensor-core kernel (tcgen05/TMEM/TMA); fp32 prefill runs the
 * token-sequential fp32 kernel; decode runs the HBM-streaming kernel.
 *
 * Ownership and execution: the caller owns every buffer (device memory for
 * all tensors and the workspace).  Calls validate their arguments on the host,
 * enqueue kernels on `stream` (a cudaStream_t passed as void*, NULL = legacy
 * default stream) and return without synchronising.  They keep no device
 * allocation between calls except the TMA descriptors, which are rebuilt per
 * call and passed by value.  Calls are reentrant; two calls that share an
 * output buffer or a workspace must be ordered by the caller.
 *
 * Errors: argument errors are returned before anything is launched; a failed
 * launch returns GDN_ERR_CUDA; errors detected on the device are recorded in
 * the workspace status word and read by gdn_read_device_status.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shape */
    GDN_ERR_UNSUPPORTED = 2,   /* valid but not implemented: head dims, dtype, no sm_103 device */
    GDN_ERR_ALIGNMENT = 3,     /* a pointer violates the alignment above */
    GDN_ERR_WORKSPACE = 4,     /* workspace missing or smaller than gdn_prefill_workspace_bytes */
    GDN_ERR_CUDA = 5,          /* a CUDA runtime/driver call or a launch failed */
    GDN_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up (status word) */
    GDN_ERR_DEVICE = 7,        /* another device-detected inconsistency (status word) */
    GDN_ERR_ALIASING = 8       /* y overlaps an input, or an output overlaps another output */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Problem shape.  T is the number of tokens per sequence (1 for decode). */
typedef struct {
    int64_t B, T;
    int32_t Hqk, Hv, dk, dv;
    int32_t dtype;              /* gdn_dtype of q, k, v and y */
} gdn_shape;

/*
 * Optional prefill controls (pass NULL for the defaults).
 *
 * segments: each head's sequence is split into this many contiguous runs of
 *   chunks that are processed in parallel (0 = chosen from the shape and the
 *   SM count; 1 = one sequential pass per head).  A run that does not start
 *   at token 0 rebuilds its entering state from a zero state over a window of
 *   preceding tokens, the shortest window (at most max_warmup_chunks chunks of
 *   64 tokens) over which sum(log alpha) <= log_eps.  With unit keys and
 *   beta in [0,1] every step is a contraction of norm <= alpha_t, so the state
 *   so rebuilt differs from the exact one by at most exp(log_eps) times the
 *   state norm at the window start.  When no such window exists (gates at
 *   or near 1) the run's entering state is computed exactly instead: each
 *   run is an affine map of the state it enters with (the product of the
 *   per-token transitions alpha_t (I - beta_t k_t k_t^T) plus the values it
 *   writes); a transition pass computes every run's map, a combine kernel
 *   chains them per head from S0, and the output pass starts each run from
 *   its exact state (four launches; the exact sequence split).  The split is
 *   taken for sequences of at least 256 chunks when the workspace holds the
 *   runs' maps (always with gdn_prefill_workspace_bytes; the fixed scratch of
 *   gdn_prefill_noalloc holds them for small shapes only); otherwise such a
 *   run restarts from token 0 and the initial state (also exact).
 * log_eps: natural log of that bound (0 = default, -20 ln 2); must be <= 0.
 * max_warmup_chunks: window limit (0 = default, 64).
 * algorithm: GDN_ALGO_AUTO (bf16 -> chunked, fp32 -> sequential),
 *   GDN_ALGO_CHUNKED (tensor-core chunked kernel; bf16 only, else
 *   GDN_ERR_UNSUPPORTED) or GDN_ALGO_SEQUENTIAL (token-sequential fp32-math
 *   kernel, one CTA per head; segments/log_eps do not apply).
 * test_stall_chunk: a fault-injection hook for tests of the device-side
 *   failure detection (chunked kernel only).  When > 0, the tiles of that
 *   chunk index are never loaded, so the kernel's bounded waits (about one
 *   second each) run out: the kernel records GDN_ERR_TIMEOUT in the workspace
 *   status word, stops, and leaves the context usable.  Outputs of such a
 *   call are undefined.  Leave 0 in normal use.
 */
typedef enum { GDN_ALGO_AUTO = 0, GDN_ALGO_CHUNKED = 1, GDN_ALGO_SEQUENTIAL = 2 } gdn_algorithm;

typedef struct {
    int32_t segments;
    float log_eps;
    int32_t max_warmup_chunks;
    int32_t algorithm;          /* gdn_algorithm */
    int32_t test_stall_chunk;   /* test hook, 0 = off: see below */
} gdn_prefill_options;

/* Text for a status code (static storage, never NULL). */
const char *gdn_status_string(gdn_status status);

/*
 * Bytes of device workspace gdn_prefill needs for this shape: a 256-byte
 * status area, B*Hv*dk*dv fp32 values used to stage S_T when it aliases S0,
 * and, for bf16 shapes of more than one chunk, the exact sequence split's
 * per-run flags and fp32 run maps (3*dk*dv values per run, for up to
 * ceil(320 / (B*Hv)) runs per head).  Returns 0 for an invalid shape.
 */
size_t gdn_prefill_workspace_bytes(const gdn_shape *shape);

/*
 * Kernels that one gdn_prefill call with this shape and these options
 * enqueues on a workspace of gdn_prefill_workspace_bytes(shape): 0 for an
 * empty problem, 4 when the chunked path takes the exact sequence split (how
 * many of its runs need it is decided on the device; runs that do not leave
 * the extra kernels at once), else 1.  Host-side copies (an in-place S_T, an
 * empty sequence's S_T) are not kernels.  Returns -1 for an invalid shape or
 * options or when no supported device is current.
 */
int gdn_prefill_launches(const gdn_shape *shape, const gdn_prefill_options *options);

/*
 * Prefill: run the recurrence over T tokens of each (batch, value head) from
 * the initial state S0 (NULL = zero state), writing every y_t and the final
 * state S_T.  S_T may equal S0 (in-place update, staged through the
 * workspace); y must not overlap any input.  ws must be device memory of at
 * least gdn_prefill_workspace_bytes(shape) bytes, 256-byte aligned; its first
 * 256 bytes must be zero before the first call (the calls leave them zero
 * unless a device error was recorded).  T == 0 copies S0 (or zeros) to S_T.
 * The chunked algebra this computes is the recurrence unrolled over chunks of
 * 64 tokens: identical up to rounding in exact arithmetic.
 */
gdn_status gdn_prefill(const gdn_shape *shape,
                       const void *q, const void *k, const void *v,
                       const float *alpha, const float *beta,
                       const float *S0, void *y, float *S_T,
                       void *ws, size_t ws_bytes, void *stream);

/* gdn_prefill with explicit options (NULL = defaults). */
gdn_status gdn_prefill_ex(const gdn_shape *shape, const gdn_prefill_options *options,
                          const void *q, const void *k, const void *v,
                          const float *alpha, const float *beta,
                          const float *S0, void *y, float *S_T,
                          void *ws, size_t ws_bytes, void *stream);

/*
 * Decode: one recurrence step (shape->T must be 1) for every (batch, value
 * head), updating S_inout in place and writing y [B, 1, Hv, dv].  Each head's
 * fp32 state is streamed once from HBM and written back once.  y must not
 * overlap any input or S_inout.
 */
gdn_status gdn_decode_step(const gdn_shape *shape,
                           const void *q, const void *k, const void *v,
                           const float *alpha, const float *beta,
                           float *S_inout, void *y, void *stream);

/*
 * Synchronise `stream`, read the status word that gdn_prefill kernels write
 * into `ws` when they detect an error on the device, clear it, and return
 * GDN_OK, GDN_ERR_TIMEOUT or GDN_ERR_DEVICE (GDN_ERR_CUDA if the sync fails).
 */
gdn_status gdn_read_device_status(void *ws, void *stream);

/*
 * Prefill for callers that cannot allocate device memory: an embedding
 * runtime, a plugin running inside someone else's process, or code under a
 * strict memory budget may have no way to call cudaMalloc for the workspace
 * gdn_prefill asks for.  (The method itself needs no such entry point.)  This
 * variant takes no workspace and allocates nothing: its scratch is a 256-byte
 * status area plus a staging area in one fixed array inside this library
 * (GDN_NOALLOC_SCRATCH_BYTES in total), which every GPU that loads the
 * library keeps until the process exits.  Inputs, outputs, layouts and
 * results are those of gdn_prefill.
 *
 * Limit: only an in-place bf16 call (S_T == S0, chunked path) stages its
 * final states in the array, so only such a call is limited: one whose
 * B*Hv*dk*dv*4 + 256 bytes exceed GDN_NOALLOC_SCRATCH_BYTES (more than 128
 * (batch, value head) pairs at d = 128, 512 at d = 64) returns
 * GDN_ERR_WORKSPACE before anything runs.  Other calls use the 256-byte status
 * area alone and take any shape gdn_prefill takes.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array, so calls whose execution overlaps
 * on the GPU (different streams without ordering between them) race on it
 * and must not be issued.  The array starts zeroed; errors detected on the
 * device (a bounded wait that timed out) accumulate in its status area until
 * gdn_prefill_noalloc_status reads and clears them.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (256u + 8u * 1024u * 1024u)

gdn_status gdn_prefill_noalloc(const gdn_shape *shape,
                               const void *q, const void *k, const void *v,
                               const float *alpha, const float *beta,
                               const float *S0, void *y, float *S_T, void *stream);

/*
 * gdn_read_device_status for the array of gdn_prefill_noalloc: synchronise
 * `stream` and return GDN_OK, GDN_ERR_TIMEOUT or GDN_ERR_DEVICE for the
 * errors the no-alloc calls recorded since the last read, clearing them.
 */
gdn_status gdn_prefill_noalloc_status(void *stream);

/*
 * Channel-wise decay: the decay gate is a vector over the key dimension,
 * alpha [B, T, Hv, dk] fp32 (16-byte aligned), and the decay step scales row
 * i of the state by alpha_t[i]: S~ = diag(alpha_t) S_{t-1}; the other three
 * lines of the recurrence are unchanged.  This is the per-channel ("diagonal")
 * gate of Kimi Delta Attention, which the reading notes name beside the delta
 * rule (section 2.1, "Why the delta rule matters").  With all channels equal
 * it is the scalar recurrence.  S_T may equal S0.  Layouts, ownership and
 * errors otherwise as gdn_prefill and gdn_decode_step.
 *
 * Prefill paths.  bf16 with dk = dv = 128 runs the chunked tensor-core path:
 * a per-chunk pre-pass forms each chunk's gated operands from per-channel
 * cumulative log decays (keys and queries scaled per channel against a
 * reference token per 16-token block, so that every exponent stays bounded;
 * a block whose own decay passes e^80 in some channel takes an element-wise
 * path), the lower-triangular inverse and the chunk's W, U~ and P, then a
 * chain kernel runs the state over the chunks, split into segments with
 * warm-up windows as in gdn_prefill (the window bound uses the largest
 * channel's decay), and the exact sequence split for the segments without
 * a window on sequences of at least 256 chunks (else they restart from
 * token 0, also exact).  Every other shape runs the token-sequential kernel (bf16 or
 * fp32, state in fp32 registers), as does the decode step.
 *
 * gdn_prefill_cw allocates the chunked path's workspace itself, in stream
 * order (cudaMallocAsync / cudaFreeAsync on `stream`); gdn_prefill_cw_ex
 * takes it from the caller: ws of at least gdn_prefill_cw_workspace_bytes
 * bytes, 256-byte aligned (a 256-byte status area, B*Hv*dk*dv fp32 for an
 * in-place S_T, and 74,244 bytes per (batch, value head, 64-token chunk); NULL
 * with 0 bytes for a token-sequential call).  options as for gdn_prefill_ex:
 * segments, log_eps and max_warmup_chunks apply to the chunked path;
 * algorithm GDN_ALGO_SEQUENTIAL forces the token-sequential kernel and
 * GDN_ALGO_CHUNKED returns GDN_ERR_UNSUPPORTED for shapes the chunked path
 * does not take; test_stall_chunk must be 0.
 */
gdn_status gdn_prefill_cw(const gdn_shape *shape, const void *q, const void *k, const void *v,
                          const float *alpha, const float *beta, const float *S0, void *y, float *S_T,
                          void *stream);

size_t gdn_prefill_cw_workspace_bytes(const gdn_shape *shape);

gdn_status gdn_prefill_cw_ex(const gdn_shape *shape, const gdn_prefill_options *options,
                             const void *q, const void *k, const void *v,
                             const float *alpha, const float *beta, const float *S0,
                             void *y, float *S_T, void *ws, size_t ws_bytes, void *stream);

gdn_status gdn_decode_step_cw(const gdn_shape *shape, const void *q, const void *k, const void *v,
                              const float *alpha, const float *beta, float *S_inout, void *y, void *stream);

/*
 * Prefill from host memory.  q, k, v, alpha, beta, S0 (NULL = zero state),
 * y and S_T (NULL = not returned) are host buffers in the layouts above; they
 * should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to
 * overlap, and are otherwise copied synchronously.  The sequence is cut into
 * pieces of tokens_per_piece tokens (0 = about an eighth of T, a multiple of
 * 64); piece p's host-to-device copy, piece p-1's prefill and piece p-2's
 * device-to-host copy of y run concurrently on two internal streams and
 * `stream`.  Each piece starts from the state the previous one left, so the
 * result is that of gdn_prefill over the whole sequence up to rounding.
 *
 * ws: device memory of gdn_prefill_host_workspace_bytes(shape,
 * tokens_per_piece) bytes, 256-byte aligned, whose first 256 bytes are zero
 * (as for gdn_prefill): two piece-sized copies of the inputs and y, two state
 * buffers and a prefill workspace.  The device status of the prefills is read
 * with gdn_read_device_status(ws, stream).  The call returns once the work is
 * queued; `stream` waits for every copy, so a synchronisation of `stream`
 * means that y and S_T are in host memory.
 */
size_t gdn_prefill_host_workspace_bytes(const gdn_shape *shape, int64_t tokens_per_piece);

gdn_status gdn_prefill_host(const gdn_shape *shape, int64_t tokens_per_piece,
                            const void *q, const void *k, const void *v,
                            const float *alpha, const float *beta, const float *S0,
                            void *y, float *S_T, void *ws, size_t ws_bytes, void *stream);

/*
 * Backward (gradients of the recurrence, for training).  Given the forward
 * inputs and the upstream gradients dy = dL/dy [B, T, Hv, dv] (dtype of the
 * shape) and dS_T = dL/dS_T [B, Hv, dk, dv] fp32 (NULL = zero), returns, for
 * the loss L whose gradients those are:
 *   dq, dk       [B, T, Hqk, dk] fp32  (summed over the value heads that share
 *                                       the query/key head)
 *   dv           [B, T, Hv, dv]  fp32
 *   dlog_alpha   [B, T, Hv]      fp32  the gradient with respect to log alpha_t,
 *                                       i.e. alpha_t * dL/dalpha_t (divide by
 *                                       alpha_t for dL/dalpha_t)
 *   dbeta        [B, T, Hv]      fp32
 *   dS0          [B, Hv, dk, dv] fp32  (NULL = not returned; may be the very
 *                                       buffer of dS_T, read before written)
 * This is the chain rule applied to the four lines of the recurrence above,
 * from t = T down to 1 (same section of the reading notes).  The decay
 * gradient is given in log space because the layer forms alpha as an
 * exponential of its gate pre-activation; the kernel obtains it from a scalar
 * recursion that never divides by alpha, so it stays finite as alpha -> 0.
 *
 * Scalar decay only; Hv * dk <= 2^24 (else GDN_ERR_UNSUPPORTED).  All
 * arithmetic is fp32 on CUDA cores, token by token:
 * the kernel recomputes the forward states from checkpoints taken every 8
 * tokens.  ws: device memory of gdn_backward_workspace_bytes(shape) bytes,
 * 256-byte aligned (no initial contents needed): the checkpoints
 * (B*Hv*ceil(T/8)*dk*dv fp32) and per-slab partial sums (2*B*T*Hv*(dv/32)*dk
 * fp32 and a little more).  Inputs q, k, v, dy, S0, dS_T and the outputs dq,
 * dk, dv, dS0 16-byte aligned; alpha, beta, dlog_alpha, dbeta 4-byte aligned.
 * No output may overlap an input, another output or the workspace (except dS0
 * == dS_T).  T == 0 writes dS0 = dS_T (or zeros).  Results are deterministic
 * (fixed summation order).  Layouts, ownership and errors otherwise as
 * gdn_prefill.
 */
size_t gdn_backward_workspace_bytes(const gdn_shape *shape);

gdn_status gdn_backward(const gdn_shape *shape,
                        const void *q, const void *k, const void *v,
                        const float *alpha, const float *beta, const float *S0,
                        const void *dy, const float *dS_T,
                        float *dq, float *dk, float *dv, float *dlog_alpha, float *dbeta, float *dS0,
                        void *ws, size_t ws_bytes, void *stream);

/*
 * Chunked backward on the tensor cores: the same gradients, arguments,
 * layouts and aliasing rules as gdn_backward, for bf16 q, k, v, dy with
 * dk = dv = 128 (else GDN_ERR_UNSUPPORTED).  It runs the chunk algebra of the
 * forward in reverse: a pre-pass forms every 64-token chunk's operands, a
 * forward chain writes the state entering every chunk, a reverse chain carries
 * dS (dU = P^T dY + Kl dS', dS = gamma_C dS' + Qp^T dY - W^T dU) and writes
 * the state gradient leaving every chunk, and a per-chunk kernel forms dq, dk,
 * dv, dbeta and dlog alpha from those (through dA = -T^T dT T^T of the chunk's
 * lower-triangular inverse T = (I + A)^{-1}).  Products take bf16 operands
 * with fp32 accumulation, so results carry bf16-level rounding (about 1e-2
 * of the largest gradient), unlike gdn_backward's fp32 arithmetic; the state
 * chains split long sequences into segments with warm-up windows, and with
 * the exact sequence split where gates do not decay, as the prefill does.  dq and dk are summed over the value heads of a group with
 * atomic additions (deterministic for up to two value heads per key head).
 * ws: device memory of gdn_backward_chunked_workspace_bytes(shape) bytes,
 * 256-byte aligned, no initial contents needed (74,244 bytes of chunk
 * operands plus two 32 KB bf16 states per (batch, value head, chunk), then
 * B*Hv*dk*dv fp32 to stage dS0 when it is dS_T's buffer).  Returns 0 bytes for
 * shapes the chunked path does not take.
 */
size_t gdn_backward_chunked_workspace_bytes(const gdn_shape *shape);

gdn_status gdn_backward_chunked(const gdn_shape *shape,
                                const void *q, const void *k, const void *v,
                                const float *alpha, const float *beta, const float *S0,
                                const void *dy, const float *dS_T,
                                float *dq, float *dk, float *dv, float *dlog_alpha, float *dbeta, float *dS0,
                                void *ws, size_t ws_bytes, void *stream);

/* 1 if the current CUDA device can run these kernels (compute capability 10.3). */
int gdn_device_supported(void);

/* ABI version of this header: major * 10000 + minor * 100 + patch. */
int gdn_abi_version(void);

#define GDN_ABI_VERSION 10000

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
