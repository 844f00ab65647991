// Internal declarations shared by the host-side entry points and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Status word written by kernels into the first bytes of the prefill workspace.
// Bit flags; 0 means no error.
enum DeviceStatusBits : uint32_t {
    kDevTimeout = 1u << 0,   // a bounded mbarrier wait gave up
    kDevBadShape = 1u << 1,  // a kernel saw parameters it cannot handle
};

struct RecurrentParams {
    int64_t B, T;
    int Hqk, Hv, group;          // group = Hv / Hqk
    const void *q, *k, *v;       // [B, T, Hqk, dk] / [B, T, Hv, dv]
    const float *alpha, *beta;   // [B, T, Hv] ([B, T, Hv, dk] for alpha when alpha_cw)
    bool alpha_cw;               // channel-wise decay: S~ = diag(alpha_t) S
    const float *S_in;           // [B, Hv, dk, dv] or nullptr (zero state)
    float *S_out;                // [B, Hv, dk, dv] or nullptr
    void *y;                     // [B, T, Hv, dv]
};

// Token-sequential kernel: decode (T == 1, S_in == S_out) and the fp32 prefill.
cudaError_t launch_recurrent(const RecurrentParams &p, int dk, int dv, gdn_dtype dtype, cudaStream_t stream);

struct ChunkedParams {
    int64_t B, T;
    int Hqk, Hv, group, d;       // d = dk = dv (64 runs as zero-padded 128)
    const void *q, *k, *v;
    const float *alpha, *beta;
    const float *S0;             // nullptr = zero state
    void *y;
    float *S_T;                  // final states (possibly the workspace staging area)
    uint32_t *status;            // device status word
    int segments;                // runs per head
    float log_eps;
    int max_warmup_chunks;
    int test_stall_chunk;        // > 0: never load this chunk (fault-injection test hook)
    // Exact sequence split (workspace, optional): per-head flags and the
    // segments' transition and entering states; used when P * pairs * 3 * d * d
    // floats fit in seg_state_bytes.
    int *exact_flag;             // [B * Hv][segments]: segment has no warm-up window
    float *seg_state;            // [B * Hv][segments][3][d][d]
    size_t seg_state_bytes;
};

// Segment count bound for which gdn_prefill_workspace_bytes reserves the
// exact-split states: segments * B * Hv stays within about two waves of a
// GPU with up to this many SMs.
constexpr int kExactSplitSmBound = 160;
// Sequences of fewer chunks (of 64 tokens) per head never take the exact split.
constexpr int kExactSplitMinChunks = 256;

// Segments per head for which a workspace reserves the exact split's maps
// (0: none needed).
inline int64_t exact_split_segments(int64_t pairs, int64_t nchunks) {
    if (pairs <= 0 || nchunks <= 1) return 0;
    const int64_t segs = (2 * kExactSplitSmBound + pairs - 1) / pairs;
    return segs > nchunks ? nchunks : segs;
}

// Number of sequence segments per (batch, value head) the chunked prefill uses
// (requested > 0 is taken as is, capped at the chunk count).
int plan_segments(int64_t pairs, int64_t nchunks, int num_sms, int requested);

// Whether a chunked prefill of P segments per head takes the exact sequence
// split (plan, transition pass, combine, then the output pass: four launches
// instead of one), given segment-state room of seg_state_bytes.
bool takes_exact_split(int64_t pairs, int64_t nchunks, int P, int d, size_t seg_state_bytes);

// Entering states of the segments of every head with a flag set: S_1 = B_0,
// S_{s+1} = M_s S_s + B_s, over seg_state [pairs][P][3][d][d] (slots B, M, In).
cudaError_t launch_segment_combine(const int *flag, float *seg_state, int64_t pairs, int P, int d,
                                   cudaStream_t stream);

// Chunked tensor-core prefill (bf16).  Builds the TMA descriptors and launches.
cudaError_t launch_chunked(const ChunkedParams &p, cudaStream_t stream, int num_sms);

// Chunked prefill with the channel-wise decay gate (bf16, d = 128): a
// per-chunk pre-pass writes each chunk's state-independent operands into the
// workspace (`ops`), then a chain kernel runs the state scan over them.
struct ChunkedCwParams {
    int64_t B, T;
    int Hqk, Hv, group, d;
    const void *q, *k, *v;
    const float *alpha, *beta;   // alpha [B, T, Hv, d]
    const float *S0;             // nullptr = zero state
    void *y;
    float *S_T;
    int segments;
    float log_eps;
    int max_warmup_chunks;
    uint8_t *ops;                // chunked_cw_ops_bytes(B, T, Hv) bytes, 16-byte aligned
    bool scalar_alpha;           // alpha is [B, T, Hv] (one decay for every channel)
    void *state_out;             // nullptr, or the state entering every chunk [B * Hv][nchunks][d][d] bf16
    // Exact sequence split (optional, as in ChunkedParams): flags and segment maps.
    int *exact_flag;
    float *seg_state;
    size_t seg_state_bytes;
};

// The per-chunk operand record the chunked pre-pass writes (bytes): -W, U~,
// Qp and Kl as bf16 [64][128], P as bf16 [64][64], e^{g_C} as fp32 [128].
namespace rec {
constexpr uint32_t kWn = 0, kUt = 16384, kQp = 32768, kKl = 49152, kP = 65536, kGc = 73728, kBytes = 74240;
}

// Bytes of one chunk's operand record in the workspace.
constexpr size_t kCwChunkBytes = 74240;
size_t chunked_cw_ops_bytes(int64_t B, int64_t T, int Hv);
cudaError_t launch_chunked_cw(const ChunkedCwParams &p, cudaStream_t stream, int num_sms);

// Tokens between two checkpoints of the backward pass (and its chunk length).
constexpr int kBackwardCheckpointTokens = 8;

struct BackwardParams {
    int64_t B, T;
    int Hqk, Hv, group;
    const void *q, *k, *v, *dy;          // dtype of the shape
    const float *alpha, *beta;           // [B, T, Hv]
    const float *S0, *dS_T;              // [B, Hv, d, d] or nullptr (zero)
    float *dq, *dk;                      // [B, T, Hqk, d]
    float *dv;                           // [B, T, Hv, d]
    float *dlog_alpha, *dbeta;           // [B, T, Hv]
    float *dS0;                          // [B, Hv, d, d] or nullptr (not returned)
    float *ckpt;                         // workspace: slab states every few tokens
    float *part_dq, *part_dk;            // workspace: [B, T, Hv, d / 32, d] per-slab partial sums
    float *part_dbeta, *part_dlog_alpha; // workspace: [B, T, Hv, d / 32]
};

// Bytes of backward workspace for this shape (d = dk = dv) and the offsets of
// its partial-sum regions (the checkpoints start at offset 0).
size_t backward_workspace_layout(int64_t B, int64_t T, int Hv, int d, size_t *off_part_dq, size_t *off_part_dk,
                                 size_t *off_part_b, size_t *off_part_g);

// Chunked tensor-core backward (bf16, d = 128): workspace bytes and launch
// (pre-pass, forward chain with the entering states, reverse chain, per-chunk
// gradients).  ws: 256-byte aligned, backward_chunked_workspace_bytes bytes.
size_t backward_chunked_workspace_bytes(int64_t B, int64_t T, int Hv);
cudaError_t launch_backward_chunked(const BackwardParams &p, uint8_t *ws, cudaStream_t stream, int num_sms);

// Backward of the recurrence: the per-slab kernel, then the reduction of its partial sums.
cudaError_t launch_backward(const BackwardParams &p, int d, gdn_dtype dtype, cudaStream_t stream, int num_sms);

}  // namespace gdn
