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
};

// Number of sequence segments per (batch, value head) the chunked prefill uses
// (requested > 0 is taken as is, capped at the chunk count).
int plan_segments(int64_t pairs, int64_t nchunks, int num_sms, int requested);

// Chunked tensor-core prefill (bf16).  Builds the TMA descriptors and launches.
cudaError_t launch_chunked(const ChunkedParams &p, cudaStream_t stream, int num_sms);

}  // namespace gdn
