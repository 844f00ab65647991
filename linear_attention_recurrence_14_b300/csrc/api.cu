// Host side of the C ABI declared in include/gdn.h: argument validation,
// aliasing and workspace checks, dispatch to the kernels.  Nothing here
// computes any part of the recurrence.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

constexpr size_t kStatusBytes = 256;
constexpr float kDefaultLogEps = -13.862943611198906f;  // -20 ln 2
constexpr int kDefaultMaxWarmupChunks = 64;

bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

// Validates the shape and returns element counts (0 on failure).
gdn_status check_shape(const gdn_shape *s, int64_t *n_qk, int64_t *n_v, int64_t *n_gate, int64_t *n_state) {
    if (!s) return GDN_ERR_INVALID_ARG;
    if (s->B < 0 || s->T < 0 || s->Hqk <= 0 || s->Hv <= 0 || s->dk <= 0 || s->dv <= 0)
        return GDN_ERR_INVALID_ARG;
    if (s->Hv % s->Hqk != 0) return GDN_ERR_INVALID_ARG;
    if (s->dtype != GDN_F32 && s->dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    int64_t bt = 0, tmp = 0;
    if (!mul_ok(s->B, s->T, &bt)) return GDN_ERR_INVALID_ARG;
    if (!mul_ok(bt, s->Hqk, &tmp) || !mul_ok(tmp, s->dk, n_qk)) return GDN_ERR_INVALID_ARG;
    if (!mul_ok(bt, s->Hv, n_gate) || !mul_ok(*n_gate, s->dv, n_v)) return GDN_ERR_INVALID_ARG;
    if (!mul_ok(s->B, s->Hv, &tmp) || !mul_ok(tmp, static_cast<int64_t>(s->dk) * s->dv, n_state))
        return GDN_ERR_INVALID_ARG;
    if (*n_qk > (INT64_MAX >> 3) || *n_v > (INT64_MAX >> 3) || *n_state > (INT64_MAX >> 3))
        return GDN_ERR_INVALID_ARG;
    if (!(s->dk == s->dv && (s->dk == 64 || s->dk == 128))) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
    const void *p;
    size_t n;
};

bool overlap(Range a, Range b) {
    if (!a.p || !b.p || a.n == 0 || b.n == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// The current device's compute capability check and SM count, queried once
// per device (the attributes do not change while the process runs).
gdn_status check_device(int *num_sms) {
    constexpr int kMaxDev = 64;
    static std::mutex lock;
    static int cached_sms[kMaxDev] = {};    // 0 = not queried, -1 = unsupported
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDev) return GDN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(lock);
    if (cached_sms[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return GDN_ERR_CUDA;
        }
        cached_sms[dev] = (major == 10 && minor == 3) ? sms : -1;
    }
    if (cached_sms[dev] < 0) return GDN_ERR_UNSUPPORTED;
    *num_sms = cached_sms[dev];
    return GDN_OK;
}

gdn_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    cudaGetLastError();
    return GDN_ERR_CUDA;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace layout of a prefill: status area, staging of in-place final states,
// then (bf16, chunked path) the exact sequence split's per-head flags and its
// segment states for up to about two waves of segments.  Returns the total.
size_t exact_split_layout(const gdn_shape &s, int64_t n_state, size_t *off_flag, size_t *off_seg, size_t *seg_bytes) {
    const size_t base = kStatusBytes + static_cast<size_t>(n_state) * sizeof(float);
    *off_flag = round256(base);
    *off_seg = *off_flag;
    *seg_bytes = 0;
    const int64_t pairs = s.B * s.Hv;
    const int64_t nchunks = (s.T + 63) / 64;
    if (s.dtype != GDN_BF16 || pairs == 0 || nchunks <= 1) return base;
    int64_t segs = (2 * gdn::kExactSplitSmBound + pairs - 1) / pairs;
    if (segs > nchunks) segs = nchunks;
    if (segs <= 1) return base;
    *off_seg = *off_flag + round256(static_cast<size_t>(pairs) * segs * sizeof(int));
    *seg_bytes = static_cast<size_t>(pairs) * segs * 3 * s.dk * s.dv * sizeof(float);
    return *off_seg + *seg_bytes;
}


// The prefill behind gdn_prefill_ex and gdn_prefill_noalloc: every argument
// check, then the launch.  ws (ws_bytes) holds the 256-byte status area and,
// after it, the staging area of an in-place chunked call; a call that needs
// the staging area and finds it too small returns GDN_ERR_WORKSPACE.
gdn_status prefill_core(const gdn_shape *shape, const gdn_prefill_options *options, const void *q, const void *k,
                        const void *v, const float *alpha, const float *beta, const float *S0, void *y, float *S_T,
                        void *ws, size_t ws_bytes, void *stream_) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    const gdn_shape &s = *shape;
    const size_t esz = s.dtype == GDN_BF16 ? 2 : 4;
    const bool has_tokens = s.B * s.T > 0;

    gdn_prefill_options opt{0, 0.f, 0, GDN_ALGO_AUTO, 0};
    if (options) opt = *options;
    if (opt.segments < 0 || opt.max_warmup_chunks < 0 || !(opt.log_eps <= 0.f)) return GDN_ERR_INVALID_ARG;
    if (opt.algorithm < GDN_ALGO_AUTO || opt.algorithm > GDN_ALGO_SEQUENTIAL) return GDN_ERR_INVALID_ARG;
    if (opt.test_stall_chunk < 0) return GDN_ERR_INVALID_ARG;
    const int algorithm = opt.algorithm;
    const int segments = opt.segments;

    if (has_tokens && (!q || !k || !v || !alpha || !beta || !y)) return GDN_ERR_INVALID_ARG;
    if (!ws || ws_bytes < kStatusBytes) return GDN_ERR_WORKSPACE;

    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(y, 16) || !aligned(S0, 16) ||
        !aligned(S_T, 16) || !aligned(alpha, 4) || !aligned(beta, 4) || !aligned(ws, 256))
        return GDN_ERR_ALIGNMENT;

    const Range rq{q, static_cast<size_t>(n_qk) * esz}, rk{k, static_cast<size_t>(n_qk) * esz};
    const Range rv{v, static_cast<size_t>(n_v) * esz}, ry{y, static_cast<size_t>(n_v) * esz};
    const Range ra{alpha, static_cast<size_t>(n_gate) * 4}, rb{beta, static_cast<size_t>(n_gate) * 4};
    const Range rs0{S0, static_cast<size_t>(n_state) * 4}, rst{S_T, static_cast<size_t>(n_state) * 4};
    const Range rws{ws, ws_bytes};
    for (const Range &in : {rq, rk, rv, ra, rb, rs0, rst, rws})
        if (overlap(ry, in)) return GDN_ERR_ALIASING;
    for (const Range &in : {rq, rk, rv, ra, rb, rws})
        if (overlap(rst, in)) return GDN_ERR_ALIASING;
    for (const Range &in : {rq, rk, rv, ra, rb, rs0})
        if (overlap(rws, in)) return GDN_ERR_ALIASING;
    const bool in_place = S0 && S_T && S0 == S_T;
    if (!in_place && overlap(rst, rs0)) return GDN_ERR_ALIASING;

    const bool chunked = algorithm == GDN_ALGO_CHUNKED || (algorithm == GDN_ALGO_AUTO && s.dtype == GDN_BF16);
    if (chunked && s.dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    // Only an in-place chunked call stages its final states.
    const bool stages = chunked && in_place && has_tokens;
    if (stages && ws_bytes < kStatusBytes + static_cast<size_t>(n_state) * sizeof(float)) return GDN_ERR_WORKSPACE;

    int num_sms = 0;
    st = check_device(&num_sms);
    if (st != GDN_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);

    if (s.B * s.Hv == 0) return GDN_OK;
    if (!has_tokens) {
        // Empty sequences: the final state is the initial state.
        if (S_T && !in_place) {
            if (S0)
                return from_cuda(cudaMemcpyAsync(S_T, S0, rst.n, cudaMemcpyDeviceToDevice, stream));
            return from_cuda(cudaMemsetAsync(S_T, 0, rst.n, stream));
        }
        return GDN_OK;
    }

    if (!chunked) {
        // Token-sequential path: each CTA reads its own head's S0 before it
        // writes that head's S_T, so in-place needs no staging.
        gdn::RecurrentParams p{};
        p.B = s.B; p.T = s.T; p.Hqk = s.Hqk; p.Hv = s.Hv; p.group = s.Hv / s.Hqk;
        p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta;
        p.S_in = S0; p.S_out = S_T; p.y = y;
        return from_cuda(gdn::launch_recurrent(p, s.dk, s.dv, static_cast<gdn_dtype>(s.dtype), stream));
    }

    gdn::ChunkedParams p{};
    p.B = s.B; p.T = s.T; p.Hqk = s.Hqk; p.Hv = s.Hv; p.group = s.Hv / s.Hqk; p.d = s.dk;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.S0 = S0; p.y = y;
    p.status = static_cast<uint32_t *>(ws);
    float *staging = reinterpret_cast<float *>(static_cast<char *>(ws) + kStatusBytes);
    // Runs of one head are processed by different CTAs, so a run that reads S0
    // may start after the head's last run wrote S_T: stage in-place results.
    p.S_T = in_place ? staging : S_T;
    p.segments = segments;
    p.log_eps = opt.log_eps < 0.f ? opt.log_eps : kDefaultLogEps;
    p.max_warmup_chunks = opt.max_warmup_chunks > 0 ? opt.max_warmup_chunks : kDefaultMaxWarmupChunks;
    p.test_stall_chunk = opt.test_stall_chunk;
    size_t off_flag = 0, off_seg = 0, seg_bytes = 0;
    const size_t full = exact_split_layout(s, n_state, &off_flag, &off_seg, &seg_bytes);
    if (seg_bytes > 0 && ws_bytes >= full) {
        p.exact_flag = reinterpret_cast<int *>(static_cast<char *>(ws) + off_flag);
        p.seg_state = reinterpret_cast<float *>(static_cast<char *>(ws) + off_seg);
        p.seg_state_bytes = seg_bytes;
    }
    st = from_cuda(gdn::launch_chunked(p, stream, num_sms));
    if (st != GDN_OK) return st;
    if (in_place) return from_cuda(cudaMemcpyAsync(S_T, staging, rst.n, cudaMemcpyDeviceToDevice, stream));
    return GDN_OK;
}

}  // namespace

extern "C" {

const char *gdn_status_string(gdn_status status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case GDN_ERR_ALIGNMENT: return "misaligned pointer";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_TIMEOUT: return "device-side wait timed out";
        case GDN_ERR_DEVICE: return "device-detected error";
        case GDN_ERR_ALIASING: return "overlapping buffers";
    }
    return "unknown status";
}

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

int gdn_device_supported(void) {
    int sms = 0;
    return check_device(&sms) == GDN_OK ? 1 : 0;
}

int gdn_prefill_launches(const gdn_shape *shape, const gdn_prefill_options *options) {
    int64_t n_qk, n_v, n_gate, n_state;
    if (check_shape(shape, &n_qk, &n_v, &n_gate, &n_state) != GDN_OK) return -1;
    const gdn_shape &s = *shape;
    gdn_prefill_options opt{0, 0.f, 0, GDN_ALGO_AUTO, 0};
    if (options) opt = *options;
    if (opt.segments < 0 || opt.algorithm < GDN_ALGO_AUTO || opt.algorithm > GDN_ALGO_SEQUENTIAL) return -1;
    if (s.B * s.T * s.Hv == 0) return 0;
    const bool chunked =
        opt.algorithm == GDN_ALGO_CHUNKED || (opt.algorithm == GDN_ALGO_AUTO && s.dtype == GDN_BF16);
    if (!chunked) return 1;
    if (s.dtype != GDN_BF16) return -1;
    int num_sms = 0;
    if (check_device(&num_sms) != GDN_OK) return -1;
    const int64_t pairs = s.B * s.Hv, nchunks = (s.T + 63) / 64;
    int P = gdn::plan_segments(pairs, nchunks, num_sms, opt.segments);
    const int64_t len = (nchunks + P - 1) / P;
    P = static_cast<int>((nchunks + len - 1) / len);
    size_t off_flag = 0, off_seg = 0, seg_bytes = 0;
    exact_split_layout(s, n_state, &off_flag, &off_seg, &seg_bytes);
    return gdn::takes_exact_split(pairs, nchunks, P, s.dk, seg_bytes) ? 4 : 1;
}

size_t gdn_prefill_workspace_bytes(const gdn_shape *shape) {
    int64_t n_qk, n_v, n_gate, n_state;
    if (check_shape(shape, &n_qk, &n_v, &n_gate, &n_state) != GDN_OK) return 0;
    size_t off_flag = 0, off_seg = 0, seg_bytes = 0;
    return exact_split_layout(*shape, n_state, &off_flag, &off_seg, &seg_bytes);
}

gdn_status gdn_prefill_ex(const gdn_shape *shape, const gdn_prefill_options *options,
                          const void *q, const void *k, const void *v,
                          const float *alpha, const float *beta,
                          const float *S0, void *y, float *S_T,
                          void *ws, size_t ws_bytes, void *stream) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    if (!ws) return GDN_ERR_WORKSPACE;
    if (ws_bytes < kStatusBytes + static_cast<size_t>(n_state) * sizeof(float)) return GDN_ERR_WORKSPACE;
    return prefill_core(shape, options, q, k, v, alpha, beta, S0, y, S_T, ws, ws_bytes, stream);
}

gdn_status gdn_prefill(const gdn_shape *shape, const void *q, const void *k, const void *v,
                       const float *alpha, const float *beta, const float *S0, void *y, float *S_T,
                       void *ws, size_t ws_bytes, void *stream) {
    return gdn_prefill_ex(shape, nullptr, q, k, v, alpha, beta, S0, y, S_T, ws, ws_bytes, stream);
}

gdn_status gdn_decode_step(const gdn_shape *shape, const void *q, const void *k, const void *v,
                           const float *alpha, const float *beta, float *S_inout, void *y, void *stream_) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    const gdn_shape &s = *shape;
    if (s.T != 1) return GDN_ERR_INVALID_ARG;
    if (s.B == 0) return GDN_OK;
    if (!q || !k || !v || !alpha || !beta || !S_inout || !y) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(y, 16) || !aligned(S_inout, 16) ||
        !aligned(alpha, 4) || !aligned(beta, 4))
        return GDN_ERR_ALIGNMENT;
    const size_t esz = s.dtype == GDN_BF16 ? 2 : 4;
    const Range rq{q, static_cast<size_t>(n_qk) * esz}, rk{k, static_cast<size_t>(n_qk) * esz};
    const Range rv{v, static_cast<size_t>(n_v) * esz}, ry{y, static_cast<size_t>(n_v) * esz};
    const Range ra{alpha, static_cast<size_t>(n_gate) * 4}, rb{beta, static_cast<size_t>(n_gate) * 4};
    const Range rs{S_inout, static_cast<size_t>(n_state) * 4};
    for (const Range &in : {rq, rk, rv, ra, rb, rs})
        if (overlap(ry, in)) return GDN_ERR_ALIASING;
    for (const Range &in : {rq, rk, rv, ra, rb})
        if (overlap(rs, in)) return GDN_ERR_ALIASING;
    int num_sms = 0;
    st = check_device(&num_sms);
    if (st != GDN_OK) return st;
    gdn::RecurrentParams p{};
    p.B = s.B; p.T = 1; p.Hqk = s.Hqk; p.Hv = s.Hv; p.group = s.Hv / s.Hqk;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta;
    p.S_in = S_inout; p.S_out = S_inout; p.y = y;
    return from_cuda(gdn::launch_recurrent(p, s.dk, s.dv, static_cast<gdn_dtype>(s.dtype),
                                           static_cast<cudaStream_t>(stream_)));
}

// Channel-wise decay (alpha [B, T, Hv, dk]): the token-sequential kernel for
// prefill (any T, dtype bf16 or fp32) and decode (T == 1); S_T may equal S0.
static gdn_status recurrence_cw(const gdn_shape *shape, bool decode, const void *q, const void *k, const void *v,
                                const float *alpha, const float *beta, const float *S0, float *S_T, void *y,
                                void *stream_) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    const gdn_shape &s = *shape;
    if (decode && s.T != 1) return GDN_ERR_INVALID_ARG;
    if (decode && !S_T) return GDN_ERR_INVALID_ARG;
    const bool has_tokens = s.B * s.T > 0;
    if (has_tokens && (!q || !k || !v || !alpha || !beta || !y)) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(y, 16) || !aligned(S0, 16) ||
        !aligned(S_T, 16) || !aligned(alpha, 16) || !aligned(beta, 4))
        return GDN_ERR_ALIGNMENT;
    const size_t esz = s.dtype == GDN_BF16 ? 2 : 4;
    const Range rq{q, static_cast<size_t>(n_qk) * esz}, rk{k, static_cast<size_t>(n_qk) * esz};
    const Range rv{v, static_cast<size_t>(n_v) * esz}, ry{y, static_cast<size_t>(n_v) * esz};
    const Range ra{alpha, static_cast<size_t>(n_gate) * s.dk * 4}, rb{beta, static_cast<size_t>(n_gate) * 4};
    const Range rs0{S0, static_cast<size_t>(n_state) * 4}, rst{S_T, static_cast<size_t>(n_state) * 4};
    for (const Range &in : {rq, rk, rv, ra, rb, rs0, rst})
        if (overlap(ry, in)) return GDN_ERR_ALIASING;
    for (const Range &in : {rq, rk, rv, ra, rb})
        if (overlap(rst, in)) return GDN_ERR_ALIASING;
    if (S0 != S_T && overlap(rst, rs0)) return GDN_ERR_ALIASING;
    int num_sms = 0;
    st = check_device(&num_sms);
    if (st != GDN_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (s.B * s.Hv == 0) return GDN_OK;
    if (!has_tokens) {
        if (S_T && S_T != S0) {
            if (S0) return from_cuda(cudaMemcpyAsync(S_T, S0, rst.n, cudaMemcpyDeviceToDevice, stream));
            return from_cuda(cudaMemsetAsync(S_T, 0, rst.n, stream));
        }
        return GDN_OK;
    }
    gdn::RecurrentParams p{};
    p.B = s.B; p.T = s.T; p.Hqk = s.Hqk; p.Hv = s.Hv; p.group = s.Hv / s.Hqk;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.alpha_cw = true;
    p.S_in = S0; p.S_out = S_T; p.y = y;
    return from_cuda(gdn::launch_recurrent(p, s.dk, s.dv, static_cast<gdn_dtype>(s.dtype), stream));
}

// Whether a channel-wise prefill of this shape takes the chunked tensor-core path.
static bool cw_chunked(const gdn_shape &s, int algorithm) {
    if (algorithm == GDN_ALGO_SEQUENTIAL) return false;
    return s.dtype == GDN_BF16 && s.dk == 128 && s.dv == 128;
}

// Segment count for which the exact split's maps are reserved: about two
// waves of a GPU with up to kExactSplitSmBound SMs (at most the chunk count).
static int64_t split_segments(const gdn_shape &s) {
    return gdn::exact_split_segments(s.B * s.Hv, (s.T + 63) / 64);
}

// Workspace of the chunked channel-wise prefill: status area, in-place
// staging, the exact split's flags and segment maps, then the per-chunk
// operand records and decay bounds.
static size_t cw_layout(const gdn_shape &s, int64_t n_state, size_t *off_ops, size_t *off_flag = nullptr,
                        size_t *off_seg = nullptr, size_t *seg_bytes = nullptr) {
    const size_t base = round256(kStatusBytes + static_cast<size_t>(n_state) * sizeof(float));
    const int64_t segs = split_segments(s), pairs = s.B * s.Hv;
    const size_t flags = round256(static_cast<size_t>(pairs) * segs * sizeof(int));
    const size_t maps = static_cast<size_t>(pairs) * segs * 3 * s.dk * s.dv * sizeof(float);
    if (off_flag) *off_flag = base;
    if (off_seg) *off_seg = base + flags;
    if (seg_bytes) *seg_bytes = maps;
    *off_ops = base + flags + round256(maps);
    return *off_ops + gdn::chunked_cw_ops_bytes(s.B, s.T, s.Hv);
}

size_t gdn_prefill_cw_workspace_bytes(const gdn_shape *shape) {
    int64_t n_qk, n_v, n_gate, n_state;
    if (check_shape(shape, &n_qk, &n_v, &n_gate, &n_state) != GDN_OK) return 0;
    if (!cw_chunked(*shape, GDN_ALGO_AUTO)) return kStatusBytes;
    size_t off = 0;
    return cw_layout(*shape, n_state, &off);
}

gdn_status gdn_prefill_cw_ex(const gdn_shape *shape, const gdn_prefill_options *options, const void *q,
                             const void *k, const void *v, const float *alpha, const float *beta, const float *S0,
                             void *y, float *S_T, void *ws, size_t ws_bytes, void *stream_) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    const gdn_shape &s = *shape;
    gdn_prefill_options opt{0, 0.f, 0, GDN_ALGO_AUTO, 0};
    if (options) opt = *options;
    if (opt.segments < 0 || opt.max_warmup_chunks < 0 || !(opt.log_eps <= 0.f)) return GDN_ERR_INVALID_ARG;
    if (opt.algorithm < GDN_ALGO_AUTO || opt.algorithm > GDN_ALGO_SEQUENTIAL) return GDN_ERR_INVALID_ARG;
    if (opt.test_stall_chunk != 0) return GDN_ERR_INVALID_ARG;
    if (opt.algorithm == GDN_ALGO_CHUNKED && !cw_chunked(s, GDN_ALGO_CHUNKED)) return GDN_ERR_UNSUPPORTED;
    if (!cw_chunked(s, opt.algorithm)) return recurrence_cw(shape, false, q, k, v, alpha, beta, S0, S_T, y, stream_);

    const bool has_tokens = s.B * s.T > 0;
    if (has_tokens && (!q || !k || !v || !alpha || !beta || !y)) return GDN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(y, 16) || !aligned(S0, 16) ||
        !aligned(S_T, 16) || !aligned(alpha, 16) || !aligned(beta, 4) || !aligned(ws, 256))
        return GDN_ERR_ALIGNMENT;
    const Range rq{q, static_cast<size_t>(n_qk) * 2}, rk{k, static_cast<size_t>(n_qk) * 2};
    const Range rv{v, static_cast<size_t>(n_v) * 2}, ry{y, static_cast<size_t>(n_v) * 2};
    const Range ra{alpha, static_cast<size_t>(n_gate) * s.dk * 4}, rb{beta, static_cast<size_t>(n_gate) * 4};
    const Range rs0{S0, static_cast<size_t>(n_state) * 4}, rst{S_T, static_cast<size_t>(n_state) * 4};
    const Range rws{ws, ws_bytes};
    for (const Range &in : {rq, rk, rv, ra, rb, rs0, rst, rws})
        if (overlap(ry, in)) return GDN_ERR_ALIASING;
    for (const Range &in : {rq, rk, rv, ra, rb, rws})
        if (overlap(rst, in)) return GDN_ERR_ALIASING;
    for (const Range &in : {rq, rk, rv, ra, rb, rs0})
        if (overlap(rws, in)) return GDN_ERR_ALIASING;
    const bool in_place = S0 && S_T && S0 == S_T;
    if (!in_place && overlap(rst, rs0)) return GDN_ERR_ALIASING;
    size_t off_ops = 0;
    const size_t need = cw_layout(s, n_state, &off_ops);
    if (has_tokens && s.Hv > 0 && (!ws || ws_bytes < need)) return GDN_ERR_WORKSPACE;
    int num_sms = 0;
    st = check_device(&num_sms);
    if (st != GDN_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (s.B * s.Hv == 0) return GDN_OK;
    if (!has_tokens) {
        if (S_T && !in_place) {
            if (S0) return from_cuda(cudaMemcpyAsync(S_T, S0, rst.n, cudaMemcpyDeviceToDevice, stream));
            return from_cuda(cudaMemsetAsync(S_T, 0, rst.n, stream));
        }
        return GDN_OK;
    }
    float *staging = reinterpret_cast<float *>(static_cast<char *>(ws) + kStatusBytes);
    gdn::ChunkedCwParams p{};
    p.B = s.B; p.T = s.T; p.Hqk = s.Hqk; p.Hv = s.Hv; p.group = s.Hv / s.Hqk; p.d = s.dk;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.S0 = S0; p.y = y;
    // segments of one head run on different CTAs: stage an in-place S_T
    p.S_T = in_place ? staging : S_T;
    p.segments = opt.segments;
    p.log_eps = opt.log_eps < 0.f ? opt.log_eps : kDefaultLogEps;
    p.max_warmup_chunks = opt.max_warmup_chunks > 0 ? opt.max_warmup_chunks : kDefaultMaxWarmupChunks;
    p.ops = static_cast<uint8_t *>(ws) + off_ops;
    {
        size_t off_flag = 0, off_seg = 0, seg_bytes = 0;
        cw_layout(s, n_state, &off_ops, &off_flag, &off_seg, &seg_bytes);
        if (seg_bytes > 0) {
            p.exact_flag = reinterpret_cast<int *>(static_cast<char *>(ws) + off_flag);
            p.seg_state = reinterpret_cast<float *>(static_cast<char *>(ws) + off_seg);
            p.seg_state_bytes = seg_bytes;
        }
    }
    st = from_cuda(gdn::launch_chunked_cw(p, stream, num_sms));
    if (st != GDN_OK) return st;
    if (in_place) return from_cuda(cudaMemcpyAsync(S_T, staging, rst.n, cudaMemcpyDeviceToDevice, stream));
    return GDN_OK;
}

gdn_status gdn_prefill_cw(const gdn_shape *shape, const void *q, const void *k, const void *v, const float *alpha,
                          const float *beta, const float *S0, void *y, float *S_T, void *stream) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    if (!cw_chunked(*shape, GDN_ALGO_AUTO) || shape->B * shape->T * shape->Hv == 0)
        return recurrence_cw(shape, false, q, k, v, alpha, beta, S0, S_T, y, stream);
    // Every argument check first (they end at the missing workspace), then the
    // chunked path's workspace, allocated and freed in stream order.
    st = gdn_prefill_cw_ex(shape, nullptr, q, k, v, alpha, beta, S0, y, S_T, nullptr, 0, stream);
    if (st != GDN_ERR_WORKSPACE) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const size_t bytes = gdn_prefill_cw_workspace_bytes(shape);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, cs) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    st = gdn_prefill_cw_ex(shape, nullptr, q, k, v, alpha, beta, S0, y, S_T, ws, bytes, stream);
    const cudaError_t fe = cudaFreeAsync(ws, cs);
    if (st == GDN_OK && fe != cudaSuccess) st = GDN_ERR_CUDA;
    return st;
}

gdn_status gdn_decode_step_cw(const gdn_shape *shape, const void *q, const void *k, const void *v,
                              const float *alpha, const float *beta, float *S_inout, void *y, void *stream) {
    return recurrence_cw(shape, true, q, k, v, alpha, beta, S_inout, S_inout, y, stream);
}

// Backward: the workspace holds the slab-state checkpoints and per-slab partial sums.
static gdn_status backward_workspace(const gdn_shape *shape, size_t *bytes) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    const int64_t nc = (shape->T + gdn::kBackwardCheckpointTokens - 1) / gdn::kBackwardCheckpointTokens;
    int64_t ck = 0;
    if (!mul_ok(n_state, nc, &ck) || ck > (INT64_MAX >> 4) || n_v > (INT64_MAX >> 6)) return GDN_ERR_INVALID_ARG;
    *bytes = gdn::backward_workspace_layout(shape->B, shape->T, shape->Hv, shape->dk, nullptr, nullptr, nullptr,
                                            nullptr);
    return GDN_OK;
}

size_t gdn_backward_workspace_bytes(const gdn_shape *shape) {
    size_t bytes = 0;
    return backward_workspace(shape, &bytes) == GDN_OK ? bytes : 0;
}

// Argument checks shared by both backward entry points (need: workspace bytes
// the chosen path requires).  Returns GDN_OK with *done set when nothing is
// left to launch (empty problem handled), else GDN_OK with *done clear.
static gdn_status backward_prologue(const gdn_shape *shape, const void *q, const void *k, const void *v,
                                    const float *alpha, const float *beta, const float *S0, const void *dy,
                                    const float *dS_T, float *dq, float *dk, float *dv, float *dlog_alpha,
                                    float *dbeta, float *dS0, void *ws, size_t ws_bytes, size_t need, void *stream_,
                                    int *num_sms, bool *done) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    *done = false;
    const gdn_shape &s = *shape;
    const bool has_tokens = s.B * s.T > 0;
    if (has_tokens && (!q || !k || !v || !alpha || !beta || !dy || !dq || !dk || !dv || !dlog_alpha || !dbeta))
        return GDN_ERR_INVALID_ARG;
    if (need > 0 && !ws) return GDN_ERR_WORKSPACE;
    if (ws_bytes < need) return GDN_ERR_WORKSPACE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dy, 16) || !aligned(S0, 16) ||
        !aligned(dS_T, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(dS0, 16) ||
        !aligned(alpha, 4) || !aligned(beta, 4) || !aligned(dlog_alpha, 4) || !aligned(dbeta, 4) ||
        !aligned(ws, 256))
        return GDN_ERR_ALIGNMENT;

    const size_t esz = s.dtype == GDN_BF16 ? 2 : 4;
    const Range rq{q, static_cast<size_t>(n_qk) * esz}, rk{k, static_cast<size_t>(n_qk) * esz};
    const Range rv{v, static_cast<size_t>(n_v) * esz}, rdy{dy, static_cast<size_t>(n_v) * esz};
    const Range ra{alpha, static_cast<size_t>(n_gate) * 4}, rb{beta, static_cast<size_t>(n_gate) * 4};
    const Range rs0{S0, static_cast<size_t>(n_state) * 4}, rdst{dS_T, static_cast<size_t>(n_state) * 4};
    const Range rdq{dq, static_cast<size_t>(n_qk) * 4}, rdk{dk, static_cast<size_t>(n_qk) * 4};
    const Range rdv{dv, static_cast<size_t>(n_v) * 4}, rdg{dlog_alpha, static_cast<size_t>(n_gate) * 4};
    const Range rdb{dbeta, static_cast<size_t>(n_gate) * 4}, rds0{dS0, static_cast<size_t>(n_state) * 4};
    const Range rws{ws, need};
    const Range outs[] = {rdq, rdk, rdv, rdg, rdb, rds0, rws};
    const Range ins[] = {rq, rk, rv, rdy, ra, rb, rs0, rdst};
    // dS0 may be the very buffer of dS_T (each element is read before it is written).
    const bool ds_in_place = dS0 && dS0 == dS_T;
    for (int o = 0; o < 7; ++o) {
        for (const Range &in : ins)
            if (!(ds_in_place && o == 5 && in.p == rdst.p) && overlap(outs[o], in)) return GDN_ERR_ALIASING;
        for (int o2 = o + 1; o2 < 7; ++o2)
            if (overlap(outs[o], outs[o2])) return GDN_ERR_ALIASING;
    }

    st = check_device(num_sms);
    if (st != GDN_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (s.B * s.Hv == 0) {
        *done = true;
        return GDN_OK;
    }
    if (!has_tokens) {
        // No tokens: dS0 = dS_T; there is nothing else to return.
        *done = true;
        if (dS0 && !ds_in_place) {
            if (dS_T) return from_cuda(cudaMemcpyAsync(dS0, dS_T, rds0.n, cudaMemcpyDeviceToDevice, stream));
            return from_cuda(cudaMemsetAsync(dS0, 0, rds0.n, stream));
        }
    }
    return GDN_OK;
}

gdn_status gdn_backward(const gdn_shape *shape, const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *S0, const void *dy, const float *dS_T, float *dq, float *dk,
                        float *dv, float *dlog_alpha, float *dbeta, float *dS0, void *ws, size_t ws_bytes,
                        void *stream_) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    // Per-token offsets inside the kernel are 32-bit: bound the head count times the head dim.
    if (static_cast<int64_t>(shape->Hv) * shape->dk > (int64_t(1) << 24)) return GDN_ERR_UNSUPPORTED;
    size_t need = 0;
    st = backward_workspace(shape, &need);
    if (st != GDN_OK) return st;
    int num_sms = 0;
    bool done = false;
    st = backward_prologue(shape, q, k, v, alpha, beta, S0, dy, dS_T, dq, dk, dv, dlog_alpha, dbeta, dS0, ws,
                           ws_bytes, need, stream_, &num_sms, &done);
    if (st != GDN_OK || done) return st;
    const gdn_shape &s = *shape;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);

    size_t o_dq = 0, o_dk = 0, o_b = 0, o_g = 0;
    gdn::backward_workspace_layout(s.B, s.T, s.Hv, s.dk, &o_dq, &o_dk, &o_b, &o_g);
    char *w = static_cast<char *>(ws);
    gdn::BackwardParams p{};
    p.B = s.B; p.T = s.T; p.Hqk = s.Hqk; p.Hv = s.Hv; p.group = s.Hv / s.Hqk;
    p.q = q; p.k = k; p.v = v; p.dy = dy; p.alpha = alpha; p.beta = beta; p.S0 = S0; p.dS_T = dS_T;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dlog_alpha = dlog_alpha; p.dbeta = dbeta; p.dS0 = dS0;
    p.ckpt = reinterpret_cast<float *>(w);
    p.part_dq = reinterpret_cast<float *>(w + o_dq);
    p.part_dk = reinterpret_cast<float *>(w + o_dk);
    p.part_dbeta = reinterpret_cast<float *>(w + o_b);
    p.part_dlog_alpha = reinterpret_cast<float *>(w + o_g);
    return from_cuda(gdn::launch_backward(p, s.dk, static_cast<gdn_dtype>(s.dtype), stream, num_sms));
}

// Chunked backward workspace: the chunk records, the states entering and the
// state gradients leaving every chunk, then (for dS0 == dS_T) dS0's staging.
size_t gdn_backward_chunked_workspace_bytes(const gdn_shape *shape) {
    int64_t n_qk, n_v, n_gate, n_state;
    if (check_shape(shape, &n_qk, &n_v, &n_gate, &n_state) != GDN_OK) return 0;
    if (shape->dtype != GDN_BF16 || shape->dk != 128 || shape->dv != 128) return 0;
    return round256(gdn::backward_chunked_workspace_bytes(shape->B, shape->T, shape->Hv)) +
           static_cast<size_t>(n_state) * sizeof(float);
}

gdn_status gdn_backward_chunked(const gdn_shape *shape, const void *q, const void *k, const void *v,
                                const float *alpha, const float *beta, const float *S0, const void *dy,
                                const float *dS_T, float *dq, float *dk, float *dv, float *dlog_alpha, float *dbeta,
                                float *dS0, void *ws, size_t ws_bytes, void *stream_) {
    int64_t n_qk, n_v, n_gate, n_state;
    gdn_status st = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st != GDN_OK) return st;
    if (shape->dtype != GDN_BF16 || shape->dk != 128 || shape->dv != 128) return GDN_ERR_UNSUPPORTED;
    const size_t need = gdn_backward_chunked_workspace_bytes(shape);
    int num_sms = 0;
    bool done = false;
    st = backward_prologue(shape, q, k, v, alpha, beta, S0, dy, dS_T, dq, dk, dv, dlog_alpha, dbeta, dS0, ws,
                           ws_bytes, need, stream_, &num_sms, &done);
    if (st != GDN_OK || done) return st;
    const gdn_shape &s = *shape;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    uint8_t *w = static_cast<uint8_t *>(ws);
    const size_t off_stage = round256(gdn::backward_chunked_workspace_bytes(s.B, s.T, s.Hv));
    // dS0 over dS_T: segments of one head run on different CTAs, so stage dS0
    const bool ds_in_place = dS0 && dS0 == dS_T;
    float *staging = reinterpret_cast<float *>(w + off_stage);
    gdn::BackwardParams p{};
    p.B = s.B; p.T = s.T; p.Hqk = s.Hqk; p.Hv = s.Hv; p.group = s.Hv / s.Hqk;
    p.q = q; p.k = k; p.v = v; p.dy = dy; p.alpha = alpha; p.beta = beta; p.S0 = S0; p.dS_T = dS_T;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dlog_alpha = dlog_alpha; p.dbeta = dbeta;
    p.dS0 = ds_in_place ? staging : dS0;
    st = from_cuda(gdn::launch_backward_chunked(p, w, stream, num_sms));
    if (st != GDN_OK) return st;
    if (ds_in_place)
        return from_cuda(cudaMemcpyAsync(dS0, staging, static_cast<size_t>(n_state) * sizeof(float),
                                         cudaMemcpyDeviceToDevice, stream));
    return GDN_OK;
}

gdn_status gdn_read_device_status(void *ws, void *stream_) {
    if (!ws) return GDN_ERR_INVALID_ARG;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    uint32_t word = 0;
    if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    if (word == 0) return GDN_OK;
    if (cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    return (word & gdn::kDevTimeout) ? GDN_ERR_TIMEOUT : GDN_ERR_DEVICE;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free prefill: its scratch is this fixed device array.  In host
// code `g_noalloc_scratch` is only a stand-in for the symbol; its device
// address comes from cudaGetSymbolAddress, looked up once per device.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_lock;
void *g_noalloc_ptr[kMaxDevices] = {};

gdn_status noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(g_noalloc_lock);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return GDN_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_prefill_noalloc(const gdn_shape *shape, const void *q, const void *k, const void *v,
                                          const float *alpha, const float *beta, const float *S0, void *y,
                                          float *S_T, void *stream) {
    int64_t n_qk, n_v, n_gate, n_state;
    const gdn_status st0 = check_shape(shape, &n_qk, &n_v, &n_gate, &n_state);
    if (st0 != GDN_OK) return st0;
    // Only an in-place chunked (bf16) call needs the staging area; the limit is checked
    // here, before anything else, so that such a shape is refused without side effects.
    const bool stages = shape->dtype == GDN_BF16 && S0 && S0 == S_T && shape->B * shape->T > 0;
    if (stages && kStatusBytes + static_cast<size_t>(n_state) * sizeof(float) > GDN_NOALLOC_SCRATCH_BYTES)
        return GDN_ERR_WORKSPACE;
    int num_sms = 0;
    gdn_status st = check_device(&num_sms);
    if (st != GDN_OK) return st;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != GDN_OK) return st;
    // The array starts zeroed and its status word is cleared only by
    // gdn_prefill_noalloc_status, so device-side errors of every call are kept.
    return prefill_core(shape, nullptr, q, k, v, alpha, beta, S0, y, S_T, scratch, GDN_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" gdn_status gdn_prefill_noalloc_status(void *stream) {
    void *scratch = nullptr;
    const gdn_status st = noalloc_scratch(&scratch);
    if (st != GDN_OK) return st;
    return gdn_read_device_status(scratch, stream);
}
