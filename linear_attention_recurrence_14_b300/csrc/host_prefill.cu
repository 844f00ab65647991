// Prefill from host memory (gdn_prefill_host, gdn.h): the sequence is cut into
// pieces of consecutive tokens; the host-to-device copy of piece p+1, the
// prefill of piece p and the device-to-host copy of piece p-1's y overlap on
// three streams.  Pieces run in order, each starting from the state the
// previous one left (the recurrence of the Qwen3.8-Next reading notes,
// section 2.1 "Gated DeltaNet", split at piece boundaries is the same map),
// so the result is that of one gdn_prefill over the whole sequence up to
// rounding.
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

constexpr size_t kAlign = 256;
constexpr int64_t kDefaultPieces = 8;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
    int64_t L;                 // tokens per piece
    size_t inner;              // gdn_prefill workspace (status word first)
    size_t state;              // one state buffer
    size_t q, v, g;            // one slot's q (= k), v (= y), gate sizes
    size_t slot;
    size_t total;
};

bool make_layout(const gdn_shape *s, int64_t tokens_per_piece, Layout *out) {
    if (!s || s->B < 0 || s->T < 0 || s->Hqk <= 0 || s->Hv <= 0 || s->dk <= 0 || s->dv <= 0) return false;
    if (tokens_per_piece < 0) return false;
    int64_t L = tokens_per_piece;
    if (L == 0) L = ((s->T + kDefaultPieces - 1) / kDefaultPieces + 63) / 64 * 64;
    if (L < 1) L = 1;
    if (L > s->T && s->T > 0) L = s->T;
    gdn_shape piece = *s;
    piece.T = L;
    const size_t inner = gdn_prefill_workspace_bytes(&piece);
    if (inner == 0) return false;
    const size_t esz = s->dtype == GDN_BF16 ? 2 : 4;
    Layout l;
    l.L = L;
    l.inner = round_up(inner);
    l.state = round_up(static_cast<size_t>(s->B) * s->Hv * s->dk * s->dv * 4);
    l.q = round_up(static_cast<size_t>(s->B) * L * s->Hqk * s->dk * esz);
    l.v = round_up(static_cast<size_t>(s->B) * L * s->Hv * s->dv * esz);
    l.g = round_up(static_cast<size_t>(s->B) * L * s->Hv * 4);
    l.slot = 2 * l.q + 2 * l.v + 2 * l.g;
    l.total = l.inner + 2 * l.state + 2 * l.slot;
    *out = l;
    return true;
}

// rows of `width` bytes: `height` of them, `spitch` apart at the source and
// `dpitch` apart at the destination
cudaError_t copy2d(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, size_t height,
                   cudaMemcpyKind kind, cudaStream_t st) {
    if (width == 0 || height == 0) return cudaSuccess;
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, st);
}

}  // namespace

extern "C" size_t gdn_prefill_host_workspace_bytes(const gdn_shape *shape, int64_t tokens_per_piece) {
    Layout l;
    return make_layout(shape, tokens_per_piece, &l) ? l.total : 0;
}

extern "C" gdn_status gdn_prefill_host(const gdn_shape *shape, int64_t tokens_per_piece,
                                       const void *q, const void *k, const void *v,
                                       const float *alpha, const float *beta, const float *S0,
                                       void *y, float *S_T, void *ws, size_t ws_bytes, void *stream_) {
    if (!shape) return GDN_ERR_INVALID_ARG;
    if (gdn_prefill_workspace_bytes(shape) == 0) {
        // invalid or unsupported shape: let the device entry point name the reason
        return gdn_prefill_ex(shape, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                              nullptr, nullptr, 0, nullptr);
    }
    Layout l;
    if (!make_layout(shape, tokens_per_piece, &l)) return GDN_ERR_INVALID_ARG;
    const gdn_shape s = *shape;
    if (!ws) return GDN_ERR_WORKSPACE;
    if (ws_bytes < l.total) return GDN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return GDN_ERR_ALIGNMENT;
    const bool has_tokens = s.B * s.T > 0;
    if (has_tokens && (!q || !k || !v || !alpha || !beta || !y)) return GDN_ERR_INVALID_ARG;
    if (s.B * s.Hv == 0) return GDN_OK;
    if (!gdn_device_supported()) return GDN_ERR_UNSUPPORTED;

    const size_t esz = s.dtype == GDN_BF16 ? 2 : 4;
    const size_t state_bytes = static_cast<size_t>(s.B) * s.Hv * s.dk * s.dv * 4;
    char *base = static_cast<char *>(ws);
    void *inner = base;
    float *S[2] = {reinterpret_cast<float *>(base + l.inner), reinterpret_cast<float *>(base + l.inner + l.state)};
    struct Slot {
        char *q, *k, *v, *a, *b, *y;
    } slot[2];
    for (int i = 0; i < 2; ++i) {
        char *p = base + l.inner + 2 * l.state + i * l.slot;
        slot[i].q = p;
        slot[i].k = p + l.q;
        slot[i].v = p + 2 * l.q;
        slot[i].y = p + 2 * l.q + l.v;
        slot[i].a = p + 2 * l.q + 2 * l.v;
        slot[i].b = p + 2 * l.q + 2 * l.v + l.g;
    }

    cudaStream_t comp = static_cast<cudaStream_t>(stream_);
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_h2d[2] = {}, ev_comp[2] = {}, ev_d2h[2] = {}, ev_done = nullptr;
    gdn_status result = GDN_OK;
    auto fail = [&](cudaError_t e) {
        if (e != cudaSuccess && result == GDN_OK) {
            cudaGetLastError();
            result = GDN_ERR_CUDA;
        }
        return e != cudaSuccess;
    };
    do {
        if (fail(cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking))) break;
        if (fail(cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking))) break;
        bool ok = true;
        for (int i = 0; i < 2 && ok; ++i)
            ok = !fail(cudaEventCreateWithFlags(&ev_h2d[i], cudaEventDisableTiming)) &&
                 !fail(cudaEventCreateWithFlags(&ev_comp[i], cudaEventDisableTiming)) &&
                 !fail(cudaEventCreateWithFlags(&ev_d2h[i], cudaEventDisableTiming));
        if (!ok || fail(cudaEventCreateWithFlags(&ev_done, cudaEventDisableTiming))) break;
        // Work the caller queued on its stream before this call comes first.
        if (fail(cudaEventRecord(ev_done, comp)) || fail(cudaStreamWaitEvent(h2d, ev_done, 0)) ||
            fail(cudaStreamWaitEvent(d2h, ev_done, 0)))
            break;

        const int64_t npieces = has_tokens ? (s.T + l.L - 1) / l.L : 0;
        const float *state_in = nullptr;
        if (S0) {
            if (fail(cudaMemcpyAsync(S[0], S0, state_bytes, cudaMemcpyHostToDevice, h2d))) break;
            state_in = S[0];
        }
        if (npieces == 0) {
            // no tokens: the final state is the initial one
            if (S_T) {
                if (S0) {
                    if (fail(cudaMemcpyAsync(S_T, S0, state_bytes, cudaMemcpyHostToHost, h2d))) break;
                } else {
                    if (fail(cudaMemsetAsync(S[0], 0, state_bytes, h2d)) ||
                        fail(cudaMemcpyAsync(S_T, S[0], state_bytes, cudaMemcpyDeviceToHost, h2d)))
                        break;
                }
            }
            if (fail(cudaEventRecord(ev_done, h2d)) || fail(cudaStreamWaitEvent(comp, ev_done, 0))) break;
            break;
        }
        const size_t row_qk = static_cast<size_t>(s.Hqk) * s.dk * esz, row_v = static_cast<size_t>(s.Hv) * s.dv * esz;
        const size_t row_g = static_cast<size_t>(s.Hv) * 4;
        for (int64_t pc = 0; pc < npieces && result == GDN_OK; ++pc) {
            const int i = static_cast<int>(pc & 1);
            const int64_t t0 = pc * l.L, tp = (t0 + l.L <= s.T ? l.L : s.T - t0);
            const size_t off_qk = static_cast<size_t>(t0) * row_qk, off_v = static_cast<size_t>(t0) * row_v;
            const size_t off_g = static_cast<size_t>(t0) * row_g;
            // inputs of this piece, once the prefill two pieces back is done with the slot
            if (pc >= 2 && fail(cudaStreamWaitEvent(h2d, ev_comp[i], 0))) break;
            const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k);
            const char *hv = static_cast<const char *>(v);
            const char *ha = reinterpret_cast<const char *>(alpha), *hb = reinterpret_cast<const char *>(beta);
            if (fail(copy2d(slot[i].q, tp * row_qk, hq + off_qk, s.T * row_qk, tp * row_qk, s.B, cudaMemcpyHostToDevice, h2d)) ||
                fail(copy2d(slot[i].k, tp * row_qk, hk + off_qk, s.T * row_qk, tp * row_qk, s.B, cudaMemcpyHostToDevice, h2d)) ||
                fail(copy2d(slot[i].v, tp * row_v, hv + off_v, s.T * row_v, tp * row_v, s.B, cudaMemcpyHostToDevice, h2d)) ||
                fail(copy2d(slot[i].a, tp * row_g, ha + off_g, s.T * row_g, tp * row_g, s.B, cudaMemcpyHostToDevice, h2d)) ||
                fail(copy2d(slot[i].b, tp * row_g, hb + off_g, s.T * row_g, tp * row_g, s.B, cudaMemcpyHostToDevice, h2d)) ||
                fail(cudaEventRecord(ev_h2d[i], h2d)))
                break;
            // the prefill of this piece, once its inputs are in and y of two pieces back is copied out
            if (fail(cudaStreamWaitEvent(comp, ev_h2d[i], 0))) break;
            if (pc >= 2 && fail(cudaStreamWaitEvent(comp, ev_d2h[i], 0))) break;
            gdn_shape ps = s;
            ps.T = tp;
            float *state_out = S[(pc + 1) & 1];
            const gdn_status st = gdn_prefill_ex(&ps, nullptr, slot[i].q, slot[i].k, slot[i].v,
                                                 reinterpret_cast<const float *>(slot[i].a),
                                                 reinterpret_cast<const float *>(slot[i].b), state_in, slot[i].y,
                                                 state_out, inner, l.inner, comp);
            if (st != GDN_OK) {
                result = st;
                break;
            }
            state_in = state_out;
            if (fail(cudaEventRecord(ev_comp[i], comp))) break;
            // y of this piece back to the host
            if (fail(cudaStreamWaitEvent(d2h, ev_comp[i], 0)) ||
                fail(copy2d(static_cast<char *>(y) + off_v, s.T * row_v, slot[i].y, tp * row_v, tp * row_v, s.B,
                            cudaMemcpyDeviceToHost, d2h)) ||
                fail(cudaEventRecord(ev_d2h[i], d2h)))
                break;
        }
        if (result != GDN_OK) break;
        if (S_T && fail(cudaMemcpyAsync(S_T, state_in, state_bytes, cudaMemcpyDeviceToHost, d2h))) break;
        // the caller's stream continues once every copy is done
        if (fail(cudaEventRecord(ev_done, d2h)) || fail(cudaStreamWaitEvent(comp, ev_done, 0))) break;
    } while (false);
    if (result != GDN_OK) {
        // The caller's stream was not chained behind the copies already queued:
        // let them finish before returning, so that no copy still reads or
        // writes the caller's host buffers once the call has failed.
        if (h2d) cudaStreamSynchronize(h2d);
        if (d2h) cudaStreamSynchronize(d2h);
        cudaGetLastError();
    }
    // Release: the runtime keeps streams and events alive until their work completes.
    for (int i = 0; i < 2; ++i) {
        if (ev_h2d[i]) cudaEventDestroy(ev_h2d[i]);
        if (ev_comp[i]) cudaEventDestroy(ev_comp[i]);
        if (ev_d2h[i]) cudaEventDestroy(ev_d2h[i]);
    }
    if (ev_done) cudaEventDestroy(ev_done);
    if (h2d) cudaStreamDestroy(h2d);
    if (d2h) cudaStreamDestroy(d2h);
    return result;
}
