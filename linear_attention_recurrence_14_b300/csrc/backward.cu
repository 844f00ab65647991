// Backward pass of the gated delta recurrence, token-sequential on CUDA cores,
// fp32 arithmetic.
//
// Forward map per (batch, value head) (Qwen3.8-Next reading notes, section
// 2.1, "Gated DeltaNet"):  S~ = a_t S_{t-1};  e_t = v_t - S~^T k_t;
// S_t = S~ + b_t k_t e_t^T;  y_t = S_t^T q_t.  Given dy_t and dS_T, with
// G = dL/dS_t walked from t = T down to 1 (G starts at dS_T), each token does
//
//   G    += q_t dy_t^T               dq_t  = S_t dy_t
//   g_k   = G^T k_t                  dv_t  = de = b_t g_k
//   dk_t  = b_t G e_t - S~ de        db_t  = g_k . e_t
//   G     = a_t (G - k_t de^T)       (G~ = G - k de^T, then through the decay)
//
// and dS_0 is the final G.  The decay gate's gradient is returned in log
// space, dlog(a_t) = a_t dL/da_t = <G~_t, S~_t>.  Because S_t = P_t S~_t +
// b_t k_t v_t^T with P_t = I - b_t k_t k_t^T and G~_t = P_t G_t, it obeys the
// scalar recursion
//
//   D_t = y_t . dy_t - b_t k_t^T G_t v_t + D_{t+1},   D_{T+1} = <dS_T, S_T>,
//
// so no term of it needs the state S_{t-1} of the reverse step.  Only dk_t
// (through S~ de) does.  The kernel evaluates the recursion once per chunk of
// kCk tokens (a suffix scan over the chunk), carrying D in fp64 from chunk to
// chunk.
//
// Work split: the columns of S (the value dimension) evolve independently in
// the forward map, so one CTA owns one (batch, value head, slab of 32 value
// columns); lane l of each warp owns column l of the slab and warp w owns key
// rows [w R, (w+1) R).  Sums over key rows (S^T k, G^T k) are per-thread sums
// plus a cross-warp sum in shared memory; sums over value columns (dk, dq) run
// as a lane reduce-scatter, are partial over the slab and are finished by the
// reduce kernel, which also sums the value heads that share a query/key head.
// All its sums run in a fixed order, so results are deterministic.
//
// States in reverse order: a forward sweep over the whole sequence stores the
// slab's state every kCk tokens (HBM checkpoints).  Then, for each chunk of
// kCk tokens from the last to the first, the CTA rebuilds the chunk's states
// from its checkpoint (kept in shared memory: kCk x 16 KB per slab at
// d = 128) and walks the chunk backwards.  The chunk's inputs are staged in
// shared memory with cp.async one chunk ahead.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kBwWarps = 8;
constexpr int kBwThreads = kBwWarps * 32;
constexpr int kSlab = 32;   // value columns per CTA, one per lane
constexpr int kCk = kBackwardCheckpointTokens;   // tokens per checkpoint interval

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Shared-memory layout of one CTA (byte offsets; every region 16-byte aligned).
template <int D, typename TIn>
struct BwLayout {
    static constexpr int R = D / kBwWarps;
    static constexpr size_t kScratch = size_t(kCk) * D * kSlab * 4;   // chunk states [kCk][R/4][256] float4
    static constexpr size_t kE = size_t(kCk) * kBwThreads * 4;        // e_t per thread [kCk][256]
    static constexpr size_t kYdy = size_t(3) * kCk * kSlab * 4;      // per-lane y.dy, g.e, g.v per token
    static constexpr size_t kRed = (2 * 2 * kBwWarps * kSlab + 2 * kBwWarps + kBwWarps) * 4;
    static constexpr size_t kStK = size_t(kCk) * D * sizeof(TIn);      // staged q or k rows
    static constexpr size_t kStV = size_t(kCk) * kSlab * sizeof(TIn);  // staged v or dy slab
    static constexpr size_t kStBuf = 2 * kStK + 2 * kStV + 2 * kCk * 4;
    static constexpr size_t kOffScratch = 0;
    static constexpr size_t kOffE = kOffScratch + kScratch;
    static constexpr size_t kOffYdy = kOffE + kE;
    static constexpr size_t kOffRed = kOffYdy + kYdy;
    static constexpr size_t kOffStage = kOffRed + ((kRed + 127) / 128) * 128;
    static constexpr bool kConvert = sizeof(TIn) != 4;                  // bf16 rows converted once per chunk
    static constexpr size_t kKQf = kConvert ? size_t(2) * kCk * D * 4 : 0;
    static constexpr size_t kOffKQf = kOffStage + 2 * kStBuf;
    static constexpr size_t kTotal = kOffKQf + kKQf;
    static_assert(kStK % 16 == 0 && kStV % 16 == 0 && kStBuf % 16 == 0, "staging regions must stay 16-byte aligned");
    static_assert(kTotal <= 227 * 1024, "shared memory over the per-CTA limit");
};

// Pointers into one staging buffer.
template <int D, typename TIn>
struct Staged {
    TIn *k, *q, *v, *dy;
    float *a, *b;
    __device__ explicit Staged(unsigned char *base) {
        using L = BwLayout<D, TIn>;
        k = reinterpret_cast<TIn *>(base);
        q = reinterpret_cast<TIn *>(base + L::kStK);
        v = reinterpret_cast<TIn *>(base + 2 * L::kStK);
        dy = reinterpret_cast<TIn *>(base + 2 * L::kStK + L::kStV);
        a = reinterpret_cast<float *>(base + 2 * L::kStK + 2 * L::kStV);
        b = a + kCk;
    }
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Issue the copies of tokens [t0, t0 + n) of this CTA's (batch, head, slab)
// into one staging buffer: the q and k rows of query/key head hk, the slab of
// v and dy, and alpha, beta.  One commit group.
template <int D, typename TIn>
__device__ __forceinline__ void stage_chunk(const BackwardParams &p, unsigned char *buf, int64_t b, int h, int hk,
                                            int slab, int64_t t0, int n) {
    constexpr int kRowPieces = D * int(sizeof(TIn)) / 16;
    constexpr int kColPieces = kSlab * int(sizeof(TIn)) / 16;
    constexpr int kPerTok = 2 * kRowPieces + 2 * kColPieces;
    using L = BwLayout<D, TIn>;
    const char *qg = static_cast<const char *>(p.q), *kg = static_cast<const char *>(p.k);
    const char *vg = static_cast<const char *>(p.v), *dyg = static_cast<const char *>(p.dy);
    for (int idx = threadIdx.x; idx < n * kPerTok; idx += kBwThreads) {
        const int s = idx / kPerTok;
        int c = idx - s * kPerTok;
        const int64_t tok = b * p.T + t0 + s;
        const int64_t qk_row = (tok * p.Hqk + hk) * D;                     // element offset of the q/k row
        const int64_t v_row = (tok * p.Hv + h) * D + int64_t(slab) * kSlab;  // element offset of the v/dy slab
        const char *src;
        unsigned char *dst;
        if (c < kRowPieces) {
            src = kg + qk_row * int64_t(sizeof(TIn)) + c * 16;
            dst = buf + size_t(s) * D * sizeof(TIn) + c * 16;
        } else if ((c -= kRowPieces) < kRowPieces) {
            src = qg + qk_row * int64_t(sizeof(TIn)) + c * 16;
            dst = buf + L::kStK + size_t(s) * D * sizeof(TIn) + c * 16;
        } else if ((c -= kRowPieces) < kColPieces) {
            src = vg + v_row * int64_t(sizeof(TIn)) + c * 16;
            dst = buf + 2 * L::kStK + size_t(s) * kSlab * sizeof(TIn) + c * 16;
        } else {
            c -= kColPieces;
            src = dyg + v_row * int64_t(sizeof(TIn)) + c * 16;
            dst = buf + 2 * L::kStK + L::kStV + size_t(s) * kSlab * sizeof(TIn) + c * 16;
        }
        cp_async16(dst, src);
    }
    float *as = reinterpret_cast<float *>(buf + 2 * L::kStK + 2 * L::kStV);
    for (int s = threadIdx.x; s < n; s += kBwThreads) {
        const int64_t g = (b * p.T + t0 + s) * p.Hv + h;
        cp_async4(as + s, p.alpha + g);
        cp_async4(as + kCk + s, p.beta + g);
    }
    cp_async_commit();
}

// R consecutive staged elements (16-byte aligned) as floats; the address is
// the same for every lane of a warp (a broadcast read).
template <typename TIn, int R>
__device__ __forceinline__ void lds_row(const TIn *src, float (&dst)[R]) {
    if constexpr (sizeof(TIn) == 2) {
        static_assert(R % 8 == 0, "bf16 rows come in groups of 8");
#pragma unroll
        for (int i = 0; i < R; i += 8) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(src + i);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&w[j]);
                dst[i + 2 * j] = __low2float(pr);
                dst[i + 2 * j + 1] = __high2float(pr);
            }
        }
    } else {
        static_assert(R % 4 == 0, "fp32 rows come in groups of 4");
#pragma unroll
        for (int i = 0; i < R; i += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(src + i);
            dst[i] = f.x; dst[i + 1] = f.y; dst[i + 2] = f.z; dst[i + 3] = f.w;
        }
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Sum over the 32 lanes of x[i] for every i, scattered: returns the total of
// index i = lane / (32 / N) (each index is held by 32 / N lanes).  log2(N)
// halving exchanges (N - 1 shuffles) and log2(32 / N) plain ones.
template <int N>
__device__ __forceinline__ float lane_reduce_scatter(float (&x)[N], int lane) {
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
#pragma unroll
    for (int s = 0; (N >> s) > 1; ++s) {
        const int o = 16 >> s;
        const int half = N >> (s + 1);
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? x[i] : x[i + half];
            const float keep = upper ? x[i + half] : x[i];
            x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = x[0];
#pragma unroll
    for (int o = (32 / N) >> 1; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

// Sum of the 8 warps' partials of one column (a fixed tree order).
__device__ __forceinline__ float sum_warps(const float *p) {
    return ((p[0] + p[kSlab]) + (p[2 * kSlab] + p[3 * kSlab])) +
           ((p[4 * kSlab] + p[5 * kSlab]) + (p[6 * kSlab] + p[7 * kSlab]));
}

template <int D, typename TIn>
__global__ void __launch_bounds__(kBwThreads, 1) backward_kernel(BackwardParams p) {
    using L = BwLayout<D, TIn>;
    constexpr int R = L::R;          // key rows per warp
    constexpr int R4 = R / 4;        // float4 groups of a thread's state column
    constexpr int NS = D / kSlab;    // slabs per head
    static_assert(R % 4 == 0 && NS * kSlab == D, "unsupported head dim");
    static_assert(kCk == 8, "the per-chunk tail scans 8 tokens");

    extern __shared__ __align__(128) unsigned char smem[];
    float4 *scratch = reinterpret_cast<float4 *>(smem + L::kOffScratch);
    float *ebuf = reinterpret_cast<float *>(smem + L::kOffE);
    float *ydl = reinterpret_cast<float *>(smem + L::kOffYdy);     // [kCk][32] y.dy per lane (warp 0)
    float *gel = ydl + kCk * kSlab;                                 // [kCk][32] g.e per lane
    float *gvl = gel + kCk * kSlab;                                 // [kCk][32] g.v per lane
    float *red_k = reinterpret_cast<float *>(smem + L::kOffRed);   // [2][8][32]
    float *red_q = red_k + 2 * kBwWarps * kSlab;                    // [2][8][32]
    float *red_kq = red_q + 2 * kBwWarps * kSlab;                   // [2][8]
    float *red_d = red_kq + 2 * kBwWarps;                           // [8]
    unsigned char *stage = smem + L::kOffStage;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t cta = blockIdx.x;   // (b * Hv + h) * NS + slab
    const int slab = static_cast<int>(cta % NS);
    const int64_t pair = cta / NS;
    const int64_t b = pair / p.Hv;
    const int h = static_cast<int>(pair % p.Hv);
    const int hk = h / p.group;
    const int r0 = warp * R;
    const int col = slab * kSlab + lane;
    const int64_t T = p.T;
    const int64_t NC = (T + kCk - 1) / kCk;
    float4 *ck = reinterpret_cast<float4 *>(p.ckpt) + cta * NC * R4 * kBwThreads;   // [NC][R4][256]
    const int64_t row_base = (b * T * p.Hv + h) * NS + slab;   // partial-sum row of token 0
    const int64_t row_step = int64_t(p.Hv) * NS;                // rows between consecutive tokens

    float S[R], G[R], Sn[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        S[r] = p.S0 ? p.S0[(pair * D + r0 + r) * D + col] : 0.f;
        G[r] = 0.f;
        Sn[r] = 0.f;
    }
    double Dc = 0.0;   // D at the first token of the chunk last walked (every lane of warp 0)
    unsigned it = 0;   // token counter: parity of the cross-warp buffers

    stage_chunk<D, TIn>(p, stage, b, h, hk, slab, 0, static_cast<int>(T < kCk ? T : kCk));

    for (int64_t i = 0; i < 2 * NC; ++i) {
        const bool fwd = i < NC;
        const int64_t ci = fwd ? i : 2 * NC - 1 - i;
        const int64_t t0 = ci * kCk;
        const int n = static_cast<int>(T - t0 < kCk ? T - t0 : kCk);
        // The last forward chunk is also the first reverse one: same buffer.
        const int bi = static_cast<int>((fwd ? i : i - 1) & 1);
        cp_async_wait_all();
        __syncthreads();
        if (i + 1 < 2 * NC && i + 1 != NC) {
            const int64_t ni = i + 1;
            const int64_t nci = ni < NC ? ni : 2 * NC - 1 - ni;
            const int nn = static_cast<int>(T - nci * kCk < kCk ? T - nci * kCk : kCk);
            stage_chunk<D, TIn>(p, stage + ((ni < NC ? ni : ni - 1) & 1) * L::kStBuf, b, h, hk, slab, nci * kCk, nn);
        }
        const Staged<D, TIn> st(stage + bi * L::kStBuf);
        // The chunk's k and q rows as fp32 ([2][kCk][D]: k then q).
        const float *kf;
        if constexpr (L::kConvert) {
            float *dst = reinterpret_cast<float *>(smem + L::kOffKQf);
            constexpr int kPieces = 2 * kCk * D / 8;   // 8 bf16 (16 bytes) per piece; k and q are adjacent
            for (int pc = tid; pc < kPieces; pc += kBwThreads) {
                const uint4 raw = reinterpret_cast<const uint4 *>(st.k)[pc];
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                float f[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162 *>(&w[j]);
                    f[2 * j] = __low2float(pr);
                    f[2 * j + 1] = __high2float(pr);
                }
                reinterpret_cast<float4 *>(dst)[2 * pc] = make_float4(f[0], f[1], f[2], f[3]);
                reinterpret_cast<float4 *>(dst)[2 * pc + 1] = make_float4(f[4], f[5], f[6], f[7]);
            }
            __syncthreads();
            kf = dst;
        } else {
            kf = reinterpret_cast<const float *>(st.k);
        }
        const float *qf = kf + kCk * D;

        if (fwd) {
            // Forward sweep: checkpoint the state entering this chunk.
            if (ci + 1 < NC) {
#pragma unroll
                for (int j = 0; j < R4; ++j)
                    ck[(ci * R4 + j) * kBwThreads + tid] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) Sn[r] = S[r];
            }
            for (int s = 0; s < n; ++s) {
                const int buf = static_cast<int>(it++ & 1);
                float kr[R];
                lds_row<float, R>(kf + s * D + r0, kr);
                const float vj = to_f(st.v[s * kSlab + lane]);
                const float a = st.a[s], bt = st.b[s];
                float pk0 = 0.f, pk1 = 0.f;
#pragma unroll
                for (int r = 0; r < R; r += 2) {
                    pk0 = fmaf(S[r], kr[r], pk0);
                    pk1 = fmaf(S[r + 1], kr[r + 1], pk1);
                }
                red_k[(buf * kBwWarps + warp) * kSlab + lane] = pk0 + pk1;
                __syncthreads();
                const float rk = sum_warps(red_k + buf * kBwWarps * kSlab + lane);
                const float be = bt * (vj - a * rk);
#pragma unroll
                for (int r = 0; r < R; ++r) S[r] = fmaf(a, S[r], kr[r] * be);
            }
            continue;
        }

        if (i == NC) {
            // S holds S_T: G starts at dS_T and D at <dS_T, S_T> (this slab).
            float part = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                G[r] = p.dS_T ? p.dS_T[(pair * D + r0 + r) * D + col] : 0.f;
                part = fmaf(G[r], S[r], part);
            }
            part = warp_sum(part);
            if (lane == 0) red_d[warp] = part;
            __syncthreads();
            if (warp == 0) {
#pragma unroll
                for (int w = 0; w < kBwWarps; ++w) Dc += static_cast<double>(red_d[w]);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) S[r] = Sn[r];
        if (ci > 0) {
#pragma unroll
            for (int j = 0; j < R4; ++j) {
                const float4 f = ck[((ci - 1) * R4 + j) * kBwThreads + tid];
                Sn[4 * j] = f.x; Sn[4 * j + 1] = f.y; Sn[4 * j + 2] = f.z; Sn[4 * j + 3] = f.w;
            }
        }

        // Rebuild the chunk: the state entering each token, e_t, and y_t . dy_t per lane.
        for (int s = 0; s < n; ++s) {
            const int buf = static_cast<int>(it++ & 1);
#pragma unroll
            for (int j = 0; j < R4; ++j)
                scratch[(s * R4 + j) * kBwThreads + tid] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
            float kr[R], qr[R];
            lds_row<float, R>(kf + s * D + r0, kr);
            lds_row<float, R>(qf + s * D + r0, qr);
            const float vj = to_f(st.v[s * kSlab + lane]);
            const float dyj = to_f(st.dy[s * kSlab + lane]);
            const float a = st.a[s], bt = st.b[s];
            float pk0 = 0.f, pk1 = 0.f, pq0 = 0.f, pq1 = 0.f, kq0 = 0.f, kq1 = 0.f;
#pragma unroll
            for (int r = 0; r < R; r += 2) {
                pk0 = fmaf(S[r], kr[r], pk0);
                pk1 = fmaf(S[r + 1], kr[r + 1], pk1);
                pq0 = fmaf(S[r], qr[r], pq0);
                pq1 = fmaf(S[r + 1], qr[r + 1], pq1);
                kq0 = fmaf(kr[r], qr[r], kq0);
                kq1 = fmaf(kr[r + 1], qr[r + 1], kq1);
            }
            red_k[(buf * kBwWarps + warp) * kSlab + lane] = pk0 + pk1;
            red_q[(buf * kBwWarps + warp) * kSlab + lane] = pq0 + pq1;
            if (lane == 0) red_kq[buf * kBwWarps + warp] = kq0 + kq1;
            __syncthreads();
            const float rk = sum_warps(red_k + buf * kBwWarps * kSlab + lane);
            const float rq = sum_warps(red_q + buf * kBwWarps * kSlab + lane);
            const float *kqp = red_kq + buf * kBwWarps;
            const float kqa = ((kqp[0] + kqp[1]) + (kqp[2] + kqp[3])) + ((kqp[4] + kqp[5]) + (kqp[6] + kqp[7]));
            const float e = vj - a * rk;
            const float be = bt * e;
            const float y = fmaf(kqa, be, a * rq);
            ebuf[s * kBwThreads + tid] = e;
            if (warp == 0) ydl[s * kSlab + lane] = y * dyj;
#pragma unroll
            for (int r = 0; r < R; ++r) S[r] = fmaf(a, S[r], kr[r] * be);
        }

        // Walk the chunk backwards.  The column sums of token s (the dk and dq
        // partials) are finished during token s-1, before its barrier.
        float xp[2 * R];
#pragma unroll
        for (int r = 0; r < 2 * R; ++r) xp[r] = 0.f;
        int pend = -1;   // token (within the chunk) whose column sums are pending
        const bool writer = lane % (32 / (2 * R)) == 0;
        const int idx = lane / (32 / (2 * R));
        // Partial-sum rows and dv of the chunk's first token; consecutive tokens are row_step rows apart.
        const int64_t prow0 = row_base + t0 * row_step;
        const int row_stride = static_cast<int>(row_step) * D;
        float *const pdk0 = p.part_dk + prow0 * D + r0;
        float *const pdq0 = p.part_dq + prow0 * D + r0;
        float *const dv0 = p.dv + ((b * T + t0) * p.Hv + h) * D + col;
        const int dv_stride = p.Hv * D;
        for (int s = n - 1; s >= 0; --s) {
            const int buf = static_cast<int>(it++ & 1);
            float Sp[R];
#pragma unroll
            for (int j = 0; j < R4; ++j) {
                const float4 f = scratch[(s * R4 + j) * kBwThreads + tid];
                Sp[4 * j] = f.x; Sp[4 * j + 1] = f.y; Sp[4 * j + 2] = f.z; Sp[4 * j + 3] = f.w;
            }
            const float e = ebuf[s * kBwThreads + tid];
            float kr[R], qr[R];
            lds_row<float, R>(kf + s * D + r0, kr);
            lds_row<float, R>(qf + s * D + r0, qr);
            const float vj = to_f(st.v[s * kSlab + lane]);
            const float dyj = to_f(st.dy[s * kSlab + lane]);
            const float a = st.a[s], bt = st.b[s];

            float pg0 = 0.f, pg1 = 0.f;
#pragma unroll
            for (int r = 0; r < R; r += 2) {
                G[r] = fmaf(qr[r], dyj, G[r]);
                G[r + 1] = fmaf(qr[r + 1], dyj, G[r + 1]);
                pg0 = fmaf(G[r], kr[r], pg0);
                pg1 = fmaf(G[r + 1], kr[r + 1], pg1);
            }
            red_k[(buf * kBwWarps + warp) * kSlab + lane] = pg0 + pg1;
            {
                const float xs = lane_reduce_scatter<2 * R>(xp, lane);
                if (pend >= 0 && writer) {
                    if (idx < R)
                        pdk0[pend * row_stride + idx] = xs;
                    else
                        pdq0[pend * row_stride + idx - R] = xs;
                }
            }
            __syncthreads();
            const float gk = sum_warps(red_k + buf * kBwWarps * kSlab + lane);
            const float de = bt * gk;

            // Column-local parts of dk_t = b G e - a S_{t-1} de (rows 0..R-1) and of
            // dq_t = S_t dy = (a S_{t-1} + b k e^T) dy (rows R..2R-1).
            const float be = bt * e, ade = a * de, ady = a * dyj, bedy = be * dyj;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                xp[r] = fmaf(G[r], be, -(Sp[r] * ade));
                xp[R + r] = fmaf(Sp[r], ady, kr[r] * bedy);
            }
            pend = s;
#pragma unroll
            for (int r = 0; r < R; ++r) G[r] = a * fmaf(-kr[r], de, G[r]);

            if (warp == 0) {
                dv0[s * dv_stride] = de;
                gel[s * kSlab + lane] = gk * e;
                gvl[s * kSlab + lane] = gk * vj;
            }
        }
        {
            const float xs = lane_reduce_scatter<2 * R>(xp, lane);
            if (writer) {
                if (idx < R)
                    pdk0[pend * row_stride + idx] = xs;
                else
                    pdq0[pend * row_stride + idx - R] = xs;
            }
        }

        // Per-chunk tail (warp 0): lane sums of y.dy, g.e, g.v for the n
        // tokens, then dbeta and D_t = D_{t+1} + y.dy - beta g.v by a suffix
        // scan over the chunk, carried in fp64 from chunk to chunk.
        if (warp == 0) {
            float z[32];
#pragma unroll
            for (int s = 0; s < kCk; ++s) {
                z[s] = s < n ? ydl[s * kSlab + lane] : 0.f;
                z[kCk + s] = s < n ? gel[s * kSlab + lane] : 0.f;
                z[2 * kCk + s] = s < n ? gvl[s * kSlab + lane] : 0.f;
                z[3 * kCk + s] = 0.f;
            }
            const float tot = lane_reduce_scatter<32>(z, lane);   // lane l: quantity l / 8 of token l % 8
            const int s = lane & (kCk - 1);
            const float ge = __shfl_sync(0xffffffffu, tot, s + kCk);
            const float gv = __shfl_sync(0xffffffffu, tot, s + 2 * kCk);
            float c = (lane < kCk && s < n) ? tot - st.b[s] * gv : 0.f;
#pragma unroll
            for (int o = 1; o < kCk; o <<= 1) {
                const float u = __shfl_down_sync(0xffffffffu, c, o);
                if (s + o < kCk) c += u;
            }
            const double Dt = Dc + static_cast<double>(c);
            if (lane < n) {
                const int64_t row = row_base + (t0 + lane) * row_step;
                p.part_dlog_alpha[row] = static_cast<float>(Dt);
                p.part_dbeta[row] = ge;
            }
            Dc = __shfl_sync(0xffffffffu, Dt, 0);
        }
    }

    if (p.dS0) {
#pragma unroll
        for (int r = 0; r < R; ++r) p.dS0[(pair * D + r0 + r) * D + col] = G[r];
    }
}

// Sums the per-slab partials: dq and dk over slabs and over the value heads
// of each query/key head, dbeta and dlog(alpha) over slabs.
template <int D>
__global__ void __launch_bounds__(256) backward_reduce_kernel(BackwardParams p) {
    constexpr int NS = D / kSlab;
    constexpr int V4 = D / 4;
    const int64_t nvec = p.B * p.T * p.Hqk * V4;
    const int64_t nsc = p.B * p.T * p.Hv;
    const int64_t total = 2 * nvec + nsc;
    for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += int64_t(gridDim.x) * blockDim.x) {
        if (idx < 2 * nvec) {
            const bool is_k = idx >= nvec;
            const int64_t vi = is_k ? idx - nvec : idx;
            const int64_t row = vi / V4;   // (b * T + t) * Hqk + hk
            const int c4 = static_cast<int>(vi - row * V4);
            const int64_t bt = row / p.Hqk;
            const int hk = static_cast<int>(row - bt * p.Hqk);
            const float4 *src = reinterpret_cast<const float4 *>(is_k ? p.part_dk : p.part_dq);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int g = 0; g < p.group; ++g) {
                const int64_t h = int64_t(hk) * p.group + g;
#pragma unroll
                for (int s = 0; s < NS; ++s) {
                    const float4 f = src[((bt * p.Hv + h) * NS + s) * V4 + c4];
                    acc.x += f.x; acc.y += f.y; acc.z += f.z; acc.w += f.w;
                }
            }
            reinterpret_cast<float4 *>(is_k ? p.dk : p.dq)[row * V4 + c4] = acc;
        } else {
            const int64_t r = idx - 2 * nvec;   // (b * T + t) * Hv + h
            float sb = 0.f, sg = 0.f;
#pragma unroll
            for (int s = 0; s < NS; ++s) {
                sb += p.part_dbeta[r * NS + s];
                sg += p.part_dlog_alpha[r * NS + s];
            }
            p.dbeta[r] = sb;
            p.dlog_alpha[r] = sg;
        }
    }
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

template <int D, typename TIn>
cudaError_t launch_typed(const BackwardParams &p, cudaStream_t stream, int num_sms) {
    using L = BwLayout<D, TIn>;
    constexpr int NS = D / kSlab;
    const int64_t ctas = p.B * p.Hv * NS;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(backward_kernel<D, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(L::kTotal));
    if (e != cudaSuccess) return e;
    backward_kernel<D, TIn><<<static_cast<unsigned>(ctas), kBwThreads, L::kTotal, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t total = 2 * p.B * p.T * p.Hqk * (D / 4) + p.B * p.T * p.Hv;
    const int64_t want = (total + 255) / 256, cap = int64_t(num_sms) * 16;
    const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
    backward_reduce_kernel<D><<<blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t backward_workspace_layout(int64_t B, int64_t T, int Hv, int d, size_t *off_part_dq, size_t *off_part_dk,
                                 size_t *off_part_b, size_t *off_part_g) {
    const int64_t NS = d / kSlab;
    const int64_t NC = (T + kCk - 1) / kCk;
    const size_t ckpt = round256(size_t(B) * Hv * NC * d * d * 4);
    const size_t pvec = round256(size_t(B) * T * Hv * NS * d * 4);
    const size_t psc = round256(size_t(B) * T * Hv * NS * 4);
    if (off_part_dq) *off_part_dq = ckpt;
    if (off_part_dk) *off_part_dk = ckpt + pvec;
    if (off_part_b) *off_part_b = ckpt + 2 * pvec;
    if (off_part_g) *off_part_g = ckpt + 2 * pvec + psc;
    return ckpt + 2 * pvec + 2 * psc;
}

cudaError_t launch_backward(const BackwardParams &p, int d, gdn_dtype dtype, cudaStream_t stream, int num_sms) {
    if (p.B * p.Hv == 0 || p.T == 0) return cudaSuccess;
    if (d == 128) {
        return dtype == GDN_BF16 ? launch_typed<128, __nv_bfloat16>(p, stream, num_sms)
                                 : launch_typed<128, float>(p, stream, num_sms);
    }
    if (d == 64) {
        return dtype == GDN_BF16 ? launch_typed<64, __nv_bfloat16>(p, stream, num_sms)
                                 : launch_typed<64, float>(p, stream, num_sms);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
