// Token-sequential gated delta recurrence on CUDA cores, fp32 arithmetic.
//
// One CTA owns one (batch, value head).  Its fp32 state S [dk x dv] lives in
// registers for the whole call: warp w owns rows [w*R, (w+1)*R) (R = dk / 8)
// and lane l owns columns [l*C, (l+1)*C) (C = dv / 32), so every row of the
// state is read and written by one warp as one coalesced 128-bit (d = 128) or
// 64-bit (d = 64) access per lane.
//
// Per token (Qwen3.8-Next reading notes, section 2.1, "Gated DeltaNet"):
//   r_k = S^T k and r_q = S^T q      (one pass over the registers, partial
//                                     sums over the warp's rows, then a
//                                     cross-warp sum through shared memory)
//   e   = v - alpha r_k              (= v - S~^T k with S~ = alpha S)
//   y   = alpha r_q + beta (k.q) e   (= S_t^T q, read after the write)
//   S   = alpha S + beta k e^T
//
// Used for decode (T = 1: the state is streamed HBM -> registers -> HBM
// once, the kernel is bound by HBM bandwidth) and for fp32 prefill, where the
// state stays in registers across all T tokens.
//
// Channel-wise decay (CW): alpha_t is a vector over the key dimension and
// S~ = diag(alpha_t) S, so row i of the state decays by alpha_t[i]:
//   r_k = S^T (alpha o k),  r_q = S^T (alpha o q),  e = v - r_k,
//   y = r_q + beta (k.q) e,  S = diag(alpha) S + beta k e^T.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// Load N consecutive elements (N * sizeof(T) a multiple of 8 bytes) as floats.
template <typename T, int N>
__device__ __forceinline__ void load_row(const T *__restrict__ src, float (&dst)[N]) {
    if constexpr (sizeof(T) == 2 && N == 2) {
        const __nv_bfloat162 pr = __ldg(reinterpret_cast<const __nv_bfloat162 *>(src));
        dst[0] = __low2float(pr);
        dst[1] = __high2float(pr);
    } else if constexpr (sizeof(T) == 2) {
        static_assert(N % 4 == 0, "bf16 loads come in groups of 4");
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(src + i));
            const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
            const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
            dst[i + 0] = __low2float(lo);
            dst[i + 1] = __high2float(lo);
            dst[i + 2] = __low2float(hi);
            dst[i + 3] = __high2float(hi);
        }
    } else {
        static_assert(N % 2 == 0, "fp32 loads come in pairs");
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float2 f = __ldg(reinterpret_cast<const float2 *>(src + i));
            dst[i] = f.x;
            dst[i + 1] = f.y;
        }
    }
}

template <typename T, int N>
__device__ __forceinline__ void store_row(T *__restrict__ dst, const float (&src)[N]) {
    if constexpr (sizeof(T) == 2) {
        if constexpr (N == 4) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(src[0], src[1]);
            __nv_bfloat162 hi = __floats2bfloat162_rn(src[2], src[3]);
            uint2 raw;
            raw.x = *reinterpret_cast<uint32_t *>(&lo);
            raw.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(dst) = raw;
        } else {
#pragma unroll
            for (int i = 0; i < N; i += 2)
                *reinterpret_cast<__nv_bfloat162 *>(dst + i) = __floats2bfloat162_rn(src[i], src[i + 1]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; i += 2)
            *reinterpret_cast<float2 *>(dst + i) = make_float2(src[i], src[i + 1]);
    }
}

template <int C>
__device__ __forceinline__ void load_state_row(const float *__restrict__ src, float (&dst)[C]) {
    if constexpr (C == 4) {
        const float4 f = __ldcs(reinterpret_cast<const float4 *>(src));
        dst[0] = f.x; dst[1] = f.y; dst[2] = f.z; dst[3] = f.w;
    } else {
        static_assert(C == 2, "two or four columns per lane");
        const float2 f = __ldcs(reinterpret_cast<const float2 *>(src));
        dst[0] = f.x; dst[1] = f.y;
    }
}

template <int C>
__device__ __forceinline__ void store_state_row(float *__restrict__ dst, const float (&src)[C]) {
    if constexpr (C == 4) {
        __stcs(reinterpret_cast<float4 *>(dst), make_float4(src[0], src[1], src[2], src[3]));
    } else {
        __stcs(reinterpret_cast<float2 *>(dst), make_float2(src[0], src[1]));
    }
}

template <int DK, int DV, typename TIn, bool CW>
__global__ void __launch_bounds__(kThreads, 2) recurrent_kernel(RecurrentParams p) {
    constexpr int R = DK / kWarps;   // state rows per warp
    constexpr int C = DV / 32;       // state columns per lane
    static_assert(R * kWarps == DK && C * 32 == DV, "unsupported head dims");

    // Cross-warp partial sums, double-buffered by token parity so one barrier
    // per token suffices.
    __shared__ float red_k[2][kWarps][DV];
    __shared__ float red_q[2][kWarps][DV];
    __shared__ float red_kq[2][kWarps];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t pair = blockIdx.x;            // b * Hv + hv
    const int64_t b = pair / p.Hv;
    const int hv = static_cast<int>(pair % p.Hv);
    const int hk = hv / p.group;
    const int row0 = warp * R;
    const int col0 = lane * C;

    float S[R][C];
    const size_t state_off = static_cast<size_t>(pair) * DK * DV;
    if (p.S_in) {
        const float *src = p.S_in + state_off;
#pragma unroll
        for (int r = 0; r < R; ++r)
            load_state_row<C>(src + static_cast<size_t>(row0 + r) * DV + col0, S[r]);
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) S[r][c] = 0.f;
    }

    const TIn *q = static_cast<const TIn *>(p.q);
    const TIn *k = static_cast<const TIn *>(p.k);
    const TIn *v = static_cast<const TIn *>(p.v);
    TIn *y = static_cast<TIn *>(p.y);

    for (int64_t t = 0; t < p.T; ++t) {
        const int64_t tok = b * p.T + t;
        const int buf = static_cast<int>(t & 1);
        float kr[R], qr[R], vr[C];
        load_row<TIn, R>(k + (tok * p.Hqk + hk) * DK + row0, kr);
        load_row<TIn, R>(q + (tok * p.Hqk + hk) * DK + row0, qr);
        load_row<TIn, C>(v + (tok * p.Hv + hv) * DV + col0, vr);
        const float bt = __ldg(p.beta + tok * p.Hv + hv);
        // a: the scalar gate; ar: the gate of each of this warp's rows (CW)
        float a = 1.f, ar[R];
        if constexpr (CW) {
            load_row<float, R>(p.alpha + (tok * p.Hv + hv) * DK + row0, ar);
        } else {
            a = __ldg(p.alpha + tok * p.Hv + hv);
        }

        float pk[C], pq[C];
#pragma unroll
        for (int c = 0; c < C; ++c) { pk[c] = 0.f; pq[c] = 0.f; }
        float kq = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            kq = fmaf(kr[r], qr[r], kq);
            const float ka = CW ? ar[r] * kr[r] : kr[r], qa = CW ? ar[r] * qr[r] : qr[r];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                pk[c] = fmaf(S[r][c], ka, pk[c]);
                pq[c] = fmaf(S[r][c], qa, pq[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < C; ++c) {
            red_k[buf][warp][col0 + c] = pk[c];
            red_q[buf][warp][col0 + c] = pq[c];
        }
        if (lane == 0) red_kq[buf][warp] = kq;
        __syncthreads();

        float rk[C], rq[C];
#pragma unroll
        for (int c = 0; c < C; ++c) { rk[c] = 0.f; rq[c] = 0.f; }
        float kq_all = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            kq_all += red_kq[buf][w];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                rk[c] += red_k[buf][w][col0 + c];
                rq[c] += red_q[buf][w][col0 + c];
            }
        }

        float e[C], yv[C];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            e[c] = vr[c] - a * rk[c];
            yv[c] = a * rq[c] + bt * kq_all * e[c];
        }
        if (warp == 0) store_row<TIn, C>(y + (tok * p.Hv + hv) * DV + col0, yv);

#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float w = bt * kr[r];
            const float ad = CW ? ar[r] : a;
#pragma unroll
            for (int c = 0; c < C; ++c) S[r][c] = fmaf(ad, S[r][c], w * e[c]);
        }
    }

    if (p.S_out) {
        float *dst = p.S_out + state_off;
#pragma unroll
        for (int r = 0; r < R; ++r)
            store_state_row<C>(dst + static_cast<size_t>(row0 + r) * DV + col0, S[r]);
    }
}

template <int DK, int DV>
cudaError_t launch_dims(const RecurrentParams &p, gdn_dtype dtype, cudaStream_t stream) {
    const int64_t pairs = p.B * p.Hv;
    if (pairs == 0) return cudaSuccess;
    if (pairs > 0x7fffffffLL) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(pairs));
    if (p.alpha_cw) {
        if (dtype == GDN_BF16)
            recurrent_kernel<DK, DV, __nv_bfloat16, true><<<grid, kThreads, 0, stream>>>(p);
        else
            recurrent_kernel<DK, DV, float, true><<<grid, kThreads, 0, stream>>>(p);
    } else {
        if (dtype == GDN_BF16)
            recurrent_kernel<DK, DV, __nv_bfloat16, false><<<grid, kThreads, 0, stream>>>(p);
        else
            recurrent_kernel<DK, DV, float, false><<<grid, kThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentParams &p, int dk, int dv, gdn_dtype dtype, cudaStream_t stream) {
    if (dk == 128 && dv == 128) return launch_dims<128, 128>(p, dtype, stream);
    if (dk == 64 && dv == 64) return launch_dims<64, 64>(p, dtype, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
