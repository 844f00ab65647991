// GDN layer steps on either side of the recurrence (gdn_layer.h): the fused
// prologue (short causal depthwise convolution, SiLU, L2Norm of q and k, the
// decay and write gates) and the fused epilogue (sigmoid output gate times a
// zero-centred RMSNorm), following the Qwen3.8-Next reading notes, section 2.1
// "Gated DeltaNet" ("Feature parameterization", "Gating dynamics").
//
// Both are single HBM passes, one warp per row of d channels (a (token, head)
// row is 128 or 256 contiguous bytes of bf16, so a warp's loads and stores are
// fully coalesced), fp32 arithmetic, bf16 outputs rounded to nearest even.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn_internal.h"
#include "gdn_layer.h"

namespace gdn {
namespace {

constexpr int kTile = 64;          // tokens per prologue warp
constexpr int kMaxConv = 4;
constexpr float kL2Eps = 1e-6f;

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// sigma(u) with the fast exponential and the approximate (MUFU) division:
// about 2 ulp, far below the bf16 rounding of the outputs; the kernels are
// otherwise limited by these per-element instructions, not by HBM.
__device__ __forceinline__ float sigmoidf_(float u) { return __fdividef(1.f, 1.f + __expf(-u)); }

// log(1 + e^u), stable for either sign of u.
__device__ __forceinline__ float softplusf_(float u) { return fmaxf(u, 0.f) + log1pf(__expf(-fabsf(u))); }

// CPL consecutive bf16 channels <-> floats (CPL = 2: one 32-bit word; 4: two).
template <int CPL>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16 *p, float (&f)[CPL]) {
    // read-only path (the inputs never alias the outputs), so loads may be
    // issued ahead of earlier stores
    if constexpr (CPL == 4) {
        const uint2 r = __ldg(reinterpret_cast<const uint2 *>(p));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
        const unsigned int r = __ldg(reinterpret_cast<const unsigned int *>(p));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r));
        f[0] = a.x; f[1] = a.y;
    }
}

template <int CPL>
struct RawOf {
    using type = uint32_t;
};
template <>
struct RawOf<4> {
    using type = uint2;
};

// CPL bf16 channels from shared memory.
template <int CPL>
__device__ __forceinline__ void load_smem(const __nv_bfloat16 *p, float (&f)[CPL]) {
    const typename RawOf<CPL>::type r = *reinterpret_cast<const typename RawOf<CPL>::type *>(p);
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
    for (int e = 0; e < CPL / 2; ++e) {
        const float2 a = __bfloat1622float2(h2[e]);
        f[2 * e] = a.x;
        f[2 * e + 1] = a.y;
    }
}

template <int CPL>
__device__ __forceinline__ void store_bf16(__nv_bfloat16 *p, const float (&f)[CPL]) {
    if constexpr (CPL == 4) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]), b = __floats2bfloat162_rn(f[2], f[3]);
        uint2 r;
        r.x = *reinterpret_cast<const uint32_t *>(&a);
        r.y = *reinterpret_cast<const uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = r;
    } else {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(f[0], f[1]);
    }
}

struct ProloguePlan {
    int64_t B, T;
    int Hqk, Hv, d, kconv, ntiles;
    gdn_prologue_io io;
};

// One CTA (4 warps): one (batch, head) row of one of q, k, v over a tile of
// kTile tokens.  The tile's input rows, with kMaxConv-1 rows of history in
// front, are first copied into shared memory with asynchronous 16-byte copies
// (all in flight at once: the kernel is HBM-bound, not latency-bound); then
// each warp computes kTile/4 tokens from shared memory, one row per step, and
// stores its rows straight to global memory.  CTAs are ordered by memory
// (consecutive CTAs take consecutive heads of one tile).
constexpr int kHalo = kMaxConv - 1;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <int CPL>
__global__ void __launch_bounds__(128) prologue_kernel(ProloguePlan p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __nv_bfloat16 *rows = reinterpret_cast<__nv_bfloat16 *>(smem_raw);   // [kHalo + kTile][d]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t job = blockIdx.x;
    const int nrows = 2 * p.Hqk + p.Hv;
    const int row = static_cast<int>(job % nrows);
    const int tile = static_cast<int>((job / nrows) % p.ntiles);
    const int64_t b = job / (static_cast<int64_t>(p.ntiles) * nrows);
    const int which = row < p.Hqk ? 0 : (row < 2 * p.Hqk ? 1 : 2);   // q, k, v
    const int h = which == 0 ? row : (which == 1 ? row - p.Hqk : row - 2 * p.Hqk);
    const int H = which == 2 ? p.Hv : p.Hqk;
    const int d = p.d, K = p.kconv;
    const int64_t C = static_cast<int64_t>(H) * d;
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(which == 0 ? p.io.xq : which == 1 ? p.io.xk : p.io.xv);
    const float *w = which == 0 ? p.io.wq : which == 1 ? p.io.wk : p.io.wv;
    const __nv_bfloat16 *sin = static_cast<const __nv_bfloat16 *>(
        which == 0 ? p.io.state_q_in : which == 1 ? p.io.state_k_in : p.io.state_v_in);
    __nv_bfloat16 *sout = static_cast<__nv_bfloat16 *>(
        which == 0 ? p.io.state_q_out : which == 1 ? p.io.state_k_out : p.io.state_v_out);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(which == 0 ? p.io.q : which == 1 ? p.io.k : p.io.v);
    const int64_t t0 = static_cast<int64_t>(tile) * kTile;
    const int64_t t1 = t0 + kTile < p.T ? t0 + kTile : p.T;
    const int nr = static_cast<int>(t1 - t0) + kHalo;   // rows in shared memory: tokens t0-kHalo .. t1-1

    // Stage the rows: 16-byte pieces, d/8 per row.
    const int per_row = d / 8;
    for (int idx = tid; idx < nr * per_row; idx += 128) {
        const int i = idx / per_row, c = idx % per_row;
        const int64_t t = t0 - kHalo + i;
        __nv_bfloat16 *dst = rows + i * d + c * 8;
        const int64_t off = static_cast<int64_t>(h) * d + c * 8;
        if (t >= 0) {
            cp_async16(dst, x + (b * p.T + t) * C + off);
        } else if (sin && t >= -(K - 1)) {
            *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(sin + (b * (K - 1) + (K - 1 + t)) * C + off);
        } else {
            *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    cp_async_wait_all();
    __syncthreads();

    const int64_t ch = static_cast<int64_t>(h) * d + lane * CPL;   // first channel of this lane
    const int cl = lane * CPL;                                      // ... within the head
    // back[e][j]: the tap applied to the input j tokens back (0 = current; 0 beyond K)
    float back[CPL][kMaxConv];
#pragma unroll
    for (int e = 0; e < CPL; ++e)
#pragma unroll
        for (int j = 0; j < kMaxConv; ++j) back[e][j] = (j < K && t1 > t0) ? w[(ch + e) * K + (K - 1 - j)] : 0.f;
    const bool normalise = which < 2;
    constexpr int kPerWarp = kTile / 4;
    const int64_t ta = t0 + warp * kPerWarp;
    const int64_t tb = ta + kPerWarp < t1 ? ta + kPerWarp : t1;
    // win[j][e]: the input j+1 tokens back; one shared-memory row read per token
    float win[kMaxConv - 1][CPL];
    if (ta < tb) {
#pragma unroll
        for (int j = 0; j < kMaxConv - 1; ++j) load_smem<CPL>(rows + (static_cast<int>(ta - t0) + kHalo - 1 - j) * d + cl, win[j]);
    }
#pragma unroll 1
    for (int64_t t = ta; t < tb; ++t) {
        const int i = static_cast<int>(t - t0) + kHalo;
        float u[CPL];
        float acc[CPL], cur[CPL];
        load_smem<CPL>(rows + i * d + cl, cur);
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
            acc[e] = back[e][0] * cur[e];
#pragma unroll
            for (int j = 0; j < kMaxConv - 1; ++j) acc[e] = fmaf(back[e][j + 1], win[j][e], acc[e]);
        }
#pragma unroll
        for (int j = kMaxConv - 2; j > 0; --j)
#pragma unroll
            for (int e = 0; e < CPL; ++e) win[j][e] = win[j - 1][e];
#pragma unroll
        for (int e = 0; e < CPL; ++e) win[0][e] = cur[e];
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
            u[e] = acc[e] * sigmoidf_(acc[e]);
            ss = fmaf(u[e], u[e], ss);
        }
        if (normalise) {
            const float inv = rsqrtf(warp_allsum(ss) + kL2Eps);
#pragma unroll
            for (int e = 0; e < CPL; ++e) u[e] *= inv;
        }
        store_bf16<CPL>(out + ((b * p.T + t) * C + ch), u);
    }
    if (sout && t1 >= p.T && warp == 0) {
        // the last K-1 inputs of the sequence, oldest first
        for (int j = 0; j < K - 1; ++j) {
            const int i = nr - (K - 1) + j;
            *reinterpret_cast<typename RawOf<CPL>::type *>(sout + (b * (K - 1) + j) * C + ch) =
                *reinterpret_cast<const typename RawOf<CPL>::type *>(rows + i * d + cl);
        }
    }
    if (which == 2 && t1 > t0 && tid < kTile) {
        // decay and write gates of this value head over the tile
        const int64_t t = t0 + tid;
        if (t < t1) {
            const float eA = __expf(p.io.A[h]), ba = p.io.b_alpha[h];
            const int64_t gi = (b * p.T + t) * p.Hv + h;
            p.io.alpha[gi] = __expf(-eA * softplusf_(__ldg(p.io.a_raw + gi) + ba));
            p.io.beta[gi] = sigmoidf_(__ldg(p.io.b_raw + gi));
        }
    }
}

struct EpiloguePlan {
    int64_t rows;          // B * T * Hv
    int d;
    float eps;
    const __nv_bfloat16 *y, *z;
    const float *w;
    __nv_bfloat16 *o;
};

// 16-byte accesses: a lane handles 8 channels, a row of d channels takes
// d/8 lanes (16 for d = 128, 8 for d = 64), so a warp covers 32*8/d rows per
// access; two such row sets are in flight per iteration; grid-stride.
template <int LPR>   // lanes per row
__global__ void __launch_bounds__(256) epilogue_kernel(EpiloguePlan p) {
    constexpr int RPW = 32 / LPR;   // rows per warp access
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, cl = lane % LPR;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t w0 = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    float g[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) g[e] = 1.f + p.w[cl * 8 + e];
    const float inv_d = 1.f / static_cast<float>(p.d);
    const int64_t nsets = (p.rows + RPW - 1) / RPW;
#pragma unroll 1
    for (int64_t s0 = w0; s0 < nsets; s0 += 2 * warps) {
        uint4 yr[2], zr[2];
        int64_t r[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            r[j] = (s0 + j * warps) * RPW + sub;
            if (r[j] < p.rows) {
                yr[j] = *reinterpret_cast<const uint4 *>(p.y + r[j] * p.d + cl * 8);
                zr[j] = *reinterpret_cast<const uint4 *>(p.z + r[j] * p.d + cl * 8);
            } else {
                yr[j] = zr[j] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __nv_bfloat162 *yh = reinterpret_cast<const __nv_bfloat162 *>(&yr[j]);
            const __nv_bfloat162 *zh = reinterpret_cast<const __nv_bfloat162 *>(&zr[j]);
            float y[8], z[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a = __bfloat1622float2(yh[e]), c = __bfloat1622float2(zh[e]);
                y[2 * e] = a.x; y[2 * e + 1] = a.y; z[2 * e] = c.x; z[2 * e + 1] = c.y;
            }
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
            for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = rsqrtf(ss * inv_d + p.eps);
            uint4 orow;
            uint32_t *ow = reinterpret_cast<uint32_t *>(&orow);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 v = __floats2bfloat162_rn(sigmoidf_(z[2 * e]) * y[2 * e] * inv * g[2 * e],
                                                               sigmoidf_(z[2 * e + 1]) * y[2 * e + 1] * inv * g[2 * e + 1]);
                ow[e] = *reinterpret_cast<const uint32_t *>(&v);
            }
            if (r[j] < p.rows) *reinterpret_cast<uint4 *>(p.o + r[j] * p.d + cl * 8) = orow;
        }
    }
}

bool aligned(const void *q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; }

struct Span {
    const void *p;
    int64_t n;
};

bool overlap(Span a, Span b) {
    if (!a.p || !b.p || a.n <= 0 || b.n <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + static_cast<uintptr_t>(b.n) && b0 < a0 + static_cast<uintptr_t>(a.n);
}

gdn_status check_layer_shape(const gdn_layer_shape *s) {
    if (!s || s->B < 0 || s->T < 0 || s->Hqk <= 0 || s->Hv <= 0 || s->Hv % s->Hqk != 0) return GDN_ERR_INVALID_ARG;
    if (s->kconv < 1 || s->kconv > kMaxConv) return GDN_ERR_INVALID_ARG;
    if (s->d != 64 && s->d != 128) return GDN_ERR_UNSUPPORTED;
    // element counts must stay far from int64 overflow
    if (s->B > (int64_t{1} << 24) || s->T > (int64_t{1} << 34) || s->Hv > 4096) return GDN_ERR_INVALID_ARG;
    if (s->B * s->T > (int64_t{1} << 36)) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

gdn_status device_ok() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    return (major == 10 && minor == 3) ? GDN_OK : GDN_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_layer_prologue(const gdn_layer_shape *shape, const gdn_prologue_io *io, void *stream) {
    const gdn_status st = check_layer_shape(shape);
    if (st != GDN_OK) return st;
    if (!io) return GDN_ERR_INVALID_ARG;
    const gdn_layer_shape s = *shape;
    const gdn_prologue_io &a = *io;
    // With no tokens only the convolution states are touched; the token
    // tensors may then be empty (NULL).
    if (s.B > 0 && s.T > 0 &&
        (!a.xq || !a.xk || !a.xv || !a.wq || !a.wk || !a.wv || !a.a_raw || !a.b_raw || !a.A || !a.b_alpha || !a.q ||
         !a.k || !a.v || !a.alpha || !a.beta))
        return GDN_ERR_INVALID_ARG;
    const void *bf[] = {a.xq, a.xk, a.xv, a.q, a.k, a.v, a.state_q_in, a.state_k_in, a.state_v_in,
                        a.state_q_out, a.state_k_out, a.state_v_out};
    for (const void *ptr : bf)
        if (!aligned(ptr, 16)) return GDN_ERR_ALIGNMENT;
    const void *fp[] = {a.wq, a.wk, a.wv, a.a_raw, a.b_raw, a.A, a.b_alpha, a.alpha, a.beta};
    for (const void *ptr : fp)
        if (!aligned(ptr, 4)) return GDN_ERR_ALIGNMENT;

    const int64_t nq = s.B * s.T * s.Hqk * s.d * 2, nv = s.B * s.T * s.Hv * s.d * 2, ng = s.B * s.T * s.Hv * 4;
    const int64_t sq = s.B * (s.kconv - 1) * s.Hqk * s.d * 2, sv = s.B * (s.kconv - 1) * s.Hv * s.d * 2;
    const Span ins[] = {{a.xq, nq}, {a.xk, nq}, {a.xv, nv}, {a.wq, int64_t{s.Hqk} * s.d * s.kconv * 4},
                        {a.wk, int64_t{s.Hqk} * s.d * s.kconv * 4}, {a.wv, int64_t{s.Hv} * s.d * s.kconv * 4},
                        {a.state_q_in, sq}, {a.state_k_in, sq}, {a.state_v_in, sv}, {a.a_raw, ng}, {a.b_raw, ng},
                        {a.A, s.Hv * 4}, {a.b_alpha, s.Hv * 4}};
    const Span outs[] = {{a.q, nq}, {a.k, nq}, {a.v, nv}, {a.alpha, ng}, {a.beta, ng},
                         {a.state_q_out, sq}, {a.state_k_out, sq}, {a.state_v_out, sv}};
    for (const Span &o : outs) {
        for (const Span &i : ins)
            if (overlap(o, i)) return GDN_ERR_ALIASING;
        for (const Span &o2 : outs)
            if (&o2 != &o && overlap(o, o2)) return GDN_ERR_ALIASING;
    }
    const gdn_status dev = device_ok();
    if (dev != GDN_OK) return dev;
    if (s.B == 0) return GDN_OK;

    ProloguePlan p;
    p.B = s.B;
    p.T = s.T;
    p.Hqk = s.Hqk;
    p.Hv = s.Hv;
    p.d = s.d;
    p.kconv = s.kconv;
    p.ntiles = static_cast<int>(s.T == 0 ? 1 : (s.T + kTile - 1) / kTile);
    p.io = a;
    const int64_t ctas = s.B * (2 * s.Hqk + s.Hv) * p.ntiles;
    if (ctas > 0x7fffffff) return GDN_ERR_INVALID_ARG;
    const dim3 grid(static_cast<unsigned>(ctas));
    const size_t smem = static_cast<size_t>(kHalo + kTile) * s.d * 2;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (s.d == 128)
        prologue_kernel<4><<<grid, 128, smem, cs>>>(p);
    else
        prologue_kernel<2><<<grid, 128, smem, cs>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_layer_epilogue(const gdn_layer_shape *shape, const void *y, const void *z,
                                         const float *norm_w, float eps, void *o, void *stream) {
    const gdn_status st = check_layer_shape(shape);
    if (st != GDN_OK) return st;
    if (!(eps > 0.f)) return GDN_ERR_INVALID_ARG;
    if (shape->B * shape->T == 0) return GDN_OK;
    if (!y || !z || !norm_w || !o) return GDN_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(z, 16) || !aligned(o, 16) || !aligned(norm_w, 4)) return GDN_ERR_ALIGNMENT;
    const gdn_layer_shape s = *shape;
    const int64_t n = s.B * s.T * s.Hv * s.d * 2;
    if (overlap({o, n}, {y, n}) || overlap({o, n}, {z, n}) || overlap({o, n}, {norm_w, s.d * 4}))
        return GDN_ERR_ALIASING;
    const gdn_status dev = device_ok();
    if (dev != GDN_OK) return dev;
    EpiloguePlan p;
    p.rows = s.B * s.T * s.Hv;
    if (p.rows == 0) return GDN_OK;
    p.d = s.d;
    p.eps = eps;
    p.y = static_cast<const __nv_bfloat16 *>(y);
    p.z = static_cast<const __nv_bfloat16 *>(z);
    p.w = norm_w;
    p.o = static_cast<__nv_bfloat16 *>(o);
    int dev_id = 0, sms = 148;
    cudaGetDevice(&dev_id);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev_id);
    // 8 resident CTAs of 8 warps per SM; each warp covers 2 * 256 / d rows per iteration
    const int64_t rows_per_cta = 8 * 2 * (256 / s.d);
    const int64_t want = (p.rows + rows_per_cta - 1) / rows_per_cta;
    const unsigned grid = static_cast<unsigned>(want < int64_t{sms} * 8 ? want : int64_t{sms} * 8);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (s.d == 128)
        epilogue_kernel<16><<<grid, 256, 0, cs>>>(p);
    else
        epilogue_kernel<8><<<grid, 256, 0, cs>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
