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
#include <mutex>

#include "gdn_internal.h"
#include "gdn_layer.h"

namespace gdn {
namespace {

constexpr int kTile = 64;          // tokens per prologue warp
constexpr int kMaxConv = 4;
constexpr float kL2Eps = 1e-6f;

// sigma(u) with the fast exponential and the approximate (MUFU) division:
// about 2 ulp, far below the bf16 rounding of the outputs; the kernels are
// otherwise limited by these per-element instructions, not by HBM.
__device__ __forceinline__ float sigmoidf_(float u) { return __fdividef(1.f, 1.f + __expf(-u)); }

// The PTX approximate instructions with denormals flushed to zero (no
// denormal fix-up code around them): 2^x, 1/x and 1/sqrt(x).
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rsqrt_ftz(float x) {
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// sigma(u) = 1 / (1 + 2^(-u log2 e)) from those instructions: for very
// negative u the power overflows to +inf and sigma is 0; for very positive u
// it flushes to 0 and sigma is 1.
__device__ __forceinline__ float sigmoid_ftz(float u) {
    constexpr float kLog2e = 1.4426950408889634f;
    return rcp_ftz(1.f + ex2_ftz(-kLog2e * u));
}

// log(1 + e^u), stable for either sign of u.
__device__ __forceinline__ float softplusf_(float u) { return fmaxf(u, 0.f) + log1pf(__expf(-fabsf(u))); }

// Eight bf16 channels (one 16-byte word) -> floats.
__device__ __forceinline__ void unpack8(const uint4 &r, float (&f)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}

// Eight floats -> bf16 (round to nearest even), one 16-byte word.
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

struct ProloguePlan {
    int64_t B, T;
    int Hqk, Hv, d, kconv, ntiles;
    int gq, gv, ngroups;   // head groups of q (and of k), of v, and their sum
    int64_t items;         // B * ntiles * ngroups
    gdn_prologue_io io;
};

constexpr int kWarps = 8;   // prologue warps per CTA
constexpr int kRing = 24;   // input rows in flight per lane (a multiple of 4)
constexpr size_t kPrologueSmem = static_cast<size_t>(kWarps) * kRing * 32 * sizeof(uint4);

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One token of the prologue for this lane's eight channels: the new input row
// goes into ring slot S (token mod 4); the convolution reads the three
// previous rows from the other slots; then SiLU, the L2 norm over the head
// (a sum over the LPR lanes of the head) when NORM, and the bf16 store.
template <int LPR, int S, bool NORM>
__device__ __forceinline__ void prologue_token(float (&ring)[4][8], const float (&tap)[kMaxConv][8], const uint4 &raw,
                                               bool store, __nv_bfloat16 *dst) {
    float cur[8], u[8];
    unpack8(raw, cur);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float a = tap[0][e] * cur[e];
        a = fmaf(tap[1][e], ring[(S + 3) & 3][e], a);
        a = fmaf(tap[2][e], ring[(S + 2) & 3][e], a);
        a = fmaf(tap[3][e], ring[(S + 1) & 3][e], a);
        ring[S][e] = cur[e];
        u[e] = a * sigmoid_ftz(a);
        if constexpr (NORM) ss = fmaf(u[e], u[e], ss);
    }
    if constexpr (NORM) {
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = rsqrt_ftz(ss + kL2Eps);
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] *= inv;
    }
    if (store) *reinterpret_cast<uint4 *>(dst) = pack8(u);
}

// The first kRing - 4 input rows of a tile for one lane, in commit groups of
// four rows (rows past n are not copied), issued before the item's other
// loads so that their latency overlaps them.
__device__ __forceinline__ void prologue_start(uint4 *lane_ring, const __nv_bfloat16 *xp, int rs, int n) {
#pragma unroll
    for (int g0 = 0; g0 < kRing - 4; g0 += 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (g0 + i < n) cp_async16(lane_ring + (g0 + i) * 32, xp + static_cast<int64_t>(g0 + i) * rs);
        cp_async_commit();
    }
}

// The rows of one tile for one lane, four tokens per step.  The lane streams
// its own 16 bytes of every input row through a private ring of kRing rows
// in shared memory (asynchronous copies, one commit group per four rows),
// kRing - 4 rows ahead of the rows it computes.  n: tokens this lane loads
// and stores (0 for an idle lane); len: tokens of the tile (the same for the
// whole warp, so the shuffles of the L2 norm see every lane).  FULL: a whole
// tile (len == n == kTile), taken with one check per group of four rows (the
// groups fetched ahead of the tile's end are not copied: they may lie past
// the end of the sequence).
template <int LPR, bool NORM, bool FULL>
__device__ __forceinline__ void prologue_rows(float (&ring)[4][8], const float (&tap)[kMaxConv][8], uint4 *lane_ring,
                                              const __nv_bfloat16 *xp, __nv_bfloat16 *op, int rs, int n, int len) {
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const int64_t rs1 = rs;
    // rows 0 .. kRing-5 were issued by prologue_start
    const __nv_bfloat16 *src = xp + (kRing - 4) * rs1;   // next row to copy
    int wslot = kRing - 4;                               // its ring slot (a multiple of 4)
    auto issue = [&](int i0) {       // rows i0 .. i0+3 of the tile, one commit group
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (FULL ? i0 < kTile : i0 + i < n) cp_async16(lane_ring + (wslot + i) * 32, src + i * rs1);
        cp_async_commit();
        src += 4 * rs1;
        wslot = wslot + 4 == kRing ? 0 : wslot + 4;
    };
    int rslot = 0;                   // ring slot of the rows computed next
    __nv_bfloat16 *o = op;
#pragma unroll 1
    for (int i0 = 0; i0 < (FULL ? kTile : len); i0 += 4) {
        issue(i0 + kRing - 4);
        cp_async_wait<kRing / 4 - 1>();   // rows i0 .. i0+3 have landed
        uint4 cur[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cur[i] = (FULL || i0 + i < n) ? lane_ring[(rslot + i) * 32] : zero;
        prologue_token<LPR, 0, NORM>(ring, tap, cur[0], FULL || i0 < n, o);
        prologue_token<LPR, 1, NORM>(ring, tap, cur[1], FULL || i0 + 1 < n, o + rs1);
        prologue_token<LPR, 2, NORM>(ring, tap, cur[2], FULL || i0 + 2 < n, o + 2 * rs1);
        prologue_token<LPR, 3, NORM>(ring, tap, cur[3], FULL || i0 + 3 < n, o + 3 * rs1);
        o += 4 * rs1;
        rslot = rslot + 4 == kRing ? 0 : rslot + 4;
    }
    cp_async_wait<0>();
}

// One warp per item: a tile of kTile tokens of one group of adjacent heads of
// one of q, k, v.  LPR = d/8 lanes cover a head (8 channels and one 16-byte
// load per lane per token), so a warp covers 32/LPR heads, which lie next to
// each other in memory: every token row of the group is one contiguous
// 512-byte access.  The convolution window lives in registers as a ring of
// four token rows indexed by token mod 4, so the taps never move data; the
// next four input rows are loaded while the current four are computed.
// Items are handed out in memory order (heads, then tiles, then batches) by
// a grid-stride loop over a grid of two CTAs per SM.
template <int LPR>
__global__ void __launch_bounds__(kWarps * 32, 2) prologue_kernel(ProloguePlan p) {
    constexpr int HPW = 32 / LPR;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;           // head within the group
    const int c0 = (lane % LPR) * 8;      // first channel of this lane within its head
    const int d = p.d, K = p.kconv;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    extern __shared__ uint4 prologue_ring[];
    // this lane's ring: row slot r at lane_ring[r * 32]
    uint4 *lane_ring = prologue_ring + (threadIdx.x >> 5) * kRing * 32 + lane;

#pragma unroll 1
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); item < p.items;
         item += nwarps) {
        const int grp = static_cast<int>(item % p.ngroups);
        const int64_t rest = item / p.ngroups;
        const int tile = static_cast<int>(rest % p.ntiles);
        const int64_t b = rest / p.ntiles;
        const int which = grp < p.gq ? 0 : (grp < 2 * p.gq ? 1 : 2);   // q, k, v
        const int g = which == 0 ? grp : (which == 1 ? grp - p.gq : grp - 2 * p.gq);
        const int H = which == 2 ? p.Hv : p.Hqk;
        const int h = g * HPW + sub;
        const bool on = h < H;   // lanes past the last head of a partial group stay idle
        const __nv_bfloat16 *x =
            static_cast<const __nv_bfloat16 *>(which == 0 ? p.io.xq : which == 1 ? p.io.xk : p.io.xv);
        const float *w = which == 0 ? p.io.wq : which == 1 ? p.io.wk : p.io.wv;
        const __nv_bfloat16 *sin = static_cast<const __nv_bfloat16 *>(
            which == 0 ? p.io.state_q_in : which == 1 ? p.io.state_k_in : p.io.state_v_in);
        __nv_bfloat16 *sout = static_cast<__nv_bfloat16 *>(
            which == 0 ? p.io.state_q_out : which == 1 ? p.io.state_k_out : p.io.state_v_out);
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(which == 0 ? p.io.q : which == 1 ? p.io.k : p.io.v);
        const int64_t rowstride = static_cast<int64_t>(H) * d;          // elements between tokens
        const int64_t col = static_cast<int64_t>(h) * d + c0;            // this lane's channels in a row
        const int64_t ta = static_cast<int64_t>(tile) * kTile;
        const int64_t tb = ta + kTile < p.T ? ta + kTile : p.T;
        const __nv_bfloat16 *xb = x + b * p.T * rowstride + col;
        __nv_bfloat16 *ob = out + b * p.T * rowstride + col;

        // Input row of token t (t may lie before the sequence: the convolution
        // state, else zeros).
        auto row_at = [&](int64_t t) -> uint4 {
            if (!on) return zero;
            if (t >= 0) return __ldg(reinterpret_cast<const uint4 *>(xb + t * rowstride));
            if (sin && t >= -(K - 1))
                return *reinterpret_cast<const uint4 *>(sin + (b * (K - 1) + (K - 1 + t)) * rowstride + col);
            return zero;
        };

        // Start streaming the tile's rows.  n: tokens of the tile this lane
        // loads and stores (0 for an idle lane).
        const int len = static_cast<int>(tb - ta);
        const int n = on ? len : 0;
        const int rs = static_cast<int>(rowstride);
        const __nv_bfloat16 *xp = xb + ta * rowstride;
        __nv_bfloat16 *op = ob + ta * rowstride;
        prologue_start(lane_ring, xp, rs, n);

        if (which == 2) {
            // decay and write gates of this group's value heads over the tile
            const float *A = p.io.A, *ba = p.io.b_alpha;
            for (int idx = lane; idx < len * HPW; idx += 32) {
                const int64_t t = ta + idx / HPW;
                const int hh = g * HPW + idx % HPW;
                if (hh < p.Hv) {
                    const int64_t gi = (b * p.T + t) * p.Hv + hh;
                    p.io.alpha[gi] = __expf(-__expf(A[hh]) * softplusf_(__ldg(p.io.a_raw + gi) + ba[hh]));
                    p.io.beta[gi] = sigmoidf_(__ldg(p.io.b_raw + gi));
                }
            }
        }

        // tap[j][e]: the weight applied to the input j tokens back (zero beyond K)
        float tap[kMaxConv][8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
            for (int j = 0; j < kMaxConv; ++j)
                tap[j][e] = (on && j < K) ? __ldg(w + (col + e) * K + (K - 1 - j)) : 0.f;

        // ring[s]: the input row of the token t with (t - ta) mod 4 == s
        float ring[4][8];
        {
            float f[8];
#pragma unroll
            for (int j = 1; j < kMaxConv; ++j) {   // tokens ta-3 .. ta-1 -> slots 1 .. 3
                const uint4 r = j >= kMaxConv - (K - 1) ? row_at(ta - kMaxConv + j) : zero;
                unpack8(r, f);
#pragma unroll
                for (int e = 0; e < 8; ++e) ring[j][e] = f[e];
            }
        }

        if (n == kTile) {
            if (which < 2)
                prologue_rows<LPR, true, true>(ring, tap, lane_ring, xp, op, rs, n, len);
            else
                prologue_rows<LPR, false, true>(ring, tap, lane_ring, xp, op, rs, n, len);
        } else {
            if (which < 2)
                prologue_rows<LPR, true, false>(ring, tap, lane_ring, xp, op, rs, n, len);
            else
                prologue_rows<LPR, false, false>(ring, tap, lane_ring, xp, op, rs, n, len);
        }

        if (sout && tb >= p.T && on) {
            // the last K-1 inputs of the sequence, oldest first
            for (int j = 0; j < K - 1; ++j)
                *reinterpret_cast<uint4 *>(sout + (b * (K - 1) + j) * rowstride + col) = row_at(p.T - (K - 1) + j);
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
constexpr int kEpiRows = 4;   // row sets in flight per warp

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
    for (int64_t s0 = w0; s0 < nsets; s0 += kEpiRows * warps) {
        uint4 yr[kEpiRows], zr[kEpiRows];
        int64_t r[kEpiRows];
#pragma unroll
        for (int j = 0; j < kEpiRows; ++j) {
            r[j] = (s0 + j * warps) * RPW + sub;
            if (r[j] < p.rows) {
                yr[j] = *reinterpret_cast<const uint4 *>(p.y + r[j] * p.d + cl * 8);
                zr[j] = *reinterpret_cast<const uint4 *>(p.z + r[j] * p.d + cl * 8);
            } else {
                yr[j] = zr[j] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < kEpiRows; ++j) {
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
            const float inv = rsqrt_ftz(ss * inv_d + p.eps);
            uint4 orow;
            uint32_t *ow = reinterpret_cast<uint32_t *>(&orow);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 v = __floats2bfloat162_rn(sigmoid_ftz(z[2 * e]) * y[2 * e] * inv * g[2 * e],
                                                               sigmoid_ftz(z[2 * e + 1]) * y[2 * e + 1] * inv * g[2 * e + 1]);
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

// The current device's SM count, after checking that it is an sm_103 part.
gdn_status num_sms(int *sms) {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_CUDA;
    }
    return (major == 10 && minor == 3) ? GDN_OK : GDN_ERR_UNSUPPORTED;
}

gdn_status device_ok() {
    int sms = 0;
    return num_sms(&sms);
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
    const int hpw = 32 / (s.d / 8);
    p.gq = (s.Hqk + hpw - 1) / hpw;
    p.gv = (s.Hv + hpw - 1) / hpw;
    p.ngroups = 2 * p.gq + p.gv;
    p.items = s.B * p.ntiles * p.ngroups;
    p.io = a;
    int sms = 0;
    if (num_sms(&sms) != GDN_OK) return GDN_ERR_CUDA;
    const int64_t want = (p.items + kWarps - 1) / kWarps;
    const unsigned grid = static_cast<unsigned>(want < int64_t{sms} * 2 ? want : int64_t{sms} * 2);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(prologue_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kPrologueSmem));
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(prologue_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(kPrologueSmem));
    });
    if (attr_err != cudaSuccess) return GDN_ERR_CUDA;
    if (s.d == 128)
        prologue_kernel<16><<<grid, kWarps * 32, kPrologueSmem, cs>>>(p);
    else
        prologue_kernel<8><<<grid, kWarps * 32, kPrologueSmem, cs>>>(p);
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
    // 8 resident CTAs of 8 warps per SM; each warp covers kEpiRows * 256 / d rows per iteration
    const int64_t rows_per_cta = 8 * kEpiRows * (256 / s.d);
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
