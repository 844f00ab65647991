// Chunked backward of the gated delta recurrence (bf16 inputs, d = 128) on
// the tensor cores: the gradients of L = <dy, y> + <dS_T, S_T> with respect to
// q, k, v, log alpha, beta and S0.
//
// Algebra (the recurrence of the Qwen3.8-Next reading notes, section 2.1,
// "Gated DeltaNet", unrolled over a chunk of 64 tokens in the WY/UT form).
// With S the state entering a chunk, its forward is
//     U = U~ + (-W) S,  Y = Qp S + P U,  S' = diag(gamma_C) S + Kl^T U
// (Qp = diag(gamma) Q, Kl = diag(lambda) K, P = M (.) Q K^T), so the gradient
// of the entering state follows from that of the leaving one by
//     dU = P^T dY + Kl dS',   dS = gamma_C dS' + Qp^T dY + (-W)^T dU,
// a reverse scan over chunks with two d-sized products per chunk, the same
// shape as the forward's state scan.  Given S and dS' of a chunk, everything
// else is local to the chunk: the gradients of U~, W, P, the gates and the
// lower-triangular inverse T = (I + A)^{-1} (dA = -T^T dT T^T) down to q, k,
// v, beta and log alpha.
//
// Four launches: the chunked pre-pass (per chunk: -W, U~, Qp, Kl, P,
// gamma_C), the forward chain writing the state entering every chunk, the
// reverse chain below writing dS' of every chunk and dS0, and the per-chunk
// gradient kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn_internal.h"
#include "warp_mma.cuh"

namespace gdn {
namespace {

using namespace wm;

constexpr int kC = 64;
constexpr int kD = 128;

struct BwDev {
    int64_t T;
    int B, Hqk, Hv, group, nchunks;
    int seg_chunks, max_warmup;
    float log_eps;
    const __nv_bfloat16 *q, *k, *v, *dy;
    const float *alpha, *beta;
    const float *dS_T;        // nullptr = zero
    const uint8_t *rec;       // chunk records [B * Hv][nchunks][rec::kBytes]
    const float *bound;       // per-chunk decay bounds [B * Hv][nchunks]
    const __nv_bfloat16 *state;   // state entering every chunk [B * Hv][nchunks][d][d] (bf16, the products' operand)
    __nv_bfloat16 *dstate;        // gradient of the state leaving every chunk, same layout
    float *dS0;               // nullptr = not returned
    float *dq, *dk;           // [B, T, Hqk, d] (summed over the value heads of a group)
    float *dv;                // [B, T, Hv, d]
    float *dlog_alpha, *dbeta;   // [B, T, Hv]
    // Exact sequence split of the reverse chain (heads whose segments reach no
    // window): pass 1 runs the transitions (kind 0: from dS = 0 with dY, or
    // from dS_T for the last segment; kind 1: from the identity with dY
    // zero), pass 0 the output pass.  Segment s's maps are stored at index
    // nseg - 1 - s, so that the forward combine chains them from the last
    // segment down: seg_state [pairs][nseg][3][d][d].
    int nseg, pass;
    const int *exact_flag;
    float *seg_state;
};

// Reverse-chain plan: flag[pair][nseg - 1 - s] = 1 when segment s < nseg - 1
// reaches neither a window of later chunks nor the sequence's end within the
// limit.  One thread per (pair, segment).
__global__ void bw_plan_kernel(const BwDev p, int *flag) {
    const int pairs = p.B * p.Hv;
    const int idx = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
    if (idx >= pairs * (p.nseg - 1)) return;
    const int pr = idx % pairs, seg = idx / pairs;   // seg = 0 .. nseg - 2
    const int c_end = (seg + 1) * p.seg_chunks;
    float acc = 0.f;
    int v = 1;
    for (int m = 0; m < p.max_warmup; ++m) {
        const int cc = c_end + m;
        if (cc >= p.nchunks) {
            v = 0;
            break;
        }
        acc += p.bound[static_cast<int64_t>(pr) * p.nchunks + cc];
        if (acc <= p.log_eps) {
            v = 0;
            break;
        }
    }
    flag[static_cast<int64_t>(pr) * p.nseg + (p.nseg - 1 - seg)] = v;
}

__device__ __forceinline__ bool bw_head_split(const int *flag, int pr, int nseg) {
    int any = 0;
    for (int sg = 1; sg < nseg; ++sg) any |= flag[static_cast<int64_t>(pr) * nseg + sg];
    return any != 0;
}

// ------------------------------------------------------------ reverse chain
// Stage: a chunk record, then the chunk's dY tile (swizzled [64][128] bf16).
constexpr uint32_t RC_DY = rec::kBytes;
constexpr uint32_t RC_STAGE = rec::kBytes + 16384;
constexpr uint32_t RC_SB = 2 * RC_STAGE;          // bf16 copy of dS' [dk][dv]
constexpr uint32_t RC_UB = RC_SB + kD * kD * 2;   // bf16 dU [tokens][dv]
constexpr uint32_t RC_MISC = RC_UB + kC * kD * 2;
constexpr uint32_t kRevSmem = RC_MISC + 64;
static_assert(kRevSmem <= 232448, "reverse chain shared memory");

// One (batch, value head, segment): the segment's chunks in reverse order,
// dS in fp32 registers as MMA accumulator fragments (warp w: rows dk = 16w ..
// 16w+15).  A segment other than the last starts from dS = 0 after a window
// of later chunks whose decay bound reaches exp(log_eps) (the reverse map is
// the transpose of the forward one, so the same contraction bound holds);
// without such a window within the limit it starts from dS_T at the last
// chunk (exact).
__global__ void __launch_bounds__(256, 1) bw_reverse_chain_kernel(const BwDev p) {
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int pairs = p.B * p.Hv;
    const unsigned per_pass = static_cast<unsigned>(pairs * p.nseg);
    const int bx = static_cast<int>(blockIdx.x % per_pass);
    const int kind = p.pass == 1 ? static_cast<int>(blockIdx.x / per_pass) : -1;
    const int pr = bx % pairs;
    const int seg = bx / pairs;
    const int b = pr / p.Hv, hv = pr % p.Hv;
    const int c_begin = seg * p.seg_chunks;
    const int c_end = c_begin + p.seg_chunks < p.nchunks ? c_begin + p.seg_chunks : p.nchunks;
    int *misc = reinterpret_cast<int *>(sm + RC_MISC);
    const int sp = p.nseg - 1 - seg;   // where this segment's maps are stored
    const bool split = p.exact_flag != nullptr && bw_head_split(p.exact_flag, pr, p.nseg);
    if (p.pass == 1 && (!split || seg == 0 || (kind == 1 && seg == p.nseg - 1))) return;

    if (tid == 0) {
        int cs = p.nchunks - 1;   // exact start
        if (p.pass == 1 || split) {
            cs = -1 - (c_end - 1);   // the segment's own last chunk (encoded as a windowed start)
            if (c_end == p.nchunks && kind != 1) cs = p.nchunks - 1;   // the last segment from dS_T
        } else if (c_end < p.nchunks) {
            float acc = 0.f;
            for (int m = 0;; ++m) {
                const int cc = c_end + m;
                if (cc >= p.nchunks || m >= p.max_warmup) break;
                acc += p.bound[static_cast<int64_t>(pr) * p.nchunks + cc];
                if (acc <= p.log_eps) {
                    cs = -1 - cc;   // windowed start at chunk cc (encoded negative)
                    break;
                }
            }
        }
        misc[0] = cs;
    }
    __syncthreads();
    const bool exact = misc[0] >= 0;
    const int c_start = exact ? misc[0] : -1 - misc[0];

    float S[16][4];   // dS
    {
        // dS_T for an exact start; the combined gradient for a split head's other segments
        // (output pass); the identity for a kind-1 transition; else zero
        const float *s0 = nullptr;
        if (kind == 1)
            s0 = nullptr;
        else if (exact)
            s0 = p.dS_T ? p.dS_T + static_cast<int64_t>(pr) * kD * kD : nullptr;
        else if (p.pass == 0 && split)
            s0 = p.seg_state + ((static_cast<int64_t>(pr) * p.nseg + sp) * 3 + 2) * kD * kD;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int r = 16 * warp + g, col = 8 * nt + 2 * t4;
            float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
            if (s0) {
                lo = *reinterpret_cast<const float2 *>(s0 + r * kD + col);
                hi = *reinterpret_cast<const float2 *>(s0 + (r + 8) * kD + col);
            } else if (kind == 1) {
                lo = make_float2(r == col ? 1.f : 0.f, r == col + 1 ? 1.f : 0.f);
                hi = make_float2(r + 8 == col ? 1.f : 0.f, r + 8 == col + 1 ? 1.f : 0.f);
            }
            S[nt][0] = lo.x;
            S[nt][1] = lo.y;
            S[nt][2] = hi.x;
            S[nt][3] = hi.y;
        }
    }

    const uint8_t *recs = p.rec + static_cast<int64_t>(pr) * p.nchunks * rec::kBytes;
    auto load_chunk = [&](int cc, int stage) {
        const uint8_t *src = recs + static_cast<int64_t>(cc) * rec::kBytes;
        const uint32_t dst = sb + stage * RC_STAGE;
        for (int e = tid; e < 4 * 1024 + 512 + 32; e += 256) {
            if (e < 4096) {
                const int tile = e >> 10, r = (e >> 4) & 63, pc = e & 15;
                cp_async16(dst + tile * 16384 + sw256(r, pc), src + tile * 16384 + r * 256 + pc * 16);
            } else if (e < 4608) {
                const int e2 = e - 4096, r = e2 >> 3, pc = e2 & 7;
                cp_async16(dst + rec::kP + sw128(r, pc), src + rec::kP + r * 128 + pc * 16);
            } else {
                const int e3 = e - 4608;
                cp_async16(dst + rec::kGc + e3 * 16, src + rec::kGc + e3 * 16);
            }
        }
        for (int e = tid; e < kC * 16; e += 256) {
            const int r = e >> 4, pc = e & 15;
            const int64_t t = static_cast<int64_t>(cc) * kC + r;
            if (t < p.T)
                cp_async16(dst + RC_DY + sw256(r, pc), p.dy + ((static_cast<int64_t>(b) * p.T + t) * p.Hv + hv) * kD + pc * 8);
            else
                *reinterpret_cast<uint4 *>(sm + stage * RC_STAGE + RC_DY + sw256(r, pc)) = make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_commit();
    };

    const int mt = warp & 3, nh = warp >> 2;
    load_chunk(c_start, 0);
#pragma unroll 1
    for (int cc = c_start; cc >= c_begin; --cc) {
        const int st = (c_start - cc) & 1;
        const uint32_t stg = sb + st * RC_STAGE;
        const uint8_t *stp = sm + st * RC_STAGE;
        if (cc < c_end && p.pass == 0) {
            __nv_bfloat16 *so = p.dstate + (static_cast<int64_t>(pr) * p.nchunks + cc) * kD * kD;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const int r = 16 * warp + g, col = 8 * nt + 2 * t4;
                *reinterpret_cast<uint32_t *>(so + r * kD + col) = pack2(S[nt][0], S[nt][1]);
                *reinterpret_cast<uint32_t *>(so + (r + 8) * kD + col) = pack2(S[nt][2], S[nt][3]);
            }
        }
        // A: bf16 copy of dS'
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int r = 16 * warp + g;
            *reinterpret_cast<uint32_t *>(sm + RC_SB + sw256(r, nt) + 4 * t4) = pack2(S[nt][0], S[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + RC_SB + sw256(r + 8, nt) + 4 * t4) = pack2(S[nt][2], S[nt][3]);
        }
        cp_async_wait_all();
        __syncthreads();
        if (cc - 1 >= c_begin) load_chunk(cc - 1, st ^ 1);

        // B: dU = P^T dY + Kl dS'  (warp: tokens 16 mt, columns 64 nh)
        float du[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) du[nt][e] = 0.f;
#pragma unroll 1
        for (int kk = mt; kk < 4 && kind != 1; ++kk) {   // P^T[t][s] is zero for s below the row block
            uint32_t ap[4];
            ldsm_x4_t(ap, stg + rec::kP + sw128(16 * kk + at_row(lane), 2 * mt + at_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t by[4];
                ldsm_x4_t(by, stg + RC_DY + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(du[2 * np], ap, by[0], by[1]);
                mma16816(du[2 * np + 1], ap, by[2], by[3]);
            }
        }
#pragma unroll 2
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t ak[4];
            ldsm_x4(ak, stg + rec::kKl + sw256(16 * mt + a_row(lane), 2 * kk + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bs[4];
                ldsm_x4_t(bs, sb + RC_SB + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(du[2 * np], ak, bs[0], bs[1]);
                mma16816(du[2 * np + 1], ak, bs[2], bs[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int t = 16 * mt + g;
            *reinterpret_cast<uint32_t *>(sm + RC_UB + sw256(t, 8 * nh + nt) + 4 * t4) = pack2(du[nt][0], du[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + RC_UB + sw256(t + 8, 8 * nh + nt) + 4 * t4) = pack2(du[nt][2], du[nt][3]);
        }
        __syncthreads();

        // C: dS = gamma_C dS' + Qp^T dY + (-W)^T dU  (warp: rows dk 16 w)
        {
            const float *gce = reinterpret_cast<const float *>(stp + rec::kGc);
            const float f0 = gce[16 * warp + g], f1 = gce[16 * warp + g + 8];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                S[nt][0] *= f0;
                S[nt][1] *= f0;
                S[nt][2] *= f1;
                S[nt][3] *= f1;
            }
        }
#pragma unroll 1
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t aq[4], aw[4];
            ldsm_x4_t(aq, stg + rec::kQp + sw256(16 * kk + at_row(lane), 2 * warp + at_ch(lane)));
            ldsm_x4_t(aw, stg + rec::kWn + sw256(16 * kk + at_row(lane), 2 * warp + at_ch(lane)));
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t by[4], bu[4];
                ldsm_x4_t(by, stg + RC_DY + sw256(16 * kk + bt_row(lane), 2 * np + bt_ch(lane)));
                ldsm_x4_t(bu, sb + RC_UB + sw256(16 * kk + bt_row(lane), 2 * np + bt_ch(lane)));
                if (kind != 1) {   // dY zero on a kind-1 transition
                    mma16816(S[2 * np], aq, by[0], by[1]);
                    mma16816(S[2 * np + 1], aq, by[2], by[3]);
                }
                mma16816(S[2 * np], aw, bu[0], bu[1]);
                mma16816(S[2 * np + 1], aw, bu[2], bu[3]);
            }
        }
    }

    float *s_end = nullptr;   // where this run's final gradient goes
    if (p.pass == 1)
        s_end = p.seg_state + ((static_cast<int64_t>(pr) * p.nseg + sp) * 3 + kind) * kD * kD;
    else if (c_begin == 0 && p.dS0)
        s_end = p.dS0 + static_cast<int64_t>(pr) * kD * kD;
    if (s_end) {
        float *so = s_end;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int r = 16 * warp + g, col = 8 * nt + 2 * t4;
            *reinterpret_cast<float2 *>(so + r * kD + col) = make_float2(S[nt][0], S[nt][1]);
            *reinterpret_cast<float2 *>(so + (r + 8) * kD + col) = make_float2(S[nt][2], S[nt][3]);
        }
    }
}

// ------------------------------------------------------- per-chunk gradients
// Shared memory (bytes).  bf16 tiles: [64][128] with 256-byte rows, [64][64]
// with 128-byte rows, [128][128] for the two states; all XOR-swizzled.
constexpr uint32_t BG_Q = 0;
constexpr uint32_t BG_K = 16384;
constexpr uint32_t BG_V = 32768;
constexpr uint32_t BG_DY = 49152;
constexpr uint32_t BG_S = 65536;        // S entering the chunk [dk][dv]
constexpr uint32_t BG_DS = 98304;       // dS' leaving it [dk][dv]
constexpr uint32_t BG_U = 131072;       // U [t][dv]          (A and T of the solve before it)
constexpr uint32_t BG_DU = 147456;      // dU [t][dv]
constexpr uint32_t BG_W = 163840;       // W, then dW [t][dk]
constexpr uint32_t BG_TT = 180224;      // T [t][s]
constexpr uint32_t BG_SA = 188416;      // T diag(beta gamma), then P, then X = T^T dT
constexpr uint32_t BG_SB = 196608;      // T diag(beta), then dQK = dP (.) M
constexpr uint32_t BG_SC = 204800;      // dT, then dKK = dA (.) beta (.) M
constexpr uint32_t BG_SMALL = 212992;   // per-token gates and reductions
constexpr uint32_t kGradSmem = BG_SMALL + 4096;
constexpr uint32_t BG_AT = BG_U;
constexpr uint32_t BG_TM = BG_U + kBlkFloats * 4;
static_assert(BG_TM + kBlkFloats * 4 <= BG_W, "A and T of the solve fit over U and dU");
static_assert(kGradSmem <= 232448, "per-chunk gradient shared memory");

// Small area (floats): g, gamma, lambda, beta, beta gamma [64] each; row and
// column partial sums; per-warp scalars.
constexpr int SM_G = 0, SM_GAM = 64, SM_LAM = 128, SM_BETA = 192, SM_BG = 256;
constexpr int SM_ROW = 320;     // [2][64] dg row sums per column half
constexpr int SM_DB = 448;      // [2][64] dbeta row sums
constexpr int SM_DLAM = 576;    // [2][64] dlambda row sums
constexpr int SM_COL = 704;     // [4][64] dg column sums per row block
constexpr int SM_RED = 960;     // [8] per-warp sums of S (.) dS'
constexpr int SM_WS = 968;      // [2] warp totals of the gate scan

// Row sums of a thread's fragment rows (16 mt + g and + 8) over the 4 lanes of
// a quad, then written per column half; column sums over the 8 quads of a warp.
__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}
__device__ __forceinline__ float col_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    return v;
}

// One CTA (256 threads) per (batch, value head, chunk).  Warp w takes rows
// 16 (w & 3) of every 64-row product and columns 64 (w >> 2) (N = 128) or
// 32 (w >> 2) (N = 64); the fragments of the 64 x 64 products K K^T and
// Q K^T stay in registers for the whole kernel.
__global__ void __launch_bounds__(256, 1) bw_chunk_grad_kernel(const BwDev p) {
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sb = smem_u32(sm);
    float *fs = reinterpret_cast<float *>(sm + BG_SMALL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int mt = warp & 3, nh = warp >> 2;
    const int hv = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.Hv));
    const int64_t rest = blockIdx.x / static_cast<unsigned>(p.Hv);
    const int c = static_cast<int>(rest % p.nchunks);
    const int b = static_cast<int>(rest / p.nchunks);
    const int hk = hv / p.group;
    const int64_t t0 = static_cast<int64_t>(c) * kC;
    const int nvalid = p.T - t0 < kC ? static_cast<int>(p.T - t0) : kC;
    const int64_t pr = static_cast<int64_t>(b) * p.Hv + hv;
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);

    // ---- loads: q, k, v, dy tiles (rows past T as zero), S and dS' to bf16
    for (int e = tid; e < kC * 16; e += 256) {
        const int r = e >> 4, pc = e & 15;
        const uint32_t off = sw256(r, pc);
        if (r < nvalid) {
            const int64_t tq = ((static_cast<int64_t>(b) * p.T + t0 + r) * p.Hqk + hk) * kD + pc * 8;
            const int64_t tv = ((static_cast<int64_t>(b) * p.T + t0 + r) * p.Hv + hv) * kD + pc * 8;
            cp_async16(sb + BG_Q + off, p.q + tq);
            cp_async16(sb + BG_K + off, p.k + tq);
            cp_async16(sb + BG_V + off, p.v + tv);
            cp_async16(sb + BG_DY + off, p.dy + tv);
        } else {
            *reinterpret_cast<uint4 *>(sm + BG_Q + off) = zero4;
            *reinterpret_cast<uint4 *>(sm + BG_K + off) = zero4;
            *reinterpret_cast<uint4 *>(sm + BG_V + off) = zero4;
            *reinterpret_cast<uint4 *>(sm + BG_DY + off) = zero4;
        }
    }
    {
        // the entering state and the leaving state gradient, bf16 [dk][dv] rows, into their tiles
        const __nv_bfloat16 *Sg = p.state + (pr * p.nchunks + c) * kD * kD;
        const __nv_bfloat16 *Dg = p.dstate + (pr * p.nchunks + c) * kD * kD;
        for (int e = tid; e < kD * 16; e += 256) {   // 128 rows x 16 pieces of 8
            const int r = e >> 4, pc = e & 15;
            cp_async16(sb + BG_S + sw256(r, pc), Sg + r * kD + pc * 8);
            cp_async16(sb + BG_DS + sw256(r, pc), Dg + r * kD + pc * 8);
        }
    }
    cp_async_commit();
    // gates: g = inclusive cumsum of log alpha (tokens past T: alpha = 1, beta = 0)
    if (tid < kC) {
        const int64_t gi = (static_cast<int64_t>(b) * p.T + t0 + tid) * p.Hv + hv;
        float la = tid < nvalid ? logf(__ldg(p.alpha + gi)) : 0.f;
        const float bt = tid < nvalid ? __ldg(p.beta + gi) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, la, o);
            if (lane >= o) la += v;
        }
        if (lane == 31) fs[SM_WS + warp] = la;
        fs[SM_G + tid] = la;
        fs[SM_BETA + tid] = bt;
    }
    cp_async_wait_all();
    __syncthreads();
    {
        // sum of S (.) dS' over the bf16 tiles (the same values the products use)
        float sds = 0.f;
        for (int e = tid; e < kD * 16; e += 256) {
            const int r = e >> 4, pc = e & 15;
            const uint4 a = *reinterpret_cast<const uint4 *>(sm + BG_S + sw256(r, pc));
            const uint4 d = *reinterpret_cast<const uint4 *>(sm + BG_DS + sw256(r, pc));
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 x = unpack2(aw[j]), y = unpack2(dw[j]);
                sds = fmaf(x.x, y.x, fmaf(x.y, y.y, sds));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sds += __shfl_xor_sync(0xffffffffu, sds, o);
        if (lane == 0) fs[SM_RED + warp] = sds;
    }
    if (tid < kC) {
        const float gv = fs[SM_G + tid] + (tid >= 32 ? fs[SM_WS] : 0.f);
        const float glast = fs[SM_WS] + fs[SM_WS + 1];
        fs[SM_G + tid] = gv;
        fs[SM_GAM + tid] = __expf(gv);
        fs[SM_LAM + tid] = __expf(glast - gv);
        fs[SM_BG + tid] = fs[SM_BETA + tid] * __expf(gv);
    }
    __syncthreads();
    const float *gg = fs + SM_G, *gam = fs + SM_GAM, *lam = fs + SM_LAM, *bet = fs + SM_BETA, *bg = fs + SM_BG;
    const int r0 = 16 * mt + g, r1 = r0 + 8;   // this thread's fragment rows

    // ---- K K^T and Q K^T (64 x 64): rows 16 mt, columns 32 nh .. + 31
    float kk[4][4], qk[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) kk[nt][e] = qk[nt][e] = 0.f;
#pragma unroll 2
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t ak[4], aq[4];
        ldsm_x4(ak, sb + BG_K + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
        ldsm_x4(aq, sb + BG_Q + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
#pragma unroll
        for (int np = 0; np < 2; ++np) {
            uint32_t bk[4];
            ldsm_x4(bk, sb + BG_K + sw256(32 * nh + 16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
            mma16816(kk[2 * np], ak, bk[0], bk[1]);
            mma16816(kk[2 * np + 1], ak, bk[2], bk[3]);
            mma16816(qk[2 * np], aq, bk[0], bk[1]);
            mma16816(qk[2 * np + 1], aq, bk[2], bk[3]);
        }
    }
    // gate factors of this thread's 64 x 64 fragment elements: M_ij = e^{g_i - g_j} (j <= i)
    float mi[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = e < 2 ? r0 : r1, j = 32 * nh + 8 * nt + 2 * t4 + (e & 1);
            mi[nt][e] = j <= i ? __expf(gg[i] - gg[j]) : 0.f;
        }
    // A = diag(beta) (M o K K^T), strictly lower, into the block-packed solve layout
    {
        float *At = reinterpret_cast<float *>(sm + BG_AT);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = e < 2 ? r0 : r1, j = 32 * nh + 8 * nt + 2 * t4 + (e & 1);
                if (j < i) At[blk(i >> 4, j >> 4) * kBlk + (j & 15) * kBS + (i & 15)] = bet[i] * mi[nt][e] * kk[nt][e];
            }
    }
    __syncthreads();
    {
        float *At = reinterpret_cast<float *>(sm + BG_AT);
        float *Tm = reinterpret_cast<float *>(sm + BG_TM);
        if (warp < 4 && lane < 16) diag_solve(warp, lane, At, Tm);
        __syncthreads();
        if (warp < 4) solve_factors(warp, At, Tm, lane);
        __syncthreads();
        if (warp == 0 || warp == 3)
            solve_column<1>(0, warp == 3 ? 1 : 0, At, Tm, lane);
        else if (warp < 3)
            solve_column<2>(warp, 0, At, Tm, lane);
        __syncthreads();
        // T, T diag(beta gamma), T diag(beta) in bf16 [t][s]
        for (int e = tid; e < kC * 8; e += 256) {
            const int t = e >> 3, pc = e & 7, I = t >> 4, J = pc >> 1;
            uint4 o0 = zero4, o1 = zero4, o2 = zero4;
            if (J <= I) {
                const float *src = Tm + blk(I, J) * kBlk + (t & 15) * kBS + (pc & 1) * 8;
                const float *bc = bg + pc * 8, *bb = bet + pc * 8;
                o0 = make_uint4(pack2(src[0], src[1]), pack2(src[2], src[3]), pack2(src[4], src[5]), pack2(src[6], src[7]));
                o1 = make_uint4(pack2(src[0] * bc[0], src[1] * bc[1]), pack2(src[2] * bc[2], src[3] * bc[3]),
                                pack2(src[4] * bc[4], src[5] * bc[5]), pack2(src[6] * bc[6], src[7] * bc[7]));
                o2 = make_uint4(pack2(src[0] * bb[0], src[1] * bb[1]), pack2(src[2] * bb[2], src[3] * bb[3]),
                                pack2(src[4] * bb[4], src[5] * bb[5]), pack2(src[6] * bb[6], src[7] * bb[7]));
            }
            *reinterpret_cast<uint4 *>(sm + BG_TT + sw128(t, pc)) = o0;
            *reinterpret_cast<uint4 *>(sm + BG_SA + sw128(t, pc)) = o1;
            *reinterpret_cast<uint4 *>(sm + BG_SB + sw128(t, pc)) = o2;
        }
    }
    __syncthreads();

    // ---- W = T diag(beta gamma) K -> bf16; U~ = T diag(beta) V (rows 16 mt, columns 64 nh)
    float u[8][4];
    {
        float w[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) w[nt][e] = u[nt][e] = 0.f;
#pragma unroll 1
        for (int kk = 0; kk <= mt; ++kk) {   // T is lower triangular by blocks
            uint32_t a1[4], a2[4];
            ldsm_x4(a1, sb + BG_SA + sw128(16 * mt + a_row(lane), 2 * kk + a_ch(lane)));
            ldsm_x4(a2, sb + BG_SB + sw128(16 * mt + a_row(lane), 2 * kk + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bk[4], bv[4];
                ldsm_x4_t(bk, sb + BG_K + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                ldsm_x4_t(bv, sb + BG_V + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(w[2 * np], a1, bk[0], bk[1]);
                mma16816(w[2 * np + 1], a1, bk[2], bk[3]);
                mma16816(u[2 * np], a2, bv[0], bv[1]);
                mma16816(u[2 * np + 1], a2, bv[2], bv[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            *reinterpret_cast<uint32_t *>(sm + BG_W + sw256(r0, 8 * nh + nt) + 4 * t4) = pack2(w[nt][0], w[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + BG_W + sw256(r1, 8 * nh + nt) + 4 * t4) = pack2(w[nt][2], w[nt][3]);
        }
    }
    __syncthreads();
    // U = U~ - W S -> bf16; P = M (.) Q K^T -> bf16 (over T diag(beta gamma), no longer read)
    {
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t aw[4];
            ldsm_x4(aw, sb + BG_W + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
#pragma unroll
            for (int e = 0; e < 4; ++e) aw[e] ^= 0x80008000u;   // -W: flip both bf16 signs
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bs[4];
                ldsm_x4_t(bs, sb + BG_S + sw256(16 * ks + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(u[2 * np], aw, bs[0], bs[1]);
                mma16816(u[2 * np + 1], aw, bs[2], bs[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            *reinterpret_cast<uint32_t *>(sm + BG_U + sw256(r0, 8 * nh + nt) + 4 * t4) = pack2(u[nt][0], u[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + BG_U + sw256(r1, 8 * nh + nt) + 4 * t4) = pack2(u[nt][2], u[nt][3]);
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int col = 32 * nh + 8 * nt + 2 * t4;
            *reinterpret_cast<uint32_t *>(sm + BG_SA + sw128(r0, col >> 3) + 2 * (col & 7)) =
                pack2(mi[nt][0] * qk[nt][0], mi[nt][1] * qk[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + BG_SA + sw128(r1, col >> 3) + 2 * (col & 7)) =
                pack2(mi[nt][2] * qk[nt][2], mi[nt][3] * qk[nt][3]);
        }
    }
    __syncthreads();

    // Per-thread sums over this thread's fragment rows (r0, r1) and 64 x 64 columns.
    float dg_r[2] = {0.f, 0.f}, db_r[2] = {0.f, 0.f}, dl_r[2] = {0.f, 0.f};
    float dg_c[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) dg_c[nt][0] = dg_c[nt][1] = 0.f;
    auto tile_f2 = [&](uint32_t base, int row, int col) {   // two bf16 of a [64][128] tile
        return unpack2(*reinterpret_cast<const uint32_t *>(sm + base + sw256(row, col >> 3) + 2 * (col & 7)));
    };

    // ---- dU = lambda (.) K dS' + P^T dY -> bf16; dlambda_j = (K dS')_j . u_j
    {
        float du[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) du[nt][e] = 0.f;
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t ak[4];
            ldsm_x4(ak, sb + BG_K + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bs[4];
                ldsm_x4_t(bs, sb + BG_DS + sw256(16 * ks + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(du[2 * np], ak, bs[0], bs[1]);
                mma16816(du[2 * np + 1], ak, bs[2], bs[3]);
            }
        }
        const float l0 = lam[r0], l1 = lam[r1];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            dl_r[0] += du[nt][0] * u[nt][0] + du[nt][1] * u[nt][1];
            dl_r[1] += du[nt][2] * u[nt][2] + du[nt][3] * u[nt][3];
            du[nt][0] *= l0;
            du[nt][1] *= l0;
            du[nt][2] *= l1;
            du[nt][3] *= l1;
        }
#pragma unroll 1
        for (int kk = mt; kk < 4; ++kk) {   // P^T[t][s] is zero for s below the row block
            uint32_t ap[4];
            ldsm_x4_t(ap, sb + BG_SA + sw128(16 * kk + at_row(lane), 2 * mt + at_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t by[4];
                ldsm_x4_t(by, sb + BG_DY + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(du[2 * np], ap, by[0], by[1]);
                mma16816(du[2 * np + 1], ap, by[2], by[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            *reinterpret_cast<uint32_t *>(sm + BG_DU + sw256(r0, 8 * nh + nt) + 4 * t4) = pack2(du[nt][0], du[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + BG_DU + sw256(r1, 8 * nh + nt) + 4 * t4) = pack2(du[nt][2], du[nt][3]);
        }
    }

    // ---- dK = lambda (.) U dS'^T;  dQ = gamma (.) dY S^T;  dg += gamma (.) rowsum(dY (.) Q S)
    float dkf[8][4], dqf[8][4];
    {
        float qs[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dkf[nt][e] = dqf[nt][e] = qs[nt][e] = 0.f;
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t au[4], ay[4], aq[4];
            ldsm_x4(au, sb + BG_U + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
            ldsm_x4(ay, sb + BG_DY + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
            ldsm_x4(aq, sb + BG_Q + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bd[4], bs[4], bst[4];
                // dS'^T and S^T: [dk][dv] storage read as [n][k] (no transpose)
                ldsm_x4(bd, sb + BG_DS + sw256(64 * nh + 16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
                ldsm_x4(bs, sb + BG_S + sw256(64 * nh + 16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
                // S for Q S: [dk][dv] as [k][n]
                ldsm_x4_t(bst, sb + BG_S + sw256(16 * ks + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(dkf[2 * np], au, bd[0], bd[1]);
                mma16816(dkf[2 * np + 1], au, bd[2], bd[3]);
                mma16816(dqf[2 * np], ay, bs[0], bs[1]);
                mma16816(dqf[2 * np + 1], ay, bs[2], bs[3]);
                mma16816(qs[2 * np], aq, bst[0], bst[1]);
                mma16816(qs[2 * np + 1], aq, bst[2], bst[3]);
            }
        }
        const float l0 = lam[r0], l1 = lam[r1], g0 = gam[r0], g1 = gam[r1];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int col = 64 * nh + 8 * nt + 2 * t4;
            const float2 y0 = tile_f2(BG_DY, r0, col), y1 = tile_f2(BG_DY, r1, col);
            s0 += y0.x * qs[nt][0] + y0.y * qs[nt][1];
            s1 += y1.x * qs[nt][2] + y1.y * qs[nt][3];
            dkf[nt][0] *= l0;
            dkf[nt][1] *= l0;
            dkf[nt][2] *= l1;
            dkf[nt][3] *= l1;
            dqf[nt][0] *= g0;
            dqf[nt][1] *= g0;
            dqf[nt][2] *= g1;
            dqf[nt][3] *= g1;
        }
        dg_r[0] += g0 * s0;
        dg_r[1] += g1 * s1;
    }

    // ---- dP = dY U^T (64 x 64); dQK = dP (.) M -> bf16 (over T diag(beta)); dM terms of dg
    {
        float dp[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dp[nt][e] = 0.f;
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t ay[4];
            ldsm_x4(ay, sb + BG_DY + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bu[4];
                ldsm_x4(bu, sb + BG_U + sw256(32 * nh + 16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
                mma16816(dp[2 * np], ay, bu[0], bu[1]);
                mma16816(dp[2 * np + 1], ay, bu[2], bu[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int col = 32 * nh + 8 * nt + 2 * t4;
            float m[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                m[e] = dp[nt][e] * mi[nt][e];               // dQK
                const float dm = m[e] * qk[nt][e];          // dM_ij (M_ij = 0 above the diagonal)
                dg_r[e >> 1] += dm;
                dg_c[nt][e & 1] -= dm;
            }
            *reinterpret_cast<uint32_t *>(sm + BG_SB + sw128(r0, col >> 3) + 2 * (col & 7)) = pack2(m[0], m[1]);
            *reinterpret_cast<uint32_t *>(sm + BG_SB + sw128(r1, col >> 3) + 2 * (col & 7)) = pack2(m[2], m[3]);
        }
    }
    __syncthreads();

    // ---- dQ += dQK K, dK += dQK^T Q; dQ complete
#pragma unroll 1
    for (int kk = 0; kk < 4; ++kk) {
        uint32_t ad[4], adt[4];
        ldsm_x4(ad, sb + BG_SB + sw128(16 * mt + a_row(lane), 2 * kk + a_ch(lane)));
        ldsm_x4_t(adt, sb + BG_SB + sw128(16 * kk + at_row(lane), 2 * mt + at_ch(lane)));
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t bk[4], bq[4];
            ldsm_x4_t(bk, sb + BG_K + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
            ldsm_x4_t(bq, sb + BG_Q + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
            if (kk <= mt) {
                mma16816(dqf[2 * np], ad, bk[0], bk[1]);
                mma16816(dqf[2 * np + 1], ad, bk[2], bk[3]);
            }
            if (kk >= mt) {
                mma16816(dkf[2 * np], adt, bq[0], bq[1]);
                mma16816(dkf[2 * np + 1], adt, bq[2], bq[3]);
            }
        }
    }
    auto store_qk_grad = [&](float *dst, const float (&f)[8][4]) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = hr ? r1 : r0;
            if (r >= nvalid) continue;
            float *row = dst + ((static_cast<int64_t>(b) * p.T + t0 + r) * p.Hqk + hk) * kD + 64 * nh + 2 * t4;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                if (p.group == 1) {
                    *reinterpret_cast<float2 *>(row + 8 * nt) = make_float2(f[nt][2 * hr], f[nt][2 * hr + 1]);
                } else {
                    atomicAdd(row + 8 * nt, f[nt][2 * hr]);
                    atomicAdd(row + 8 * nt + 1, f[nt][2 * hr + 1]);
                }
            }
        }
    };
    store_qk_grad(p.dq, dqf);

    // ---- dW = -dU S^T -> bf16 (over W);  T^T dU -> dV = beta (.) T^T dU, dbeta terms
    {
        float dw[8][4], tdu[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dw[nt][e] = tdu[nt][e] = 0.f;
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t au[4];
            ldsm_x4(au, sb + BG_DU + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
#pragma unroll
            for (int e = 0; e < 4; ++e) au[e] ^= 0x80008000u;   // -dU
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bs[4];
                ldsm_x4(bs, sb + BG_S + sw256(64 * nh + 16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
                mma16816(dw[2 * np], au, bs[0], bs[1]);
                mma16816(dw[2 * np + 1], au, bs[2], bs[3]);
            }
        }
#pragma unroll 1
        for (int kk = mt; kk < 4; ++kk) {   // T^T[t][s] is zero for s below the row block
            uint32_t at[4];
            ldsm_x4_t(at, sb + BG_TT + sw128(16 * kk + at_row(lane), 2 * mt + at_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bu[4];
                ldsm_x4_t(bu, sb + BG_DU + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(tdu[2 * np], at, bu[0], bu[1]);
                mma16816(tdu[2 * np + 1], at, bu[2], bu[3]);
            }
        }
        const float b0 = bet[r0], b1 = bet[r1];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int col = 64 * nh + 8 * nt + 2 * t4;
            *reinterpret_cast<uint32_t *>(sm + BG_W + sw256(r0, 8 * nh + nt) + 4 * t4) = pack2(dw[nt][0], dw[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + BG_W + sw256(r1, 8 * nh + nt) + 4 * t4) = pack2(dw[nt][2], dw[nt][3]);
            const float2 v0 = tile_f2(BG_V, r0, col), v1 = tile_f2(BG_V, r1, col);
            db_r[0] += tdu[nt][0] * v0.x + tdu[nt][1] * v0.y;
            db_r[1] += tdu[nt][2] * v1.x + tdu[nt][3] * v1.y;
        }
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = hr ? r1 : r0;
            const float bb = hr ? b1 : b0;
            if (r >= nvalid) continue;
            float *row = p.dv + ((static_cast<int64_t>(b) * p.T + t0 + r) * p.Hv + hv) * kD + 64 * nh + 2 * t4;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
                *reinterpret_cast<float2 *>(row + 8 * nt) = make_float2(bb * tdu[nt][2 * hr], bb * tdu[nt][2 * hr + 1]);
        }
    }
    __syncthreads();

    // ---- T^T dW: dK += (beta gamma) (.) T^T dW, dbeta and dg terms;
    // dT = (dW K^T) diag(beta gamma) + (dU V^T) diag(beta) -> bf16
    {
        float tdw[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) tdw[nt][e] = 0.f;
#pragma unroll 1
        for (int kk = mt; kk < 4; ++kk) {
            uint32_t at[4];
            ldsm_x4_t(at, sb + BG_TT + sw128(16 * kk + at_row(lane), 2 * mt + at_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bw[4];
                ldsm_x4_t(bw, sb + BG_W + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(tdw[2 * np], at, bw[0], bw[1]);
                mma16816(tdw[2 * np + 1], at, bw[2], bw[3]);
            }
        }
        const float bg0 = bg[r0], bg1 = bg[r1];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int col = 64 * nh + 8 * nt + 2 * t4;
            const float2 k0 = tile_f2(BG_K, r0, col), k1 = tile_f2(BG_K, r1, col);
            s0 += tdw[nt][0] * k0.x + tdw[nt][1] * k0.y;
            s1 += tdw[nt][2] * k1.x + tdw[nt][3] * k1.y;
            dkf[nt][0] += bg0 * tdw[nt][0];
            dkf[nt][1] += bg0 * tdw[nt][1];
            dkf[nt][2] += bg1 * tdw[nt][2];
            dkf[nt][3] += bg1 * tdw[nt][3];
        }
        db_r[0] += gam[r0] * s0;
        db_r[1] += gam[r1] * s1;
        dg_r[0] += bg0 * s0;
        dg_r[1] += bg1 * s1;

        float dt[4][4], dv2[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dt[nt][e] = dv2[nt][e] = 0.f;
#pragma unroll 2
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t aw[4], au[4];
            ldsm_x4(aw, sb + BG_W + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
            ldsm_x4(au, sb + BG_DU + sw256(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bk[4], bv[4];
                ldsm_x4(bk, sb + BG_K + sw256(32 * nh + 16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
                ldsm_x4(bv, sb + BG_V + sw256(32 * nh + 16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
                mma16816(dt[2 * np], aw, bk[0], bk[1]);
                mma16816(dt[2 * np + 1], aw, bk[2], bk[3]);
                mma16816(dv2[2 * np], au, bv[0], bv[1]);
                mma16816(dv2[2 * np + 1], au, bv[2], bv[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int col = 32 * nh + 8 * nt + 2 * t4;
            const float c0 = bg[col], c1 = bg[col + 1], e0 = bet[col], e1 = bet[col + 1];
            *reinterpret_cast<uint32_t *>(sm + BG_SC + sw128(r0, col >> 3) + 2 * (col & 7)) =
                pack2(dt[nt][0] * c0 + dv2[nt][0] * e0, dt[nt][1] * c1 + dv2[nt][1] * e1);
            *reinterpret_cast<uint32_t *>(sm + BG_SC + sw128(r1, col >> 3) + 2 * (col & 7)) =
                pack2(dt[nt][2] * c0 + dv2[nt][2] * e0, dt[nt][3] * c1 + dv2[nt][3] * e1);
        }
    }
    __syncthreads();

    // ---- X = T^T dT -> bf16 (over P)
    {
        float x[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) x[nt][e] = 0.f;
#pragma unroll 1
        for (int kk = mt; kk < 4; ++kk) {
            uint32_t at[4];
            ldsm_x4_t(at, sb + BG_TT + sw128(16 * kk + at_row(lane), 2 * mt + at_ch(lane)));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bd[4];
                ldsm_x4_t(bd, sb + BG_SC + sw128(16 * kk + bt_row(lane), 4 * nh + 2 * np + bt_ch(lane)));
                mma16816(x[2 * np], at, bd[0], bd[1]);
                mma16816(x[2 * np + 1], at, bd[2], bd[3]);
            }
        }
        __syncthreads();   // every warp has read dT and P before X and dKK overwrite them
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int col = 32 * nh + 8 * nt + 2 * t4;
            *reinterpret_cast<uint32_t *>(sm + BG_SA + sw128(r0, col >> 3) + 2 * (col & 7)) = pack2(x[nt][0], x[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + BG_SA + sw128(r1, col >> 3) + 2 * (col & 7)) = pack2(x[nt][2], x[nt][3]);
        }
    }
    __syncthreads();

    // ---- dA = -X T^T (strictly lower); dbeta, dKK = dA (.) beta (.) M -> bf16 (over dT), dM terms
    {
        float da[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) da[nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t ax[4];
            ldsm_x4(ax, sb + BG_SA + sw128(16 * mt + a_row(lane), 2 * ks + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bt[4];
                ldsm_x4(bt, sb + BG_TT + sw128(32 * nh + 16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
                mma16816(da[2 * np], ax, bt[0], bt[1]);
                mma16816(da[2 * np + 1], ax, bt[2], bt[3]);
            }
        }
        const float be0 = bet[r0], be1 = bet[r1];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int col = 32 * nh + 8 * nt + 2 * t4;
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = e < 2 ? r0 : r1, j = col + (e & 1);
                const float a = j < i ? -da[nt][e] * mi[nt][e] : 0.f;   // dA (.) M_s
                db_r[e >> 1] += a * kk[nt][e];
                const float bb = e < 2 ? be0 : be1;
                o[e] = a * bb;                                         // dKK
                const float dm = o[e] * kk[nt][e];                      // dM_s
                dg_r[e >> 1] += dm;
                dg_c[nt][e & 1] -= dm;
            }
            *reinterpret_cast<uint32_t *>(sm + BG_SC + sw128(r0, col >> 3) + 2 * (col & 7)) = pack2(o[0], o[1]);
            *reinterpret_cast<uint32_t *>(sm + BG_SC + sw128(r1, col >> 3) + 2 * (col & 7)) = pack2(o[2], o[3]);
        }
    }
    __syncthreads();

    // ---- dK += (dKK + dKK^T) K; dK complete
#pragma unroll 1
    for (int kk = 0; kk < 4; ++kk) {
        uint32_t a1[4], a2[4];
        ldsm_x4(a1, sb + BG_SC + sw128(16 * mt + a_row(lane), 2 * kk + a_ch(lane)));
        ldsm_x4_t(a2, sb + BG_SC + sw128(16 * kk + at_row(lane), 2 * mt + at_ch(lane)));
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t bk[4];
            ldsm_x4_t(bk, sb + BG_K + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
            if (kk <= mt) {
                mma16816(dkf[2 * np], a1, bk[0], bk[1]);
                mma16816(dkf[2 * np + 1], a1, bk[2], bk[3]);
            }
            if (kk >= mt) {
                mma16816(dkf[2 * np], a2, bk[0], bk[1]);
                mma16816(dkf[2 * np + 1], a2, bk[2], bk[3]);
            }
        }
    }
    store_qk_grad(p.dk, dkf);

    // ---- per-token sums in a fixed order, then d log alpha = reverse cumulative sum of dg
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const float sg = quad_sum(dg_r[hr]), sbv = quad_sum(db_r[hr]), sl = quad_sum(dl_r[hr]);
        if (t4 == 0) {
            const int r = hr ? r1 : r0;
            fs[SM_ROW + 64 * nh + r] = sg;
            fs[SM_DB + 64 * nh + r] = sbv;
            fs[SM_DLAM + 64 * nh + r] = sl;
        }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float v = col_sum(dg_c[nt][h]);
            if (g == 0) fs[SM_COL + 64 * mt + 32 * nh + 8 * nt + 2 * t4 + h] = v;
        }
    __syncthreads();
    if (tid < kC) {
        const int i = tid;
        const float dl = fs[SM_DLAM + i] + fs[SM_DLAM + 64 + i];
        float dgi = fs[SM_ROW + i] + fs[SM_ROW + 64 + i] + fs[SM_COL + i] + fs[SM_COL + 64 + i] + fs[SM_COL + 128 + i] +
                    fs[SM_COL + 192 + i] - dl * lam[i];
        float tot = dl * lam[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        const float dbi = fs[SM_DB + i] + fs[SM_DB + 64 + i];
        // dg at the chunk's last token: gamma_C <S, dS'> and the sum over j of dlambda_j lambda_j
        __syncwarp();
        if (lane == 0) fs[SM_WS + warp] = tot;   // warps 0 and 1
        // suffix sums within each warp
        float sfx = dgi;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_down_sync(0xffffffffu, sfx, o);
            if (lane + o < 32) sfx += v;
        }
        fs[SM_ROW + i] = sfx;      // reused: suffix sum within the warp
        fs[SM_DB + i] = dbi;
    }
    __syncthreads();
    if (tid < kC) {
        const int i = tid;
        float sred = 0.f;
        for (int w = 0; w < 8; ++w) sred += fs[SM_RED + w];
        const float last = gam[kC - 1] * sred + fs[SM_WS] + fs[SM_WS + 1];   // added to dg[63]
        // dla_i = sum_{j >= i} dg_j: the warp's suffix, the upper warp's total, and dg[63]'s extra
        float dla = fs[SM_ROW + i] + (i < 32 ? fs[SM_ROW + 32] : 0.f) + last;
        if (i < nvalid) {
            const int64_t gi = (static_cast<int64_t>(b) * p.T + t0 + i) * p.Hv + hv;
            p.dlog_alpha[gi] = dla;
            p.dbeta[gi] = fs[SM_DB + i];
        }
    }
}

}  // namespace

namespace {
cudaError_t set_bw_attributes() {
    static cudaError_t result = [] {
        cudaError_t e = cudaFuncSetAttribute(bw_reverse_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kRevSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bw_chunk_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kGradSmem));
        return e;
    }();
    return result;
}
}  // namespace

// Workspace: the chunk records and decay bounds, then (256-byte aligned) the
// states entering and the state gradients leaving every chunk (bf16).
static size_t states_offset(int64_t B, int64_t T, int Hv) {
    return (chunked_cw_ops_bytes(B, T, Hv) + 255) / 256 * 256;
}

// After the states: the exact split's flags and segment maps (used by the
// forward chain, then by the reverse chain, in stream order).
static size_t split_offset(int64_t B, int64_t T, int Hv) {
    const int64_t nchunks = (T + kC - 1) / kC;
    const size_t states = static_cast<size_t>(B) * Hv * nchunks * kD * kD * sizeof(__nv_bfloat16);
    return (states_offset(B, T, Hv) + 2 * states + 255) / 256 * 256;
}

static void split_sizes(int64_t B, int64_t T, int Hv, size_t *flag_bytes, size_t *map_bytes) {
    const int64_t pairs = B * Hv, segs = exact_split_segments(pairs, (T + kC - 1) / kC);
    *flag_bytes = (static_cast<size_t>(pairs) * segs * sizeof(int) + 255) / 256 * 256;
    *map_bytes = static_cast<size_t>(pairs) * segs * 3 * kD * kD * sizeof(float);
}

size_t backward_chunked_workspace_bytes(int64_t B, int64_t T, int Hv) {
    size_t fb = 0, mb = 0;
    split_sizes(B, T, Hv, &fb, &mb);
    return split_offset(B, T, Hv) + fb + mb;
}

cudaError_t launch_backward_chunked(const BackwardParams &p, uint8_t *ws, cudaStream_t stream, int num_sms) {
    const int64_t nchunks = (p.T + kC - 1) / kC;
    const int64_t pairs = p.B * p.Hv;
    if (nchunks <= 0 || pairs <= 0) return cudaSuccess;
    if (nchunks > 0x7fffffffLL || p.B * nchunks * p.Hv > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t e = set_bw_attributes();
    if (e != cudaSuccess) return e;
    const size_t ops = states_offset(p.B, p.T, p.Hv);
    const size_t states = static_cast<size_t>(pairs) * nchunks * kD * kD * sizeof(__nv_bfloat16);
    __nv_bfloat16 *state = reinterpret_cast<__nv_bfloat16 *>(ws + ops);
    __nv_bfloat16 *dstate = reinterpret_cast<__nv_bfloat16 *>(ws + ops + states);

    // forward: chunk records and the state entering every chunk
    ChunkedCwParams f{};
    f.B = p.B; f.T = p.T; f.Hqk = p.Hqk; f.Hv = p.Hv; f.group = p.group; f.d = kD;
    f.q = p.q; f.k = p.k; f.v = p.v; f.alpha = p.alpha; f.beta = p.beta; f.S0 = p.S0;
    f.y = nullptr; f.S_T = nullptr;
    f.segments = 0; f.log_eps = -13.862943611198906f; f.max_warmup_chunks = 64;
    f.ops = ws; f.scalar_alpha = true; f.state_out = state;
    size_t flag_bytes = 0, map_bytes = 0;
    split_sizes(p.B, p.T, p.Hv, &flag_bytes, &map_bytes);
    int *flags = reinterpret_cast<int *>(ws + split_offset(p.B, p.T, p.Hv));
    float *maps = reinterpret_cast<float *>(ws + split_offset(p.B, p.T, p.Hv) + flag_bytes);
    if (map_bytes > 0) {
        f.exact_flag = flags;
        f.seg_state = maps;
        f.seg_state_bytes = map_bytes;
    }
    e = launch_chunked_cw(f, stream, num_sms);
    if (e != cudaSuccess) return e;

    BwDev dv{};
    dv.T = p.T;
    dv.B = static_cast<int>(p.B);
    dv.Hqk = p.Hqk;
    dv.Hv = p.Hv;
    dv.group = p.group;
    dv.nchunks = static_cast<int>(nchunks);
    int P = plan_segments(pairs, nchunks, num_sms, 0);
    const int64_t len = (nchunks + P - 1) / P;
    P = static_cast<int>((nchunks + len - 1) / len);
    dv.seg_chunks = static_cast<int>(len);
    dv.max_warmup = 64;
    dv.log_eps = -13.862943611198906f;
    dv.q = static_cast<const __nv_bfloat16 *>(p.q);
    dv.k = static_cast<const __nv_bfloat16 *>(p.k);
    dv.v = static_cast<const __nv_bfloat16 *>(p.v);
    dv.dy = static_cast<const __nv_bfloat16 *>(p.dy);
    dv.alpha = p.alpha;
    dv.beta = p.beta;
    dv.dS_T = p.dS_T;
    dv.rec = ws;
    dv.bound = reinterpret_cast<const float *>(ws + static_cast<size_t>(pairs) * nchunks * rec::kBytes);
    dv.state = state;
    dv.dstate = dstate;
    dv.dS0 = p.dS0;
    dv.dq = p.dq;
    dv.dk = p.dk;
    dv.dv = p.dv;
    dv.dlog_alpha = p.dlog_alpha;
    dv.dbeta = p.dbeta;
    dv.nseg = P;
    dv.pass = 0;
    dv.exact_flag = nullptr;
    dv.seg_state = nullptr;
    if (map_bytes > 0 && takes_exact_split(pairs, nchunks, P, kD, map_bytes)) {
        // the reverse chain's exact split: plan, transitions, combine (maps stored in reverse
        // segment order, so the forward combine applies), then the output pass
        dv.exact_flag = flags;
        dv.seg_state = maps;
        const int nplan = static_cast<int>(pairs * (P - 1));
        bw_plan_kernel<<<static_cast<unsigned>((nplan + 127) / 128), 128, 0, stream>>>(dv, flags);
        dv.pass = 1;
        bw_reverse_chain_kernel<<<static_cast<unsigned>(2 * pairs * P), 256, kRevSmem, stream>>>(dv);
        if ((e = launch_segment_combine(flags, maps, pairs, P, kD, stream)) != cudaSuccess) return e;
        dv.pass = 0;
    }
    bw_reverse_chain_kernel<<<static_cast<unsigned>(pairs * P), 256, kRevSmem, stream>>>(dv);
    if (p.group > 1) {   // dq, dk accumulate over the value heads of a group
        const size_t nqk = static_cast<size_t>(p.B) * p.T * p.Hqk * kD * sizeof(float);
        if ((e = cudaMemsetAsync(p.dq, 0, nqk, stream)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(p.dk, 0, nqk, stream)) != cudaSuccess) return e;
    }
    bw_chunk_grad_kernel<<<static_cast<unsigned>(p.B * nchunks * p.Hv), 256, kGradSmem, stream>>>(dv);
    return cudaGetLastError();
}

}  // namespace gdn
