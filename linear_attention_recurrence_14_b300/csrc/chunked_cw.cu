// Chunked prefill with the channel-wise decay gate (bf16 q/k/v, d = 128):
// S~ = diag(alpha_t) S with alpha_t in (0, 1]^{dk}, the other three lines of the
// recurrence unchanged (Qwen3.8-Next reading notes, section 2.1, "Why the
// delta rule matters": the per-channel decay of Kimi Delta Attention).
//
// Chunk algebra.  Over a chunk of C = 64 tokens let G[t][c] be the cumulative
// sum of log alpha of channel c up to and including token t, and write
// Qp = Q (.) e^G, Kp = K (.) e^G, Kl = K (.) e^{g_C - G} (g_C the last row of G).
// Unrolling the transition form S_t = diag(alpha_t)(I - beta_t k_t k_t^T) S_{t-1}
// + beta_t k_t v_t^T over the chunk gives, for the state S entering it:
//     A_ts = beta_t sum_c k_tc k_sc e^{G_tc - G_sc}      (s < t),   T = (I + A)^{-1}
//     W = T diag(beta) Kp,  U~ = T diag(beta) V,  U = U~ - W S
//     P_ts = sum_c q_tc k_sc e^{G_tc - G_sc}              (s <= t)
//     Y = Qp S + P U,       S_next = diag(e^{g_C}) S + Kl^T U.
// With a scalar gate the factors e^{G_t - G_s} come out of the channel sums;
// here they stay inside, so A and P are Gram products of per-channel scaled
// keys and queries.  Every factor used is bounded by 1 except inside a
// 16-token block: row block I uses the reference R_I = G at the token before
// the block, so (t in block I, s <= t)
//     e^{G_t - G_s} = e^{G_t - R_I} * e^{R_I - G_s},
// the first factor <= 1 and the second <= 1 for s before the block and at most
// the block's own decay for s inside it.  A block whose decay exceeds e^80 in
// some channel (far beyond any gate of a trained layer) has its diagonal part
// computed element by element instead, so the result holds for every gate.
// The pre-pass keeps G in base 2 (cumulative log2 alpha) and takes every
// power with one ex2.
//
// Two kernels.  cw_prepass_kernel, one CTA per (batch, value head, chunk),
// computes everything that does not depend on the state and writes it to the
// workspace: -W, U~, Qp, Kl and P in bf16, e^{g_C}, and a per-chunk bound on
// the state's decay (the sum over tokens of max_c log alpha) for the warm-up
// windows.  cw_chain_kernel, one CTA per (batch, value head, segment), runs the
// state through the chunks: three products per chunk on the tensor cores
// (warp-level bf16 MMAs, fp32 accumulation), the state in fp32 registers as
// the accumulator of its own update, y written per chunk.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn_internal.h"
#include "warp_mma.cuh"

namespace gdn {
namespace {

using namespace wm;

constexpr int kC = 64;             // tokens per chunk
constexpr int kD = 128;            // head dimension (dk = dv)
// Exponents are kept in base 2 (G holds cumulative log2 alpha): the largest
// power of two taken through a bf16 operand is 2^115 (about e^80).
constexpr float kMaxExp2 = 115.f;
constexpr float kLn2 = 0.6931471805599453f;

// Chunk record in the workspace, per (batch, value head, chunk); tiles are
// row-major bf16 [64][128] (P: [64][64]), rows 256 (128) bytes.
constexpr uint32_t REC_WN = 0;          // -W
constexpr uint32_t REC_UT = 16384;      // U~
constexpr uint32_t REC_QP = 32768;      // Qp
constexpr uint32_t REC_KL = 49152;      // Kl
constexpr uint32_t REC_P = 65536;       // P (zero above the diagonal)
constexpr uint32_t REC_GC = 73728;      // e^{g_C}, fp32 [128]
constexpr uint32_t kRecBytes = 74240;
static_assert(kRecBytes == kCwChunkBytes, "chunk record size");

// ------------------------------------------------------------- parameters

struct CwDev {
    int64_t T;
    int B, Hqk, Hv, group, nchunks;
    int seg_chunks, max_warmup;
    float log_eps;
    const __nv_bfloat16 *q, *k, *v;
    const float *alpha, *beta, *S0;
    __nv_bfloat16 *y;
    float *S_T;
    uint8_t *rec;     // [B * Hv][nchunks][kRecBytes]
    float *bound;     // [B * Hv][nchunks]
    int scalar_alpha; // alpha is [B, T, Hv], the same decay for every channel
    __nv_bfloat16 *state_out; // nullptr, or the state entering every chunk [B * Hv][nchunks][d][d] bf16
    // Exact sequence split (chain): nseg segments per head; pass 1 runs the
    // transitions of the heads with a flag set (kind 0: from the zero state,
    // or S0 for segment 0, with the values; kind 1: from the identity with
    // the values zero), pass 0 the output pass, where those heads start every
    // segment from the state the combine wrote.  seg_state: [pairs][nseg][3][d][d].
    int nseg, pass;
    const int *exact_flag;
    float *seg_state;
};

// Segments (of every head) whose preceding chunks reach no window within the
// limit: flag[pair][seg] = 1 (one thread per (pair, segment >= 1)).  Walking
// back to chunk 0 within the limit needs no split (that start is exact).
__global__ void cw_plan_kernel(const CwDev p, int *flag) {
    const int pairs = p.B * p.Hv;
    const int idx = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
    if (idx >= pairs * (p.nseg - 1)) return;
    const int pr = idx % pairs, seg = 1 + idx / pairs;
    const int c_begin = seg * p.seg_chunks;
    float acc = 0.f;
    int v = 1;
    for (int m = 1; m <= p.max_warmup; ++m) {
        const int cc = c_begin - m;
        if (cc < 0) {
            v = 0;
            break;
        }
        acc += p.bound[static_cast<int64_t>(pr) * p.nchunks + cc];
        if (acc <= p.log_eps) {
            v = 0;
            break;
        }
    }
    flag[static_cast<int64_t>(pr) * p.nseg + seg] = v;
}

__device__ __forceinline__ bool cw_head_split(const int *flag, int pr, int nseg) {
    int any = 0;
    for (int sg = 1; sg < nseg; ++sg) any |= flag[static_cast<int64_t>(pr) * nseg + sg];
    return any != 0;
}

// Pre-pass shared memory (bytes).  After the A and P products the q/k tiles
// hold A and T, the G tile holds T diag(beta) and the Kn tile holds V.
constexpr uint32_t PP_G = 0;            // G, fp32 [64][128]    | later T2 bf16 [64][64]
constexpr uint32_t PP_QT = 32768;       // q, then Qloc         | later A (fp32, block-packed)
constexpr uint32_t PP_KT = 49152;       // k                    | later T (from PP_QT + 15360)
constexpr uint32_t PP_KL = 65536;       // Kloc
constexpr uint32_t PP_KN = 81920;       // Kn of the current row block | later V
constexpr uint32_t PP_FIX = 98304;      // element-wise diagonal blocks [4][2][16][16] fp32
constexpr uint32_t PP_BETA = 106496;    // beta [64]
constexpr uint32_t PP_R = 106752;       // R_I [4][128]
constexpr uint32_t PP_ER = 108800;      // e^{R_I} [4][128]
constexpr uint32_t PP_GC = 110848;      // g_C [128]
constexpr uint32_t PP_VIOL = 111360;    // [4] int: block exceeds e^kMaxExp in some channel
constexpr uint32_t PP_WRED = 111376;    // [8] per-warp partial sums
constexpr uint32_t kPrepassSmem = 111408;
constexpr uint32_t PP_AT = PP_QT;
constexpr uint32_t PP_TM = PP_QT + kBlkFloats * 4;
constexpr uint32_t PP_T2 = PP_G;
static_assert(PP_TM + kBlkFloats * 4 <= PP_KL, "A and T fit in the q/k tiles");

__device__ __forceinline__ float tile_elem(const uint8_t *tile, int row, int col) {
    const uint16_t h = *reinterpret_cast<const uint16_t *>(tile + sw256(row, col >> 3) + 2 * (col & 7));
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__global__ void __launch_bounds__(256, 2) cw_prepass_kernel(const CwDev p) {
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sb = smem_u32(sm);
    float *G = reinterpret_cast<float *>(sm + PP_G);
    float *beta_s = reinterpret_cast<float *>(sm + PP_BETA);
    float *R = reinterpret_cast<float *>(sm + PP_R);
    float *eR = reinterpret_cast<float *>(sm + PP_ER);
    float *gC = reinterpret_cast<float *>(sm + PP_GC);
    int *viol = reinterpret_cast<int *>(sm + PP_VIOL);
    float *wred = reinterpret_cast<float *>(sm + PP_WRED);
    float *fix = reinterpret_cast<float *>(sm + PP_FIX);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int hv = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.Hv));
    const int64_t rest = blockIdx.x / static_cast<unsigned>(p.Hv);
    const int c = static_cast<int>(rest % p.nchunks);
    const int b = static_cast<int>(rest / p.nchunks);
    const int hk = hv / p.group;
    const int64_t t0 = static_cast<int64_t>(c) * kC;
    const int nvalid = p.T - t0 < kC ? static_cast<int>(p.T - t0) : kC;
    const int64_t pr = static_cast<int64_t>(b) * p.Hv + hv;
    uint8_t *rec = p.rec + (pr * p.nchunks + c) * static_cast<int64_t>(kRecBytes);
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);

    // ---- loads: alpha (tokens past T as 1), q and k (as 0), beta (as 0)
    for (int e = tid; e < kC * 32; e += 256) {
        const int r = e >> 5, pc = e & 31;
        float *dst = G + r * kD + pc * 4;
        if (r < nvalid && !p.scalar_alpha) {
            cp_async16(smem_u32(dst), p.alpha + ((static_cast<int64_t>(b) * p.T + t0 + r) * p.Hv + hv) * kD + pc * 4);
        } else {
            const float a = r < nvalid ? __ldg(p.alpha + (static_cast<int64_t>(b) * p.T + t0 + r) * p.Hv + hv) : 1.f;
            *reinterpret_cast<float4 *>(dst) = make_float4(a, a, a, a);
        }
    }
    for (int e = tid; e < kC * 16; e += 256) {
        const int r = e >> 4, pc = e & 15;
        const uint32_t off = sw256(r, pc);
        if (r < nvalid) {
            const int64_t gi = ((static_cast<int64_t>(b) * p.T + t0 + r) * p.Hqk + hk) * kD + pc * 8;
            cp_async16(sb + PP_QT + off, p.q + gi);
            cp_async16(sb + PP_KT + off, p.k + gi);
        } else {
            *reinterpret_cast<uint4 *>(sm + PP_QT + off) = zero4;
            *reinterpret_cast<uint4 *>(sm + PP_KT + off) = zero4;
        }
    }
    if (tid < kC) beta_s[tid] = tid < nvalid ? __ldg(p.beta + (static_cast<int64_t>(b) * p.T + t0 + tid) * p.Hv + hv) : 0.f;
    if (tid < 4) viol[tid] = 0;
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();

    // ---- G = cumulative log2 alpha per channel (two halves of 32 tokens, then
    // the second half offset by the first); block references R_I = G before
    // block I; e^{g_C} into the record; blocks whose own decay passes 2^kMaxExp2
    {
        const int ch = tid & (kD - 1), h = tid >> 7;
        float run = 0.f;
#pragma unroll 8
        for (int t = 32 * h; t < 32 * h + 32; ++t) {
            run += log2_approx(G[t * kD + ch]);
            G[t * kD + ch] = run;
        }
    }
    __syncthreads();
    {
        const int ch = tid & (kD - 1), h = tid >> 7;
        const float off = G[31 * kD + ch];
#pragma unroll 8
        for (int t = 32 + 16 * h; t < 48 + 16 * h; ++t) G[t * kD + ch] += off;
    }
    __syncthreads();
    if (tid < kD) {
        const int ch = tid;
        const float gc = G[63 * kD + ch];
        gC[ch] = gc;
        reinterpret_cast<float *>(rec + REC_GC)[ch] = exp2_ftz(gc);
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            const float r = I == 0 ? 0.f : G[(16 * I - 1) * kD + ch];
            R[I * kD + ch] = r;
            eR[I * kD + ch] = exp2_ftz(r);
            if (r - G[(16 * I + 15) * kD + ch] > kMaxExp2) viol[I] = 1;
        }
    }
    __syncthreads();

    // ---- decay bound of the chunk: sum over tokens of max_c log alpha (natural log).
    // Warp w: tokens 8w..8w+7; four lanes per token, each over 32 channels
    // 32 (lane % 4) + i, visited from i = lane so that a step reads 32 banks.
    {
        const int t = warp * 8 + (lane >> 2), cb = 32 * (lane & 3);
        float m = -INFINITY;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
            const int ch = cb + ((lane + i) & 31);
            m = fmaxf(m, G[t * kD + ch] - (t > 0 ? G[(t - 1) * kD + ch] : 0.f));
        }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        float part = m;   // then the sum over the warp's 8 tokens
        part += __shfl_xor_sync(0xffffffffu, part, 4);
        part += __shfl_xor_sync(0xffffffffu, part, 8);
        part += __shfl_xor_sync(0xffffffffu, part, 16);
        if (lane == 0) wred[warp] = part;
    }
    // ---- diagonal blocks past the bf16 range, element by element (t >= s in the block)
#pragma unroll 1
    for (int I = 0; I < 4; ++I) {
        if (!viol[I]) continue;
        const int t = 16 * I + (tid >> 4), s = 16 * I + (tid & 15);
        float a = 0.f, pp = 0.f;
        if (s <= t) {
#pragma unroll 4
            for (int ch = 0; ch < kD; ++ch) {
                const float e = exp2_ftz(G[t * kD + ch] - G[s * kD + ch]);
                const float ks = tile_elem(sm + PP_KT, s, ch) * e;
                a = fmaf(tile_elem(sm + PP_KT, t, ch), ks, a);
                pp = fmaf(tile_elem(sm + PP_QT, t, ch), ks, pp);
            }
        }
        fix[(2 * I) * 256 + (tid >> 4) * 16 + (tid & 15)] = s < t ? a : 0.f;
        fix[(2 * I + 1) * 256 + (tid >> 4) * 16 + (tid & 15)] = s <= t ? pp : 0.f;
    }
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < 8; ++w) s += wred[w];
        p.bound[pr * p.nchunks + c] = s * kLn2;
    }

    // ---- per-token operands: Qp, Kl to the record; Qloc (in place of q), Kloc
    #pragma unroll 2
    for (int e = tid; e < kC * 16; e += 256) {
        const int t = e >> 4, pc = e & 15, I = t >> 4;
        const uint32_t off = sw256(t, pc);
        const uint4 qr = *reinterpret_cast<const uint4 *>(sm + PP_QT + off);
        const uint4 kr = *reinterpret_cast<const uint4 *>(sm + PP_KT + off);
        const uint32_t qw[4] = {qr.x, qr.y, qr.z, qr.w}, kw[4] = {kr.x, kr.y, kr.z, kr.w};
        float gr[8], rr[8], gc[8];
        *reinterpret_cast<float4 *>(gr) = *reinterpret_cast<const float4 *>(G + t * kD + pc * 8);
        *reinterpret_cast<float4 *>(gr + 4) = *reinterpret_cast<const float4 *>(G + t * kD + pc * 8 + 4);
        *reinterpret_cast<float4 *>(rr) = *reinterpret_cast<const float4 *>(R + I * kD + pc * 8);
        *reinterpret_cast<float4 *>(rr + 4) = *reinterpret_cast<const float4 *>(R + I * kD + pc * 8 + 4);
        *reinterpret_cast<float4 *>(gc) = *reinterpret_cast<const float4 *>(gC + pc * 8);
        *reinterpret_cast<float4 *>(gc + 4) = *reinterpret_cast<const float4 *>(gC + pc * 8 + 4);
        // end of this token's block: R_{I+1} (g_C for the last block)
        float re[8];
        const float *rn = I < 3 ? R + (I + 1) * kD + pc * 8 : gC + pc * 8;
        *reinterpret_cast<float4 *>(re) = *reinterpret_cast<const float4 *>(rn);
        *reinterpret_cast<float4 *>(re + 4) = *reinterpret_cast<const float4 *>(rn + 4);
        uint32_t oqp[4], okl[4], oql[4], okq[4], okn[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 qf = unpack2(qw[j]), kf = unpack2(kw[j]);
            float e1[2], el[2], eo[2], en[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float gv = gr[2 * j + h];
                e1[h] = exp2_ftz(gv);
                el[h] = exp2_ftz(gc[2 * j + h] - gv);
                eo[h] = exp2_ftz(gv - rr[2 * j + h]);
                en[h] = exp2_ftz(re[2 * j + h] - gv);   // <= 1: the block's end is no later than the token
            }
            oqp[j] = pack2(qf.x * e1[0], qf.y * e1[1]);
            okl[j] = pack2(kf.x * el[0], kf.y * el[1]);
            oql[j] = pack2(qf.x * eo[0], qf.y * eo[1]);
            okq[j] = pack2(kf.x * eo[0], kf.y * eo[1]);
            okn[j] = pack2(kf.x * en[0], kf.y * en[1]);
        }
        *reinterpret_cast<uint4 *>(rec + REC_QP + t * 256 + pc * 16) = make_uint4(oqp[0], oqp[1], oqp[2], oqp[3]);
        *reinterpret_cast<uint4 *>(rec + REC_KL + t * 256 + pc * 16) = make_uint4(okl[0], okl[1], okl[2], okl[3]);
        *reinterpret_cast<uint4 *>(sm + PP_QT + off) = make_uint4(oql[0], oql[1], oql[2], oql[3]);
        *reinterpret_cast<uint4 *>(sm + PP_KL + off) = make_uint4(okq[0], okq[1], okq[2], okq[3]);
        *reinterpret_cast<uint4 *>(sm + PP_KT + off) = make_uint4(okn[0], okn[1], okn[2], okn[3]);
    }
    __syncthreads();

    // ---- A and P by row block I with Kn_I = K (.) 2^{R_I - G} on the key rows s < 16(I+1).
    // The raw k tile now holds Knend = K (.) 2^{R_{J+1} - G} (J the block of s, bounded by 1), so
    // Kn_I = Knend (.) 2^{R_I - R_{J+1}}: the factor is at most 1 before block I and the block's
    // own decay inside it (rows of a block past 2^kMaxExp2 left zero for the element-wise path).
    // All four Kn_I are built at once (into the G tile and the Kn tile); then each warp runs its
    // product tasks of every row block without further barriers, one task per (product, pair of
    // 8-column tiles).  Warp w keeps the A tile pair np = w of every block I >= w in registers
    // until the q/k tiles are free.
    auto kn_base = [](int I) -> uint32_t {   // rows 0..16(I+1)-1 of Kn_I
        return I == 3 ? PP_KN : PP_G + static_cast<uint32_t>(I * (I + 1) / 2) * 16u * 256u;
    };
    // the factors 2^{R_I - R_{J+1}} for the ten (I, J <= I) pairs, per channel, in the G tile's
    // last 8 KB (the Kn_I use its first 24 KB)
    float *fac = reinterpret_cast<float *>(sm + PP_G + 24576);
    for (int e = tid; e < 10 * kD; e += 256) {
        const int pair = e >> 7, ch = e & (kD - 1);
        const int I = pair < 1 ? 0 : (pair < 3 ? 1 : (pair < 6 ? 2 : 3));
        const int J = pair - I * (I + 1) / 2;
        const float rj = J < 3 ? R[(J + 1) * kD + ch] : gC[ch];
        fac[e] = exp2_ftz(R[I * kD + ch] - rj);
    }
    __syncthreads();
    #pragma unroll 2
    for (int e = tid; e < 160 * 16; e += 256) {   // 16 + 32 + 48 + 64 rows
        const int row = e >> 4, pc = e & 15;
        const int I = row < 16 ? 0 : (row < 48 ? 1 : (row < 96 ? 2 : 3));
        const int s = row - 16 * (I * (I + 1) / 2);
        const int J = s >> 4;
        uint4 out = zero4;
        if (!(J == I && viol[I] != 0)) {
            const uint4 kr = *reinterpret_cast<const uint4 *>(sm + PP_KT + sw256(s, pc));
            const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
            float f[8];
            const float *fp = fac + (I * (I + 1) / 2 + J) * kD + pc * 8;
            *reinterpret_cast<float4 *>(f) = *reinterpret_cast<const float4 *>(fp);
            *reinterpret_cast<float4 *>(f + 4) = *reinterpret_cast<const float4 *>(fp + 4);
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 kf = unpack2(kw[j]);
                o[j] = pack2(kf.x * f[2 * j], kf.y * f[2 * j + 1]);
            }
            out = make_uint4(o[0], o[1], o[2], o[3]);
        }
        *reinterpret_cast<uint4 *>(sm + kn_base(I) + sw256(s, pc)) = out;
    }
    __syncthreads();
    float aacc[4][2][4];
#pragma unroll
    for (int I = 0; I < 4; ++I) {
#pragma unroll
        for (int e = 0; e < 8; ++e) aacc[I][e >> 2][e & 3] = 0.f;
        const bool vI = viol[I] != 0;
        const int ntask = 2 * (I + 1);
        if (warp < ntask) {
            const bool is_a = warp <= I;
            const int np = is_a ? warp : warp - (I + 1);
            const uint32_t xa = sb + (is_a ? PP_KL : PP_QT);
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t af[4], bf[4];
                ldsm_x4(af, xa + sw256(16 * I + a_row(lane), 2 * ks + a_ch(lane)));
                ldsm_x4(bf, sb + kn_base(I) + sw256(16 * np + bn_row(lane), 2 * ks + bn_ch(lane)));
                mma16816(acc[0], af, bf[0], bf[1]);
                mma16816(acc[1], af, bf[2], bf[3]);
            }
            if (is_a) {
#pragma unroll
                for (int e = 0; e < 8; ++e) aacc[I][e >> 2][e & 3] = acc[e >> 2][e & 3];
            } else {
                // P rows t = 16I + g (+8), columns s = 16np + 8j + 2t4 (+1), s <= t
#pragma unroll
                for (int j = 0; j < 2; ++j) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int t = 16 * I + g + 8 * hr;
                        const int s = 16 * np + 8 * j + 2 * t4;
                        float v0 = acc[j][2 * hr], v1 = acc[j][2 * hr + 1];
                        if (vI && np == I) {
                            v0 = fix[(2 * I + 1) * 256 + (t & 15) * 16 + (s & 15)];
                            v1 = fix[(2 * I + 1) * 256 + (t & 15) * 16 + ((s + 1) & 15)];
                        }
                        v0 = s <= t ? v0 : 0.f;
                        v1 = s + 1 <= t ? v1 : 0.f;
                        *reinterpret_cast<uint32_t *>(rec + REC_P + t * 128 + s * 2) = pack2(v0, v1);
                    }
                }
            }
        } else if (warp - ntask < 3 - I) {
            // a block (I, np > I) of P above the diagonal blocks: zeros, 16 bytes per lane
            const int np = I + 1 + (warp - ntask);
            const int t = 16 * I + (lane >> 1), s = 16 * np + 8 * (lane & 1);
            *reinterpret_cast<uint4 *>(rec + REC_P + t * 128 + s * 2) = zero4;
        }
    }
    __syncthreads();

    // ---- A into the block-packed solve layout (over the q/k tiles), V into the Kn tile
    float *At = reinterpret_cast<float *>(sm + PP_AT);
    float *Tm = reinterpret_cast<float *>(sm + PP_TM);
#pragma unroll
    for (int I = 0; I < 4; ++I) {
        if (warp <= I) {
            const bool vdiag = warp == I && viol[I] != 0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int t = 16 * I + g + 8 * hr;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int s = 16 * warp + 8 * j + 2 * t4 + h;
                        if (s < t) {
                            const float a = vdiag ? fix[(2 * I) * 256 + (t & 15) * 16 + (s & 15)] : aacc[I][j][2 * hr + h];
                            At[blk(I, warp) * kBlk + (s & 15) * kBS + (t & 15)] = beta_s[t] * a;
                        }
                    }
                }
            }
        }
    }
    for (int e = tid; e < kC * 16; e += 256) {
        const int r = e >> 4, pc = e & 15;
        const uint32_t off = sw256(r, pc);
        if (r < nvalid)
            cp_async16(sb + PP_KN + off, p.v + ((static_cast<int64_t>(b) * p.T + t0 + r) * p.Hv + hv) * kD + pc * 8);
        else
            *reinterpret_cast<uint4 *>(sm + PP_KN + off) = zero4;
    }
    cp_async_commit();
    __syncthreads();

    // ---- T = (I + A)^{-1} (warps 0-3)
    if (warp < 4 && lane < 16) diag_solve(warp, lane, At, Tm);
    __syncthreads();
    if (warp < 4) solve_factors(warp, At, Tm, lane);
    __syncthreads();
    if (warp == 0 || warp == 3)
        solve_column<1>(0, warp == 3 ? 1 : 0, At, Tm, lane);
    else if (warp < 3)
        solve_column<2>(warp, 0, At, Tm, lane);
    __syncthreads();

    // ---- T2 = T diag(beta) in bf16 over the G tile (rows of 64 columns)
    for (int e = tid; e < kC * 8; e += 256) {
        const int t = e >> 3, pc = e & 7, I = t >> 4, J = pc >> 1;
        uint4 out = zero4;
        if (J <= I) {
            const float *src = Tm + blk(I, J) * kBlk + (t & 15) * kBS + (pc & 1) * 8;
            const float *bc = beta_s + pc * 8;
            out = make_uint4(pack2(src[0] * bc[0], src[1] * bc[1]), pack2(src[2] * bc[2], src[3] * bc[3]),
                             pack2(src[4] * bc[4], src[5] * bc[5]), pack2(src[6] * bc[6], src[7] * bc[7]));
        }
        *reinterpret_cast<uint4 *>(sm + PP_T2 + sw128(t, pc)) = out;
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- W = sum_J (T2[:, J] Kloc[J]) (.) e^{R_J} (Kp = Kloc (.) e^{R_J} on block J)
    // and U~ = T2 V: warp w takes columns 16 w .. 16 w + 15 of every row block (the
    // ten nonzero blocks of T2 give each warp the same work).
    {
        float aw[4][2][4], au[4][2][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int e = 0; e < 8; ++e) aw[mt][e >> 2][e & 3] = au[mt][e >> 2][e & 3] = 0.f;
#pragma unroll
        for (int J = 0; J < 4; ++J) {
            uint32_t bk[4], bv[4];
            ldsm_x4_t(bk, sb + PP_KL + sw256(16 * J + bt_row(lane), 2 * warp + bt_ch(lane)));
            ldsm_x4_t(bv, sb + PP_KN + sw256(16 * J + bt_row(lane), 2 * warp + bt_ch(lane)));
            float e[2][2];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int col = 16 * warp + 8 * jj + 2 * t4;
                e[jj][0] = eR[J * kD + col];
                e[jj][1] = eR[J * kD + col + 1];
            }
#pragma unroll
            for (int mt = J; mt < 4; ++mt) {   // T2 is zero above the diagonal blocks
                uint32_t af[4];
                ldsm_x4(af, sb + PP_T2 + sw128(16 * mt + a_row(lane), 2 * J + a_ch(lane)));
                float tw[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                mma16816(tw[0], af, bk[0], bk[1]);
                mma16816(tw[1], af, bk[2], bk[3]);
                mma16816(au[mt][0], af, bv[0], bv[1]);
                mma16816(au[mt][1], af, bv[2], bv[3]);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    aw[mt][jj][0] = fmaf(tw[jj][0], e[jj][0], aw[mt][jj][0]);
                    aw[mt][jj][1] = fmaf(tw[jj][1], e[jj][1], aw[mt][jj][1]);
                    aw[mt][jj][2] = fmaf(tw[jj][2], e[jj][0], aw[mt][jj][2]);
                    aw[mt][jj][3] = fmaf(tw[jj][3], e[jj][1], aw[mt][jj][3]);
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = 16 * warp + 8 * nt + 2 * t4;
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int t = 16 * mt + g + 8 * hr;
                    *reinterpret_cast<uint32_t *>(rec + REC_WN + t * 256 + col * 2) =
                        pack2(-aw[mt][nt][2 * hr], -aw[mt][nt][2 * hr + 1]);
                    *reinterpret_cast<uint32_t *>(rec + REC_UT + t * 256 + col * 2) =
                        pack2(au[mt][nt][2 * hr], au[mt][nt][2 * hr + 1]);
                }
            }
        }
    }
}

// Chain shared memory: two stages of a chunk record (tiles swizzled), the bf16
// copy of the state [dk][dv] and the bf16 U [tokens][dv].
constexpr uint32_t CH_SB = 2 * kRecBytes;
constexpr uint32_t CH_UB = CH_SB + kD * kD * 2;
constexpr uint32_t CH_MISC = CH_UB + kC * kD * 2;
constexpr uint32_t kChainSmem = CH_MISC + 64;

// State scan of one (batch, value head, segment).  Warp w holds state rows
// dk = 16w .. 16w+15 (all 128 dv columns) as MMA accumulator fragments.  Per
// chunk, with the state S entering it:
//   A: the bf16 copy of S to shared memory;
//   B: U = U~ + (-W) S and Y = Qp S (warp w: tokens 16 (w & 3), columns 64 (w >> 2));
//   C: Y += P U, y stored; S = diag(e^{g_C}) S + Kl^T U into the fragments.
// Chunk records stream in with asynchronous copies one chunk ahead.
// WITH_Y = false (no y requested, only states): the Y products are skipped.
template <bool WITH_Y>
__global__ void __launch_bounds__(256, 1) cw_chain_kernel(const CwDev p) {
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
    int *misc = reinterpret_cast<int *>(sm + CH_MISC);
    const bool exact = p.exact_flag != nullptr && cw_head_split(p.exact_flag, pr, p.nseg);
    // transition pass: heads that need the split, segments whose maps are used
    if (p.pass == 1 && (!exact || seg == p.nseg - 1 || (kind == 1 && seg == 0))) return;

    // Warm-up window: walk back from the segment start until the decay bound
    // reaches exp(log_eps) (start there from a zero state); at chunk 0 or past
    // the window limit, start at chunk 0 from S0 (exact).  The transition pass
    // and the heads that take the split start every segment at its first chunk.
    if (tid == 0) {
        int cw = 0;
        if (p.pass == 1 || exact) {
            cw = c_begin;
        } else if (seg > 0) {
            float acc = 0.f;
            for (int m = 1;; ++m) {
                const int cc = c_begin - m;
                if (cc < 0 || m > p.max_warmup) break;
                acc += p.bound[static_cast<int64_t>(pr) * p.nchunks + cc];
                if (acc <= p.log_eps) {
                    cw = cc;
                    break;
                }
            }
        }
        misc[0] = cw;
    }
    __syncthreads();
    const int c_w = misc[0];

    float S[16][4];
    {
        // the starting state: S0 at chunk 0, a combined entering state for a split head,
        // the identity for a kind-1 transition, else zero
        const float *s0 = nullptr;
        if (kind == 1)
            s0 = nullptr;
        else if (c_w == 0)
            s0 = p.S0 ? p.S0 + static_cast<int64_t>(pr) * kD * kD : nullptr;
        else if (p.pass == 0 && exact)
            s0 = p.seg_state + ((static_cast<int64_t>(pr) * p.nseg + seg) * 3 + 2) * kD * kD;
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

    const uint8_t *recs = p.rec + static_cast<int64_t>(pr) * p.nchunks * kRecBytes;
    auto load_chunk = [&](int cc, int stage) {
        const uint8_t *src = recs + static_cast<int64_t>(cc) * kRecBytes;
        const uint32_t dst = sb + stage * kRecBytes;
        for (int e = tid; e < 4 * 1024 + 512 + 32; e += 256) {
            if (e < 4096) {
                const int tile = e >> 10, r = (e >> 4) & 63, pc = e & 15;
                cp_async16(dst + tile * 16384 + sw256(r, pc), src + tile * 16384 + r * 256 + pc * 16);
            } else if (e < 4608) {
                const int e2 = e - 4096, r = e2 >> 3, pc = e2 & 7;
                cp_async16(dst + REC_P + sw128(r, pc), src + REC_P + r * 128 + pc * 16);
            } else {
                const int e3 = e - 4608;
                cp_async16(dst + REC_GC + e3 * 16, src + REC_GC + e3 * 16);
            }
        }
        cp_async_commit();
    };

    const int mt = warp & 3, nh = warp >> 2;
    if (c_w < c_end) load_chunk(c_w, 0);
#pragma unroll 1
    for (int cc = c_w; cc < c_end; ++cc) {
        const int st = (cc - c_w) & 1;
        const uint32_t stg = sb + st * kRecBytes;
        const uint8_t *stp = sm + st * kRecBytes;
        if (p.state_out && p.pass == 0 && cc >= c_begin) {
            __nv_bfloat16 *so = p.state_out + (static_cast<int64_t>(pr) * p.nchunks + cc) * kD * kD;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const int r = 16 * warp + g, col = 8 * nt + 2 * t4;
                *reinterpret_cast<uint32_t *>(so + r * kD + col) = pack2(S[nt][0], S[nt][1]);
                *reinterpret_cast<uint32_t *>(so + (r + 8) * kD + col) = pack2(S[nt][2], S[nt][3]);
            }
        }
        // A: bf16 copy of the state
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int r = 16 * warp + g;
            *reinterpret_cast<uint32_t *>(sm + CH_SB + sw256(r, nt) + 4 * t4) = pack2(S[nt][0], S[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + CH_SB + sw256(r + 8, nt) + 4 * t4) = pack2(S[nt][2], S[nt][3]);
        }
        cp_async_wait_all();
        __syncthreads();
        if (cc + 1 < c_end) load_chunk(cc + 1, st ^ 1);

        // B: U = U~ + (-W) S, Y = Qp S
        float u[8][4], ys[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int t = 16 * mt + g + 8 * hr;
                const float2 f = kind == 1 ? make_float2(0.f, 0.f)   // values zero: U~ = 0
                    : unpack2(*reinterpret_cast<const uint32_t *>(stp + REC_UT + sw256(t, 8 * nh + nt) + 4 * t4));
                u[nt][2 * hr] = f.x;
                u[nt][2 * hr + 1] = f.y;
                ys[nt][2 * hr] = 0.f;
                ys[nt][2 * hr + 1] = 0.f;
            }
        }
#pragma unroll 2
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t aw[4], aq[4] = {0u, 0u, 0u, 0u};
            ldsm_x4(aw, stg + REC_WN + sw256(16 * mt + a_row(lane), 2 * kk + a_ch(lane)));
            if constexpr (WITH_Y) ldsm_x4(aq, stg + REC_QP + sw256(16 * mt + a_row(lane), 2 * kk + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bs[4];
                ldsm_x4_t(bs, sb + CH_SB + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(u[2 * np], aw, bs[0], bs[1]);
                mma16816(u[2 * np + 1], aw, bs[2], bs[3]);
                if constexpr (WITH_Y) {
                    mma16816(ys[2 * np], aq, bs[0], bs[1]);
                    mma16816(ys[2 * np + 1], aq, bs[2], bs[3]);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int t = 16 * mt + g;
            *reinterpret_cast<uint32_t *>(sm + CH_UB + sw256(t, 8 * nh + nt) + 4 * t4) = pack2(u[nt][0], u[nt][1]);
            *reinterpret_cast<uint32_t *>(sm + CH_UB + sw256(t + 8, 8 * nh + nt) + 4 * t4) = pack2(u[nt][2], u[nt][3]);
        }
        __syncthreads();

        // C: Y += P U (P is zero above the diagonal blocks)
#pragma unroll 1
        for (int kk = 0; WITH_Y && kk <= mt; ++kk) {
            uint32_t ap[4];
            ldsm_x4(ap, stg + REC_P + sw128(16 * mt + a_row(lane), 2 * kk + a_ch(lane)));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bu[4];
                ldsm_x4_t(bu, sb + CH_UB + sw256(16 * kk + bt_row(lane), 8 * nh + 2 * np + bt_ch(lane)));
                mma16816(ys[2 * np], ap, bu[0], bu[1]);
                mma16816(ys[2 * np + 1], ap, bu[2], bu[3]);
            }
        }
        if (WITH_Y && cc >= c_begin) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int64_t t = static_cast<int64_t>(cc) * kC + 16 * mt + g + 8 * hr;
                if (t < p.T) {
                    __nv_bfloat16 *yr = p.y + ((static_cast<int64_t>(b) * p.T + t) * p.Hv + hv) * kD + 64 * nh + 2 * t4;
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
                        *reinterpret_cast<uint32_t *>(yr + 8 * nt) = pack2(ys[nt][2 * hr], ys[nt][2 * hr + 1]);
                }
            }
        }
        // S = diag(e^{g_C}) S + Kl^T U
        {
            const float *gce = reinterpret_cast<const float *>(stp + REC_GC);
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
            uint32_t ak[4];
            ldsm_x4_t(ak, stg + REC_KL + sw256(16 * kk + at_row(lane), 2 * warp + at_ch(lane)));
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t bu[4];
                ldsm_x4_t(bu, sb + CH_UB + sw256(16 * kk + bt_row(lane), 2 * np + bt_ch(lane)));
                mma16816(S[2 * np], ak, bu[0], bu[1]);
                mma16816(S[2 * np + 1], ak, bu[2], bu[3]);
            }
        }
    }

    float *s_end = nullptr;   // where this run's final state goes
    if (p.pass == 1)
        s_end = p.seg_state + ((static_cast<int64_t>(pr) * p.nseg + seg) * 3 + kind) * kD * kD;
    else if (c_end == p.nchunks)
        s_end = p.S_T;
    if (s_end) {
        float *so = p.pass == 1 ? s_end : s_end + static_cast<int64_t>(pr) * kD * kD;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int r = 16 * warp + g, col = 8 * nt + 2 * t4;
            *reinterpret_cast<float2 *>(so + r * kD + col) = make_float2(S[nt][0], S[nt][1]);
            *reinterpret_cast<float2 *>(so + (r + 8) * kD + col) = make_float2(S[nt][2], S[nt][3]);
        }
    }
}

cudaError_t set_cw_attributes() {
    static cudaError_t result = [] {
        cudaError_t e = cudaFuncSetAttribute(cw_prepass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kPrepassSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(cw_chain_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kChainSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(cw_chain_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kChainSmem));
        return e;
    }();
    return result;
}

}  // namespace

size_t chunked_cw_ops_bytes(int64_t B, int64_t T, int Hv) {
    const int64_t nchunks = (T + kC - 1) / kC;
    return static_cast<size_t>(B) * Hv * nchunks * (kRecBytes + sizeof(float));
}

cudaError_t launch_chunked_cw(const ChunkedCwParams &p, cudaStream_t stream, int num_sms) {
    if (p.d != kD) return cudaErrorInvalidValue;
    const int64_t nchunks = (p.T + kC - 1) / kC;
    const int64_t pairs = p.B * p.Hv;
    if (nchunks <= 0 || pairs <= 0) return cudaSuccess;
    if (nchunks > 0x7fffffffLL || pairs > 0x7fffffffLL || p.B * nchunks * p.Hv > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    int P = plan_segments(pairs, nchunks, num_sms, p.segments);
    const int64_t len = (nchunks + P - 1) / P;
    P = static_cast<int>((nchunks + len - 1) / len);
    if (pairs * P > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t e = set_cw_attributes();
    if (e != cudaSuccess) return e;
    CwDev dv{};
    dv.T = p.T;
    dv.B = static_cast<int>(p.B);
    dv.Hqk = p.Hqk;
    dv.Hv = p.Hv;
    dv.group = p.group;
    dv.nchunks = static_cast<int>(nchunks);
    dv.seg_chunks = static_cast<int>(len);
    dv.max_warmup = p.max_warmup_chunks;
    dv.log_eps = p.log_eps;
    dv.q = static_cast<const __nv_bfloat16 *>(p.q);
    dv.k = static_cast<const __nv_bfloat16 *>(p.k);
    dv.v = static_cast<const __nv_bfloat16 *>(p.v);
    dv.alpha = p.alpha;
    dv.beta = p.beta;
    dv.S0 = p.S0;
    dv.y = static_cast<__nv_bfloat16 *>(p.y);
    dv.S_T = p.S_T;
    dv.rec = p.ops;
    dv.bound = reinterpret_cast<float *>(p.ops + static_cast<size_t>(pairs) * nchunks * kRecBytes);
    dv.scalar_alpha = p.scalar_alpha ? 1 : 0;
    dv.state_out = static_cast<__nv_bfloat16 *>(p.state_out);
    dv.nseg = P;
    dv.pass = 0;
    dv.exact_flag = nullptr;
    dv.seg_state = nullptr;
    cw_prepass_kernel<<<static_cast<unsigned>(p.B * nchunks * p.Hv), 256, kPrepassSmem, stream>>>(dv);
    // Exact sequence split for the heads whose segments reach no window (as the
    // scalar prefill does): plan, transition runs, combine, then the output pass.
    if (p.exact_flag && p.seg_state && takes_exact_split(pairs, nchunks, P, kD, p.seg_state_bytes)) {
        dv.exact_flag = p.exact_flag;
        dv.seg_state = p.seg_state;
        const int nplan = static_cast<int>(pairs * (P - 1));
        cw_plan_kernel<<<static_cast<unsigned>((nplan + 127) / 128), 128, 0, stream>>>(dv, p.exact_flag);
        dv.pass = 1;
        cw_chain_kernel<false><<<static_cast<unsigned>(2 * pairs * P), 256, kChainSmem, stream>>>(dv);
        e = launch_segment_combine(p.exact_flag, p.seg_state, pairs, P, kD, stream);
        if (e != cudaSuccess) return e;
        dv.pass = 0;
    }
    if (p.y)
        cw_chain_kernel<true><<<static_cast<unsigned>(pairs * P), 256, kChainSmem, stream>>>(dv);
    else
        cw_chain_kernel<false><<<static_cast<unsigned>(pairs * P), 256, kChainSmem, stream>>>(dv);
    return cudaGetLastError();
}

}  // namespace gdn
