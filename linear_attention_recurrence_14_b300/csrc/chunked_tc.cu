// Chunked tensor-core prefill of the gated delta recurrence (bf16 inputs,
// fp32 state), one fused kernel for sm_103a: TMA loads, tcgen05 MMAs with
// TMEM accumulators, the state carried in fp32 registers across chunks.
//
// Algebra (Qwen3.8-Next reading notes, section 2.1 "Gated DeltaNet": the
// four-line recurrence and its transition-matrix form
// S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, unrolled
// over a chunk of C = 64 tokens).  With S0 the state entering the chunk, local
// positions i, j in [0, 64) and g_i = sum_{s <= i} log alpha_s, gamma_i = e^{g_i}:
//   A_ij = beta_i e^{g_i - g_j} (k_i . k_j)   (j < i),   T = (I + A)^{-1}
//   W    = T diag(beta gamma) K,                 U~ = T diag(beta) V
//   U    = U~ - W S0                             (the per-token writes u_i)
//   P_ij = e^{g_i - g_j} (q_i . k_j)   (j <= i)
//   Y    = diag(gamma) Q S0 + P U                (y_i = S_i^T q_i)
//   S_C  = gamma_C S0 + K~^T U,   K~_i = e^{g_C - g_i} k_i
// Every contraction runs as an M = 128 tcgen05 MMA in the value-major
// (transposed) orientation, so the state's value dimension is the TMEM lane:
//   Gram   [K;Q] K^T            -> KK^T (lanes 0-63), QK^T (lanes 64-127)
//   W^T  = K^T (T diag(beta gamma))^T,   U~^T = V^T (T diag(beta))^T
//   U^T  = U~^T + S^T (-W)^T              (accumulated onto U~^T)
//   Y^T  = S^T Q~^T + U^T P^T             (Q~ = diag(gamma) Q)
//   dS^T = U^T K~,   S^T <- gamma_C S^T + dS^T   (fp32, in registers)
// S^T and U^T are fed to the tensor core from TMEM as bf16 (A operand).
//
// Work item: one (batch, value head, segment of chunks).  A segment that does
// not start at token 0 rebuilds its entering state from a zero state over a
// warm-up window of preceding chunks chosen so that the product of the decay
// gates over the window is below exp(log_eps); with unit keys and beta in
// [0, 1] each step is a contraction of norm <= alpha_t, which bounds the
// difference to the exact state by that factor times the state norm.
//
// Warp roles (512 threads):
//   warp 0        TMA producer (one thread): K, Q, V tiles of each chunk
//   warp 1        MMA issuer (one thread); owns the TMEM allocation
//   warps 2-3     gates of each chunk (one chunk ahead of the local warpgroup)
//   warps 4-7     "local" warpgroup: gated Gram products, the triangular
//                 solve, the T, P and -W operands (Q~, K~ on the exact path)
//   warps 8-15    "chain" warpgroups: the fp32 state (dv lane x dk half),
//                 U conversion, state update, y output
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kC = 64;          // chunk length
constexpr int kStages = 3;
constexpr int kThreads = 512;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s

// Shared-memory layout (offsets from a 1024-byte aligned base).  Operand
// tiles use the 128-byte swizzle: rows of 128 bytes (64 bf16), 16-byte chunk
// c of row r stored at chunk position c ^ (r & 7).
constexpr uint32_t kKQBytes = 2 * 128 * 128;  // [kb][128 rows][64]: K rows 0-63, Q rows 64-127
constexpr uint32_t kVWBytes = 2 * 64 * 128;   // [kb][64 rows][64]: V, later -W
constexpr uint32_t kPBytes = 64 * 128;        // [64 rows][64]
constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_VW = OFF_KQ + kStages * kKQBytes;
constexpr uint32_t OFF_P = OFF_VW + kStages * kVWBytes;
constexpr uint32_t OFF_T1 = OFF_P + kStages * kPBytes;
constexpr uint32_t OFF_T2 = OFF_T1 + 64 * 128;
// Solve matrices, block-packed: the ten 16 x 16 blocks (I, J), J <= I, of a
// 64 x 64 lower-triangular matrix, block (I, J) at index I (I + 1) / 2 + J,
// rows of kBS floats (the padding makes the warp-MMA fragment loads
// conflict-free).  A is stored column-major within a block, T row-major.
constexpr int kBS = 24;
constexpr int kBlk = 16 * kBS;
constexpr uint32_t OFF_AT = OFF_T2 + 64 * 128;
constexpr uint32_t OFF_TM = OFF_AT + 10 * kBlk * 4;
constexpr uint32_t OFF_R = OFF_TM + 10 * kBlk * 4;      // 3 warps x [16][kBS]
constexpr uint32_t OFF_GATES = OFF_R + 3 * kBlk * 4;
// gates, double-buffered by chunk parity: g, u = gamma, w = 1/gamma, beta,
// beta gamma (64 floats each), misc (64)
constexpr int kGateFloats = 6 * 64;
constexpr uint32_t OFF_CHAIN = OFF_GATES + 2 * kGateFloats * 4;
// ring of 4 chunks: lambda[64], gamma[64], gamma_C for the chain warpgroups
constexpr int kChainFloats = 132;
constexpr int kChainSlots = 4;
constexpr uint32_t OFF_BAR = OFF_CHAIN + kChainSlots * kChainFloats * 4;
constexpr int kNumBars = 22;
constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr uint32_t kSmemUsed = OFF_MISC + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

enum Bar {
    B_FULL = 0,           // + stage: TMA landed
    B_EMPTY = B_FULL + kStages,  // + stage: all MMAs reading the stage are done
    B_GRAM = B_EMPTY + kStages,  // + GW buffer: Gram product in TMEM (one barrier per buffer, so
                                 //   two Grams issued back to back cannot alias one phase)
    B_TREADY = B_GRAM + 2,  // T1, T2, P, Q~ written; Gram region read (local, 128 arrivals)
    B_WU,                 // W^T and U~^T in TMEM
    B_OPS,                // -W, K~ written (local, 128 arrivals)
    B_SREADY,             // S^T bf16 in TMEM (chain, 256 arrivals)
    B_UFULL,              // U^T fp32 in TMEM
    B_USMEM,              // U^T bf16 packed in TMEM (chain, 256 arrivals)
    B_DFULL,              // dS^T in TMEM
    B_YFULL,              // Y^T in TMEM
    B_YFREE,              // Y^T read (chain, 256 arrivals)
    B_FINAL,              // every MMA issued is complete
    B_GFULL,              // + buffer: gates of a chunk written (gate warps, 64 arrivals)
    B_GEMPTY = B_GFULL + 2,  // + buffer: gates of a chunk consumed (local, 128 arrivals)
};
static_assert(B_GEMPTY + 2 == kNumBars, "barrier count");

struct Misc {
    uint32_t tmem_base;
    int abort;
    int c_w;
    int dec;
    float wsum[8];
};

// TMEM columns (512 allocated).  S^T bf16 is double-buffered: Y^T of chunk j
// reads the state entering chunk j after the chain has produced the next one.
constexpr uint32_t TM_GW = 0;     // 2 x 64: Gram, then W^T
constexpr uint32_t TM_ZU = 128;   // 64: U~^T, accumulated to U^T; bf16 U^T packed in place
constexpr uint32_t TM_Y = 192;    // 64: Y^T
constexpr uint32_t TM_D = 256;    // 128: dS^T
constexpr uint32_t TM_SB = 384;   // 2 x 64: S^T bf16 packed

struct Dev {
    int64_t T;
    int B, Hqk, Hv, group, d;
    int nchunks, seg_chunks, nseg, max_warmup;
    float log_eps;
    const float *alpha, *beta, *S0;
    __nv_bfloat16 *y;
    float *S_T;
    uint32_t *status;
};

__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t parity, volatile int *abort, uint32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(status, kDevTimeout);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (teardown).
__device__ __forceinline__ void bwait_teardown(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

// All lanes of the warp agree: true only if every lane's wait succeeded.
__device__ __forceinline__ bool warp_ok(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t lane_addr(uint32_t base, uint32_t quadrant, uint32_t col) {
    return base + ((quadrant * 32u) << 16) + col;
}

// Byte offset of element (row, col) of a 128-byte-swizzled bf16 tile with 64 columns.
__device__ __forceinline__ uint32_t sw128_elem(int row, int col) {
    return static_cast<uint32_t>(row) * 128u + ((static_cast<uint32_t>((col >> 3) ^ (row & 7))) << 4) +
           static_cast<uint32_t>(col & 7) * 2u;
}

__constant__ int kBlkIdx[4][4] = {{0, 0, 0, 0}, {1, 2, 0, 0}, {3, 4, 5, 0}, {6, 7, 8, 9}};

// Chunks whose total log decay is at least this use the factored gates.
constexpr float kFastLogDecay = -40.f;

__device__ __forceinline__ uint32_t f2tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// d (16 x 8, fp32) += a (16 x 8, tf32, row) * b (8 x 8, tf32, col): one warp.
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Off-diagonal blocks of block column J of T = (I + A)^{-1} (one warp):
// T_IJ = -T_II R, R = sum_{K=J}^{I-1} A_IK T_KJ, for I = J+1..3, with tf32 warp
// MMAs (m16n8k8, fp32 accumulation; fp32 operands are passed as is, the
// tensor core reads their tf32 part).  Writes T_IJ as fp32 (row-major block)
// and as bf16 T1 = T diag(beta gamma), T2 = T diag(beta).
template <int J>
__device__ __forceinline__ void merge_column(const float *At, float *Tm, float *Rw, uint8_t *t1b, uint8_t *t2b,
                                             const float *s_b, const float *s_bu, int lane) {
    const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int I = J + 1; I < 4; ++I) {
        float acc[3][2][4];
#pragma unroll
        for (int K = 0; K < 3; ++K)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[K][nt][e] = 0.f;
#pragma unroll
        for (int K = J; K < I; ++K) {
            const float *Ab = At + (I * (I + 1) / 2 + K) * kBlk;   // A[r][k] at k*kBS + r
            const float *Bb = Tm + (K * (K + 1) / 2 + J) * kBlk;   // T[k][n] at k*kBS + n
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int k0 = 8 * ks;
                const uint32_t a0 = __float_as_uint(Ab[(k0 + t4) * kBS + gq]);
                const uint32_t a1 = __float_as_uint(Ab[(k0 + t4) * kBS + gq + 8]);
                const uint32_t a2 = __float_as_uint(Ab[(k0 + t4 + 4) * kBS + gq]);
                const uint32_t a3 = __float_as_uint(Ab[(k0 + t4 + 4) * kBS + gq + 8]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    mma_tf32(acc[K - J][nt], a0, a1, a2, a3, __float_as_uint(Bb[(k0 + t4) * kBS + 8 * nt + gq]),
                             __float_as_uint(Bb[(k0 + t4 + 4) * kBS + 8 * nt + gq]));
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float c[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) c[e] = acc[0][nt][e] + acc[1][nt][e] + acc[2][nt][e];
            *reinterpret_cast<float2 *>(Rw + gq * kBS + 8 * nt + 2 * t4) = make_float2(c[0], c[1]);
            *reinterpret_cast<float2 *>(Rw + (gq + 8) * kBS + 8 * nt + 2 * t4) = make_float2(c[2], c[3]);
        }
        __syncwarp();
        float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const float *Td = Tm + (I * (I + 1) / 2 + I) * kBlk;       // T[r][k] at r*kBS + k
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int k0 = 8 * ks;
            const uint32_t a0 = __float_as_uint(Td[gq * kBS + k0 + t4]);
            const uint32_t a1 = __float_as_uint(Td[(gq + 8) * kBS + k0 + t4]);
            const uint32_t a2 = __float_as_uint(Td[gq * kBS + k0 + t4 + 4]);
            const uint32_t a3 = __float_as_uint(Td[(gq + 8) * kBS + k0 + t4 + 4]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
                mma_tf32(d[nt], a0, a1, a2, a3, __float_as_uint(Rw[(k0 + t4) * kBS + 8 * nt + gq]),
                         __float_as_uint(Rw[(k0 + t4 + 4) * kBS + 8 * nt + gq]));
        }
        float *Tb = Tm + (I * (I + 1) / 2 + J) * kBlk;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int cn = 8 * nt + 2 * t4;
            const int C = 16 * J + cn;
            const float sa0 = s_bu[C], sa1 = s_bu[C + 1], sb0 = s_b[C], sb1 = s_b[C + 1];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = gq + 8 * hr;
                const float v0 = -d[nt][2 * hr], v1 = -d[nt][2 * hr + 1];
                *reinterpret_cast<float2 *>(Tb + r * kBS + cn) = make_float2(v0, v1);
                const uint32_t off = sw128_elem(16 * I + r, C);
                *reinterpret_cast<uint32_t *>(t1b + off) = pack_bf16(v0 * sa0, v1 * sa1);
                *reinterpret_cast<uint32_t *>(t2b + off) = pack_bf16(v0 * sb0, v1 * sb1);
            }
        }
        __syncwarp();
    }
}

// bf16 T1, T2 of the four diagonal blocks from their fp32 copies (one warp).
__device__ __forceinline__ void diag_to_bf16(const float *Tm, uint8_t *t1b, uint8_t *t2b, const float *s_b,
                                             const float *s_bu, int lane) {
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int e = lane + 32 * u;             // 512 column pairs
        const int blk = e >> 7, r = (e >> 3) & 15, cp = e & 7;
        const int C = 16 * blk + 2 * cp;
        const float2 v = *reinterpret_cast<const float2 *>(Tm + (blk * (blk + 1) / 2 + blk) * kBlk + r * kBS + 2 * cp);
        const uint32_t off = sw128_elem(16 * blk + r, C);
        *reinterpret_cast<uint32_t *>(t1b + off) = pack_bf16(v.x * s_bu[C], v.y * s_bu[C + 1]);
        *reinterpret_cast<uint32_t *>(t2b + off) = pack_bf16(v.x * s_b[C], v.y * s_b[C + 1]);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    gdn_chunked_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const Dev p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    Misc *misc = reinterpret_cast<Misc *>(sm + OFF_MISC);
    volatile int *abort_flag = &misc->abort;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    const int pairs = p.B * p.Hv;
    const int seg = blockIdx.x / pairs;
    const int pr = blockIdx.x % pairs;
    const int b = pr / p.Hv;
    const int hv = pr % p.Hv;
    const int hk = hv / p.group;
    const int c_begin = seg * p.seg_chunks;
    const int c_end = min(p.nchunks, c_begin + p.seg_chunks);
    const bool last_seg = seg == p.nseg - 1;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars[B_FULL + s], 1);
            mbar_init(&bars[B_EMPTY + s], 1);
        }
        mbar_init(&bars[B_GRAM + 0], 1);
        mbar_init(&bars[B_GRAM + 1], 1);
        mbar_init(&bars[B_TREADY], 128);
        mbar_init(&bars[B_WU], 1);
        mbar_init(&bars[B_OPS], 128);
        mbar_init(&bars[B_SREADY], 256);
        mbar_init(&bars[B_UFULL], 1);
        mbar_init(&bars[B_USMEM], 256);
        mbar_init(&bars[B_DFULL], 1);
        mbar_init(&bars[B_YFULL], 1);
        mbar_init(&bars[B_YFREE], 256);
        mbar_init(&bars[B_FINAL], 1);
        for (int e = 0; e < 2; ++e) {
            mbar_init(&bars[B_GFULL + e], 64);
            mbar_init(&bars[B_GEMPTY + e], 128);
        }
        misc->abort = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(&misc->tmem_base, 512);
        tmem_relinquish();
    }

    // Warm-up window of this segment (warps 4-11): walk back from the segment
    // start, eight chunks per round, until the decay over the window reaches
    // exp(log_eps), chunk 0 is reached (exact start from S0) or the window
    // limit is hit (exact restart from token 0).
    if (tid == 128 && seg == 0) misc->c_w = 0;
    if (warp >= 4 && warp < 12 && seg > 0) {
        const int gw = warp - 4;
        float acc = 0.f;
        for (int r = 0;; ++r) {
            const int m = r * 8 + gw + 1;
            const int cc = c_begin - m;
            float part = 0.f;
            if (cc >= 0 && m <= p.max_warmup) {
                const int64_t t = static_cast<int64_t>(cc) * kC + lane;
                const float *al = p.alpha + (static_cast<int64_t>(b) * p.T + t) * p.Hv + hv;
                part = logf(__ldg(al)) + logf(__ldg(al + 32 * static_cast<int64_t>(p.Hv)));
            }
            part = warp_sum(part);
            if (lane == 0) misc->wsum[gw] = part;
            named_bar(3, 256);
            if (tid == 128) {
                int dec = -1;
                for (int w = 0; w < 8; ++w) {
                    const int mm = r * 8 + w + 1;
                    if (c_begin - mm < 0 || mm > p.max_warmup) {
                        dec = 0;
                        break;
                    }
                    acc += misc->wsum[w];
                    if (acc <= p.log_eps) {
                        dec = c_begin - mm;
                        break;
                    }
                    if (c_begin - mm == 0) {
                        dec = 0;
                        break;
                    }
                }
                misc->dec = dec;
            }
            named_bar(3, 256);
            const int dec = misc->dec;
            if (dec >= 0) {
                if (tid == 128) misc->c_w = dec;
                break;
            }
        }
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = misc->tmem_base;
    const int c_w = misc->c_w;
    const int n = c_end - c_w;
    const bool use_s0 = c_w == 0 && p.S0 != nullptr;

    const uint32_t smb = smem_u32(sm);
    auto kq_addr = [&](int s) { return smb + OFF_KQ + s * kKQBytes; };
    auto vw_addr = [&](int s) { return smb + OFF_VW + s * kVWBytes; };
    auto p_addr = [&](int s) { return smb + OFF_P + s * kPBytes; };

    uint32_t loads_issued[kStages] = {0, 0, 0};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int j = 0; j < n; ++j) {
                const int s = j % kStages;
                const uint32_t ph = (j / kStages) & 1;
                if (!bwait(&bars[B_EMPTY + s], ph ^ 1, abort_flag, p.status)) break;
                const int t0 = (c_w + j) * kC;
                mbar_arrive_expect_tx(&bars[B_FULL + s], kKQBytes + kVWBytes);
                uint8_t *kq = sm + OFF_KQ + s * kKQBytes;
                uint8_t *vw = sm + OFF_VW + s * kVWBytes;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_4d(kq + kb * 16384, &tm_k, &bars[B_FULL + s], kb * 64, hk, t0, b);
                    tma_load_4d(kq + kb * 16384 + 8192, &tm_q, &bars[B_FULL + s], kb * 64, hk, t0, b);
                    tma_load_4d(vw + kb * 8192, &tm_v, &bars[B_FULL + s], kb * 64, hv, t0, b);
                }
                loads_issued[s] = j + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_KK = idesc_bf16(128, 64, false, false);   // A, B K-major
            constexpr uint32_t ID_MK = idesc_bf16(128, 64, true, false);    // A MN-major
            constexpr uint32_t ID_TS = idesc_bf16(128, 64, false, false);   // A in TMEM, B K-major
            constexpr uint32_t ID_TD = idesc_bf16(128, 128, false, true);   // A in TMEM, B MN-major
            const uint32_t t1 = smb + OFF_T1, t2 = smb + OFF_T2;
            auto gram = [&](int j) {
                const uint32_t base = kq_addr(j % kStages);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint64_t d = sw128_desc(base + off, 16, 1024);
                    mma_bf16(tb + TM_GW + (j & 1) * 64, d, d, ID_KK, kk > 0);
                }
            };
            auto wu = [&](int j) {
                const int s = j % kStages;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t a = sw128_desc(kq_addr(s) + kk * 2048, 16384, 1024);
                    mma_bf16(tb + TM_GW + (j & 1) * 64, a, sw128_desc(t1 + kk * 32, 16, 1024), ID_MK, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t a = sw128_desc(vw_addr(s) + kk * 2048, 8192, 1024);
                    mma_bf16(tb + TM_ZU, a, sw128_desc(t2 + kk * 32, 16, 1024), ID_MK, kk > 0);
                }
            };
            bool ok = true;
            do {
                if (!(ok = bwait(&bars[B_FULL + 0], 0, abort_flag, p.status))) break;
                tc_fence_after();
                gram(0);
                mma_commit(&bars[B_GRAM + 0]);
                if (n > 1) {
                    if (!(ok = bwait(&bars[B_FULL + 1 % kStages], (1 / kStages) & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    gram(1);
                    mma_commit(&bars[B_GRAM + 1]);
                }
                if (!(ok = bwait(&bars[B_TREADY], 0, abort_flag, p.status))) break;
                tc_fence_after();
                wu(0);
                mma_commit(&bars[B_WU]);
                for (int j = 0; j < n && ok; ++j) {
                    const int s = j % kStages;
                    const uint32_t zu = tb + TM_ZU;
                    const uint32_t sb = tb + TM_SB + (j & 1) * 64;
                    if (!(ok = bwait(&bars[B_OPS], j & 1, abort_flag, p.status))) break;
                    if (!(ok = bwait(&bars[B_SREADY], j & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    // U^T = U~^T + S^T (-W)^T
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t bd = sw128_desc(vw_addr(s) + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
                        mma_bf16_ts(zu, sb + kk * 8, bd, ID_TS, 1);
                    }
                    mma_commit(&bars[B_UFULL]);
                    // Gram of chunk j+2 into the GW buffer W^T(j) occupied (read before
                    // OPS(j)); it runs while the chain converts U^T, before MMA2 is issued.
                    if (j + 2 < n) {
                        const int s2 = (j + 2) % kStages;
                        if (!(ok = bwait(&bars[B_FULL + s2], ((j + 2) / kStages) & 1, abort_flag, p.status))) break;
                        tc_fence_after();
                        gram(j + 2);
                        mma_commit(&bars[B_GRAM + (j & 1)]);
                    }
                    if (!(ok = bwait(&bars[B_USMEM], j & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    // dS^T = U^T K~   (U^T bf16: tokens 0-31 at columns 0-15, 32-63 at 32-47)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = sw128_desc(kq_addr(s) + kk * 2048, 16384, 1024);
                        mma_bf16_ts(tb + TM_D, zu + kk * 8 + (kk >= 2 ? 16 : 0), bd, ID_TD, kk > 0);
                    }
                    mma_commit(&bars[B_DFULL]);
                    if (j > 0 && !(ok = bwait(&bars[B_YFREE], (j - 1) & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    // Y^T = S^T Q~^T + U^T P^T
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t bd =
                            sw128_desc(kq_addr(s) + (kk >> 2) * 16384 + 8192 + (kk & 3) * 32, 16, 1024);
                        mma_bf16_ts(tb + TM_Y, sb + kk * 8, bd, ID_TS, kk > 0);
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = sw128_desc(p_addr(s) + kk * 32, 16, 1024);
                        mma_bf16_ts(tb + TM_Y, zu + kk * 8 + (kk >= 2 ? 16 : 0), bd, ID_TS, 1);
                    }
                    mma_commit(&bars[B_YFULL]);
                    mma_commit(&bars[B_EMPTY + s]);
                    if (j + 1 < n) {
                        if (!(ok = bwait(&bars[B_TREADY], (j + 1) & 1, abort_flag, p.status))) break;
                        tc_fence_after();
                        wu(j + 1);
                        mma_commit(&bars[B_WU]);
                    }
                }
            } while (false);
            mma_commit(&bars[B_FINAL]);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ gate warps (2, 3)
        const int gt = tid - 64;
        const float *alpha_h = p.alpha + static_cast<int64_t>(b) * p.T * p.Hv + hv;
        const float *beta_h = p.beta + static_cast<int64_t>(b) * p.T * p.Hv + hv;
        float a_nxt = 1.f, b_nxt = 0.f;
        auto load_gates = [&](int j) {
            a_nxt = 1.f;
            b_nxt = 0.f;
            const int64_t t = static_cast<int64_t>(c_w + j) * kC + gt;
            if (j < n && t < p.T) {
                a_nxt = __ldg(alpha_h + t * p.Hv);
                b_nxt = __ldg(beta_h + t * p.Hv);
            }
        };
        load_gates(0);
        for (int j = 0; j < n; ++j) {
            const int buf = j & 1;
            float *sg = reinterpret_cast<float *>(sm + OFF_GATES) + buf * kGateFloats;
            float *s_g = sg, *s_u = sg + 64, *s_w = sg + 128, *s_b = sg + 192, *s_bu = sg + 256, *s_misc = sg + 320;
            float *cs = reinterpret_cast<float *>(sm + OFF_CHAIN) + (j % kChainSlots) * kChainFloats;
            const bool ok = bwait(&bars[B_GEMPTY + buf], ((j >> 1) & 1) ^ 1, abort_flag, p.status);
            if (!warp_ok(ok)) break;
            const float a_cur = a_nxt, b_cur = b_nxt;
            load_gates(j + 1);
            // g = inclusive cumsum of log alpha over the chunk
            float g = logf(a_cur);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, g, o);
                if (lane >= o) g += v;
            }
            if (gt == 31) s_misc[0] = g;
            named_bar(4, 64);
            if (gt >= 32) g += s_misc[0];
            s_g[gt] = g;
            named_bar(4, 64);
            // Fast path (chunk decay >= e^kFastLogDecay): gates factor as
            // e^{g_i - g_j} = u_i w_j with u = e^g, w = e^-g, all finite.
            const float g63 = s_g[63];
            const bool fastc = g63 >= kFastLogDecay;
            const float u = expf(g);
            s_u[gt] = u;
            s_b[gt] = b_cur;
            s_bu[gt] = b_cur * u;
            s_w[gt] = fastc ? expf(-g) : 0.f;
            cs[gt] = fastc ? expf(g63 - g) : 1.f;   // lambda: U^T columns
            cs[64 + gt] = fastc ? u : 1.f;          // gamma: y columns
            if (gt == 63) {
                cs[128] = u;                         // gamma_C
                s_misc[1] = fastc ? expf(-g63) : 0.f;
                s_misc[2] = fastc ? 1.f : 0.f;
            }
            mbar_arrive(&bars[B_GFULL + buf]);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ local warpgroup
        const int l = tid - 128;
        const int lw = warp - 4;
        const uint32_t q = lw;
        float *At = reinterpret_cast<float *>(sm + OFF_AT);
        float *Tm = reinterpret_cast<float *>(sm + OFF_TM);
        float *Rw = reinterpret_cast<float *>(sm + OFF_R) + lw * 16 * kBS;
        uint8_t *t1b = sm + OFF_T1, *t2b = sm + OFF_T2;
        // Blocks of T1, T2 above the block diagonal are never written: zero them once.
        for (int e = l; e < 2 * 64 * 128 / 16; e += 128)
            reinterpret_cast<uint4 *>(t1b)[e] = make_uint4(0u, 0u, 0u, 0u);
        // AP(j): gated Gram readout of chunk j -> A (warps 4-5, which then invert
        // their two diagonal blocks) and P (warps 6-7).  Runs one chunk ahead of
        // the W readout so the W^T MMA of chunk j overlaps it.
        auto ap = [&](int j) -> bool {
            const int s = j % kStages;
            const int gbuf = j & 1;
            const float *sg = reinterpret_cast<const float *>(sm + OFF_GATES) + gbuf * kGateFloats;
            const float *s_g = sg, *s_u = sg + 64, *s_w = sg + 128, *s_b = sg + 192, *s_bu = sg + 256,
                        *s_misc = sg + 320;
            bool ok = bwait(&bars[B_GFULL + gbuf], (j >> 1) & 1, abort_flag, p.status);
            ok = ok && bwait(&bars[B_FULL + s], (j / kStages) & 1, abort_flag, p.status);
            ok = ok && bwait(&bars[B_GRAM + (j & 1)], (j >> 1) & 1, abort_flag, p.status);
            if (!warp_ok(ok)) return false;
            const bool fast = s_misc[2] != 0.f;
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float gr[32];
                tmem_ld32(lane_addr(tb + TM_GW + (j & 1) * 64, q, 32 * half), gr);
                tmem_wait_ld();
                if (l < 64) {
                    // A row i = l (beta_i e^{g_i - g_j} k_i.k_j, j < i) into the block-packed,
                    // column-major-within-block layout: A[i][j] at blk(i/16, j/16) + (j%16)*kBS + i%16.
                    const int i = l, bi = i >> 4;
                    float *abase = At + kBlkIdx[bi][0] * kBlk + (i & 15);
                    if (fast) {
                        // all loads of the half first: the stores below may alias them
                        const float ci = s_bu[i];
                        float wv[32];
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 f = *reinterpret_cast<const float4 *>(s_w + 32 * half + 4 * c4);
                            wv[4 * c4] = f.x * ci;
                            wv[4 * c4 + 1] = f.y * ci;
                            wv[4 * c4 + 2] = f.z * ci;
                            wv[4 * c4 + 3] = f.w * ci;
                        }
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) {
                            const int c = 32 * half + cc;
                            if (c < i) abase[(c >> 4) * kBlk + (c & 15) * kBS] = gr[cc] * wv[cc];
                        }
                    } else {
                        const float bi_ = s_b[i], gi = s_g[i];
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) {
                            const int c = 32 * half + cc;
                            if (c < i) abase[(c >> 4) * kBlk + (c & 15) * kBS] = bi_ * expf(gi - s_g[c]) * gr[cc];
                        }
                    }
                } else {
                    // P row i = l - 64, bf16: fast path (q_i.k_j) / gamma_C (the gates are
                    // applied to U and y by the chain), else e^{g_i - g_j} (q_i.k_j).
                    const int i = l - 64;
                    uint8_t *prow = sm + OFF_P + s * kPBytes + i * 128;
                    float v[32];
                    if (fast) {
                        const float pinv = s_misc[1];
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) v[cc] = (32 * half + cc <= i) ? gr[cc] * pinv : 0.f;
                    } else {
                        const float gi = s_g[i];
#pragma unroll
                        for (int cc = 0; cc < 32; ++cc) {
                            const int c = 32 * half + cc;
                            v[cc] = c <= i ? expf(gi - s_g[c]) * gr[cc] : 0.f;
                        }
                    }
#pragma unroll
                    for (int ch4 = 0; ch4 < 4; ++ch4) {
                        const int ch = 4 * half + ch4;
                        *reinterpret_cast<uint4 *>(prow + ((ch ^ (i & 7)) << 4)) =
                            make_uint4(pack_bf16(v[8 * ch4], v[8 * ch4 + 1]), pack_bf16(v[8 * ch4 + 2], v[8 * ch4 + 3]),
                                       pack_bf16(v[8 * ch4 + 4], v[8 * ch4 + 5]),
                                       pack_bf16(v[8 * ch4 + 6], v[8 * ch4 + 7]));
                    }
                }
            }
            tc_fence_before();
            if (l < 64) {
                // Diagonal blocks of T = (I + A)^{-1} by forward substitution, one
                // column per thread; this warp wrote both blocks' rows.
                __syncwarp();
                const int blk = l >> 4, col = l & 15;
                const float *Ab = At + kBlkIdx[blk][blk] * kBlk;
                float t[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) t[r] = (r == col) ? 1.f : 0.f;
#pragma unroll
                for (int mb = 0; mb < 2; ++mb) {
                    constexpr int kSplit = 5;   // columns 0-4 hold 65 values, 5-14 hold 55
                    float av[65];
                    const int m0 = mb ? kSplit : 0, m1 = mb ? 15 : kSplit;
#pragma unroll
                    for (int m = m0; m < m1; ++m)
#pragma unroll
                        for (int r = m + 1; r < 16; ++r)
                            av[(m * 16 - (m * (m + 1)) / 2 + (r - m - 1)) - (m0 * 16 - (m0 * (m0 + 1)) / 2)] =
                                Ab[m * kBS + r];
#pragma unroll
                    for (int m = m0; m < m1; ++m)
#pragma unroll
                        for (int r = m + 1; r < 16; ++r)
                            t[r] = fmaf(-av[(m * 16 - (m * (m + 1)) / 2 + (r - m - 1)) - (m0 * 16 - (m0 * (m0 + 1)) / 2)],
                                        t[m], t[r]);
                }
                float *Tb = Tm + kBlkIdx[blk][blk] * kBlk + col;
#pragma unroll
                for (int r = 0; r < 16; ++r) Tb[r * kBS] = t[r];
            } else if (!fast) {
                // Q~ = diag(gamma) Q in place (exact path)
                const int i = l - 64;
                const float gam = s_u[i];
                uint8_t *qrow = sm + OFF_KQ + s * kKQBytes + (64 + i) * 128;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint4 *ptr = reinterpret_cast<uint4 *>(qrow + kb * 16384 + ch * 16);
                        uint4 raw = *ptr;
                        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&raw);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(h2[e]);
                            h2[e] = __floats2bfloat162_rn(f.x * gam, f.y * gam);
                        }
                        *ptr = raw;
                    }
                }
            }
            return true;
        };

        if (ap(0)) {
            for (int j = 0; j < n; ++j) {
                const int s = j % kStages;
                const int gbuf = j & 1;
                const float *sg = reinterpret_cast<const float *>(sm + OFF_GATES) + gbuf * kGateFloats;
                const float *s_g = sg, *s_b = sg + 192, *s_bu = sg + 256, *s_misc = sg + 320;
                const bool fast = s_misc[2] != 0.f;
                named_bar(1, 128);   // A, diagonal T blocks and P of chunk j are written
                // Off-diagonal blocks T_IJ = -T_II sum_{K=J}^{I-1} A_IK T_KJ (warp J of 0-2),
                // and the bf16 T1 = T diag(beta gamma), T2 = T diag(beta) of the diagonal blocks (warp 3).
                if (lw == 0)
                    merge_column<0>(At, Tm, Rw, t1b, t2b, s_b, s_bu, lane);
                else if (lw == 1)
                    merge_column<1>(At, Tm, Rw, t1b, t2b, s_b, s_bu, lane);
                else if (lw == 2)
                    merge_column<2>(At, Tm, Rw, t1b, t2b, s_b, s_bu, lane);
                else
                    diag_to_bf16(Tm, t1b, t2b, s_b, s_bu, lane);
                fence_proxy_async();
                mbar_arrive(&bars[B_TREADY]);
                named_bar(1, 128);   // A and T of chunk j are no longer read
                if (j + 1 < n && !ap(j + 1)) break;

                // ---- -W (token-major, K-major operand) into the V slot (exact path: K~ in place)
                bool ok = bwait(&bars[B_WU], j & 1, abort_flag, p.status);
                if (!warp_ok(ok)) break;
                tc_fence_after();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float w[32];
                    tmem_ld32(lane_addr(tb + TM_GW + (j & 1) * 64, q, 32 * half), w);
                    tmem_wait_ld();
                    const int kb = l >> 6, col = l & 63;
                    uint8_t *base = sm + OFF_VW + s * kVWBytes + kb * 8192 + (col & 7) * 2;
#pragma unroll
                    for (int ii = 0; ii < 32; ++ii) {
                        const int i = 32 * half + ii;
                        *reinterpret_cast<__nv_bfloat16 *>(base + i * 128 + (((col >> 3) ^ (i & 7)) << 4)) =
                            __float2bfloat16_rn(-w[ii]);
                    }
                }
                if (!fast) {
                    const float g63 = s_g[63];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int idx = l + 128 * u;
                        const int kb = idx >> 9, r = (idx >> 3) & 63, ch = idx & 7;
                        uint4 *ptr =
                            reinterpret_cast<uint4 *>(sm + OFF_KQ + s * kKQBytes + kb * 16384 + r * 128 + ch * 16);
                        const float lam = expf(g63 - s_g[r]);
                        uint4 raw = *ptr;
                        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&raw);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(h2[e]);
                            h2[e] = __floats2bfloat162_rn(f.x * lam, f.y * lam);
                        }
                        *ptr = raw;
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(&bars[B_OPS]);
                mbar_arrive(&bars[B_GEMPTY + gbuf]);
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ chain warpgroups
        const int h = (warp - 8) >> 2;          // dk half
        const uint32_t q = warp & 3;             // TMEM lane quadrant
        const int x = 32 * q + lane;             // value index (TMEM lane)
        const int d = p.d;
        float S[64];
        if (use_s0 && x < d) {
            const float *src = p.S0 + (static_cast<int64_t>(b) * p.Hv + hv) * d * d + x;
#pragma unroll
            for (int m = 0; m < 64; ++m) {
                const int dk = 64 * h + m;
                S[m] = dk < d ? __ldg(src + static_cast<int64_t>(dk) * d) : 0.f;
            }
        } else {
#pragma unroll
            for (int m = 0; m < 64; ++m) S[m] = 0.f;
        }
        auto write_sb = [&](int buf) {
#pragma unroll
            for (int piece = 0; piece < 2; ++piece) {
                uint32_t u[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) u[c] = pack_bf16(S[32 * piece + 2 * c], S[32 * piece + 2 * c + 1]);
                tmem_st16(lane_addr(tb + TM_SB + 64 * buf + 32 * h + 16 * piece, q, 0), u);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars[B_SREADY]);
        };
        write_sb(0);
        for (int j = 0; j < n; ++j) {
            const int c = c_w + j;
            const float *cs = reinterpret_cast<const float *>(sm + OFF_CHAIN) + (j % kChainSlots) * kChainFloats;
            const uint32_t zu = tb + TM_ZU;
            bool ok = bwait(&bars[B_UFULL], j & 1, abort_flag, p.status);
            ok = ok && bwait(&bars[B_OPS], j & 1, abort_flag, p.status);  // per-chunk scales
            if (!warp_ok(ok)) break;
            tc_fence_after();
            {
                // U^T scaled by lambda, bf16: this half's 32 tokens packed into 16 columns
                uint32_t pk[16];
#pragma unroll
                for (int piece = 0; piece < 2; ++piece) {
                    float u[16];
                    tmem_ld16(lane_addr(zu, q, 32 * h + 16 * piece), u);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pk[8 * piece + e] = pack_bf16(u[2 * e] * cs[32 * h + 16 * piece + 2 * e],
                                                      u[2 * e + 1] * cs[32 * h + 16 * piece + 2 * e + 1]);
                }
                tmem_st16(lane_addr(zu, q, 32 * h), pk);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&bars[B_USMEM]);
            const float gC = cs[128];
            ok = bwait(&bars[B_DFULL], j & 1, abort_flag, p.status);
            if (!warp_ok(ok)) break;
            tc_fence_after();
#pragma unroll
            for (int piece = 0; piece < 4; ++piece) {
                float dd[16];
                tmem_ld16(lane_addr(tb + TM_D + 64 * h + 16 * piece, q, 0), dd);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) S[16 * piece + e] = fmaf(gC, S[16 * piece + e], dd[e]);
            }
            write_sb((j + 1) & 1);
            ok = bwait(&bars[B_YFULL], j & 1, abort_flag, p.status);
            if (!warp_ok(ok)) break;
            tc_fence_after();
            uint32_t yb[16];   // y of this lane's 32 tokens, bf16 pairs
#pragma unroll
            for (int piece = 0; piece < 2; ++piece) {
                float yv[16];
                tmem_ld16(lane_addr(tb + TM_Y + 32 * h + 16 * piece, q, 0), yv);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    yb[8 * piece + e] = pack_bf16(yv[2 * e] * cs[64 + 32 * h + 16 * piece + 2 * e],
                                                  yv[2 * e + 1] * cs[64 + 32 * h + 16 * piece + 2 * e + 1]);
            }
            tc_fence_before();
            mbar_arrive(&bars[B_YFREE]);
            if (c >= c_begin && x < d) {
                __nv_bfloat16 *yp = p.y + ((static_cast<int64_t>(b) * p.T + static_cast<int64_t>(c) * kC + 32 * h) *
                                               p.Hv + hv) * d + x;
                const int64_t tstart = static_cast<int64_t>(c) * kC + 32 * h;
                const int64_t ystride = static_cast<int64_t>(p.Hv) * d;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint32_t pr = yb[i >> 1];
                    const uint16_t bits = (i & 1) ? static_cast<uint16_t>(pr >> 16) : static_cast<uint16_t>(pr & 0xffffu);
                    if (tstart + i < p.T) *reinterpret_cast<uint16_t *>(yp + i * ystride) = bits;
                }
            }
        }
        if (last_seg && !*abort_flag && x < d) {
            float *dst = p.S_T + (static_cast<int64_t>(b) * p.Hv + hv) * d * d + x;
#pragma unroll
            for (int m = 0; m < 64; ++m) {
                const int dk = 64 * h + m;
                if (dk < d) dst[static_cast<int64_t>(dk) * d] = S[m];
            }
        }
    }

    // ------------------------------------------------------------ teardown
    __syncthreads();
    if (warp == 0 && lane == 0 && *abort_flag) {
        // Let any load still in flight land before the CTA exits.
        for (int s = 0; s < kStages; ++s)
            if (loads_issued[s] > 0) bwait_teardown(&bars[B_FULL + s], ((loads_issued[s] - 1) / kStages) & 1);
    }
    if (warp == 1 && lane == 0) bwait_teardown(&bars[B_FINAL], 0);
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// 4-D bf16 map over [B, T, H, d] (d innermost), box 64 (d) x 1 x 64 (tokens) x 1,
// 128-byte swizzle, out-of-range elements read as zero.
bool make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *ptr, int d, int H, int64_t T,
              int64_t B) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                                   static_cast<cuuint64_t>(T) * H * d * 2};
    const cuuint32_t box[4] = {64, 1, 64, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int plan_segments(int64_t pairs, int64_t nchunks, int num_sms, int requested) {
    if (requested > 0) return static_cast<int>(requested < nchunks ? requested : nchunks);
    // Minimise waves x (chunks per segment + assumed warm-up) over segment counts.
    const int64_t warm = 8;
    int best = 1;
    int64_t best_cost = INT64_MAX;
    const int64_t limit = nchunks < 4096 ? nchunks : 4096;
    for (int64_t P = 1; P <= limit; ++P) {
        const int64_t len = (nchunks + P - 1) / P;
        const int64_t Peff = (nchunks + len - 1) / len;
        if (Peff != P) continue;
        const int64_t ctas = pairs * P;
        if (ctas > 0x7fffffffLL) break;
        const int64_t waves = (ctas + num_sms - 1) / num_sms;
        const int64_t cost = waves * (len + (P > 1 ? warm : 0));
        if (cost < best_cost) {
            best_cost = cost;
            best = static_cast<int>(P);
        }
    }
    return best;
}

cudaError_t launch_chunked(const ChunkedParams &p, cudaStream_t stream, int num_sms) {
    if (p.d != 64 && p.d != 128) return cudaErrorInvalidValue;
    if (p.T > 0xffffffffLL || p.B > 0x7fffffffLL) return cudaErrorInvalidValue;
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encoder();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv;
    if (!make_map(enc, &mq, p.q, p.d, p.Hqk, p.T, p.B) || !make_map(enc, &mk, p.k, p.d, p.Hqk, p.T, p.B) ||
        !make_map(enc, &mv, p.v, p.d, p.Hv, p.T, p.B))
        return cudaErrorInvalidValue;
    const int64_t nchunks = (p.T + kC - 1) / kC;
    const int64_t pairs = p.B * p.Hv;
    if (nchunks > 0x7fffffffLL || pairs > 0x7fffffffLL) return cudaErrorInvalidValue;
    int P = plan_segments(pairs, nchunks, num_sms, p.segments);
    const int64_t len = (nchunks + P - 1) / P;
    P = static_cast<int>((nchunks + len - 1) / len);
    const int64_t grid = pairs * P;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;

    Dev dv{};
    dv.T = p.T;
    dv.B = static_cast<int>(p.B);
    dv.Hqk = p.Hqk;
    dv.Hv = p.Hv;
    dv.group = p.group;
    dv.d = p.d;
    dv.nchunks = static_cast<int>(nchunks);
    dv.seg_chunks = static_cast<int>(len);
    dv.nseg = P;
    dv.max_warmup = p.max_warmup_chunks;
    dv.log_eps = p.log_eps;
    dv.alpha = p.alpha;
    dv.beta = p.beta;
    dv.S0 = p.S0;
    dv.y = static_cast<__nv_bfloat16 *>(p.y);
    dv.S_T = p.S_T;
    dv.status = p.status;

    cudaError_t e = cudaFuncSetAttribute(gdn_chunked_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    gdn_chunked_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(mq, mk, mv, dv);
    return cudaGetLastError();
}

}  // namespace gdn
