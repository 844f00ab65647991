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
//   Gram   [Q;K] K^T            -> QK^T (lanes 0-63), KK^T (lanes 64-127)
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
//   warp 0        TMA producer (one thread): Q, K, V tiles of each chunk
//   warp 1        MMA issuer (the whole warp runs the control flow, lane 0
//                 issues); owns the TMEM allocation
//   warps 2-3     gates of each chunk, then its A rows (KK^T, TMEM lanes
//                 64-127) and the diagonal blocks of T = (I + A)^{-1}
//   warps 4-7     "local" warpgroup: the off-diagonal blocks of T and the
//                 bf16 T operands, the P rows (QK^T), the -W operand (Q~, K~
//                 on the exact path)
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
constexpr uint32_t kKQBytes = 2 * 128 * 128;  // [kb][128 rows][64]: Q rows 0-63, K rows 64-127
constexpr uint32_t kVWBytes = 2 * 64 * 128;   // [kb][64 rows][64]: V; later -W^T as [128 dk][64 tokens]
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
constexpr uint32_t OFF_GATES = OFF_TM + 10 * kBlk * 4;
// gates, double-buffered by chunk parity: g, u = gamma, w = 1/gamma, beta,
// beta gamma (64 floats each), misc (64)
constexpr int kGateFloats = 6 * 64;
constexpr uint32_t OFF_CHAIN = OFF_GATES + 2 * kGateFloats * 4;
// ring of 4 chunks: lambda[64], gamma[64], gamma_C for the chain warpgroups
constexpr int kChainFloats = 132;
constexpr int kChainSlots = 4;
constexpr uint32_t OFF_BAR = OFF_CHAIN + kChainSlots * kChainFloats * 4;
constexpr int kNumBars = 23;
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
    B_SOLVED = B_GEMPTY + 2,  // A and the diagonal T blocks of a chunk written (gate warps, 64 arrivals)
};
static_assert(B_SOLVED + 1 == kNumBars, "barrier count");

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
    int nchunks, seg_chunks, nseg, max_warmup, test_stall_chunk;
    float log_eps;
    const float *alpha, *beta, *S0;
    __nv_bfloat16 *y;
    float *S_T;
    uint32_t *status;
    // Exact sequence split (see launch_chunked): pass 1 runs every segment's
    // transition (kind 0: from the zero state, or S0 for segment 0, with the
    // real values; kind 1: from the identity with the values zero), pass 0 is
    // the output pass; heads with exact_flag set start each segment from the
    // state the combine kernel wrote.  seg_state: [pairs][nseg][3][d][d] fp32,
    // slots B (kind 0 end), M (kind 1 end), In (entering state).
    int pass;
    const int *exact_flag;
    float *seg_state;
};

// Slow path of a bounded wait (out of line: one copy for every call site).
__device__ __noinline__ bool bwait_slow(uint64_t *bar, uint32_t parity, volatile int *abort, uint32_t *status) {
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

__device__ __forceinline__ bool bwait(uint64_t *bar, uint32_t parity, volatile int *abort, uint32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    return bwait_slow(bar, parity, abort, status);
}

// Bounded wait that ignores the abort flag (teardown).
__device__ __forceinline__ void bwait_teardown(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

// True when some segment of head `pr` has no warm-up window (flags of the plan).
__device__ __forceinline__ bool head_needs_split(const int *flag, int pr, int nseg) {
    int any = 0;
    for (int sgm = 1; sgm < nseg; ++sgm) any |= flag[static_cast<int64_t>(pr) * nseg + sgm];
    return any != 0;
}

// All lanes of the warp agree: true only if every lane's wait succeeded.
__device__ __forceinline__ bool warp_ok(bool ok) { return __all_sync(0xffffffffu, ok); }

// All `count` threads of named barrier `id` agree (the barrier's AND
// reduction, which is also a barrier): warps that meet at that named barrier
// take every abort decision together, so none of them is left waiting there
// for a warp that has already left its loop.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t count, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(ok)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

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

// Off-diagonal blocks of T = (I + A)^{-1} from its diagonal blocks T_II, in
// left-factor form: with F_IK = T_II A_IK (K < I),
//   T_IJ = -sum_{K=J}^{I-1} F_IK T_KJ      (I > J),
// so each block column is a chain of plain products once every F is known.
// Warp MMAs m16n8k8 tf32 with fp32 accumulation (fp32 operands are passed as
// is; the tensor core reads their tf32 part).
//
// Step 1 (solve_factors): the six F_IK, as twelve 8-column tiles, three per
// warp, written in place of A_IK (column-major within the block: a warp only
// reads and writes the columns of its own tiles).
struct FactorJob {
    uint8_t I, K, nt;
};
__constant__ FactorJob kFactorJobs[4][3] = {
    {{1, 0, 0}, {1, 0, 1}, {2, 0, 0}},
    {{2, 1, 0}, {2, 1, 1}, {2, 0, 1}},
    {{3, 2, 0}, {3, 2, 1}, {3, 1, 0}},
    {{3, 0, 0}, {3, 0, 1}, {3, 1, 1}},
};

__device__ __forceinline__ void solve_factors(int lw, float *At, const float *Tm, int lane) {
    const int gq = lane >> 2, t4 = lane & 3;
    float acc[3][2][4];
    float *fb[3];
    int col[3];
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const FactorJob jb = kFactorJobs[lw][u];
        const int I = jb.I, K = jb.K;
        const float *Td = Tm + (I * (I + 1) / 2 + I) * kBlk;   // T_II[r][k] at r*kBS + k
        fb[u] = At + (I * (I + 1) / 2 + K) * kBlk;             // A_IK[k][n] at n*kBS + k
        col[u] = 8 * jb.nt + gq;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int k0 = 8 * ks;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[u][ks][e] = 0.f;
            mma_tf32(acc[u][ks], __float_as_uint(Td[gq * kBS + k0 + t4]), __float_as_uint(Td[(gq + 8) * kBS + k0 + t4]),
                     __float_as_uint(Td[gq * kBS + k0 + t4 + 4]), __float_as_uint(Td[(gq + 8) * kBS + k0 + t4 + 4]),
                     __float_as_uint(fb[u][col[u] * kBS + k0 + t4]), __float_as_uint(fb[u][col[u] * kBS + k0 + t4 + 4]));
        }
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        // accumulator (row gq (+8), column 2 t4 (+1) of the tile) -> F[r][n] at n*kBS + r
        float *f = fb[u] + (col[u] - gq + 2 * t4) * kBS + gq;
        f[0] = acc[u][0][0] + acc[u][1][0];
        f[kBS] = acc[u][0][1] + acc[u][1][1];
        f[8] = acc[u][0][2] + acc[u][1][2];
        f[kBS + 8] = acc[u][0][3] + acc[u][1][3];
    }
}

// Step 2: block column J (NNT = 2: both 8-column tiles; NNT = 1: tile nt0 only),
// T_IJ for I = J+1..3 in order.  Writes T_IJ as fp32 (row-major, for the next
// block of the column) and as bf16 T1 = T diag(beta gamma), T2 = T diag(beta).
template <int NNT>
__device__ __forceinline__ void solve_column(int J, int nt0, const float *At, float *Tm, uint8_t *t1b, uint8_t *t2b,
                                             const float *s_b, const float *s_bu, int lane) {
    const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll 1
    for (int I = J + 1; I < 4; ++I) {
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int K = J; K < I; ++K) {
            const float *Fb = At + (I * (I + 1) / 2 + K) * kBlk;   // F[r][k] at k*kBS + r
            const float *Bb = Tm + (K * (K + 1) / 2 + J) * kBlk;   // T[k][n] at k*kBS + n
            // k-steps 0 and 1 into separate accumulators: two independent MMA chains
            uint32_t a[2][4], b[2][2][2];
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int k0 = 8 * ks;
                a[ks][0] = __float_as_uint(Fb[(k0 + t4) * kBS + gq]);
                a[ks][1] = __float_as_uint(Fb[(k0 + t4) * kBS + gq + 8]);
                a[ks][2] = __float_as_uint(Fb[(k0 + t4 + 4) * kBS + gq]);
                a[ks][3] = __float_as_uint(Fb[(k0 + t4 + 4) * kBS + gq + 8]);
#pragma unroll
                for (int nt = 0; nt < NNT; ++nt) {
                    b[ks][nt][0] = __float_as_uint(Bb[(k0 + t4) * kBS + 8 * (nt0 + nt) + gq]);
                    b[ks][nt][1] = __float_as_uint(Bb[(k0 + t4 + 4) * kBS + 8 * (nt0 + nt) + gq]);
                }
            }
            mma_tf32(c0, a[0][0], a[0][1], a[0][2], a[0][3], b[0][0][0], b[0][0][1]);
            mma_tf32(e0, a[1][0], a[1][1], a[1][2], a[1][3], b[1][0][0], b[1][0][1]);
            if (NNT == 2) {
                mma_tf32(c1, a[0][0], a[0][1], a[0][2], a[0][3], b[0][NNT - 1][0], b[0][NNT - 1][1]);
                mma_tf32(e1, a[1][0], a[1][1], a[1][2], a[1][3], b[1][NNT - 1][0], b[1][NNT - 1][1]);
            }
        }
        float *Tb = Tm + (I * (I + 1) / 2 + J) * kBlk;
#pragma unroll
        for (int nt = 0; nt < NNT; ++nt) {
            const float *cc = nt ? c1 : c0;
            const float *ee = nt ? e1 : e0;
            const int cn = 8 * (nt0 + nt) + 2 * t4;
            const int C = 16 * J + cn;
            const float sa0 = s_bu[C], sa1 = s_bu[C + 1], sb0 = s_b[C], sb1 = s_b[C + 1];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = gq + 8 * hr;
                const float v0 = -(cc[2 * hr] + ee[2 * hr]), v1 = -(cc[2 * hr + 1] + ee[2 * hr + 1]);
                if (I < 3) *reinterpret_cast<float2 *>(Tb + r * kBS + cn) = make_float2(v0, v1);
                const uint32_t off = sw128_elem(16 * I + r, C);
                *reinterpret_cast<uint32_t *>(t1b + off) = pack_bf16(v0 * sa0, v1 * sa1);
                *reinterpret_cast<uint32_t *>(t2b + off) = pack_bf16(v0 * sb0, v1 * sb1);
            }
        }
        __syncwarp();
    }
}

// bf16 T1, T2 of diagonal block blk from its fp32 copy (one warp).
__device__ __forceinline__ void diag_block_to_bf16(int blk, const float *Tm, uint8_t *t1b, uint8_t *t2b,
                                                   const float *s_b, const float *s_bu, int lane) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = lane + 32 * u;             // 128 column pairs of the block
        const int r = e >> 3, cp = e & 7;
        const int C = 16 * blk + 2 * cp;
        const float2 v = *reinterpret_cast<const float2 *>(Tm + (blk * (blk + 1) / 2 + blk) * kBlk + r * kBS + 2 * cp);
        const uint32_t off = sw128_elem(16 * blk + r, C);
        *reinterpret_cast<uint32_t *>(t1b + off) = pack_bf16(v.x * s_bu[C], v.y * s_bu[C + 1]);
        *reinterpret_cast<uint32_t *>(t2b + off) = pack_bf16(v.x * s_b[C], v.y * s_b[C + 1]);
    }
}

// Operand of a run of K=16 MMAs.  Offsets advance as
// (kk >> shift) * big + (kk & ((1 << shift) - 1)) * small bytes (TMEM A: columns);
// a start address inside a descriptor moves by adding offset >> 4.
struct MmaOperand {
    uint64_t desc;      // shared-memory descriptor (unused for a TMEM A operand)
    uint32_t tmem;      // TMEM address of A (0: A from shared memory)
    uint32_t big, small, shift;
};

__device__ __forceinline__ uint32_t operand_offset(const MmaOperand &o, uint32_t kk) {
    return (kk >> o.shift) * o.big + (kk & ((1u << o.shift) - 1u)) * o.small;
}

// NK consecutive K=16 MMAs of one product, issued warp-wide (a rolled loop:
// the issuing warp's code stays small; each step adds a constant offset to
// the descriptors).  TMEM_A:
// A is read from tensor memory (a.tmem) instead of shared memory (a.desc).
template <int NK, bool TMEM_A>
__device__ __forceinline__ void mma_run_t(uint32_t d, const MmaOperand &a, const MmaOperand &b, uint32_t idesc, uint32_t acc) {
#pragma unroll 1
    for (int kk = 0; kk < NK; ++kk) {
        const uint64_t bd = b.desc + (operand_offset(b, kk) >> 4);
        const uint32_t accumulate = acc | (kk > 0 ? 1u : 0u);
        if constexpr (TMEM_A)
            mma_bf16_ts_w(d, a.tmem + operand_offset(a, kk), bd, idesc, accumulate);
        else
            mma_bf16_w(d, a.desc + (operand_offset(a, kk) >> 4), bd, idesc, accumulate);
    }
}

// A product with a lower-triangular right factor over the chunk's tokens:
// D[:, i] (+)= sum_{j <= i} A[:, j] B[i][j] with B stored K-major ([i rows][j],
// 128-byte rows) and N = 64.  The K step over tokens 16 kk .. 16 kk + 15 only
// reaches columns i >= 16 kk, so it is issued with N = 64 - 16 kk from column
// 16 kk of D and row 16 kk of B: the zero blocks above B's block diagonal are
// not multiplied.  idesc0: the instruction descriptor without its N field.
template <bool TMEM_A>
__device__ __forceinline__ void mma_run_tri(uint32_t d, const MmaOperand &a, const MmaOperand &b, uint32_t idesc0, uint32_t acc) {
#pragma unroll 1
    for (int kk = 0; kk < 4; ++kk) {
        const uint32_t idesc = idesc0 | (static_cast<uint32_t>((64 - 16 * kk) >> 3) << 17);
        const uint64_t bd = b.desc + ((operand_offset(b, kk) + 2048u * kk) >> 4);
        const uint32_t accumulate = acc | (kk > 0 ? 1u : 0u);
        if constexpr (TMEM_A)
            mma_bf16_ts_w(d + 16u * kk, a.tmem + operand_offset(a, kk), bd, idesc, accumulate);
        else
            mma_bf16_w(d + 16u * kk, a.desc + (operand_offset(a, kk) >> 4), bd, idesc, accumulate);
    }
}

// A rows of a chunk (gate warps): row i of K K^T is TMEM lane 64 + i.  Written
// into the block-packed layout, A[i][j] at blk(i/16, j/16) + (j%16)*kBS + i%16,
// for j < i.  Fast gates: A_ij = (beta_i gamma_i) (1/gamma_j) (k_i.k_j).
__device__ __forceinline__ void fast_a_rows(int i, uint32_t q, uint32_t gw, float *At, const float *s_w, const float *s_bu) {
    const float ci = s_bu[i];
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        float gr[32];
        tmem_ld32(lane_addr(gw, q, 32 * half), gr);
        tmem_wait_ld();
        float *abase = At + (kBlkIdx[i >> 4][0] + 2 * half) * kBlk + (i & 15);
        float wv[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
            const float4 f = *reinterpret_cast<const float4 *>(s_w + 32 * half + 4 * c4);
            wv[4 * c4] = f.x * ci;
            wv[4 * c4 + 1] = f.y * ci;
            wv[4 * c4 + 2] = f.z * ci;
            wv[4 * c4 + 3] = f.w * ci;
        }
        const int lim = i - 32 * half;
#pragma unroll
        for (int cc = 0; cc < 32; ++cc)
            if (cc < lim) abase[(cc >> 4) * kBlk + (cc & 15) * kBS] = gr[cc] * wv[cc];
    }
}

// Exact gate path (a chunk whose decay is below e^kFastLogDecay), A rows:
// A_ij = beta_i e^{g_i - g_j} (k_i.k_j) per element.  Cold code.
__device__ __noinline__ void exact_a_rows(int i, uint32_t q, uint32_t gw, float *At, const float *s_g, const float *s_b) {
    const float bi = s_b[i], gi = s_g[i];
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        float gr[32];
        tmem_ld32(lane_addr(gw, q, 32 * half), gr);
        tmem_wait_ld();
        float *abase = At + (kBlkIdx[i >> 4][0] + 2 * half) * kBlk + (i & 15);
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) {
            const int c = 32 * half + cc;
            if (c < i) abase[(cc >> 4) * kBlk + (cc & 15) * kBS] = bi * expf(gi - s_g[c]) * gr[cc];
        }
    }
}

// Exact gate path, P rows (row i of Q K^T is TMEM lane i): P_ij = e^{g_i - g_j}
// (q_i.k_j) for j <= i, and Q~ = diag(gamma) Q in place.  Cold code.
__device__ __noinline__ void exact_p_rows(int i, uint32_t q, uint32_t gw, uint8_t *pbuf, uint8_t *kq, const float *s_g,
                                          const float *s_u) {
    const float gi = s_g[i];
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
        float gr[32];
        tmem_ld32(lane_addr(gw, q, 32 * half), gr);
        tmem_wait_ld();
        uint8_t *prow = pbuf + i * 128;
#pragma unroll
        for (int ch4 = 0; ch4 < 4; ++ch4) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int cc = 8 * ch4 + 2 * e, c = 32 * half + cc;
                w4[e] = pack_bf16(c <= i ? expf(gi - s_g[c]) * gr[cc] : 0.f,
                                  c + 1 <= i ? expf(gi - s_g[c + 1]) * gr[cc + 1] : 0.f);
            }
            *reinterpret_cast<uint4 *>(prow + (((4 * half + ch4) ^ (i & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
    }
    const float gam = s_u[i];
    uint8_t *qrow = kq + i * 128;
#pragma unroll 1
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

// Diagonal blocks of T = (I + A)^{-1} by forward substitution, one column per
// thread (thread i: block i/16, column i%16; the calling warp wrote both of its
// blocks' rows).  The block's strictly lower part (column m: rows m+1..15) is
// loaded in two batches ahead of the arithmetic.
__device__ __forceinline__ void diag_solve(int i, const float *At, float *Tm) {
    const int blk = i >> 4, col = i & 15;
    const float *Ab = At + kBlkIdx[blk][blk] * kBlk;
    float t[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) t[r] = (r == col) ? 1.f : 0.f;
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
        constexpr int kSplit = 5;
        float av[65];
        const int m0 = mb ? kSplit : 0, m1 = mb ? 15 : kSplit;
#pragma unroll
        for (int m = m0; m < m1; ++m)
#pragma unroll
            for (int r = m + 1; r < 16; ++r)
                av[(m * 16 - (m * (m + 1)) / 2 + (r - m - 1)) - (m0 * 16 - (m0 * (m0 + 1)) / 2)] = Ab[m * kBS + r];
#pragma unroll
        for (int m = m0; m < m1; ++m)
#pragma unroll
            for (int r = m + 1; r < 16; ++r)
                t[r] = fmaf(-av[(m * 16 - (m * (m + 1)) / 2 + (r - m - 1)) - (m0 * 16 - (m0 * (m0 + 1)) / 2)], t[m], t[r]);
    }
    float *Tb = Tm + kBlkIdx[blk][blk] * kBlk + col;
#pragma unroll
    for (int r = 0; r < 16; ++r) Tb[r * kBS] = t[r];
}

// Exact gate path: K~ = diag(lambda) K in place, lambda_r = e^{g_C - g_r}.  Cold code.
__device__ __noinline__ void exact_scale_k(int l, uint8_t *kq, const float *s_g) {
    const float g63 = s_g[63];
#pragma unroll 1
    for (int u = 0; u < 8; ++u) {
        const int idx = l + 128 * u;
        const int kb = idx >> 9, r = (idx >> 3) & 63, ch = idx & 7;
        uint4 *ptr = reinterpret_cast<uint4 *>(kq + kb * 16384 + 8192 + r * 128 + ch * 16);
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
    const int bx = static_cast<int>(blockIdx.x % static_cast<unsigned>(pairs * p.nseg));
    const int kind = p.pass == 1 ? static_cast<int>(blockIdx.x / static_cast<unsigned>(pairs * p.nseg)) : -1;
    const int seg = bx / pairs;
    const int pr = bx % pairs;
    const bool exact = p.exact_flag != nullptr && head_needs_split(p.exact_flag, pr, p.nseg);
    // Transition pass: only heads that need the exact split, only segments whose
    // transition is used (not the last; segment 0 starts from S0, so no M).
    if (p.pass == 1 && (!exact || seg == p.nseg - 1 || (kind == 1 && seg == 0))) return;
    const int b = pr / p.Hv;
    const int hv = pr % p.Hv;
    const int hk = hv / p.group;
    const int c_begin = seg * p.seg_chunks;
    const int c_end = min(p.nchunks, c_begin + p.seg_chunks);

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
        mbar_init(&bars[B_SOLVED], 64);

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
    // (No window on the transition pass or for an exactly split head: each
    // segment starts at its own first chunk.)
    const bool windowed = p.pass == 0 && !exact;
    if (tid == 128 && (seg == 0 || !windowed)) misc->c_w = windowed ? 0 : c_begin;
    if (warp >= 4 && warp < 12 && seg > 0 && windowed) {
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
    const uint32_t tb_s = tb;
    const int c_w = misc->c_w;
    const int n = c_end - c_w;
    const int n_s = n;
    const bool use_s0 = c_w == 0 && p.S0 != nullptr && kind != 1;
    const bool zero_v = kind == 1;   // the identity run propagates the state with v = 0

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
                if (p.test_stall_chunk > 0 && c_w + j == p.test_stall_chunk) continue;  // fault injection
                mbar_arrive_expect_tx(&bars[B_FULL + s], kKQBytes + kVWBytes);
                uint8_t *kq = sm + OFF_KQ + s * kKQBytes;
                uint8_t *vw = sm + OFF_VW + s * kVWBytes;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    tma_load_4d(kq + kb * 16384, &tm_q, &bars[B_FULL + s], kb * 64, hk, t0, b);
                    tma_load_4d(kq + kb * 16384 + 8192, &tm_k, &bars[B_FULL + s], kb * 64, hk, t0, b);
                    tma_load_4d(vw + kb * 8192, &tm_v, &bars[B_FULL + s], kb * 64, hv, t0, b);
                }
                loads_issued[s] = j + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this role's control flow, so descriptors and TMEM
        // addresses stay warp-uniform; one elected lane issues each MMA and commit.
        {
            auto wait = [&](uint64_t *bar, uint32_t parity) {
                return warp_ok(bwait(bar, parity, abort_flag, p.status));
            };
            // Values read from shared memory, broadcast so that the compiler treats
            // them (and every descriptor derived from them) as warp-uniform.
            const uint32_t tb = __shfl_sync(0xffffffffu, tb_s, 0);
            const int n = __shfl_sync(0xffffffffu, n_s, 0);
            constexpr uint32_t ID_KK = idesc_bf16(128, 64, false, false);   // A, B K-major
            constexpr uint32_t ID_TS = idesc_bf16(128, 64, false, false);   // A in TMEM, B K-major
            constexpr uint32_t ID_TD = idesc_bf16(128, 128, false, true);   // A in TMEM, B MN-major
            constexpr uint32_t ID_TSM = idesc_bf16(128, 64, false, true);   // A in TMEM, B MN-major, N = 64
            const uint32_t t1 = smb + OFF_T1, t2 = smb + OFF_T2;
            // K-major tiles split in two 64-column sub-tiles (16 KB apart for [K;Q]);
            // MN-major tiles advance 2048 bytes (16 rows) per K step.
            auto smem_kmajor = [](uint32_t addr, uint32_t subtile) {
                return MmaOperand{sw128_desc(addr, 16, 1024), 0u, subtile, 32u, 2u};
            };
            auto smem_mnmajor = [](uint32_t addr, uint32_t lbo) {
                return MmaOperand{sw128_desc(addr, lbo, 1024), 0u, 8192u, 2048u, 2u};
            };
            auto gram = [&](int j) {
                // [Q;K] K^T: Q K^T in lanes 0-63, K K^T in lanes 64-127
                const uint32_t a = kq_addr(j % kStages);
                mma_run_t<8, false>(tb + TM_GW + (j & 1) * 64, smem_kmajor(a, 16384u), smem_kmajor(a + 8192, 16384u), ID_KK, 0u);
            };
            // W^T = K^T T1^T and U~^T = V^T T2^T: T1, T2 are lower triangular by blocks
            constexpr uint32_t ID_MK0 = idesc_bf16(128, 0, true, false);
            constexpr uint32_t ID_TS0 = idesc_bf16(128, 0, false, false);
            auto wu = [&](int j) {
                const int s = j % kStages;
                mma_run_tri<false>(tb + TM_GW + (j & 1) * 64, smem_mnmajor(kq_addr(s) + 8192, 16384u), smem_kmajor(t1, 0u), ID_MK0, 0u);
                if (!zero_v)
                    mma_run_tri<false>(tb + TM_ZU, smem_mnmajor(vw_addr(s), 8192u), smem_kmajor(t2, 0u), ID_MK0, 0u);
            };
            bool ok = true;
            do {
                if (!(ok = wait(&bars[B_FULL + 0], 0))) break;
                tc_fence_after();
                gram(0);
                mma_commit_w(&bars[B_GRAM + 0]);
                if (n > 1) {
                    if (!(ok = wait(&bars[B_FULL + 1 % kStages], (1 / kStages) & 1))) break;
                    tc_fence_after();
                    gram(1);
                    mma_commit_w(&bars[B_GRAM + 1]);
                }
                if (!(ok = wait(&bars[B_TREADY], 0))) break;
                tc_fence_after();
                wu(0);
                mma_commit_w(&bars[B_WU]);
                for (int j = 0; j < n && ok; ++j) {
                    const int s = j % kStages;
                    const uint32_t zu = tb + TM_ZU;
                    const uint32_t sb = tb + TM_SB + (j & 1) * 64;
                    if (!(ok = wait(&bars[B_OPS], j & 1))) break;
                    if (!(ok = wait(&bars[B_SREADY], j & 1))) break;
                    tc_fence_after();
                    // U^T = U~^T + S^T (-W)^T   (-W^T stored [dk][tokens], MN-major)
                    const MmaOperand sa{0ull, sb, 0u, 8u, 3u};          // S^T bf16: 8 columns per K step
                    const MmaOperand ua{0ull, zu, 32u, 8u, 1u};         // U^T bf16: tokens 0-31 at 0-15, 32-63 at 32-47
                    mma_run_t<8, true>(zu, sa, smem_mnmajor(vw_addr(s), 16u), ID_TSM, zero_v ? 0u : 1u);
                    mma_commit_w(&bars[B_UFULL]);
                    // Gram of chunk j+2 into the GW buffer W^T(j) occupied (read before
                    // OPS(j)); it runs while the chain converts U^T, before MMA2 is issued.
                    if (j + 2 < n) {
                        const int s2 = (j + 2) % kStages;
                        if (!(ok = wait(&bars[B_FULL + s2], ((j + 2) / kStages) & 1))) break;
                        tc_fence_after();
                        gram(j + 2);
                        mma_commit_w(&bars[B_GRAM + (j & 1)]);
                    }
                    if (!(ok = wait(&bars[B_USMEM], j & 1))) break;
                    tc_fence_after();
                    // dS^T = U^T K~
                    mma_run_t<4, true>(tb + TM_D, ua, smem_mnmajor(kq_addr(s) + 8192, 16384u), ID_TD, 0u);
                    mma_commit_w(&bars[B_DFULL]);
                    if (j > 0 && !(ok = wait(&bars[B_YFREE], (j - 1) & 1))) break;
                    tc_fence_after();
                    // Y^T = S^T Q~^T + U^T P^T, for the chunks whose y is stored (not the
                    // warm-up window, not a transition pass)
                    if (p.pass == 0 && c_w + j >= c_begin) {
                        mma_run_t<8, true>(tb + TM_Y, sa, smem_kmajor(kq_addr(s), 16384u), ID_TS, 0u);
                        mma_run_tri<true>(tb + TM_Y, ua, smem_kmajor(p_addr(s), 0u), ID_TS0, 1u);   // P^ lower triangular
                    }
                    mma_commit_w(&bars[B_YFULL]);
                    mma_commit_w(&bars[B_EMPTY + s]);
                    if (j + 1 < n) {
                        if (!(ok = wait(&bars[B_TREADY], (j + 1) & 1))) break;
                        tc_fence_after();
                        wu(j + 1);
                        mma_commit_w(&bars[B_WU]);
                    }
                }
            } while (false);
            mma_commit_w(&bars[B_FINAL]);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ gate warps (2, 3)
        const int gt = tid - 64;
        float *At = reinterpret_cast<float *>(sm + OFF_AT);
        float *Tm = reinterpret_cast<float *>(sm + OFF_TM);
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
            // Abort decisions are reduced over both gate warps (named barrier 4).
            const bool ok = bwait(&bars[B_GEMPTY + buf], ((j >> 1) & 1) ^ 1, abort_flag, p.status);
            if (!bar_and(4, 64, ok)) break;
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
            named_bar(4, 64);   // this chunk's gates are visible to both gate warps
            // A rows of chunk j (K K^T, TMEM lanes 64-127: row gt) and the diagonal
            // blocks of T, once the local warpgroup is done with chunk j-1's A and
            // T (TREADY(j-1)).
            bool ok2 = j == 0 || bwait(&bars[B_TREADY], (j - 1) & 1, abort_flag, p.status);
            ok2 = ok2 && bwait(&bars[B_GRAM + (j & 1)], (j >> 1) & 1, abort_flag, p.status);
            if (!bar_and(4, 64, ok2)) break;
            tc_fence_after();
            const uint32_t gw = tb + TM_GW + (j & 1) * 64;
            if (fastc)
                fast_a_rows(gt, warp, gw, At, s_w, s_bu);
            else
                exact_a_rows(gt, warp, gw, At, s_g, s_b);
            tc_fence_before();
            __syncwarp();
            diag_solve(gt, At, Tm);
            mbar_arrive(&bars[B_SOLVED]);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ local warpgroup
        const int l = tid - 128;
        const int lw = warp - 4;
        const uint32_t q = lw;
        float *At = reinterpret_cast<float *>(sm + OFF_AT);
        float *Tm = reinterpret_cast<float *>(sm + OFF_TM);
        uint8_t *t1b = sm + OFF_T1, *t2b = sm + OFF_T2;
        // Blocks of T1, T2 above the block diagonal are never written: zero them once.
        for (int e = l; e < 2 * 64 * 128 / 16; e += 128)
            reinterpret_cast<uint4 *>(t1b)[e] = make_uint4(0u, 0u, 0u, 0u);
        // P rows of chunk j (Q K^T, TMEM lanes 0-63: warps 4-5, row l) as the bf16
        // operand P^ = mask(Q K^T) / gamma_C (fast gates; y is scaled by the chain)
        // or P = mask(e^{g_i - g_j} q_i.k_j) with Q~ = diag(gamma) Q (exact gates).
        auto p_readout = [&](int j) -> bool {
            const int s = j % kStages;
            const int gbuf = j & 1;
            const float *sg = reinterpret_cast<const float *>(sm + OFF_GATES) + gbuf * kGateFloats;
            const float *s_g = sg, *s_u = sg + 64, *s_misc = sg + 320;
            bool ok = bwait(&bars[B_GFULL + gbuf], (j >> 1) & 1, abort_flag, p.status);
            ok = ok && bwait(&bars[B_FULL + s], (j / kStages) & 1, abort_flag, p.status);
            ok = ok && bwait(&bars[B_GRAM + (j & 1)], (j >> 1) & 1, abort_flag, p.status);
            if (!bar_and(2, 128, ok)) return false;
            if (l >= 64 || p.pass != 0 || c_w + j < c_begin) return true;   // P^ (and Q~) feed y only
            const uint32_t gw = tb + TM_GW + (j & 1) * 64;
            uint8_t *pbuf = sm + OFF_P + s * kPBytes;
            tc_fence_after();
            if (s_misc[2] != 0.f) {
                const int i = l;
                const float pinv = s_misc[1];
                uint8_t *prow = pbuf + i * 128;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float gr[32];
                    tmem_ld32(lane_addr(gw, q, 32 * half), gr);
                    tmem_wait_ld();
                    const int lim = i - 32 * half;
#pragma unroll
                    for (int ch4 = 0; ch4 < 4; ++ch4) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int cc = 8 * ch4 + 2 * e;
                            w4[e] = pack_bf16(cc <= lim ? gr[cc] * pinv : 0.f, cc + 1 <= lim ? gr[cc + 1] * pinv : 0.f);
                        }
                        *reinterpret_cast<uint4 *>(prow + (((4 * half + ch4) ^ (i & 7)) << 4)) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            } else {
                exact_p_rows(l, q, gw, pbuf, sm + OFF_KQ + s * kKQBytes, s_g, s_u);
            }
            tc_fence_before();
            return true;
        };

        // Chunk j: merges (once the gate warps have written A and the diagonal T
        // blocks), the next chunk's P rows, then chunk j's -W operand.
#pragma unroll 1
        for (int j = -1; j < n; ++j) {
            if (j >= 0) {
                const int s = j % kStages;
                const int gbuf = j & 1;
                const float *sg = reinterpret_cast<const float *>(sm + OFF_GATES) + gbuf * kGateFloats;
                const float *s_g = sg, *s_b = sg + 192, *s_bu = sg + 256, *s_misc = sg + 320;
                const bool fast = s_misc[2] != 0.f;
                // Abort decisions of this warpgroup are reduced over its 128 threads
                // (named barrier 2, which the merges below also use).
                if (!bar_and(2, 128, bwait(&bars[B_SOLVED], j & 1, abort_flag, p.status))) break;
                // The factors F_IK (three tiles per warp) and bf16 T1, T2 of diagonal
                // block lw; then the off-diagonal blocks T_IJ by block column: column 0
                // split over warps 0 and 3 (one 8-column tile each), column 1 on warp 1,
                // column 2 on warp 2.
                solve_factors(lw, At, Tm, lane);
                diag_block_to_bf16(lw, Tm, t1b, t2b, s_b, s_bu, lane);
                named_bar(2, 128);   // every F_IK is written
                if (lw == 0 || lw == 3)
                    solve_column<1>(0, lw == 3 ? 1 : 0, At, Tm, t1b, t2b, s_b, s_bu, lane);
                else
                    solve_column<2>(lw, 0, At, Tm, t1b, t2b, s_b, s_bu, lane);
                fence_proxy_async();
                mbar_arrive(&bars[B_TREADY]);
                if (j + 1 < n && !p_readout(j + 1)) break;

                // The W^T, U~^T MMAs of chunk j have read T1, T2 (rewritten by the next
                // merges) and K (exact path: K~ = diag(lambda) K in place).  Waiting here
                // also keeps this warpgroup at most one TREADY phase ahead of the MMA thread.
                if (!bar_and(2, 128, bwait(&bars[B_WU], j & 1, abort_flag, p.status))) break;
                tc_fence_after();
                {
                    // -W^T row l (key index l, 64 tokens) as one swizzled 128-byte row of
                    // the MN-major operand [dk][tokens] in the V slot
                    uint8_t *wrow = sm + OFF_VW + s * kVWBytes + l * 128;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        float w[32];
                        tmem_ld32(lane_addr(tb + TM_GW + (j & 1) * 64, q, 32 * half), w);
                        tmem_wait_ld();
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const int ch = 4 * half + c4;
                            *reinterpret_cast<uint4 *>(wrow + ((ch ^ (l & 7)) << 4)) = make_uint4(
                                pack_bf16(-w[8 * c4], -w[8 * c4 + 1]), pack_bf16(-w[8 * c4 + 2], -w[8 * c4 + 3]),
                                pack_bf16(-w[8 * c4 + 4], -w[8 * c4 + 5]), pack_bf16(-w[8 * c4 + 6], -w[8 * c4 + 7]));
                        }
                    }
                }
                if (!fast) exact_scale_k(l, sm + OFF_KQ + s * kKQBytes, s_g);
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(&bars[B_OPS]);
                mbar_arrive(&bars[B_GEMPTY + gbuf]);
            } else if (!p_readout(0)) {
                break;
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ chain warpgroups
        const int h = (warp - 8) >> 2;          // dk half
        const uint32_t q = warp & 3;             // TMEM lane quadrant
        const int x = 32 * q + lane;             // value index (TMEM lane)
        const int d = p.d;
        // S[m] = S[64 h + m][x] (this thread's value column, this warpgroup's key half)
        float S[64];
#pragma unroll
        for (int m = 0; m < 64; ++m) S[m] = 0.f;
        const float *s_in = nullptr;   // state entering this run, [d][d]
        if (use_s0) s_in = p.S0 + (static_cast<int64_t>(b) * p.Hv + hv) * d * d;
        if (p.pass == 0 && exact && seg > 0)
            s_in = p.seg_state + ((static_cast<int64_t>(pr) * p.nseg + seg) * 3 + 2) * d * d;
        if (s_in && x < d && 64 * h < d) {
            const float *src = s_in + static_cast<int64_t>(64 * h) * d + x;
#pragma unroll
            for (int m = 0; m < 64; ++m) {
                S[m] = __ldg(src);
                src += d;
            }
        }
        if (kind == 1) {
#pragma unroll
            for (int m = 0; m < 64; ++m) S[m] = (64 * h + m == x && x < d) ? 1.f : 0.f;
        }
        // j = -1 writes the initial state; j >= 0 processes chunk j and writes the next state.
#pragma unroll 1
        for (int j = -1; j < n; ++j) {
            const float *cs = reinterpret_cast<const float *>(sm + OFF_CHAIN) + ((j + kChainSlots) % kChainSlots) * kChainFloats;
            if (j >= 0) {
                const uint32_t zu = tb + TM_ZU;
                bool ok = bwait(&bars[B_UFULL], j & 1, abort_flag, p.status);
                ok = ok && bwait(&bars[B_OPS], j & 1, abort_flag, p.status);  // per-chunk scales
                if (!warp_ok(ok)) break;
                tc_fence_after();
                {
                    // U^T scaled by lambda, bf16: this half's 32 tokens packed into 16 columns
                    float u[32];
                    tmem_ld32(lane_addr(zu, q, 32 * h), u);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 lam = *reinterpret_cast<const float4 *>(cs + 32 * h + 4 * e4);
                        pk[2 * e4] = pack_bf16(u[4 * e4] * lam.x, u[4 * e4 + 1] * lam.y);
                        pk[2 * e4 + 1] = pack_bf16(u[4 * e4 + 2] * lam.z, u[4 * e4 + 3] * lam.w);
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
                for (int piece = 0; piece < 2; ++piece) {
                    float dd[32];
                    tmem_ld32(lane_addr(tb + TM_D + 64 * h + 32 * piece, q, 0), dd);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) S[32 * piece + e] = fmaf(gC, S[32 * piece + e], dd[e]);
                }
            }
            {
                // S^T bf16 for the next chunk's products (double-buffered)
                const int buf = (j + 1) & 1;
#pragma unroll
                for (int piece = 0; piece < 2; ++piece) {
                    uint32_t u[16];
#pragma unroll
                    for (int c2 = 0; c2 < 16; ++c2) u[c2] = pack_bf16(S[32 * piece + 2 * c2], S[32 * piece + 2 * c2 + 1]);
                    tmem_st16(lane_addr(tb + TM_SB + 64 * buf + 32 * h + 16 * piece, q, 0), u);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[B_SREADY]);
            }
            if (j < 0) continue;
            const int c = c_w + j;
            bool ok = bwait(&bars[B_YFULL], j & 1, abort_flag, p.status);
            if (!warp_ok(ok)) break;
            tc_fence_after();
            uint32_t yb[16];   // y of this lane's 32 tokens, bf16 pairs
            {
                float yv[32];
                tmem_ld32(lane_addr(tb + TM_Y + 32 * h, q, 0), yv);
                tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 gm = *reinterpret_cast<const float4 *>(cs + 64 + 32 * h + 4 * e4);
                    yb[2 * e4] = pack_bf16(yv[4 * e4] * gm.x, yv[4 * e4 + 1] * gm.y);
                    yb[2 * e4 + 1] = pack_bf16(yv[4 * e4 + 2] * gm.z, yv[4 * e4 + 3] * gm.w);
                }
            }
            tc_fence_before();
            mbar_arrive(&bars[B_YFREE]);
            if (c >= c_begin && x < d && p.pass == 0) {
                const int64_t tstart = static_cast<int64_t>(c) * kC + 32 * h;
                uint16_t *yp = reinterpret_cast<uint16_t *>(p.y) + ((static_cast<int64_t>(b) * p.T + tstart) * p.Hv + hv) * d + x;
                const int ystride = p.Hv * d;
                const int nvalid = static_cast<int>(min(static_cast<int64_t>(32), p.T - tstart));
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint32_t pr = yb[i >> 1];
                    if (i < nvalid) yp[i * ystride] = (i & 1) ? static_cast<uint16_t>(pr >> 16) : static_cast<uint16_t>(pr);
                }
            }
        }
        // Where this run's final state goes.  The indices are recomputed from a
        // fresh read of the block index, so that they are not kept in registers
        // across the chunk loop above.
        float *s_out = nullptr;
        {
            uint32_t cta;
            asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(cta));
            const uint32_t per_pass = static_cast<uint32_t>(p.B * p.Hv * p.nseg);
            const int bxr = static_cast<int>(cta % per_pass), pr_r = bxr % (p.B * p.Hv), seg_r = bxr / (p.B * p.Hv);
            if (p.pass == 1)
                s_out = p.seg_state + ((static_cast<int64_t>(pr_r) * p.nseg + seg_r) * 3 + cta / per_pass) * d * d;
            else if (seg_r == p.nseg - 1)
                s_out = p.S_T + static_cast<int64_t>(pr_r) * d * d;
        }
        if (s_out && !*abort_flag && x < d && 64 * h < d) {
            float *dst = s_out + static_cast<int64_t>(64 * h) * d + x;
#pragma unroll
            for (int m = 0; m < 64; ++m) {
                *dst = S[m];
                dst += d;
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

// Which segments have no warm-up window: one CTA (8 warps) per (batch, value
// head, segment after the first), walking back from the segment start eight
// chunks per round as the chunk kernel's warm-up search does.  flag[pair][seg]
// is set when no window of at most max_warmup chunks reaches exp(log_eps)
// (and token 0 is not reached within the limit); a head with any flag set
// takes the exact split.
__global__ void __launch_bounds__(256) segment_plan_kernel(const Dev p, int *flag) {
    const int pairs = p.B * p.Hv;
    const int pr = blockIdx.x % pairs, seg = 1 + static_cast<int>(blockIdx.x / pairs);
    const int b = pr / p.Hv, hv = pr % p.Hv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c_begin = seg * p.seg_chunks;
    __shared__ float wsum[8];
    __shared__ int verdict;
    float acc = 0.f;
    for (int r = 0;; ++r) {
        const int m = r * 8 + warp + 1;
        const int cc = c_begin - m;
        float part = 0.f;
        if (cc >= 0 && m <= p.max_warmup) {
            const int64_t t = static_cast<int64_t>(cc) * kC + lane;
            const float *al = p.alpha + (static_cast<int64_t>(b) * p.T + t) * p.Hv + hv;
            part = logf(__ldg(al)) + logf(__ldg(al + 32 * static_cast<int64_t>(p.Hv)));
        }
        part = warp_sum(part);
        if (lane == 0) wsum[warp] = part;
        __syncthreads();
        if (threadIdx.x == 0) {
            int v = -1;   // -1 undecided, 0 window found (or token 0 reached), 1 none within the limit
            for (int w = 0; w < 8 && v < 0; ++w) {
                const int mm = r * 8 + w + 1;
                if (mm > p.max_warmup) {
                    v = 1;
                    break;
                }
                acc += wsum[w];
                if (acc <= p.log_eps || c_begin - mm == 0) v = 0;
            }
            verdict = v;
        }
        __syncthreads();
        const int v = verdict;
        if (v >= 0) {
            if (threadIdx.x == 0) flag[static_cast<int64_t>(pr) * p.nseg + seg] = v;
            return;
        }
        __syncthreads();
    }
}

// Entering states of the segments of each flagged head: with B_s and M_s the
// ends of segment s's two transition runs (B_0 from the true initial state),
// S_1 = B_0 and S_{s+1} = M_s S_s + B_s, each state [d][d] fp32, row-major.
// One CTA (512 threads) per (batch, value head); S_s and M_s are staged in
// shared memory; each thread owns one column x and the rows r0 + (512/d) u.
template <int D>
__global__ void __launch_bounds__(512) segment_combine_kernel(const int *flag, float *seg_state, int nseg) {
    extern __shared__ float4 smem4[];
    float *st = reinterpret_cast<float *>(smem4);   // S_s, D x D
    float *mt = st + D * D;                         // M_s, D x D
    const int pr = blockIdx.x;
    if (!head_needs_split(flag, pr, nseg)) return;
    constexpr int kRows = D * D / 512;              // rows per thread
    constexpr int kStep = 512 / D;
    const int tid = threadIdx.x;
    const int64_t dd = static_cast<int64_t>(D) * D;
    float *base = seg_state + static_cast<int64_t>(pr) * nseg * 3 * dd;
    for (int e = tid; e < D * D; e += 512) st[e] = base[e];   // S_1 = B_0
    __syncthreads();
    const int x = tid % D, r0 = tid / D;
    for (int sgm = 1; sgm < nseg; ++sgm) {
        float *slot = base + static_cast<int64_t>(sgm) * 3 * dd;
        for (int e = tid; e < D * D; e += 512) {
            slot[2 * dd + e] = st[e];   // entering state of segment sgm
            mt[e] = slot[dd + e];       // M_sgm
        }
        if (sgm == nseg - 1) break;
        __syncthreads();
        float acc[kRows];
#pragma unroll
        for (int u = 0; u < kRows; ++u) acc[u] = slot[static_cast<int64_t>(r0 + kStep * u) * D + x];   // B_sgm
#pragma unroll 1
        for (int k = 0; k < D; k += 4) {
            const float s0 = st[k * D + x], s1 = st[(k + 1) * D + x], s2 = st[(k + 2) * D + x], s3 = st[(k + 3) * D + x];
#pragma unroll
            for (int u = 0; u < kRows; ++u) {
                const float4 m4 = *reinterpret_cast<const float4 *>(mt + (r0 + kStep * u) * D + k);
                acc[u] = fmaf(m4.x, s0, fmaf(m4.y, s1, fmaf(m4.z, s2, fmaf(m4.w, s3, acc[u]))));
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kRows; ++u) st[(r0 + kStep * u) * D + x] = acc[u];
        __syncthreads();
    }
}

// Dynamic shared memory limits of the kernels above, set once per device.
cudaError_t set_smem_attributes() {
    constexpr int kMaxDevices = 64;
    static std::once_flag once[kMaxDevices];
    static cudaError_t result[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        cudaError_t r = cudaFuncSetAttribute(gdn_chunked_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(segment_combine_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     2 * 128 * 128 * 4);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(segment_combine_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     2 * 64 * 64 * 4);
        result[dev] = r;
    });
    return result[dev];
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

cudaError_t launch_segment_combine(const int *flag, float *seg_state, int64_t pairs, int P, int d,
                                   cudaStream_t stream) {
    cudaError_t e = set_smem_attributes();
    if (e != cudaSuccess) return e;
    const size_t comb_smem = 2 * static_cast<size_t>(d) * d * sizeof(float);
    if (d == 128)
        segment_combine_kernel<128><<<static_cast<unsigned>(pairs), 512, comb_smem, stream>>>(flag, seg_state, P);
    else
        segment_combine_kernel<64><<<static_cast<unsigned>(pairs), 512, comb_smem, stream>>>(flag, seg_state, P);
    return cudaGetLastError();
}

bool takes_exact_split(int64_t pairs, int64_t nchunks, int P, int d, size_t seg_state_bytes) {
    // Only for long sequences: below kExactSplitMinChunks chunks per head a
    // restart from token 0 costs less than the split's three extra launches.
    const size_t need = static_cast<size_t>(pairs) * P * 3 * d * d * sizeof(float);
    return P > 1 && nchunks >= kExactSplitMinChunks && need <= seg_state_bytes;
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
    dv.test_stall_chunk = p.test_stall_chunk;
    dv.log_eps = p.log_eps;
    dv.alpha = p.alpha;
    dv.beta = p.beta;
    dv.S0 = p.S0;
    dv.y = static_cast<__nv_bfloat16 *>(p.y);
    dv.S_T = p.S_T;
    dv.status = p.status;

    dv.pass = 0;
    dv.exact_flag = nullptr;
    dv.seg_state = nullptr;

    cudaError_t e = set_smem_attributes();
    if (e != cudaSuccess) return e;
    // Exact sequence split, for the heads whose gates do not decay within the
    // warm-up limit: each segment is an affine map of its entering state, so its
    // two transition runs and a short combine give every segment its exact start.
    // Heads that do not need it leave the extra passes at once.
    if (p.exact_flag && p.seg_state && takes_exact_split(pairs, nchunks, P, p.d, p.seg_state_bytes)) {
        dv.exact_flag = p.exact_flag;
        dv.seg_state = p.seg_state;
        segment_plan_kernel<<<static_cast<unsigned>(pairs * (P - 1)), 256, 0, stream>>>(dv, p.exact_flag);
        dv.pass = 1;
        gdn_chunked_kernel<<<static_cast<unsigned>(2 * grid), kThreads, kSmemBytes, stream>>>(mq, mk, mv, dv);
        const size_t comb_smem = 2 * static_cast<size_t>(p.d) * p.d * sizeof(float);
        if (p.d == 128)
            segment_combine_kernel<128><<<static_cast<unsigned>(pairs), 512, comb_smem, stream>>>(p.exact_flag,
                                                                                                 p.seg_state, P);
        else
            segment_combine_kernel<64><<<static_cast<unsigned>(pairs), 512, comb_smem, stream>>>(p.exact_flag,
                                                                                                p.seg_state, P);
        dv.pass = 0;
    }
    gdn_chunked_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(mq, mk, mv, dv);
    return cudaGetLastError();
}

}  // namespace gdn
