// Warp-level tensor-core helpers shared by the kernels built on mma.sync:
// swizzled bf16 tiles in shared memory, ldmatrix lane addresses, bf16 and
// tf32 MMAs, asynchronous copies, and the blocked lower-triangular inverse of
// a 64 x 64 chunk matrix used by the WY/UT form of the chunked recurrence.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace gdn {
namespace wm {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of the 16-byte piece `ch` of row `row` in a tile of 256-byte
// rows (16 pieces) or 128-byte rows (8 pieces), XOR-swizzled by the row so
// that eight rows read at the same column fall in different banks.
__device__ __forceinline__ uint32_t sw256(int row, int ch) { return row * 256 + ((ch ^ (row & 7)) << 4); }
__device__ __forceinline__ uint32_t sw128(int row, int ch) { return row * 128 + ((ch ^ (row & 7)) << 4); }

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void *g) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t a) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t a) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

// d (16 x 8 fp32) += a (16 x 16 bf16, row) * b (16 x 8 bf16, col).
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d (16 x 8 fp32) += a (16 x 8 tf32, row) * b (8 x 8 tf32, col).
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x with the PTX approximation, denormal results flushed to zero.
__device__ __forceinline__ float exp2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) with the PTX approximation (absolute error about 2^-22 near 1).
__device__ __forceinline__ float log2_approx(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Lane addresses of ldmatrix x4 loads (16 x 16 pieces of bf16 tiles).
//  A, row-major [m][k] storage: matrices (m 0-7, k 0-7), (m 8-15, k 0-7), (m 0-7, k 8-15), (m 8-15, k 8-15).
__device__ __forceinline__ int a_row(int lane) { return (lane & 7) + 8 * ((lane >> 3) & 1); }
__device__ __forceinline__ int a_ch(int lane) { return lane >> 4; }
//  B from [n][k] storage (no transpose), two n-tiles: (n 0-7, k 0-7), (n 0-7, k 8-15), (n 8-15, k 0-7), (n 8-15, k 8-15).
__device__ __forceinline__ int bn_row(int lane) { return (lane & 7) + 8 * (lane >> 4); }
__device__ __forceinline__ int bn_ch(int lane) { return (lane >> 3) & 1; }
//  B from [k][n] storage (transposed load), two n-tiles: (k 0-7, n 0-7), (k 8-15, n 0-7), (k 0-7, n 8-15), (k 8-15, n 8-15).
__device__ __forceinline__ int bt_row(int lane) { return (lane & 7) + 8 * ((lane >> 3) & 1); }
__device__ __forceinline__ int bt_ch(int lane) { return lane >> 4; }
//  A from [k][m] storage (transposed load): (k 0-7, m 0-7), (k 0-7, m 8-15), (k 8-15, m 0-7), (k 8-15, m 8-15).
__device__ __forceinline__ int at_row(int lane) { return (lane & 7) + 8 * (lane >> 4); }
__device__ __forceinline__ int at_ch(int lane) { return (lane >> 3) & 1; }

// ------------------------------------------------ lower-triangular inverse
// T = (I + A)^{-1} of the chunk's 64 x 64 strictly lower A by 16 x 16 blocks:
// the four diagonal blocks by forward substitution, then with the left factors
// F_IK = T_II A_IK each off-diagonal block T_IJ = -sum_{K=J}^{I-1} F_IK T_KJ.
// Matrices are block-packed: block (I, J), J <= I, at index I (I + 1) / 2 + J,
// rows of kBS floats; A is column-major within a block, T row-major.
constexpr int kBS = 24;
constexpr int kBlk = 16 * kBS;
constexpr int kBlkFloats = 10 * kBlk;
__device__ __forceinline__ int blk(int I, int J) { return I * (I + 1) / 2 + J; }

// Column `col` of the diagonal block b of T: t[r] = delta(r, col) - sum_{m<r} A[r][m] t[m].
__device__ __forceinline__ void diag_solve(int b, int col, const float *At, float *Tm) {
    const float *Ab = At + blk(b, b) * kBlk;
    float t[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) t[r] = (r == col) ? 1.f : 0.f;
#pragma unroll
    for (int m = 0; m < 15; ++m) {
        const float tm = t[m];
#pragma unroll
        for (int r = m + 1; r < 16; ++r) t[r] = fmaf(-Ab[m * kBS + r], tm, t[r]);
    }
    float *Tb = Tm + blk(b, b) * kBlk + col;
#pragma unroll
    for (int r = 0; r < 16; ++r) Tb[r * kBS] = t[r];
}

// The six left factors as twelve 8-column tiles, three per warp (warps 0-3),
// written in place of A_IK (a warp reads and writes only its own columns).
struct FactorJob {
    uint8_t I, K, nt;
};
static __constant__ FactorJob kFactorJobs[4][3] = {
    {{1, 0, 0}, {1, 0, 1}, {2, 0, 0}},
    {{2, 1, 0}, {2, 1, 1}, {2, 0, 1}},
    {{3, 2, 0}, {3, 2, 1}, {3, 1, 0}},
    {{3, 0, 0}, {3, 0, 1}, {3, 1, 1}},
};

__device__ __forceinline__ void solve_factors(int w, float *At, const float *Tm, int lane) {
    const int gq = lane >> 2, t4 = lane & 3;
    float acc[3][2][4];
    float *fb[3];
    int col[3];
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const FactorJob jb = kFactorJobs[w][u];
        const float *Td = Tm + blk(jb.I, jb.I) * kBlk;
        fb[u] = At + blk(jb.I, jb.K) * kBlk;
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
        float *f = fb[u] + (col[u] - gq + 2 * t4) * kBS + gq;
        f[0] = acc[u][0][0] + acc[u][1][0];
        f[kBS] = acc[u][0][1] + acc[u][1][1];
        f[8] = acc[u][0][2] + acc[u][1][2];
        f[kBS + 8] = acc[u][0][3] + acc[u][1][3];
    }
}

// Off-diagonal blocks of block column J (NNT = 2: both 8-column tiles, NNT = 1:
// tile nt0): T_IJ = -sum_{K=J}^{I-1} F_IK T_KJ for I = J+1..3 in order.
template <int NNT>
__device__ __forceinline__ void solve_column(int J, int nt0, const float *At, float *Tm, int lane) {
    const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll 1
    for (int I = J + 1; I < 4; ++I) {
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float e[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 1
        for (int K = J; K < I; ++K) {
            const float *Fb = At + blk(I, K) * kBlk;   // F[r][k] at k*kBS + r
            const float *Bb = Tm + blk(K, J) * kBlk;   // T[k][n] at k*kBS + n
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int k0 = 8 * ks;
                const uint32_t a0 = __float_as_uint(Fb[(k0 + t4) * kBS + gq]);
                const uint32_t a1 = __float_as_uint(Fb[(k0 + t4) * kBS + gq + 8]);
                const uint32_t a2 = __float_as_uint(Fb[(k0 + t4 + 4) * kBS + gq]);
                const uint32_t a3 = __float_as_uint(Fb[(k0 + t4 + 4) * kBS + gq + 8]);
#pragma unroll
                for (int nt = 0; nt < NNT; ++nt) {
                    const uint32_t b0 = __float_as_uint(Bb[(k0 + t4) * kBS + 8 * (nt0 + nt) + gq]);
                    const uint32_t b1 = __float_as_uint(Bb[(k0 + t4 + 4) * kBS + 8 * (nt0 + nt) + gq]);
                    mma_tf32(ks ? e[nt] : c[nt], a0, a1, a2, a3, b0, b1);
                }
            }
        }
        float *Tb = Tm + blk(I, J) * kBlk;
#pragma unroll
        for (int nt = 0; nt < NNT; ++nt) {
            const int cn = 8 * (nt0 + nt) + 2 * t4;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = gq + 8 * hr;
                *reinterpret_cast<float2 *>(Tb + r * kBS + cn) =
                    make_float2(-(c[nt][2 * hr] + e[nt][2 * hr]), -(c[nt][2 * hr + 1] + e[nt][2 * hr + 1]));
            }
        }
        __syncwarp();
    }
}

}  // namespace wm
}  // namespace gdn
