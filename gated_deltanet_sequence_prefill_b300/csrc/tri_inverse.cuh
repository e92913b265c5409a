// tri_inverse.cuh -- (I + A)^-1 for a strictly lower-triangular 64 x 64 A in
// shared memory, by four warps (the delta-system solve of one chunk).
//
// Blocked forward substitution on 16 x 16 blocks.  The four diagonal blocks
// T_bb = (I + A_bb)^-1 are solved first (one warp per block, one lane per
// column, in column order so the dependent chain is 16 FMAs long).  The
// blocks below the diagonal follow in order of their distance d = i - j from
// it, every block of one distance at once:
//     T_ij = -T_ii * sum_{k=j}^{i-1} A_ik T_kj,
// with each 16 x 8 piece a short chain of warp-level TF32 MMAs.  A block of
// distance d needs only blocks of smaller distance, so three levels finish
// the matrix.  T_ij (i > j) is written into the unused upper block (j, i) --
// element T[16i + a][16j + b] at M[16j + a][16i + b] -- so no A block is
// overwritten while still needed.  Read the result with tri_get().  The
// result is rounded to bf16 by its user, so TF32 products (10-bit mantissa)
// lose nothing that matters.
#pragma once

#include "tc_util.cuh"

namespace gdn {

constexpr int kTriLd = 68;  // row stride (floats) of the 64 x 64 matrix

// Element T[t][s] of the inverse for s <= t (layout above).
__device__ __forceinline__ const float* tri_block_row(const float* M, int t, int jb) {
    const int ib = t >> 4, a = t & 15;
    return jb == ib ? M + t * kTriLd + 16 * ib : M + (16 * jb + a) * kTriLd + 16 * ib;
}

// TF32 operand of a warp-level MMA: the fp32 bits as they are, of which the
// MMA uses the tf32 part (no separate rounding step; the result is rounded to
// bf16 by its users, far coarser than either rounding).
__device__ __forceinline__ uint32_t tf32_bits(float x) { return __float_as_uint(x); }

// On entry M holds A below the diagonal (entries on and above it are never
// read); on exit the layout above.  Called by the 128 threads of warps pw = 0..3 (warp index within the
// group) with named barrier `bar_id`; `scratch` is 4 x 128 floats.  Only the
// blocks at most `maxd` blocks below the diagonal are formed (maxd = 3: the
// whole inverse; maxd = 1: the block-adjacent solver, whose farther blocks
// are taken as zero and never read).
__device__ __forceinline__ void tri_inverse_64(float* M, float* scratch, int pw, int lane,
                                               int bar_id, int maxd) {
    {
        float* B = M + (16 * pw) * kTriLd + 16 * pw;
        const int c = lane & 15;
        // column c by forward substitution, one row of B at a time (four entries
        // per load; entries on and above the diagonal are never used)
        float y[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            float acc = (rr == c) ? 1.f : 0.f;
#pragma unroll
            for (int i4 = 0; i4 < rr; i4 += 4) {
                const float4 b = *reinterpret_cast<const float4*>(B + rr * kTriLd + i4);
                acc = fmaf(-b.x, y[i4], acc);
                if (i4 + 1 < rr) acc = fmaf(-b.y, y[i4 + 1], acc);
                if (i4 + 2 < rr) acc = fmaf(-b.z, y[i4 + 2], acc);
                if (i4 + 3 < rr) acc = fmaf(-b.w, y[i4 + 3], acc);
            }
            y[rr] = acc;
        }
        __syncwarp();
        if (lane < 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) B[i * kTriLd + c] = y[i];
        }
    }
    tc::named_bar(bar_id, 128);

    const int g = lane >> 2, t4 = lane & 3;
    float* scr = scratch + pw * 128;  // 16 x 8, row stride 8
#pragma unroll 1
    for (int d = 1; d <= maxd; ++d) {
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
            const int tile = pw + 4 * q;
            if (tile < 2 * (4 - d)) {
                const int i = d + (tile >> 1), j = i - d, n0 = 8 * (tile & 1);
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                for (int k = j; k < i; ++k) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const float* Ar = M + (16 * i + g) * kTriLd + 16 * k + 8 * kk + t4;
                        uint32_t a[4] = {tf32_bits(Ar[0]), tf32_bits(Ar[8 * kTriLd]),
                                         tf32_bits(Ar[4]), tf32_bits(Ar[8 * kTriLd + 4])};
                        // T_kj rows 8kk + t4 (+4), column n0 + g of block j
                        const float* Br = (k == j)
                                              ? M + (16 * j + 8 * kk + t4) * kTriLd + 16 * j + n0 + g
                                              : M + (16 * j + 8 * kk + t4) * kTriLd + 16 * k + n0 + g;
                        uint32_t b[2] = {tf32_bits(Br[0]), tf32_bits(Br[4 * kTriLd])};
                        tc::mma_tf32(c, a, b);
                    }
                }
                scr[g * 8 + 2 * t4] = c[0];
                scr[g * 8 + 2 * t4 + 1] = c[1];
                scr[(g + 8) * 8 + 2 * t4] = c[2];
                scr[(g + 8) * 8 + 2 * t4 + 1] = c[3];
                __syncwarp();
                float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const float* Tr = M + (16 * i + g) * kTriLd + 16 * i + 8 * kk + t4;
                    uint32_t a[4] = {tf32_bits(Tr[0]), tf32_bits(Tr[8 * kTriLd]),
                                     tf32_bits(Tr[4]), tf32_bits(Tr[8 * kTriLd + 4])};
                    uint32_t b[2] = {tf32_bits(scr[(8 * kk + t4) * 8 + g]),
                                     tf32_bits(scr[(8 * kk + t4 + 4) * 8 + g])};
                    tc::mma_tf32(e, a, b);
                }
                __syncwarp();
                // T_ij[a][b] -> M[16j + a][16i + b]
                float* Or = M + (16 * j + g) * kTriLd + 16 * i + n0 + 2 * t4;
                Or[0] = -e[0];
                Or[1] = -e[1];
                Or[8 * kTriLd] = -e[2];
                Or[8 * kTriLd + 1] = -e[3];
            }
        }
        tc::named_bar(bar_id, 128);
    }
}

}  // namespace gdn
