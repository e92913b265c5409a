// tri_inverse.cuh -- (I + A)^-1 for a strictly lower-triangular 64 x 64 A in
// shared memory, by four warps (the delta-system solve of one chunk).
//
// Forward substitution, blocked in 16 x 16 blocks: the four diagonal blocks
// T_bb = (I + A_bb)^-1 by plain substitution (one thread per column), then
// the blocks below the diagonal row by row,
//     T_ij = -T_ii * sum_{k=j}^{i-1} A_ik T_kj      (i > j),
// each 16 x 8 piece of a block a warp-level TF32 MMA.  The result is rounded
// to bf16 by its user, so TF32 products (10-bit mantissa) lose nothing that
// matters.
#pragma once

#include "tc_util.cuh"

namespace gdn {

constexpr int kTriLd = 68;  // row stride (floats) of the 64 x 64 matrix

// In place: on entry M holds A (zero on and above the diagonal), on exit
// T = (I + A)^-1.  Called by the 128 threads of warps `pw` = 0..3 (warp index
// within the group) with named barrier `bar_id`; `scratch` is 4 x 128 floats.
__device__ __forceinline__ void tri_inverse_64(float* M, float* scratch, int pw, int lane,
                                               int bar_id) {
    // diagonal blocks: warp pw inverts block pw, lane c < 16 owns column c
    {
        float* B = M + (16 * pw) * kTriLd + 16 * pw;
        const int c = lane & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < i; ++j) acc = fmaf(-B[i * kTriLd + j], x[j], acc);
            x[i] = acc;
        }
        __syncwarp();
        if (lane < 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) B[i * kTriLd + c] = x[i];
        }
    }
    tc::named_bar(bar_id, 128);

    const int g = lane >> 2, t4 = lane & 3;
    float* scr = scratch + pw * 128;  // 16 x 8, row stride 8
    for (int bi = 1; bi < 4; ++bi) {
        float res[2][4];
        int tiles[2];
        int nt = 0;
        for (int tile = pw; tile < 2 * bi; tile += 4) {
            const int j = tile >> 1, n0 = 16 * j + 8 * (tile & 1);
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            for (int kb = j; kb < bi; ++kb) {
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int kc = 16 * kb + 8 * kk;
                    const float* Ar = M + (16 * bi + g) * kTriLd + kc + t4;
                    uint32_t a[4] = {tc::to_tf32(Ar[0]), tc::to_tf32(Ar[8 * kTriLd]),
                                     tc::to_tf32(Ar[4]), tc::to_tf32(Ar[8 * kTriLd + 4])};
                    const float* Br = M + (kc + t4) * kTriLd + n0 + g;
                    uint32_t b[2] = {tc::to_tf32(Br[0]), tc::to_tf32(Br[4 * kTriLd])};
                    tc::mma_tf32(c, a, b);
                }
            }
            scr[g * 8 + 2 * t4] = c[0];
            scr[g * 8 + 2 * t4 + 1] = c[1];
            scr[(g + 8) * 8 + 2 * t4] = c[2];
            scr[(g + 8) * 8 + 2 * t4 + 1] = c[3];
            __syncwarp();
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const float* Tr = M + (16 * bi + g) * kTriLd + 16 * bi + 8 * kk + t4;
                uint32_t a[4] = {tc::to_tf32(Tr[0]), tc::to_tf32(Tr[8 * kTriLd]),
                                 tc::to_tf32(Tr[4]), tc::to_tf32(Tr[8 * kTriLd + 4])};
                uint32_t b[2] = {tc::to_tf32(scr[(8 * kk + t4) * 8 + g]),
                                 tc::to_tf32(scr[(8 * kk + t4 + 4) * 8 + g])};
                tc::mma_tf32(d, a, b);
            }
            __syncwarp();
            res[nt][0] = -d[0]; res[nt][1] = -d[1]; res[nt][2] = -d[2]; res[nt][3] = -d[3];
            tiles[nt] = tile;
            ++nt;
        }
        tc::named_bar(bar_id, 128);  // every read of block row bi is done
        for (int q = 0; q < nt; ++q) {
            const int j = tiles[q] >> 1, n0 = 16 * j + 8 * (tiles[q] & 1);
            float* Or = M + (16 * bi + g) * kTriLd + n0 + 2 * t4;
            Or[0] = res[q][0];
            Or[1] = res[q][1];
            Or[8 * kTriLd] = res[q][2];
            Or[8 * kTriLd + 1] = res[q][3];
        }
        tc::named_bar(bar_id, 128);
    }
}

}  // namespace gdn
