// decode.cu -- one decode token of the gated delta rule, state in place.
//
// Per (sequence, head), with h = S^T [dk][dv] fp32:
//   Sk_j = sum_i h[i][j] k_i,   Sq_j = sum_i h[i][j] q_i
//   delta_j = b (v_j - a Sk_j)
//   h[i][j] <- a h[i][j] + k_i delta_j
//   o_j = a Sq_j + delta_j (k . q)          (= S_t q after the update)
// which is S_t = a S (I - b k k^T) + b v k^T, o = S_t q for one token.
//
// The pass is HBM-bound: each state is read once and written once.  A block
// owns one (sequence, head); each thread holds a 4-column x R-row tile of the
// state in registers (float4 loads and stores, a warp covers whole 512-byte
// rows), the column sums are reduced across row groups in shared memory, and
// the tile is updated and written back from registers.
#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr int kDecodeThreads = 256;

template <int DK, int DV>
__global__ void __launch_bounds__(kDecodeThreads)
decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
              const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ log_alpha,
              const __nv_bfloat16* __restrict__ beta, float* __restrict__ state,
              __nv_bfloat16* __restrict__ o) {
    constexpr int kCols4 = DV / 4;                       // threads across a row
    constexpr int kGroups = kDecodeThreads / kCols4;      // row groups
    constexpr int kRows = DK / kGroups;                   // rows per thread
    static_assert(kRows * kGroups == DK, "row split");

    __shared__ float s_q[DK], s_k[DK];
    __shared__ float4 s_part[2][kGroups][kCols4];
    __shared__ float s_kq;

    const int bh = blockIdx.x, tid = threadIdx.x;
    const int c4 = tid % kCols4, grp = tid / kCols4;
    float4* st = reinterpret_cast<float4*>(state + (size_t)bh * DK * DV);

    // issue the state loads first: they are the whole cost of the step
    float4 tile[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) tile[r] = st[(size_t)(grp * kRows + r) * kCols4 + c4];

    for (int i = tid; i < DK; i += kDecodeThreads) {
        s_q[i] = __bfloat162float(q[(size_t)bh * DK + i]);
        s_k[i] = __bfloat162float(k[(size_t)bh * DK + i]);
    }
    __syncthreads();
    if (tid < 32) {
        float acc = 0.f;
        for (int i = tid; i < DK; i += 32) acc = fmaf(s_k[i], s_q[i], acc);
        for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (tid == 0) s_kq = acc;
    }

    float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sq = sk;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const float ki = s_k[grp * kRows + r], qi = s_q[grp * kRows + r];
        sk.x = fmaf(tile[r].x, ki, sk.x); sk.y = fmaf(tile[r].y, ki, sk.y);
        sk.z = fmaf(tile[r].z, ki, sk.z); sk.w = fmaf(tile[r].w, ki, sk.w);
        sq.x = fmaf(tile[r].x, qi, sq.x); sq.y = fmaf(tile[r].y, qi, sq.y);
        sq.z = fmaf(tile[r].z, qi, sq.z); sq.w = fmaf(tile[r].w, qi, sq.w);
    }
    s_part[0][grp][c4] = sk;
    s_part[1][grp][c4] = sq;
    __syncthreads();
    float4 Sk = make_float4(0.f, 0.f, 0.f, 0.f), Sq = Sk;
#pragma unroll
    for (int g2 = 0; g2 < kGroups; ++g2) {
        float4 a = s_part[0][g2][c4], b = s_part[1][g2][c4];
        Sk.x += a.x; Sk.y += a.y; Sk.z += a.z; Sk.w += a.w;
        Sq.x += b.x; Sq.y += b.y; Sq.z += b.z; Sq.w += b.w;
    }

    const float alpha = __expf(__bfloat162float(log_alpha[bh]));
    const float b = __bfloat162float(beta[bh]);
    const __nv_bfloat16* vb = v + (size_t)bh * DV + 4 * c4;
    float4 d;
    d.x = b * (__bfloat162float(vb[0]) - alpha * Sk.x);
    d.y = b * (__bfloat162float(vb[1]) - alpha * Sk.y);
    d.z = b * (__bfloat162float(vb[2]) - alpha * Sk.z);
    d.w = b * (__bfloat162float(vb[3]) - alpha * Sk.w);

#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const float ki = s_k[grp * kRows + r];
        float4 x = tile[r];
        x.x = fmaf(alpha, x.x, ki * d.x); x.y = fmaf(alpha, x.y, ki * d.y);
        x.z = fmaf(alpha, x.z, ki * d.z); x.w = fmaf(alpha, x.w, ki * d.w);
        st[(size_t)(grp * kRows + r) * kCols4 + c4] = x;
    }
    if (grp == 0) {
        const float kq = s_kq;
        __nv_bfloat16* ob = o + (size_t)bh * DV + 4 * c4;
        __nv_bfloat162 lo = __floats2bfloat162_rn(fmaf(alpha, Sq.x, d.x * kq), fmaf(alpha, Sq.y, d.y * kq));
        __nv_bfloat162 hi = __floats2bfloat162_rn(fmaf(alpha, Sq.z, d.z * kq), fmaf(alpha, Sq.w, d.w * kq));
        reinterpret_cast<__nv_bfloat162*>(ob)[0] = lo;
        reinterpret_cast<__nv_bfloat162*>(ob)[1] = hi;
    }
}

cudaError_t launch_decode(const void* q, const void* k, const void* v, const void* log_alpha,
                          const void* beta, float* state, void* o, int B, int H, int dk, int dv,
                          cudaStream_t st) {
    const unsigned n = (unsigned)B * (unsigned)H;
    if (n == 0) return cudaSuccess;
    auto* Q = (const __nv_bfloat16*)q; auto* K = (const __nv_bfloat16*)k;
    auto* V = (const __nv_bfloat16*)v; auto* LA = (const __nv_bfloat16*)log_alpha;
    auto* BE = (const __nv_bfloat16*)beta; auto* O = (__nv_bfloat16*)o;
    if (dk == 128 && dv == 128) decode_kernel<128, 128><<<n, kDecodeThreads, 0, st>>>(Q, K, V, LA, BE, state, O);
    else if (dk == 128 && dv == 64) decode_kernel<128, 64><<<n, kDecodeThreads, 0, st>>>(Q, K, V, LA, BE, state, O);
    else if (dk == 64 && dv == 128) decode_kernel<64, 128><<<n, kDecodeThreads, 0, st>>>(Q, K, V, LA, BE, state, O);
    else decode_kernel<64, 64><<<n, kDecodeThreads, 0, st>>>(Q, K, V, LA, BE, state, O);
    return cudaGetLastError();
}

}  // namespace gdn
