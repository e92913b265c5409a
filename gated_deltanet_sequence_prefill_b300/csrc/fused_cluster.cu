// fused_cluster.cu -- chunked GDN / linear-attention prefill on a pair of SMs
// (a 2-CTA thread-block cluster per (sequence, head)), sm_103a, bf16 I/O,
// dk = dv = 128, chunk 64.
//
// The chunk stages of the SparseGDN article ("Чем дорог префилл в Gated Delta
// Networks…": intra-chunk delta-system solve, sequential pass over chunks,
// outputs from chunk-start states) are split across the two SMs of the pair
// so that the long-latency solve never holds the buffers the sequential
// state pass needs:
//
//  front CTA (rank 0): the delta-system solve, one chunk ahead or more
//    TMA warp   q, k (2 x 64x64 SW128 boxes each) and the gates of the head
//               into a 3-stage ring; chunk-local cumsum g and decay factors;
//               [k; q] k^T on tcgen05 (M=128 N=64 K=128) into TMEM
//    3 solve warpgroups, chunk c on group c % 3 (one per ring stage):
//               A = beta KK^T exp(g_i - g_j) (strictly lower),
//               P = QK^T exp(g_i - g_j) (causal, diagonal included),
//               T = (I + A)^-1 (tri_inverse.cuh),
//               P staged locally; once the back has armed the chunk's slot,
//               P (64x64 bf16) and [T diag(beta e^g) | 0 | T diag(beta)] are
//               pushed into the back CTA's shared memory with st.async
//  back CTA (rank 1): everything that touches the state
//    TMA warp   k, q, v (both 64-column halves) and the gates into a 2-slot
//               ring; the gate factors the back needs
//    apply      w = T diag(beta e^g) k  -> TMEM, then -w (bf16) into the slot
//               u = T diag(beta) v      -> written by the MMA straight into
//                                          rows 64..127 of the chain's D1
//               q~ = q e^g, k~ = k e^{g_last - g} (in place)
//    chain      8 warps; h = S^T (128 x 128 fp32) in registers, each thread
//               one row and one 64-column half
//               D1 += [q~; -w] h        (M=128 N=128 K=128, accumulating onto
//                                        [0; u]: rows 64..127 become v_new)
//               v_new -> bf16 smem; D2 = k~^T v_new; D1[0:64] += P v_new
//               h <- e^{g_last} h + D2; o = D1[0:64]
//
// HBM sees q, k, v, gates, h0 in and o, h_T out; q and k are read by both
// CTAs (the second read is an L2 hit).  All waits are bounded; a wait that
// runs out sets GDN_ERR_TIMEOUT in the workspace status word and both CTAs
// unwind without skipping any barrier.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"
#include "tri_inverse.cuh"

namespace gdn {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
bool encode_token_map(CUtensorMap* m, const void* ptr, int64_t T, int H);
bool encode_gate_map(CUtensorMap* m, const float* ptr, int64_t T, int H);

namespace pair {

constexpr int kThreads = 416;  // 13 warps in both CTAs
constexpr int kD = 128;

// ---------------------------------------------------------------- front layout
constexpr uint32_t kFK0 = 0, kFQ0 = 8192, kFK1 = 16384, kFQ1 = 24576;  // [k0 q0 | k1 q1]
constexpr uint32_t kFBlk = 16384;                                         // K-block stride
constexpr uint32_t kFGRaw = 32768;                                        // la [64][4], beta [64][4]
constexpr uint32_t kFGate = 34816;                                        // derived gate arrays
constexpr uint32_t kFStage = 36864;
constexpr int kFGroups = 3;                                // = ring stages: chunk c uses both c % 3
constexpr uint32_t kFPst = kFGroups * kFStage;             // 3 x P staging (bf16 64x64, swizzled)
constexpr uint32_t kFAF = kFPst + kFGroups * 8192;         // 3 x A/T fp32 [64][68]
constexpr uint32_t kFScr = kFAF + kFGroups * 64 * kTriLd * 4;  // 3 x 4 x 128 floats
constexpr uint32_t kFBar = kFScr + kFGroups * 4 * 128 * 4;
constexpr uint32_t kFEnd = kFBar + 32 * 8 + 64;

// ---------------------------------------------------------------- back layout
constexpr uint32_t kBK0 = 0, kBQ0 = 8192, kBW0 = 16384, kBK1 = 24576, kBQ1 = 32768, kBW1 = 40960;
constexpr uint32_t kBBlk = 24576;  // stride between the two 64-column blocks of k, q, w
constexpr uint32_t kBV0 = 49152, kBV1 = 57344, kBP = 65536;
constexpr uint32_t kBGRaw = 73728, kBGate = 75776;
constexpr uint32_t kBSlot = 77824;
constexpr uint32_t kBTP = 2 * kBSlot;            // [T' | 0 | T''], 3 x 8 KB
constexpr uint32_t kBHB = kBTP + 3 * 8192;       // h bf16 [128][128]: two 64-column blocks
constexpr uint32_t kBVN = kBHB + 2 * 16384;      // v_new bf16 [64][128]: two 64-column blocks
constexpr uint32_t kBBar = kBVN + 2 * 8192;
constexpr uint32_t kBEnd = kBBar + 32 * 8 + 64;

constexpr uint32_t kSmemBytes = (kFEnd > kBEnd ? kFEnd : kBEnd);
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kFBar + 32 * 8 <= kSmemBytes && kBBar + 32 * 8 <= kSmemBytes, "barriers");

// gate arrays (float index from the gate area); scalars at kGscal:
// [0] e^{g_last}, [1] safe-factor flag, [2] n valid
constexpr int kGg = 0, kGeg = 64, kGeng = 128, kGbeg = 192, kGbb = 256, kGkdec = 320, kGscal = 384;

// ---------------------------------------------------------------- barriers
// front
enum {
    F_FULL = 0,     // [3] TMA landed
    F_GREADY = 3,   // [3] gate values derived
    F_EMPTY = 6,    // [3] stage free
    F_P1D = 9,      // [3] [k;q]k^T done in DP1[group]
    F_P1F = 12,     // [3] DP1[group] read
    F_ARMED = 15,   // [2] back slot armed for this use   (remote arrive by the back)
    F_TPF = 17,     // TP buffer consumed by the back      (remote arrive by the back)
    F_PUSHED = 18,  // [3] group pushed its chunk (orders the pushes of the three groups)
    F_FIN = 21,
    F_COUNT = 22
};
// back
enum {
    B_FULLT = 0,    // [2] own TMA landed
    B_FULLP = 2,    // [2] P and TP pushed by the front
    B_GREADY = 4,   // [2] gate values derived
    B_SLOTFREE = 6, // [2] the chain is done with the slot
    B_D1F = 8,      // [2] D1[b] read by the output epilogue (count 4 warps)
    B_P2D = 10,     // w / u MMAs done
    B_READY = 11,   // [2] slot operands ready for the chain
    B_M1 = 13,      // [q~; -w] h done
    B_M2 = 14,      // k~^T v_new done
    B_M3 = 15,      // P v_new done
    B_FIN = 16,
    B_COUNT = 17
};

// TMEM columns
constexpr uint32_t kFColP1 = 0;        // front: 3 x 64
constexpr uint32_t kFTmemCols = 256;
constexpr uint32_t kBColW = 0;         // back: w 128
constexpr uint32_t kBColD1 = 128;      // back: D1 2 x 128
constexpr uint32_t kBColD2 = 384;      // back: D2 128
constexpr uint32_t kBTmemCols = 512;

constexpr uint32_t kIdP1 = tc::idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdP2w = tc::idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdP2u = tc::idesc_bf16(128, 128, false, true);
constexpr uint32_t kId1 = tc::idesc_bf16(128, 128, false, true);
constexpr uint32_t kId2 = tc::idesc_bf16(128, 128, true, true);
constexpr uint32_t kId3 = tc::idesc_bf16(128, 128, false, true);

__device__ __forceinline__ void report_timeout(char* ws, volatile int* abort_flag) {
    atomicExch(&reinterpret_cast<WsHeader*>(ws)->status, GDN_ERR_TIMEOUT);
    *abort_flag = 1;
}

// Bounded waits that stop waiting once this CTA has aborted; every thread
// keeps executing the same sequence of named barriers after an abort.
struct Waiter {
    volatile int* abort_flag;
    char* ws;
    __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
        if (*abort_flag) return false;
        if (tc::mbar_wait(bar, parity)) return true;
        report_timeout(ws, abort_flag);
        return false;
    }
    __device__ __forceinline__ bool remote(uint32_t bar, uint32_t parity) const {
        if (*abort_flag) return false;
        if (tc::mbar_wait_cluster(bar, parity)) return true;
        report_timeout(ws, abort_flag);
        return false;
    }
};

__device__ __forceinline__ void store_row64(uint32_t tile, uint32_t r, const float* v) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        tc::st_shared_v4(tc::sw128(tile, r, j), tc::pack_bf16(v[8 * j], v[8 * j + 1]),
                         tc::pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                         tc::pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                         tc::pack_bf16(v[8 * j + 6], v[8 * j + 7]));
}
// -v as one bf16 row of a 128-byte-swizzled tile.
__device__ __forceinline__ void store_row64_neg(uint32_t tile, uint32_t r, const float* v) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        tc::st_shared_v4(tc::sw128(tile, r, j), tc::pack_bf16(-v[8 * j], -v[8 * j + 1]),
                         tc::pack_bf16(-v[8 * j + 2], -v[8 * j + 3]),
                         tc::pack_bf16(-v[8 * j + 4], -v[8 * j + 5]),
                         tc::pack_bf16(-v[8 * j + 6], -v[8 * j + 7]));
}
// The same row, written into another CTA's tile with st.async.
__device__ __forceinline__ void push_row64(uint32_t remote_tile, uint32_t r, const float* v,
                                           uint32_t remote_bar) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        tc::st_async_v4(tc::sw128(remote_tile, r, j), tc::pack_bf16(v[8 * j], v[8 * j + 1]),
                        tc::pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                        tc::pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                        tc::pack_bf16(v[8 * j + 6], v[8 * j + 7]), remote_bar);
}

__device__ __forceinline__ void scale_row(uint32_t box0, uint32_t r, float f) {
    const __nv_bfloat162 f2 = __float2bfloat162_rn(f);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t a = tc::sw128(box0 + half * kBBlk, r, j);
            uint4 x = tc::ld_shared_v4(a);
            __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&x);
            p[0] = __hmul2(p[0], f2);
            p[1] = __hmul2(p[1], f2);
            p[2] = __hmul2(p[2], f2);
            p[3] = __hmul2(p[3], f2);
            tc::st_shared_v4(a, x.x, x.y, x.z, x.w);
        }
    }
}

// Per-token gate values of a chunk (one warp): running sum g of log_alpha
// (rows past the chunk end contribute nothing), exp(g), exp(-g), beta,
// beta e^g, k decay exp(g_last - g) (0 past the end), and the scalars.
template <bool GDN>
__device__ __forceinline__ void derive_gates(const float* la_raw, const float* b_raw, int hc, int n,
                                             float* gt, int lane) {
    const int ta = lane, tb = lane + 32;
    float ga = 0.f, gb = 0.f, ba, bb;
    if (GDN) {
        ga = ta < n ? la_raw[ta * 4 + hc] : 0.f;
        gb = tb < n ? la_raw[tb * 4 + hc] : 0.f;
        ba = ta < n ? b_raw[ta * 4 + hc] : 0.f;
        bb = tb < n ? b_raw[tb * 4 + hc] : 0.f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            float xa = __shfl_up_sync(0xffffffffu, ga, off);
            float xb = __shfl_up_sync(0xffffffffu, gb, off);
            if (lane >= off) { ga += xa; gb += xb; }
        }
        gb += __shfl_sync(0xffffffffu, ga, 31);
    } else {
        ba = ta < n ? 1.f : 0.f;
        bb = tb < n ? 1.f : 0.f;
    }
    const int last = n - 1;
    const float glast = __shfl_sync(0xffffffffu, last < 32 ? ga : gb, last & 31);
    float amax = fmaxf(ta < n ? fabsf(ga) : 0.f, tb < n ? fabsf(gb) : 0.f);
#pragma unroll
    for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float ega = __expf(ga), egb = __expf(gb);
    gt[kGg + ta] = ga;
    gt[kGg + tb] = gb;
    gt[kGeg + ta] = ega;
    gt[kGeg + tb] = egb;
    gt[kGeng + ta] = __expf(-ga);
    gt[kGeng + tb] = __expf(-gb);
    gt[kGbeg + ta] = ba * ega;
    gt[kGbeg + tb] = bb * egb;
    gt[kGbb + ta] = ba;
    gt[kGbb + tb] = bb;
    gt[kGkdec + ta] = ta < n ? __expf(glast - ga) : 0.f;
    gt[kGkdec + tb] = tb < n ? __expf(glast - gb) : 0.f;
    if (lane == 0) {
        gt[kGscal + 0] = __expf(glast);
        gt[kGscal + 1] = amax <= 40.f ? 1.f : 0.f;
        gt[kGscal + 2] = (float)n;
    }
    __syncwarp();
}

template <bool GDN>
__global__ void __launch_bounds__(kThreads, 1)
pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
            const __grid_constant__ CUtensorMap tm_b, const float* __restrict__ h0,
            __nv_bfloat16* __restrict__ o, float* __restrict__ h_T, char* __restrict__ ws, int H) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    char* const sptr = reinterpret_cast<char*>(smem_raw) + pad;
    const uint32_t sbase = raw + pad;  // identical in both CTAs (same kernel, same layout)

    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    const bool dead = hdr->status != GDN_OK;  // uniform across the cluster

    const uint32_t rank = tc::cluster_rank();
    const bool front = rank == 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_seqs = hdr->n_seqs;
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* order = reinterpret_cast<const int*>(ws + L.order);
    const int unit = blockIdx.x >> 1;
    const int seq = dead ? 0 : order[unit / H];
    const int head = unit % H;
    const int start = dead ? 0 : cu[seq];
    const int len = dead ? 0 : cu[seq + 1] - start;
    const int nch = (len + kChunk - 1) / kChunk;

    const uint32_t bar_base = sbase + (front ? kFBar : kBBar);
    auto bar = [&](int i) { return bar_base + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + (front ? kFBar : kBBar) + 32 * 8);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + (front ? kFBar : kBBar) + 32 * 8 + 8);
    const Waiter wait{abort_flag, ws};

    if (tid == 0) {
        *abort_flag = 0;
        if (front) {
            for (int b = 0; b < F_COUNT; ++b) tc::mbar_init(bar(b), b == F_FIN ? 4 : 1);
        } else {
            for (int b = 0; b < B_COUNT; ++b) {
                uint32_t cnt = 1;
                if (b == B_D1F || b == B_D1F + 1) cnt = 4;
                if (b == B_FIN) cnt = 2;
                tc::mbar_init(bar(b), cnt);
            }
        }
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        if (!front) tc::prefetch_tmap(&tm_v);
        if (GDN) {
            tc::prefetch_tmap(&tm_la);
            tc::prefetch_tmap(&tm_b);
        }
    }
    if (!front) {
        // the zero block between T' and T'' (the rows 0..63 of the u MMA's A operand),
        // and w = 0 for linear attention
        for (int i = tid; i < 8192 / 16; i += kThreads) tc::st_shared_v4(sbase + kBTP + 8192 + 16 * i, 0, 0, 0, 0);
        if (!GDN)
            for (int i = tid; i < 2 * 2 * 8192 / 16; i += kThreads) {
                const int s = i / 1024, rest = i % 1024, box = rest / 512, off = (rest % 512) * 16;
                tc::st_shared_v4(sbase + s * kBSlot + (box ? kBW1 : kBW0) + off, 0, 0, 0, 0);
            }
        tc::fence_proxy_async();
    }
    if (warp == 0) tc::tmem_alloc(sbase + (front ? kFBar : kBBar) + 32 * 8 + 8, front ? kFTmemCols : kBTmemCols);
    tc::tc_fence_before();
    __syncthreads();
    tc::cluster_sync();  // both CTAs' barriers exist before any remote access
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int quad = warp & 3;
    const int row = 32 * quad + lane;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;

    // peer addresses (front -> back)
    const uint32_t peer_base = tc::map_to_rank(sbase, 1);
    const uint32_t peer_bar_b = peer_base + kBBar;  // back barrier array, as seen from the front
    const uint32_t peer_bar_f = tc::map_to_rank(sbase + kFBar, 0);  // front barriers, seen from the back

    const bool issuer0 = (warp == 0 && lane == 0);

    if (front) {
        // ============================================================ FRONT
        if (warp == 0) {
            // ---- TMA, [k; q] k^T, gates (chunk c in stage / group c % 3)
            int issued = 0;
            for (int c = 0; c < nch && !dead; ++c) {
                const int f = c % kFGroups, uf = c / kFGroups;
                const uint32_t st = sbase + f * kFStage;
                if (c >= kFGroups) wait(bar(F_EMPTY + f), (uf - 1) & 1);
                const int t0 = start + c * kChunk;
                if (lane == 0 && !*abort_flag) {
                    tc::mbar_arrive_expect_tx(bar(F_FULL + f), 32768 + (GDN ? 2048 : 0));
                    tc::tma_load_3d(st + kFK0, &tm_k, 0, head, t0, bar(F_FULL + f));
                    tc::tma_load_3d(st + kFK1, &tm_k, 64, head, t0, bar(F_FULL + f));
                    tc::tma_load_3d(st + kFQ0, &tm_q, 0, head, t0, bar(F_FULL + f));
                    tc::tma_load_3d(st + kFQ1, &tm_q, 64, head, t0, bar(F_FULL + f));
                    if (GDN) {
                        tc::tma_load_2d(st + kFGRaw, &tm_la, head & ~3, t0, bar(F_FULL + f));
                        tc::tma_load_2d(st + kFGRaw + 1024, &tm_b, head & ~3, t0, bar(F_FULL + f));
                    }
                    issued = c + 1;
                    if (c + 4 < nch) {
                        const int tp = t0 + 4 * kChunk;
                        tc::tma_prefetch_3d(&tm_k, 0, head, tp);
                        tc::tma_prefetch_3d(&tm_k, 64, head, tp);
                        tc::tma_prefetch_3d(&tm_q, 0, head, tp);
                        tc::tma_prefetch_3d(&tm_q, 64, head, tp);
                        if (GDN) {
                            tc::tma_prefetch_2d(&tm_la, head & ~3, tp);
                            tc::tma_prefetch_2d(&tm_b, head & ~3, tp);
                        }
                    }
                }
                __syncwarp();
                wait(bar(F_FULL + f), uf & 1);
                if (lane == 0) {
                    if (c >= kFGroups) wait(bar(F_P1F + f), (uf - 1) & 1);
                    if (!*abort_flag) {
                        tc::tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = (kk >> 2) * kFBlk + (kk & 3) * 32;
                            tc::mma_bf16(tmem + kFColP1 + f * 64, tc::sdesc(st + kFK0 + off, 16, 1024),
                                         tc::sdesc(st + kFK0 + off, 16, 1024), kIdP1, kk > 0);
                        }
                        tc::mma_commit(bar(F_P1D + f));
                    }
                }
                const float* la_raw = reinterpret_cast<const float*>(sptr + f * kFStage + kFGRaw);
                derive_gates<GDN>(la_raw, la_raw + 256, head & 3, min(kChunk, len - c * kChunk),
                                  reinterpret_cast<float*>(sptr + f * kFStage + kFGate), lane);
                if (lane == 0) tc::mbar_arrive(bar(F_GREADY + f));
            }
            if (lane == 0 && *abort_flag)
                for (int c = max(0, issued - kFGroups); c < issued; ++c)
                    tc::mbar_wait(bar(F_FULL + c % kFGroups), (c / kFGroups) & 1);
            if (issuer0) tc::mma_commit(bar(F_FIN));
        } else {
            // ---- solve groups: group g takes chunks c with c % 3 == g
            const int grp = (warp - 1) >> 2;  // 0, 1, 2
            const int pw = (warp - 1) & 3;    // warp within the group
            const int nb = 1 + grp;           // named barrier of the group
            const bool gissuer = (pw == 3 && lane == 0);  // row 0 of the group (quadrant 0)
            float* AF = reinterpret_cast<float*>(sptr + kFAF + grp * 64 * kTriLd * 4);
            float* scr = reinterpret_cast<float*>(sptr + kFScr + grp * 4 * 128 * 4);
            const uint32_t pst = sbase + kFPst + grp * 8192;
            for (int c = grp; c < nch && !dead; c += kFGroups) {
                const int uf = c / kFGroups, s = c & 1, us = c >> 1;
                wait(bar(F_GREADY + grp), uf & 1);
                wait(bar(F_P1D + grp), uf & 1);
                tc::tc_fence_after();
                const float* gt = reinterpret_cast<const float*>(sptr + grp * kFStage + kFGate);
                const bool safe = gt[kGscal + 1] != 0.f;
                const int n = (int)gt[kGscal + 2];
                float x[64];
                tc::tmem_ld32(tmem + lane_off + kFColP1 + grp * 64, *reinterpret_cast<float(*)[32]>(x));
                tc::tmem_ld32(tmem + lane_off + kFColP1 + grp * 64 + 32, *reinterpret_cast<float(*)[32]>(x + 32));
                tc::tmem_wait_ld();
                tc::tc_fence_before();
                tc::named_bar(nb, 128);
                if (gissuer) tc::mbar_arrive(bar(F_P1F + grp));
                // rows 0..63: K K^T -> A (fp32); rows 64..127: Q K^T -> P (staged, bf16)
                {
                    const int t = row & 63;
                    const bool is_a = row < 64;
                    if (!is_a || GDN) {
                        const float rs = (is_a ? gt[kGbb + t] : 1.f) * gt[kGeg + t];
                        const int lim = is_a ? t : t + 1;
                        const bool tok = t < n;
                        if (safe) {
#pragma unroll
                            for (int q4 = 0; q4 < 16; ++q4) {
                                const float4 en = *reinterpret_cast<const float4*>(gt + kGeng + 4 * q4);
                                const int s0 = 4 * q4;
                                x[s0 + 0] = (tok && s0 + 0 < lim) ? x[s0 + 0] * en.x * rs : 0.f;
                                x[s0 + 1] = (tok && s0 + 1 < lim) ? x[s0 + 1] * en.y * rs : 0.f;
                                x[s0 + 2] = (tok && s0 + 2 < lim) ? x[s0 + 2] * en.z * rs : 0.f;
                                x[s0 + 3] = (tok && s0 + 3 < lim) ? x[s0 + 3] * en.w * rs : 0.f;
                            }
                        } else {
                            const float gtt = gt[kGg + t], bsc = is_a ? gt[kGbb + t] : 1.f;
#pragma unroll
                            for (int sidx = 0; sidx < 64; ++sidx)
                                x[sidx] = (tok && sidx < lim) ? x[sidx] * bsc * __expf(gtt - gt[kGg + sidx]) : 0.f;
                        }
                        if (is_a) {
                            float* Ar = AF + t * kTriLd;
#pragma unroll
                            for (int q4 = 0; q4 < 16; ++q4)
                                *reinterpret_cast<float4*>(Ar + 4 * q4) =
                                    make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
                        } else {
                            store_row64(pst, t, x);
                        }
                    }
                }
                tc::named_bar(nb, 128);
                if (GDN) tri_inverse_64(AF, scr, pw, lane, nb);
                // ---- push P and [T diag(beta e^g) | 0 | T diag(beta)] in chunk order, once
                // the back has consumed the previous TP and armed this chunk's slot (the
                // pushed bytes are counted on that slot's barrier).  Waiting for chunk
                // c - 1's push first keeps every parity wait below at most one phase behind.
                if (c >= 1) {
                    wait(bar(F_PUSHED + (c - 1) % kFGroups), ((c - 1) / kFGroups) & 1);
                    wait.remote(bar(F_TPF), (c - 1) & 1);
                }
                wait.remote(bar(F_ARMED + s), us & 1);
                if (!*abort_flag) {
                    const int t = row & 63;
                    const uint32_t fb = peer_bar_b + 8u * (B_FULLP + s);
                    if (row >= 64) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 pv = tc::ld_shared_v4(tc::sw128(pst, t, j));
                            tc::st_async_v4(tc::sw128(peer_base + s * kBSlot + kBP, t, j), pv.x, pv.y, pv.z, pv.w, fb);
                        }
                    }
                    const float* cs = gt + (row < 64 ? kGbeg : kGbb);
                    const uint32_t tp = peer_base + kBTP + (row < 64 ? 0u : 16384u);
#pragma unroll
                    for (int jb = 0; jb < 4; ++jb) {
                        float v16[16];
                        if (GDN && jb <= (t >> 4)) {
                            const float* Tr = tri_block_row(AF, t, jb);
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const float4 tv = *reinterpret_cast<const float4*>(Tr + e);
                                const float4 sv = *reinterpret_cast<const float4*>(cs + 16 * jb + e);
                                v16[e] = tv.x * sv.x; v16[e + 1] = tv.y * sv.y;
                                v16[e + 2] = tv.z * sv.z; v16[e + 3] = tv.w * sv.w;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v16[e] = (!GDN && 16 * jb + e == t) ? cs[t] : 0.f;
                        }
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2)
                            tc::st_async_v4(tc::sw128(tp, t, 2 * jb + h2), tc::pack_bf16(v16[8 * h2], v16[8 * h2 + 1]),
                                            tc::pack_bf16(v16[8 * h2 + 2], v16[8 * h2 + 3]),
                                            tc::pack_bf16(v16[8 * h2 + 4], v16[8 * h2 + 5]),
                                            tc::pack_bf16(v16[8 * h2 + 6], v16[8 * h2 + 7]), fb);
                    }
                }
                tc::named_bar(nb, 128);  // AF, the P staging and the stage's gate values are free
                if (gissuer) {
                    tc::mbar_arrive(bar(F_PUSHED + grp));
                    tc::mbar_arrive(bar(F_EMPTY + grp));
                }
            }
            if (gissuer) tc::mbar_arrive(bar(F_FIN));
        }
    } else {
        // ============================================================ BACK
        if (warp == 0) {
            // ---- TMA, gates, slot arming
            int issued = 0;
            for (int c = 0; c < nch && !dead; ++c) {
                const int s = c & 1, u = c >> 1;
                const uint32_t st = sbase + s * kBSlot;
                if (c >= 2) wait(bar(B_SLOTFREE + s), (u - 1) & 1);
                const int t0 = start + c * kChunk;
                if (lane == 0 && !*abort_flag) {
                    tc::mbar_arrive_expect_tx(bar(B_FULLT + s), 3 * 16384 + (GDN ? 2048 : 0));
                    tc::tma_load_3d(st + kBK0, &tm_k, 0, head, t0, bar(B_FULLT + s));
                    tc::tma_load_3d(st + kBK1, &tm_k, 64, head, t0, bar(B_FULLT + s));
                    tc::tma_load_3d(st + kBV0, &tm_v, 0, head, t0, bar(B_FULLT + s));
                    tc::tma_load_3d(st + kBV1, &tm_v, 64, head, t0, bar(B_FULLT + s));
                    tc::tma_load_3d(st + kBQ0, &tm_q, 0, head, t0, bar(B_FULLT + s));
                    tc::tma_load_3d(st + kBQ1, &tm_q, 64, head, t0, bar(B_FULLT + s));
                    if (GDN) {
                        tc::tma_load_2d(st + kBGRaw, &tm_la, head & ~3, t0, bar(B_FULLT + s));
                        tc::tma_load_2d(st + kBGRaw + 1024, &tm_b, head & ~3, t0, bar(B_FULLT + s));
                    }
                    issued = c + 1;
                    // arm the push barrier of this slot, then tell the front
                    tc::mbar_arrive_expect_tx(bar(B_FULLP + s), 8192 + 16384);
                    tc::mbar_arrive_remote(peer_bar_f + 8u * (F_ARMED + s));
                    if (c + 2 < nch) {
                        const int tp = t0 + 2 * kChunk;
                        tc::tma_prefetch_3d(&tm_v, 0, head, tp);
                        tc::tma_prefetch_3d(&tm_v, 64, head, tp);
                    }
                }
                __syncwarp();
                wait(bar(B_FULLT + s), u & 1);
                const float* la_raw = reinterpret_cast<const float*>(sptr + s * kBSlot + kBGRaw);
                derive_gates<GDN>(la_raw, la_raw + 256, head & 3, min(kChunk, len - c * kChunk),
                                  reinterpret_cast<float*>(sptr + s * kBSlot + kBGate), lane);
                if (lane == 0) tc::mbar_arrive(bar(B_GREADY + s));
            }
            if (lane == 0 && *abort_flag)
                for (int c = max(0, issued - 2); c < issued; ++c) tc::mbar_wait(bar(B_FULLT + (c & 1)), (c >> 1) & 1);
        } else if (warp <= 4) {
            // ---- apply: w = T' k (-> -w bf16), u = T'' v (-> the chain's D1), q~, k~
            const bool aissuer = (warp == 4 && lane == 0);
            for (int c = 0; c < nch && !dead; ++c) {
                const int s = c & 1, u = c >> 1, b = c & 1;
                const uint32_t st = sbase + s * kBSlot;
                wait(bar(B_FULLT + s), u & 1);
                wait.remote(bar(B_FULLP + s), u & 1);
                if (aissuer) {
                    if (c >= 2) wait(bar(B_D1F + b), ((c >> 1) - 1) & 1);
                    if (!*abort_flag) {
                        tc::tc_fence_after();
                        if (GDN) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc::mma_bf16(tmem + kBColW, tc::sdesc(sbase + kBTP + kk * 32, 16, 1024),
                                             tc::sdesc(st + kBK0 + kk * 2048, kBBlk, 1024), kIdP2w, kk > 0);
                        }
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)  // D1 = [0; u]
                            tc::mma_bf16(tmem + kBColD1 + b * 128, tc::sdesc(sbase + kBTP + 8192 + kk * 32, 16, 1024),
                                         tc::sdesc(st + kBV0 + kk * 2048, 8192, 1024), kIdP2u, kk > 0);
                        tc::mma_commit(bar(B_P2D));
                    }
                }
                wait(bar(B_P2D), c & 1);
                tc::tc_fence_after();
                if (aissuer) tc::mbar_arrive_remote(peer_bar_f + 8u * F_TPF);  // TP buffer consumed
                wait(bar(B_GREADY + s), u & 1);
                const float* gt = reinterpret_cast<const float*>(sptr + s * kBSlot + kBGate);
                if (row < 64) {
                    if (GDN) {  // -w row -> bf16 into the w boxes
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            float x[64];
                            tc::tmem_ld32(tmem + lane_off + kBColW + 64 * half, *reinterpret_cast<float(*)[32]>(x));
                            tc::tmem_ld32(tmem + lane_off + kBColW + 64 * half + 32,
                                          *reinterpret_cast<float(*)[32]>(x + 32));
                            tc::tmem_wait_ld();
                            store_row64_neg(st + (half ? kBW1 : kBW0), row, x);
                        }
                    } else {
                        scale_row(st + kBK0, row, gt[kGkdec + row]);
                    }
                } else {
                    const int t = row - 64;
                    if (GDN) {
                        scale_row(st + kBQ0, t, gt[kGeg + t]);
                        scale_row(st + kBK0, t, gt[kGkdec + t]);
                    }
                }
                tc::fence_proxy_async();
                tc::tc_fence_before();
                tc::named_bar(1, 128);
                if (aissuer) tc::mbar_arrive(bar(B_READY + s));
            }
            if (aissuer) tc::mma_commit(bar(B_FIN));
        } else {
            // ---- the chain: 8 warps; thread = (row r of h, 64-column half hw)
            const int hw = (warp - 5) >> 2;  // 0, 1
            const int j0 = 64 * hw;
            const int r = row;
            const bool cissuer = (warp == 6 && lane == 0);  // row 64 of half 0
            const size_t hoff = (((size_t)seq * H + head) * kD + r) * kD + j0;
            const uint32_t hb = sbase + kBHB, vn = sbase + kBVN;
            float h[64];
            if (h0 && !dead) {
#pragma unroll
                for (int e = 0; e < 64; e += 4) {
                    float4 v4 = *reinterpret_cast<const float4*>(h0 + hoff + e);
                    h[e] = v4.x; h[e + 1] = v4.y; h[e + 2] = v4.z; h[e + 3] = v4.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) h[e] = 0.f;
            }
            store_row64(hb + hw * 16384, r, h);
            tc::fence_proxy_async();
            tc::named_bar(2, 256);
            for (int c = 0; c < nch && !dead; ++c) {
                const int s = c & 1, u = c >> 1, b = c & 1;
                const uint32_t st = sbase + s * kBSlot;
                const uint32_t d1 = tmem + kBColD1 + b * 128;
                wait(bar(B_READY + s), u & 1);
                const float* gt = reinterpret_cast<const float*>(sptr + s * kBSlot + kBGate);
                if (cissuer && !*abort_flag) {  // D1 = [0; u] + [q~; -w] h
                    tc::tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_bf16(d1, tc::sdesc(st + kBQ0 + (kk >> 2) * kBBlk + (kk & 3) * 32, 16, 1024),
                                     tc::sdesc(hb + kk * 2048, 16384, 1024), kId1, 1);
                    tc::mma_commit(bar(B_M1));
                }
                if (r >= 64) {  // rows 64..127 of D1 now hold v_new
                    wait(bar(B_M1), c & 1);
                    tc::tc_fence_after();
                    const int t = r - 64;
#pragma unroll
                    for (int part = 0; part < 4; ++part) {
                        float x[16];
                        tc::tmem_ld16(d1 + lane_off + j0 + 16 * part, x);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int q8 = 0; q8 < 2; ++q8)
                            tc::st_shared_v4(tc::sw128(vn + hw * 8192, t, 2 * part + q8),
                                             tc::pack_bf16(x[8 * q8], x[8 * q8 + 1]),
                                             tc::pack_bf16(x[8 * q8 + 2], x[8 * q8 + 3]),
                                             tc::pack_bf16(x[8 * q8 + 4], x[8 * q8 + 5]),
                                             tc::pack_bf16(x[8 * q8 + 6], x[8 * q8 + 7]));
                    }
                    tc::fence_proxy_async();
                    tc::tc_fence_before();
                    tc::named_bar(3, 128);
                    if (cissuer && !*abort_flag) {
                        tc::tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)  // D2 = k~^T v_new
                            tc::mma_bf16(tmem + kBColD2, tc::sdesc(st + kBK0 + kk * 2048, kBBlk, 1024),
                                         tc::sdesc(vn + kk * 2048, 8192, 1024), kId2, kk > 0);
                        tc::mma_commit(bar(B_M2));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)  // D1[0:64] += P v_new
                            tc::mma_bf16(d1, tc::sdesc(st + kBP + kk * 32, 16, 1024),
                                         tc::sdesc(vn + kk * 2048, 8192, 1024), kId3, 1);
                        tc::mma_commit(bar(B_M3));
                    }
                }
                wait(bar(B_M2), c & 1);
                tc::tc_fence_after();
                {
                    const float egl = gt[kGscal + 0];
#pragma unroll
                    for (int part = 0; part < 4; ++part) {
                        float dd[16];
                        tc::tmem_ld16(tmem + kBColD2 + lane_off + j0 + 16 * part, dd);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) h[16 * part + e] = fmaf(egl, h[16 * part + e], dd[e]);
                    }
                }
                if (c + 1 < nch) store_row64(hb + hw * 16384, r, h);
                tc::fence_proxy_async();
                tc::tc_fence_before();
                tc::named_bar(2, 256);
                if (r < 64) {  // o = rows 0..63 of D1
                    wait(bar(B_M3), c & 1);
                    tc::tc_fence_after();
                    if (r == 0 && hw == 0) tc::mbar_arrive(bar(B_SLOTFREE + s));
                    const int n = min(kChunk, len - c * kChunk);
                    const int t0 = start + c * kChunk;
#pragma unroll
                    for (int part = 0; part < 4; ++part) {
                        float oo[16];
                        tc::tmem_ld16(d1 + lane_off + j0 + 16 * part, oo);
                        tc::tmem_wait_ld();
                        if (r < n && !*abort_flag) {
                            uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(t0 + r) * H + head) * kD + j0 + 16 * part);
#pragma unroll
                            for (int q8 = 0; q8 < 2; ++q8)
                                dst[q8] = make_uint4(tc::pack_bf16(oo[8 * q8], oo[8 * q8 + 1]),
                                                     tc::pack_bf16(oo[8 * q8 + 2], oo[8 * q8 + 3]),
                                                     tc::pack_bf16(oo[8 * q8 + 4], oo[8 * q8 + 5]),
                                                     tc::pack_bf16(oo[8 * q8 + 6], oo[8 * q8 + 7]));
                        }
                    }
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(bar(B_D1F + b));
                }
            }
            if (h_T && !*abort_flag && !dead) {
#pragma unroll
                for (int e = 0; e < 64; e += 4)
                    *reinterpret_cast<float4*>(h_T + hoff + e) = make_float4(h[e], h[e + 1], h[e + 2], h[e + 3]);
            }
            if (cissuer) tc::mma_commit(bar(B_FIN));
        }
    }

    // drain this CTA's MMAs, then release TMEM; the cluster barrier keeps
    // either CTA from exiting while the other may still touch its memory
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) tc::mbar_wait(bar(front ? F_FIN : B_FIN), 0);
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, front ? kFTmemCols : kBTmemCols);
    tc::cluster_sync();
}

}  // namespace pair

bool pair_supported(const PrefillArgs& a) {
    auto al = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
    if (a.io != GDN_BF16 || a.dk != 128 || a.dv != 128) return false;
    if (a.delta_rule) {
        if (a.H % 4 != 0) return false;
        if (!al(a.log_alpha, 16) || !al(a.beta, 16)) return false;
    }
    return al(a.q, 16) && al(a.k, 16) && al(a.v, 16) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_pair(const PrefillArgs& a, cudaStream_t st) {
    using namespace pair;
    const long long units = (long long)a.n_seqs * a.H;
    if (units == 0) return cudaSuccess;
    if (2 * units > 0x7fffffffLL) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mla, mb;
    const int64_t T = a.T_total > 0 ? a.T_total : 1;
    const void* base = a.q ? a.q : a.ws;
    if (!encode_token_map(&mq, a.q ? a.q : base, T, a.H) || !encode_token_map(&mk, a.k ? a.k : base, T, a.H) ||
        !encode_token_map(&mv, a.v ? a.v : base, T, a.H))
        return cudaErrorInvalidValue;
    if (a.delta_rule) {
        if (!encode_gate_map(&mla, a.log_alpha ? a.log_alpha : (const float*)base, T, a.H) ||
            !encode_gate_map(&mb, a.beta ? a.beta : (const float*)base, T, a.H))
            return cudaErrorInvalidValue;
    } else {
        mla = mq;
        mb = mq;
    }
    auto kern = a.delta_rule ? pair_kernel<true> : pair_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * units), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mla, mb, a.h0, (__nv_bfloat16*)a.o, a.h_T, a.ws, a.H);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn
