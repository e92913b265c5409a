// fused_tc.cu -- single-kernel chunked prefill of the gated delta rule and of
// plain causal linear attention on sm_103a (bf16 I/O, dk = dv = 128, chunk 64).
//
// The chunk stages of the SparseGDN article ("Чем дорог префилл в Gated Delta
// Networks…": intra-chunk delta-system solve, sequential pass over chunks,
// outputs from chunk-start states; "Схема встраивания селектора…": the stage
// split intra-chunk / chunk_delta_h / outputs) run inside one kernel, so no
// intermediate (A, T, w, u, per-chunk state) ever reaches HBM: HBM sees q, k,
// v, gates, h0 in and o, h_T out.
//
// One CTA owns one (sequence, head, 64-column half of the state).  The state
// h = S^T (128 x 64 fp32 for this half) lives in registers of the four state
// warps (one row of h per thread) for the whole sequence.  Per chunk c, with
// g the running sum of log_alpha inside the chunk, four roles run as a
// pipeline (TMA two chunks ahead, solve one ahead of apply, apply one ahead
// of the state chain):
//   TMA warp     TMA q, k (2 x 64x64 boxes each), v (64 x 64), gates (64 x 4)
//                into stage c%2 (and an L2 prefetch three chunks ahead);
//                chunk-local cumsum g and the per-token decay factors
//   solve (4 w)  [k; q] k^T on tcgen05 (M=128 N=64 K=128), issued one chunk
//                ahead; A = beta KK^T exp(g_i - g_j) (strictly lower),
//                P = QK^T exp(g_i - g_j) (causal, diagonal included);
//                T = (I + A)^-1 (tri_inverse.cuh);
//                [T diag(beta e^g); T diag(beta)] -> TP (bf16)
//   apply (4 w)  TP x [k | v] on tcgen05 -> w = T(beta e^g k), u = T(beta v);
//                w -> smem (bf16), u -> smem (bf16), q~ = q e^g and
//                k~ = k e^{g_last - g} in place
//   state (4 w)  D1 = [q~; w] h            (M=128 N=64 K=128)
//                v_new = u - w h           (rows 64..127 of D1) -> bf16
//                D2 = k~^T v_new           (M=128 N=64 K=64, A MN-major)
//                D1[0:64] += P v_new       (M=128 N=64 K=64)
//                h <- e^{g_last} h + D2    (fp32 registers) -> bf16 for next D1
//                o = D1[0:64]              (bf16 store, rows < n)
// All waits are bounded; a wait that runs out sets GDN_ERR_TIMEOUT in the
// workspace status word and the CTA unwinds without skipping any barrier.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"
#include "tri_inverse.cuh"

namespace gdn {

namespace fused {

constexpr int kThreads = 416;  // warp 0: TMA; 1-4: solve; 5-8: apply; 9-12: state
constexpr int kNv = 64;        // state columns per CTA
constexpr int kD = 128;        // dk = dv

// per-stage layout (bytes from the stage base)
constexpr uint32_t kOffK0 = 0, kOffQ0 = 8192, kOffW0 = 16384;
constexpr uint32_t kOffK1 = 24576, kOffQ1 = 32768, kOffW1 = 40960;
constexpr uint32_t kKBlk = 24576;  // stride between the two 64-column blocks of k, q, w
constexpr uint32_t kOffV = 49152, kOffP = 57344;
constexpr uint32_t kOffGRaw = 65536;  // log_alpha box [64][4] then beta box [64][4]
constexpr uint32_t kOffGate = 67584;  // derived per-token gate values (float[64] arrays)
constexpr uint32_t kStage = 69632;
// gate arrays (float index from kOffGate)
constexpr int kGg = 0, kGeg = 64, kGeng = 128, kGbeg = 192, kGbb = 256, kGkdec = 320, kGscal = 384;
// scalars at kGscal: [0] e^{g_last}, [1] safe-factor flag, [2] n valid (as float)

// shared region
constexpr uint32_t kOffTP = 2 * kStage;          // 2 x [T'; T''] 128 x 64 bf16
constexpr uint32_t kOffHB = kOffTP + 2 * 16384;  // h bf16 [128][64]
constexpr uint32_t kOffVN = kOffHB + 16384;      // v_new bf16 [64][64]
constexpr uint32_t kOffU = kOffVN + 8192;        // u bf16 [64][64] (swizzled rows)
constexpr uint32_t kOffAF = kOffU + 8192;        // A / T fp32 [64][68]
constexpr uint32_t kOffScr = kOffAF + 64 * kTriLd * 4;
constexpr uint32_t kOffBar = kOffScr + 4 * 128 * 4;
constexpr int kNumBars = 24;  // >= B_COUNT
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 64;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// barriers
enum {
    B_FULL = 0,    // [2] TMA bytes landed                      (TMA -> all)
    B_GREADY = 2,  // [2] gate values derived                   (TMA -> solve, apply, state)
    B_EMPTY = 4,   // [2] stage free                            (state -> TMA)
    B_P1D = 6,     // [2] [k;q]k^T done in DP1[b]               (tcgen05 -> solve)
    B_P1F = 20,    // [2] DP1[b] read by the solve group        (solve -> TMA warp)
    B_TPR = 8,     // [2] TP[b] written                         (solve -> apply)
    B_TPF = 10,    // [2] TP[b] consumed                        (apply -> solve)
    B_READY = 12,  // [2] operands of the stage ready           (apply -> state)
    B_P2D = 14,    // w, u MMAs done                            (tcgen05 -> apply)
    B_UF = 15,     // u buffer read by the state                (state -> apply)
    B_M1 = 16, B_M2 = 17, B_M3 = 18,
    B_FIN = 19,    // every issuer's MMAs retired
    B_COUNT = 22
};

// TMEM columns
constexpr uint32_t kColD1 = 0;    // 2 x 64
constexpr uint32_t kColD2 = 128;  // 64
constexpr uint32_t kColP1 = 192;  // 2 x 64
constexpr uint32_t kColW = 320;   // 128
constexpr uint32_t kColU = 448;   // 64
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdP1 = tc::idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdP2w = tc::idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdP2u = tc::idesc_bf16(128, 64, false, true);
constexpr uint32_t kId1 = tc::idesc_bf16(128, 64, false, true);
constexpr uint32_t kId2 = tc::idesc_bf16(128, 64, true, true);
constexpr uint32_t kId3 = tc::idesc_bf16(128, 64, false, true);

__device__ __forceinline__ void report_timeout(char* ws, volatile int* abort_flag) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    atomicExch(&hdr->status, GDN_ERR_TIMEOUT);
    atomicCAS(&hdr->timeout_site, 0, 3000);  // this kernel records no barrier index
    *abort_flag = 1;
}

// Bounded mbarrier wait that also stops waiting once the CTA has aborted.
// Every thread keeps executing the same sequence of named barriers after an
// abort (work is skipped, barriers are not), so an abort cannot deadlock.
// The wait is one out-of-line function: inlined at every call site its loop
// and timeout path made up a large share of the kernel's instruction footprint.
// abort_flag[0] is the CTA's abort flag, abort_flag[1] the call's bound on
// polls per wait after the first (both in shared memory; the bound is read
// only when the first poll finds the phase incomplete).
static __device__ __noinline__ bool wait_bar(volatile int* abort_flag, char* ws, uint32_t bar, uint32_t parity) {
    if (*abort_flag) return false;
    if (tc::mbar_try_wait(bar, parity)) return true;
    const int limit = abort_flag[1];
    if (tc::mbar_wait(bar, parity, limit)) return true;
    report_timeout(ws, abort_flag);
    return false;
}
struct Waiter {
    volatile int* abort_flag;
    char* ws;
    __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
        return wait_bar(abort_flag, ws, bar, parity);
    }
};

// Scale the 128 bf16 of row r of a [64 x 128] operand (two 64-column boxes
// kKBlk apart) by f, in place, with packed bf16x2 multiplies (the bf16
// product of two bf16 values is rounded once, as an fp32 multiply then a
// rounding to bf16 would be; f itself is rounded to bf16 first).
__device__ __forceinline__ void scale_row(uint32_t box0, uint32_t r, float f) {
    const __nv_bfloat162 f2 = __float2bfloat162_rn(f);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t a = tc::sw128(box0 + half * kKBlk, r, j);
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

// Write 64 fp32 values as one bf16 row of a 128-byte-swizzled tile.
__device__ __forceinline__ void store_row64(uint32_t tile, uint32_t r, const float* v) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        tc::st_shared_v4(tc::sw128(tile, r, j), tc::pack_bf16(v[8 * j], v[8 * j + 1]),
                         tc::pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                         tc::pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                         tc::pack_bf16(v[8 * j + 6], v[8 * j + 7]));
}

// MAXD: farthest 16-token block below the diagonal at which the inverse of
// the delta system is formed (3: exact; 1: the block-adjacent solver).
template <bool GDN, int MAXD>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
               const __grid_constant__ CUtensorMap tm_b, const float* __restrict__ h0,
               __nv_bfloat16* __restrict__ o, float* __restrict__ h_T, char* __restrict__ ws,
               int H) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // offset to the next 1024-byte boundary; pointers stay derived from the
    // __shared__ array so every access compiles to a shared-space access
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    char* const sptr = reinterpret_cast<char*>(smem_raw) + pad;
    const uint32_t sbase = raw + pad;
    auto bar = [&](int i) { return sbase + kOffBar + 8u * (uint32_t)i; };
    auto gate = [&](int s) { return reinterpret_cast<float*>(sptr + s * kStage + kOffGate); };

    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;

    // the warp index and the TMEM base are broadcast from lane 0 so that the
    // compiler sees them as warp-uniform: role branches then stay in uniform
    // control flow and MMA descriptors are built in uniform registers
    const int tid = threadIdx.x, lane = tid & 31;
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const int n_seqs = hdr->n_seqs;
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* order = reinterpret_cast<const int*>(ws + L.order);
    const int unit = blockIdx.x;
    const int seq = order[unit / (2 * H)];
    const int rem = unit % (2 * H);
    const int head = rem >> 1, j0 = (rem & 1) * kNv;
    // loaded values, broadcast so that loops over chunks count as warp-uniform
    const int start = __shfl_sync(0xffffffffu, cu[seq], 0);
    const int len = __shfl_sync(0xffffffffu, cu[seq + 1], 0) - start;
    const int nch = (len + kChunk - 1) / kChunk;

    volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + kOffMisc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + kOffMisc + 8);
    const Waiter wait{abort_flag, ws};

    if (tid == 0) {
        abort_flag[0] = 0;
        abort_flag[1] = hdr->wait_limit;
#pragma unroll 1
        for (int b = 0; b < B_COUNT; ++b) tc::mbar_init(bar(b), b == B_FIN ? 4 : 1);
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
        if (GDN) {
            tc::prefetch_tmap(&tm_la);
            tc::prefetch_tmap(&tm_b);
        }
    }
    if (!GDN) {  // w = 0 for linear attention: zero the w boxes of both stages once
        for (int i = tid; i < 2 * 2 * 8192 / 16; i += kThreads) {
            const int s = i / 1024, rest = i % 1024, box = rest / 512, off = (rest % 512) * 16;
            tc::st_shared_v4(sbase + s * kStage + (box ? kOffW1 : kOffW0) + off, 0, 0, 0, 0);
        }
        tc::fence_proxy_async();
    }
    __syncwarp();  // lane-0-only work above: reconverge before any .aligned instruction
    if (warp == 0) tc::tmem_alloc(sbase + kOffMisc + 8, kTmemCols);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
    const int quad = warp & 3;                        // TMEM lane quadrant of this warp
    const int row = 32 * quad + lane;                 // TMEM lane / tile row
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    const bool tma_issuer = (warp == 0 && lane == 0);
    const bool solve_issuer = (warp == 4 && lane == 0);
    const bool apply_issuer = (warp == 8 && lane == 0);
    const bool state_issuer = (warp == 10 && lane == 0);  // row 64

    // ---- [k; q] k^T for chunk c into DP1[c & 1] (issued by the solve group)
    auto issue_p1 = [&](int c) {
        const uint32_t st = sbase + (c & 1) * kStage;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kKBlk + (kk & 3) * 32;
            tc::mma_bf16(tmem + kColP1 + (c & 1) * 64, tc::sdesc(st + kOffK0 + off, 16, 1024),
                         tc::sdesc(st + kOffK0 + off, 16, 1024), kIdP1, kk > 0);
        }
        tc::mma_commit(bar(B_P1D + (c & 1)));
    };

    if (warp == 0) {
        // ================================================== TMA + gates
        int issued = 0;
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1, u = c >> 1;
            const uint32_t st = sbase + s * kStage;
            if (c >= 2) wait(bar(B_EMPTY + s), (u - 1) & 1);
            const int t0 = start + c * kChunk;
            if (lane == 0 && !*abort_flag) {
                const uint32_t bytes = 2 * 16384 + 8192 + (GDN ? 2048 : 0);
                tc::mbar_arrive_expect_tx(bar(B_FULL + s), bytes);
                tc::tma_load_3d(st + kOffK0, &tm_k, 0, head, t0, bar(B_FULL + s));
                tc::tma_load_3d(st + kOffK1, &tm_k, 64, head, t0, bar(B_FULL + s));
                tc::tma_load_3d(st + kOffQ0, &tm_q, 0, head, t0, bar(B_FULL + s));
                tc::tma_load_3d(st + kOffQ1, &tm_q, 64, head, t0, bar(B_FULL + s));
                tc::tma_load_3d(st + kOffV, &tm_v, j0, head, t0, bar(B_FULL + s));
                if (GDN) {
                    tc::tma_load_2d(st + kOffGRaw, &tm_la, head & ~3, t0, bar(B_FULL + s));
                    tc::tma_load_2d(st + kOffGRaw + 1024, &tm_b, head & ~3, t0, bar(B_FULL + s));
                }
                issued = c + 1;
                if (c + 3 < nch) {  // warm L2 for a later chunk; its copy then waits less
                    const int tp = t0 + 3 * kChunk;
                    tc::tma_prefetch_3d(&tm_k, 0, head, tp);
                    tc::tma_prefetch_3d(&tm_k, 64, head, tp);
                    tc::tma_prefetch_3d(&tm_q, 0, head, tp);
                    tc::tma_prefetch_3d(&tm_q, 64, head, tp);
                    tc::tma_prefetch_3d(&tm_v, j0, head, tp);
                    if (GDN) {
                        tc::tma_prefetch_2d(&tm_la, head & ~3, tp);
                        tc::tma_prefetch_2d(&tm_b, head & ~3, tp);
                    }
                }
            }
            __syncwarp();
            wait(bar(B_FULL + s), u & 1);
            // [k; q] k^T of this chunk, once the solve group has released DP1[c & 1]
            if (tma_issuer) {
                if (c >= 2) wait(bar(B_P1F + (c & 1)), ((c >> 1) - 1) & 1);
                if (!*abort_flag) issue_p1(c);
            }
            __syncwarp();
            // derived gate values of the chunk
            const int n = min(kChunk, len - c * kChunk);
            float* gt = gate(s);
            const float* la_raw = reinterpret_cast<const float*>(sptr + s * kStage + kOffGRaw);
            const float* b_raw = la_raw + 256;
            const int hc = head & 3;
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
            if (lane == 0) tc::mbar_arrive(bar(B_GREADY + s));
            __syncwarp();
        }
        // after an abort, let copies already issued land before the CTA exits
        if (lane == 0 && *abort_flag)
            for (int c = max(0, issued - 2); c < issued; ++c)
                tc::mbar_wait(bar(B_FULL + (c & 1)), (c >> 1) & 1);
        __syncwarp();
    } else if (warp <= 4) {
        // ================================================== solve group
        const int pw = warp - 1;  // 0..3
        float* AF = reinterpret_cast<float*>(sptr + kOffAF);
        float* scr = reinterpret_cast<float*>(sptr + kOffScr);
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1, u = c >> 1;
            const uint32_t st = sbase + s * kStage;
            wait(bar(B_GREADY + s), u & 1);
            wait(bar(B_P1D + (c & 1)), u & 1);
            __syncwarp();
            tc::tc_fence_after();
            const float* gt = gate(s);
            const bool safe = gt[kGscal + 1] != 0.f;
            const int n = (int)gt[kGscal + 2];
            float x[64];
            tc::tmem_ld32(tmem + lane_off + kColP1 + (c & 1) * 64, *reinterpret_cast<float(*)[32]>(x));
            tc::tmem_ld32(tmem + lane_off + kColP1 + (c & 1) * 64 + 32,
                          *reinterpret_cast<float(*)[32]>(x + 32));
            tc::tmem_wait_ld();
            tc::tc_fence_before();
            tc::named_bar(1, 128);  // DP1[c & 1] fully read
            if (solve_issuer) tc::mbar_arrive(bar(B_P1F + (c & 1)));
            __syncwarp();
            // rows 0..63: K K^T -> A (fp32); rows 64..127: Q K^T -> P (bf16 tile)
            {
                const int t = row & 63;
                const bool is_a = row < 64;
                if (!is_a || GDN) {
                    const float rs = (is_a ? gt[kGbb + t] : 1.f) * gt[kGeg + t];
                    const int lim = is_a ? t : t + 1;  // s < lim kept
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
                        store_row64(st + kOffP, t, x);
                    }
                }
            }
            tc::fence_proxy_async();
            tc::named_bar(1, 128);
            if (GDN) tri_inverse_64(AF, scr, pw, lane, 1, MAXD);
            // ---- TP[c & 1]: rows 0..63 T diag(beta e^g), rows 64..127 T diag(beta)
            if (c >= 2) wait(bar(B_TPF + (c & 1)), ((c >> 1) - 1) & 1);
            {
                const int t = row & 63;
                const float* cs = gt + (row < 64 ? kGbeg : kGbb);
                const uint32_t tp = sbase + kOffTP + (c & 1) * 16384;
#pragma unroll
                for (int jb = 0; jb < 4; ++jb) {
                    float v16[16];
                    if (GDN && jb <= (t >> 4) && (t >> 4) - jb <= MAXD) {
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
                        tc::st_shared_v4(tc::sw128(tp, row, 2 * jb + h2),
                                         tc::pack_bf16(v16[8 * h2], v16[8 * h2 + 1]),
                                         tc::pack_bf16(v16[8 * h2 + 2], v16[8 * h2 + 3]),
                                         tc::pack_bf16(v16[8 * h2 + 4], v16[8 * h2 + 5]),
                                         tc::pack_bf16(v16[8 * h2 + 6], v16[8 * h2 + 7]));
                }
            }
            tc::fence_proxy_async();
            tc::named_bar(1, 128);
            if (solve_issuer) tc::mbar_arrive(bar(B_TPR + (c & 1)));
            __syncwarp();
        }
    } else if (warp <= 8) {
        // ================================================== apply group
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1, u = c >> 1;
            const uint32_t st = sbase + s * kStage;
            const uint32_t tp = sbase + kOffTP + (c & 1) * 16384;
            wait(bar(B_GREADY + s), u & 1);
            wait(bar(B_TPR + (c & 1)), u & 1);
            // ---- w = T' k (GDN), u = T'' v
            if (apply_issuer && !*abort_flag) {
                tc::tc_fence_after();
                if (GDN) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_bf16(tmem + kColW, tc::sdesc(tp + kk * 32, 16, 1024),
                                     tc::sdesc(st + kOffK0 + kk * 2048, kKBlk, 1024), kIdP2w, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16(tmem + kColU, tc::sdesc(tp + kk * 32, 16, 1024),
                                 tc::sdesc(st + kOffV + kk * 2048, 8192, 1024), kIdP2u, kk > 0);
                tc::mma_commit(bar(B_P2D));
            }
            __syncwarp();
            wait(bar(B_P2D), c & 1);
            __syncwarp();
            tc::tc_fence_after();
            if (apply_issuer) tc::mbar_arrive(bar(B_TPF + (c & 1)));
            __syncwarp();
            const float* gt = gate(s);
            if (row < 64) {
                if (GDN) {  // w row -> bf16 into the w boxes
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float x[64];
                        tc::tmem_ld32(tmem + lane_off + kColW + 64 * half, *reinterpret_cast<float(*)[32]>(x));
                        tc::tmem_ld32(tmem + lane_off + kColW + 64 * half + 32,
                                      *reinterpret_cast<float(*)[32]>(x + 32));
                        tc::tmem_wait_ld();
                        store_row64(st + (half ? kOffW1 : kOffW0), row, x);
                    }
                }
                scale_row(st + kOffK0, row, gt[kGkdec + row]);
            } else {
                const int t = row - 64;
                if (c >= 1) wait(bar(B_UF), (c - 1) & 1);
                float x[64];
                tc::tmem_ld32(tmem + lane_off + kColU, *reinterpret_cast<float(*)[32]>(x));
                tc::tmem_ld32(tmem + lane_off + kColU + 32, *reinterpret_cast<float(*)[32]>(x + 32));
                tc::tmem_wait_ld();
                store_row64(sbase + kOffU, t, x);
                if (GDN) scale_row(st + kOffQ0, t, gt[kGeg + t]);
            }
            tc::fence_proxy_async();
            tc::tc_fence_before();
            tc::named_bar(2, 128);
            if (apply_issuer) tc::mbar_arrive(bar(B_READY + s));
            __syncwarp();
        }
    } else {
        // ================================================== state chain
        const int r = row;  // row of h (dk index) and TMEM lane
        const size_t hoff = (((size_t)seq * H + head) * kD + r) * kD + j0;
        float h[kNv];
        if (h0) {
#pragma unroll
            for (int j = 0; j < kNv; j += 4) {
                float4 v4 = *reinterpret_cast<const float4*>(h0 + hoff + j);
                h[j] = v4.x; h[j + 1] = v4.y; h[j + 2] = v4.z; h[j + 3] = v4.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kNv; ++j) h[j] = 0.f;
        }
        store_row64(sbase + kOffHB, r, h);
        tc::fence_proxy_async();
        tc::named_bar(3, 128);

        for (int c = 0; c < nch; ++c) {
            const int s = c & 1, u = c >> 1, b = c & 1;
            const uint32_t st = sbase + s * kStage;
            wait(bar(B_READY + s), u & 1);
            const float* gt = gate(s);
            const uint32_t d1 = tmem + kColD1 + b * 64;
            // ---- D1 = [q~; w] h
            if (state_issuer && !*abort_flag) {
                tc::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16(d1, tc::sdesc(st + kOffQ0 + (kk >> 2) * kKBlk + (kk & 3) * 32, 16, 1024),
                                 tc::sdesc(sbase + kOffHB + kk * 2048, 8192, 1024), kId1, kk > 0);
                tc::mma_commit(bar(B_M1));
            }
            __syncwarp();
            if (r >= 64) {
                // ---- v_new = u - w h   (rows 64..127 of D1 are w h)
                wait(bar(B_M1), c & 1);
                __syncwarp();
                tc::tc_fence_after();
                const int t = r - 64;
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    float wh[16];
                    tc::tmem_ld16(d1 + lane_off + 16 * part, wh);
                    const uint4 ua = tc::ld_shared_v4(tc::sw128(sbase + kOffU, t, 2 * part));
                    const uint4 ub = tc::ld_shared_v4(tc::sw128(sbase + kOffU, t, 2 * part + 1));
                    tc::tmem_wait_ld();
                    const uint32_t uw[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 uu = tc::unpack_bf16(uw[e]);
                        pk[e] = tc::pack_bf16(uu.x - wh[2 * e], uu.y - wh[2 * e + 1]);
                    }
                    tc::st_shared_v4(tc::sw128(sbase + kOffVN, t, 2 * part), pk[0], pk[1], pk[2], pk[3]);
                    tc::st_shared_v4(tc::sw128(sbase + kOffVN, t, 2 * part + 1), pk[4], pk[5], pk[6], pk[7]);
                }
                tc::fence_proxy_async();
                tc::tc_fence_before();
                tc::named_bar(4, 64);
                if (state_issuer) {
                    tc::mbar_arrive(bar(B_UF));
                    if (!*abort_flag) {
                        tc::tc_fence_after();
                        // ---- D2 = k~^T v_new
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_bf16(tmem + kColD2, tc::sdesc(st + kOffK0 + kk * 2048, kKBlk, 1024),
                                         tc::sdesc(sbase + kOffVN + kk * 2048, 8192, 1024), kId2, kk > 0);
                        tc::mma_commit(bar(B_M2));
                        // ---- D1[0:64] += P v_new
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_bf16(d1, tc::sdesc(st + kOffP + kk * 32, 16, 1024),
                                         tc::sdesc(sbase + kOffVN + kk * 2048, 8192, 1024), kId3, 1);
                        tc::mma_commit(bar(B_M3));
                    }
                }
                __syncwarp();
            }
            // ---- h <- e^{g_last} h + k~^T v_new
            wait(bar(B_M2), c & 1);
            __syncwarp();
            tc::tc_fence_after();
            {
                const float egl = gt[kGscal + 0];
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    float dd[32];
                    tc::tmem_ld32(tmem + lane_off + kColD2 + 32 * part, dd);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) h[32 * part + j] = fmaf(egl, h[32 * part + j], dd[j]);
                }
            }
            if (c + 1 < nch) store_row64(sbase + kOffHB, r, h);
            tc::fence_proxy_async();
            tc::tc_fence_before();
            tc::named_bar(3, 128);
            // ---- o = rows 0..63 of D1
            if (r < 64) {
                wait(bar(B_M3), c & 1);
                __syncwarp();
                tc::tc_fence_after();
                if (r == 0) tc::mbar_arrive(bar(B_EMPTY + s));  // every MMA reading the stage has retired
                __syncwarp();
                const int n = min(kChunk, len - c * kChunk);
                const int t0 = start + c * kChunk;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    float oo[32];
                    tc::tmem_ld32(d1 + lane_off + 32 * part, oo);
                    tc::tmem_wait_ld();
                    if (r < n && !*abort_flag) {
                        uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(t0 + r) * H + head) * kD + j0 + 32 * part);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(tc::pack_bf16(oo[8 * j], oo[8 * j + 1]),
                                                tc::pack_bf16(oo[8 * j + 2], oo[8 * j + 3]),
                                                tc::pack_bf16(oo[8 * j + 4], oo[8 * j + 5]),
                                                tc::pack_bf16(oo[8 * j + 6], oo[8 * j + 7]));
                    }
                }
                tc::tc_fence_before();
            }
        }
        if (h_T && !*abort_flag) {
#pragma unroll
            for (int j = 0; j < kNv; j += 4)
                *reinterpret_cast<float4*>(h_T + hoff + j) = make_float4(h[j], h[j + 1], h[j + 2], h[j + 3]);
        }
    }

    // drain: every MMA issuer commits once more; wait (bounded) until every
    // MMA of this CTA has completed before the tensor memory is released
    if (tma_issuer || solve_issuer || apply_issuer || state_issuer) tc::mma_commit(bar(B_FIN));
    __syncwarp();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) tc::mbar_wait(bar(B_FIN), 0);
    __syncwarp();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [T][H][128] bf16, box 64 (features) x 1 (head) x 64 (tokens), 128-byte swizzle
bool map_tokens(CUtensorMap* m, const void* ptr, int64_t T, int H) {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
    cuuint32_t box[3] = {64, 1, 64}, es[3] = {1, 1, 1};
    return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T][H] fp32, box 4 (heads) x 64 (tokens)
bool map_gates(CUtensorMap* m, const float* ptr, int64_t T, int H) {
    cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)H * 4};
    cuuint32_t box[2] = {4, 64}, es[2] = {1, 1};
    return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fused

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return fused::encoder(); }
bool encode_token_map(CUtensorMap* m, const void* p, int64_t T, int H) { return fused::map_tokens(m, p, T, H); }
bool encode_gate_map(CUtensorMap* m, const float* p, int64_t T, int H) { return fused::map_gates(m, p, T, H); }

bool fused_supported(const PrefillArgs& a) {
    auto al = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
    if (a.io != GDN_BF16 || a.dk != 128 || a.dv != 128) return false;
    if (a.delta_rule) {
        if (a.H % 4 != 0) return false;  // the gate boxes need H * 4 bytes to be a multiple of 16
        if (!al(a.log_alpha, 16) || !al(a.beta, 16)) return false;
    }
    return al(a.q, 16) && al(a.k, 16) && al(a.v, 16) && fused::encoder() != nullptr;
}

cudaError_t launch_fused(const PrefillArgs& a, cudaStream_t st) {
    using namespace fused;
    const long long units = (long long)a.n_seqs * a.H * 2;
    if (units == 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mla, mb;
    const int64_t T = a.T_total > 0 ? a.T_total : 1;
    // with T_total == 0 every sequence is empty and no copy is issued; the
    // maps only need a valid address to encode
    const void* base = a.q ? a.q : a.ws;
    if (!map_tokens(&mq, a.q ? a.q : base, T, a.H) || !map_tokens(&mk, a.k ? a.k : base, T, a.H) ||
        !map_tokens(&mv, a.v ? a.v : base, T, a.H))
        return cudaErrorInvalidValue;
    if (a.delta_rule) {
        if (!map_gates(&mla, a.log_alpha ? a.log_alpha : (const float*)base, T, a.H) ||
            !map_gates(&mb, a.beta ? a.beta : (const float*)base, T, a.H))
            return cudaErrorInvalidValue;
    } else {
        mla = mq;
        mb = mq;
    }
    auto kern = !a.delta_rule ? prefill_kernel<false, 3>
                              : a.max_block_dist == 1 ? prefill_kernel<true, 1> : prefill_kernel<true, 3>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)units, kThreads, kSmemAlloc, st>>>(mq, mk, mv, mla, mb, a.h0, (__nv_bfloat16*)a.o,
                                                        a.h_T, a.ws, a.H);
    return cudaGetLastError();
}

}  // namespace gdn
