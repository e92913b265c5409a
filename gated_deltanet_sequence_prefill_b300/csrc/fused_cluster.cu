// fused_cluster.cu -- chunked GDN / linear-attention prefill on a thread-block
// cluster per (sequence, head): FR solve CTAs (FR = 1 or 2) and one state CTA,
// sm_103a, bf16 I/O, dk = dv = 128, chunk 64.
//
// The chunk stages of the SparseGDN article ("Чем дорог префилл в Gated Delta
// Networks…": intra-chunk delta-system solve, sequential pass over chunks,
// outputs from chunk-start states) are split across the SMs of the cluster so
// that the long-latency solve never holds the buffers the sequential state
// pass needs.  The state pass works on the transpose S = h^T (dv x dk), so
// that S and v_new are tensor-core A operands held in TMEM.
//
//  solve CTA r (ranks 0..FR-1): the delta-system solve of chunks r, r+FR, ...
//    TMA warp   q, k (2 x 64x64 SW128 boxes each) and the gates of the head
//               into a 4-stage ring
//    warp 13    [k; q] k^T on tcgen05 (M=128 N=64 K=128) into TMEM; the
//               chunk's cumsum g and decay factors
//    3 solve warpgroups, chunk u on group u % 3:
//               A = beta KK^T exp(g_i - g_j) (strictly lower),
//               P^ = QK^T e^{-g_last} (causal; QK^T exp(g_i - g_j) when the
//                    chunk's decay range is large),
//               T = (I + A)^-1 (tri_inverse.cuh),
//               T' = T diag(beta e^g) and T'' = T diag(beta) into the dead q tile,
//               w^T = k^T T'^T on tcgen05, -w staged as [dk][t]
//    2 store warps  bulk-copy P^, T'' and -w into the (sequence, head)'s global
//               scratch slot c % 6 (it stays in L2) and announce it to the state
//               CTA with a remote mbarrier arrive
//  state CTA (rank FR): everything that touches the state
//    TMA warp   q, k into a 3-entry ring, v and the gates into a 2-entry ring
//    loader     bulk-loads each chunk's P^, T'', -w from its scratch slot
//    gates      the gate factors the state CTA needs
//    chain      8 warps, each thread one row j of S and one 64-column half;
//               S in TMEM twice: fp32 (the accumulator of D2) and bf16 (the
//               A operand)
//               D1v  = u^T = v^T T''^T, then += S (-w)^T: v_new^T
//               D1o  = S q^T
//               v^ = e^{g_last - g} v_new (bf16, TMEM)
//               S <- e^{g_last} S (fp32, in place), then S += v^^T k on the
//               tensor core;  D1o += v^^T P^^T
//    output     4 warps: o = e^{g} D1o, staged in the dead k tile and written
//               with a TMA store
//    MMA warp   issues every MMA of the state CTA as straight-line elect.sync
//               sequences
//
// HBM sees q, k, v, gates, h0 in and o, h_T out; q and k are read by both
// kinds of CTA (the second read is an L2 hit) and the scratch ring never
// leaves L2.  All waits are bounded; a wait that runs out sets GDN_ERR_TIMEOUT
// in the workspace status word and the CTAs unwind without skipping any
// barrier.
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

constexpr int kThreads = 512;  // 16 warps in both CTAs
// run-mode bits (PrefillArgs::mode)
constexpr int kModeNoOutput = 1, kModeZeroV = 2, kModeIdentityH0 = 4;
constexpr int kD = 128;

// ---------------------------------------------------------------- front layout
constexpr uint32_t kFK0 = 0, kFQ0 = 8192, kFK1 = 16384, kFQ1 = 24576;  // [k0 q0 | k1 q1]
constexpr uint32_t kFBlk = 16384;                                         // K-block stride
constexpr uint32_t kFGRaw = 32768;                                        // la [64][4], beta [64][4]
constexpr uint32_t kFGate = 34816;                                        // derived gate arrays
constexpr uint32_t kFStage = 36864;
constexpr int kFGroups = 3;   // solve groups: chunk c goes to group c % 3
constexpr int kFStages = 4;   // TMA stages: chunk c lands in stage c % 4 (one chunk of lookahead)
// Once [k; q] k^T is done the stage's q tile is dead: its first box then holds
// T' = T diag(beta e^g) (the B operand of the w MMA), its second T'' = T diag(beta).
constexpr uint32_t kFT1 = kFQ0, kFT2 = kFQ1;
constexpr uint32_t kFPst = kFStages * kFStage;             // 3 x P^ staging (bf16 64x64, swizzled)
constexpr uint32_t kFAF = kFPst + kFGroups * 8192;         // 3 x A/T fp32 [64][68]; later -w staging
constexpr uint32_t kFScr = kFAF + kFGroups * 64 * kTriLd * 4;  // 3 x 4 x 128 floats
constexpr int kBarSlots = 40;
constexpr uint32_t kFBar = kFScr + kFGroups * 4 * 128 * 4;
constexpr uint32_t kFEnd = kFBar + kBarSlots * 8 + 64;

// ---------------------------------------------------------------- back layout
// Chain ring (3 entries, chunk c in entry c % 3): q and k as two 64-column
// SW128 boxes each (the k tile later stages o), -w as [128 i][64 t] (the
// MN-major B operand of the w MMA), P^, the derived gate values.
constexpr uint32_t kBBox = 8192;  // stride between the two 64-column boxes
constexpr uint32_t kCQ = 0, kCK = 16384, kCW = 32768, kCP = 49152, kCGate = 57344;
constexpr uint32_t kCEntry = 59392;
// Apply ring (2 entries, chunk c in entry c % 2): v (two boxes), T'' loaded
// from the scratch slot, the raw log-decay of four heads.
constexpr uint32_t kARing = 3 * kCEntry;
constexpr uint32_t kAV = 0, kAT2 = 16384, kALa = 24576;
constexpr uint32_t kAEntry = 25600;
constexpr uint32_t kBBar = kARing + 2 * kAEntry;
constexpr uint32_t kBEnd = kBBar + kBarSlots * 8 + 64;

// Global scratch per (sequence, head): six 32 KB slots (chunk c in slot c % 6)
// holding P^ [64 t][64 s], T'' [64 t][64 s] and -w [128 i][64 t] (bf16, rows of
// 128 bytes already in the 128-byte swizzle of the state CTA's tiles).
constexpr int kSlots = 6;
constexpr uint32_t kScratchSlot = 32768;
constexpr uint32_t kScratchUnit = kSlots * kScratchSlot;

constexpr uint32_t kSmemBytes = (kFEnd > kBEnd ? kFEnd : kBEnd);
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kFBar + kBarSlots * 8 <= kSmemBytes && kBBar + kBarSlots * 8 <= kSmemBytes, "barriers");
static_assert(kCEntry % 1024 == 0 && kARing % 1024 == 0 && kAEntry % 1024 == 0, "tile alignment");

// gate arrays (float index from the gate area); scalars at kGscal:
// [0] e^{g_last}, [1] safe-factor flag, [2] n valid, [3] e^{-g_last}; kGone holds ones
constexpr int kGg = 0, kGeg = 64, kGeng = 128, kGbeg = 192, kGbb = 256, kGkdec = 320, kGscal = 384, kGone = 448;

// ---------------------------------------------------------------- barriers
// front
enum {
    F_FULL = 0,     // [4] TMA landed in stage c % 4
    F_EMPTY = 4,    // [4] stage free (a store warp has read T'' out of it)
    F_GREADY = 8,   // [3] gate values of the group's chunk derived
    F_P1D = 11,     // [3] [k;q]k^T done in DP1[group]
    F_P1F = 14,     // [3] DP1[group] read
    F_STAGED = 17,  // [3] group staged P^, T'', -w of its chunk for the store warps
    F_WD = 20,      // [3] w^T MMA of the group done
    F_FIN = 23,
    F_SFREE = 24,   // [3] a store warp has read the group's staging (P^, -w in AF)
    F_ARMED = 27,   // [6] scratch slot read by the state CTA (remote arrive by the back)
    F_COUNT = 33
};
// back
enum {
    B_FULLC = 0,    // [3] q, k landed in the chain entry
    B_FULLA = 3,    // [2] v, log-decay landed in the apply entry
    B_FULLP = 5,    // [3] -w, P^, T'' loaded from the scratch slot (counted on the chain entry)
    B_GREADY = 8,   // [3] gate values derived into the chain entry
    B_CFREE = 11,   // [3] chain entry free (o store has read its staging)
    B_AFREE = 14,   // [2] apply entry free (u MMA done)
    B_D1OF = 16,    // [2] D1o[b] read by the output warps
    B_M3 = 18,      // [2] D1o[b] complete
    B_M1W = 20,     // D1v = v_new^T
    B_M2 = 21,      // S += v^^T k done
    B_SREADY = 22,  // S (bf16) of the next chunk in TMEM (chain -> issuer)
    B_VREADY = 23,  // v^ in TMEM (chain -> issuer)
    B_FIN = 24,
    B_STORED = 25,  // [6] the solve CTA's chunk is in its global scratch slot (remote arrive)
    B_COUNT = 31
};

// TMEM columns
constexpr uint32_t kFColP1 = 0;        // front: 3 x 64
constexpr uint32_t kFColW = 256;       // front: 3 x 64, w^T (lane = dk row i)
constexpr uint32_t kFTmemCols = 512;
// back (lane = dv row j of the state)
constexpr uint32_t kTD1o = 0;          // 2 x 64: o^T accumulators (fp32)
constexpr uint32_t kTD1v = 128;        // 2 x 64: u^T - S w^T = v_new^T (fp32)
constexpr uint32_t kTD2 = 256;         // S (fp32), 128 cols: S += v^^T k accumulates here
constexpr uint32_t kTS = 384;          // S (bf16 pairs), 64 cols: A operand
constexpr uint32_t kTVN = 448;         // v^ (bf16 pairs), 32 cols: A operand
constexpr uint32_t kBTmemCols = 512;

constexpr uint32_t kIdP1 = tc::idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdWU = tc::idesc_bf16(128, 64, true, false);   // A = k^T / v^T (MN-major), B = T (K-major)
constexpr uint32_t kId1w = tc::idesc_bf16(128, 64, false, true);   // A = S (TMEM), B = -w [i][t]
constexpr uint32_t kId1q = tc::idesc_bf16(128, 64, false, false);  // A = S (TMEM), B = q [t][i]
constexpr uint32_t kId2 = tc::idesc_bf16(128, 128, false, true);   // A = v^T (TMEM), B = k [t][i]
constexpr uint32_t kId3 = tc::idesc_bf16(128, 64, false, false);   // A = v^T (TMEM), B = P^ [t][s]

// A wait that ran out: GDN_ERR_TIMEOUT in the status word, and the first
// barrier that gave up (1000 + index on the solve CTA, 2000 + index on the
// state CTA) in the header's first spare word, for diagnosis.
__device__ __forceinline__ void report_timeout(char* ws, volatile int* abort_flag, int site) {
    WsHeader* h = reinterpret_cast<WsHeader*>(ws);
    atomicExch(&h->status, GDN_ERR_TIMEOUT);
    atomicCAS(&h->timeout_site, 0, site);
    *abort_flag = 1;
}

// Bounded waits that stop waiting once this CTA has aborted; every thread
// keeps executing the same sequence of named barriers after an abort.  The
// wait is one out-of-line function: inlined at every call site its loop and
// timeout path made up a large share of the kernel's instruction footprint.
// abort_flag[0] is the CTA's abort flag and abort_flag[1] the call's bound on
// polls per wait after the first (both in shared memory, so no call site
// carries the bound; it is read only when the first poll finds the phase
// incomplete).
static __device__ __noinline__ bool wait_bar(volatile int* abort_flag, char* ws, uint32_t bar, uint32_t parity,
                                             int site, bool cluster_scope) {
    if (*abort_flag) return false;
    if (cluster_scope ? tc::mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity)) return true;
    const int limit = abort_flag[1];
    if (cluster_scope ? tc::mbar_wait_cluster(bar, parity, limit) : tc::mbar_wait(bar, parity, limit)) return true;
    report_timeout(ws, abort_flag, site);
    return false;
}
struct Waiter {
    volatile int* abort_flag;
    char* ws;
    uint32_t bar_base;
    int site_base;
    __device__ __forceinline__ bool operator()(uint32_t bar, uint32_t parity) const {
        return wait_bar(abort_flag, ws, bar, parity, site_base + (int)((bar - bar_base) >> 3), false);
    }
    __device__ __forceinline__ bool remote(uint32_t bar, uint32_t parity) const {
        return wait_bar(abort_flag, ws, bar, parity, site_base + (int)((bar - bar_base) >> 3), true);
    }
};

// An opaque copy of a flag: branching on it inside a loop keeps the compiler
// from cloning the loop once per flag value (loop unswitching), which would
// multiply the kernel's instruction footprint.
__device__ __forceinline__ bool opaque(bool f) {
    uint32_t v = f;
    asm volatile("" : "+r"(v));
    return v != 0;
}
__device__ __forceinline__ int opaque_i(int x) {
    asm volatile("" : "+r"(x));
    return x;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Per-token gate values of a chunk (one warp): running sum g of log_alpha
// (rows past the chunk end contribute nothing), exp(g), exp(-g), beta,
// beta e^g, k decay exp(g_last - g) (0 past the end), and the scalars.
template <bool GDN>
__device__ __noinline__ void derive_gates(const float* la_raw, const float* b_raw, int hc, int n,
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
    gt[kGone + ta] = 1.f;
    gt[kGone + tb] = 1.f;
    if (lane == 0) {
        gt[kGscal + 0] = __expf(glast);
        gt[kGscal + 1] = amax <= 40.f ? 1.f : 0.f;
        gt[kGscal + 2] = (float)n;
        gt[kGscal + 3] = __expf(-glast);
    }
    __syncwarp();
}

// MAXD: farthest 16-token block below the diagonal at which the inverse of
// the delta system is formed (3: exact; 1: the block-adjacent solver).
// MODE: run-mode bits of the two-level state scan (0 for an ordinary call).
template <bool GDN, int FR, int MAXD, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_la,
            const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_o,
            const float* __restrict__ h0, __nv_bfloat16* __restrict__ o, float* __restrict__ h_T,
            char* __restrict__ ws, char* __restrict__ scratch, int H) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    char* const sptr = reinterpret_cast<char*>(smem_raw) + pad;
    const uint32_t sbase = raw + pad;  // identical in both CTAs (same kernel, same layout)

    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    // loaded values are broadcast from lane 0 so that the compiler treats them,
    // and the loops over chunks they bound, as warp-uniform
    const bool dead = __shfl_sync(0xffffffffu, hdr->status, 0) != GDN_OK;  // uniform across the cluster

    // cluster of FR solve CTAs (ranks 0 .. FR-1; solve CTA r takes the chunks
    // c = r, r + FR, ...) and one state CTA (rank FR)
    const uint32_t rank = tc::cluster_rank();
    const bool front = rank < (uint32_t)FR;
    const int fr = opaque_i(front ? (int)rank : 0);
    // the warp index and the TMEM base are broadcast from lane 0 so that the
    // compiler sees them as warp-uniform: role branches then stay in uniform
    // control flow and MMA descriptors are built in uniform registers
    const int tid = threadIdx.x, lane = tid & 31;
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const int n_seqs = hdr->n_seqs;
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* order = reinterpret_cast<const int*>(ws + L.order);
    const int unit = blockIdx.x / (FR + 1);
    const int seq = dead ? 0 : __shfl_sync(0xffffffffu, order[unit / H], 0);
    const int head = unit % H;
    const int start = dead ? 0 : __shfl_sync(0xffffffffu, cu[seq], 0);
    const int len = dead ? 0 : __shfl_sync(0xffffffffu, cu[seq + 1], 0) - start;
    const int nch = (len + kChunk - 1) / kChunk;
    const int nu = opaque_i(front ? (nch - fr + FR - 1) / FR : 0);  // this solve CTA's chunks

    const uint32_t bar_base = sbase + (front ? kFBar : kBBar);
    auto bar = [&](int i) { return bar_base + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + (front ? kFBar : kBBar) + kBarSlots * 8);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sptr + (front ? kFBar : kBBar) + kBarSlots * 8 + 8);
    const Waiter wait{abort_flag, ws, bar_base, front ? 1000 : 2000};
    // run modes of the two-level state scan (0 for an ordinary call): no o
    // stores; v taken as zero; h0 taken as the identity
    constexpr bool no_o = (MODE & kModeNoOutput) != 0;
    constexpr bool vzero = (MODE & kModeZeroV) != 0;
    constexpr bool h0eye = (MODE & kModeIdentityH0) != 0;

    if (!front && vzero) {  // the v tiles of both apply entries hold zeros for the whole run
        for (uint32_t x = tid; x < 2 * 2 * kBBox / 16; x += kThreads) {
            const uint32_t ent = x / (2 * kBBox / 16), off = (x % (2 * kBBox / 16)) * 16;
            tc::st_shared_v4(sbase + kARing + ent * kAEntry + kAV + off, 0u, 0u, 0u, 0u);
        }
        tc::fence_proxy_async();
    }
    if (tid == 0) {
        abort_flag[0] = 0;
        abort_flag[1] = hdr->wait_limit;
#pragma unroll 1
        for (int b = 0; b < (front ? (int)F_COUNT : (int)B_COUNT); ++b)
            tc::mbar_init(bar(b), (front && b == F_FIN) ? 4 : 1);
        tc::fence_mbar_init();
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        if (!front) {
            tc::prefetch_tmap(&tm_v);
            tc::prefetch_tmap(&tm_o);
        }
        if (GDN) {
            tc::prefetch_tmap(&tm_la);
            tc::prefetch_tmap(&tm_b);
        }
    }
    __syncwarp();  // lane-0-only work above: reconverge before any .aligned instruction
    if (warp == 0) tc::tmem_alloc(sbase + (front ? kFBar : kBBar) + kBarSlots * 8 + 8, front ? kFTmemCols : kBTmemCols);
    tc::tc_fence_before();
    __syncthreads();
    tc::cluster_sync();  // both CTAs' barriers exist before any remote access
    tc::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
    const int quad = warp & 3;
    const int row = 32 * quad + lane;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;

    // peer addresses
    const uint32_t peer_bar_b = tc::map_to_rank(sbase + kBBar, FR);  // state CTA's barriers
    const uint32_t peer_bar_f0 = tc::map_to_rank(sbase + kFBar, 0);  // solve CTAs' barriers
    const uint32_t peer_bar_f1 = tc::map_to_rank(sbase + kFBar, FR - 1);


    if (front) {
        // ============================================================ FRONT
        if (warp == 0) {
            // ---- TMA issue only (this CTA's u-th chunk in stage u % 4): runs ahead as
            // far as the ring allows; [k; q] k^T and the gate values are warp 13's
            int issued = 0;
            for (int u = 0; u < nu && !dead; ++u) {
                const int f = u % kFStages, uf = u / kFStages;
                const uint32_t st = sbase + f * kFStage;
                if (u >= kFStages) wait(bar(F_EMPTY + f), (uf - 1) & 1);
                const int t0 = start + (fr + FR * u) * kChunk;
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
                    issued = u + 1;
                    if (u + 4 < nu) {
                        const int tp = t0 + 4 * FR * kChunk;
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
            }
            if (lane == 0 && *abort_flag)
                for (int u = max(0, issued - kFStages); u < issued; ++u)
                    tc::mbar_wait(bar(F_FULL + u % kFStages), (u / kFStages) & 1);
            __syncwarp();
        } else if (warp <= 12) {
            // ---- solve groups: group g takes this CTA's chunks u with u % 3 == g
            const int grp = (warp - 1) >> 2;  // 0, 1, 2
            const int pw = (warp - 1) & 3;    // warp within the group
            const int nb = 1 + grp;           // named barrier of the group
            const bool gissuer = (pw == 3 && lane == 0);  // row 0 of the group (quadrant 0)
            float* AF = reinterpret_cast<float*>(sptr + kFAF + grp * 64 * kTriLd * 4);
            float* scr = reinterpret_cast<float*>(sptr + kFScr + grp * 4 * 128 * 4);
            const uint32_t pst = sbase + kFPst + grp * 8192;
            for (int u = grp; u < nu && !dead; u += kFGroups) {
                const int uf = u / kFGroups;
                const uint32_t stg = sbase + (u % kFStages) * kFStage;
                wait(bar(F_GREADY + grp), uf & 1);
                wait(bar(F_P1D + grp), uf & 1);
                // P^ staging and AF are rewritten below: the store warp must have read
                // this group's previous chunk out of them
                if (u >= kFGroups) wait(bar(F_SFREE + grp), (uf - 1) & 1);
                __syncwarp();
                tc::tc_fence_after();
                const float* gt = reinterpret_cast<const float*>(sptr + (u % kFStages) * kFStage + kFGate);
                const bool safe = gt[kGscal + 1] != 0.f;
                const int n = (int)gt[kGscal + 2];
                const int t = row & 63;
                // rows 0..63: K K^T -> A (fp32); rows 64..127: Q K^T -> P^ (staged, bf16),
                // in four parts of 16 columns (a short loop keeps this code small).
                // When the chunk's decay range is moderate, P^ = (q k^T)_causal e^{-g_last};
                // the back then scales v_new by e^{g_last - g} and o by e^{g}, which gives
                // the same o and h.
                {
                    const bool is_a = row < 64;
                    // safe factors: A[t][s] = KK[t][s] beta_t e^{g_t} e^{-g_s} (row t >= n of
                    // the chunk zeroed; entries on and above the diagonal are never read by the
                    // inverse, so they are not masked), P^[t][s] = QK[t][s] e^{-g_last} for
                    // s <= t (rows t >= n produce outputs that are never stored)
                    const bool tok = t < n;
                    const float rs = is_a ? (tok ? gt[kGbb + t] * gt[kGeg + t] : 0.f) : gt[kGscal + 3];
                    const float* const en = gt + (is_a ? kGeng : kGone);
                    const float gtt = gt[kGg + t], bsc = is_a ? gt[kGbb + t] : 1.f;
                    const int lim = is_a ? t : t + 1;
#pragma unroll 1
                    for (int part = 0; part < 4; ++part) {
                        float x[16];
                        tc::tmem_ld16(tmem + lane_off + kFColP1 + grp * 64 + 16 * part, x);
                        tc::tmem_wait_ld();
                        const int s0 = 16 * part;
                        if (!is_a || GDN) {
                            if (safe) {
#pragma unroll
                                for (int q4 = 0; q4 < 4; ++q4) {
                                    const float4 f = *reinterpret_cast<const float4*>(en + s0 + 4 * q4);
                                    x[4 * q4 + 0] *= f.x * rs;
                                    x[4 * q4 + 1] *= f.y * rs;
                                    x[4 * q4 + 2] *= f.z * rs;
                                    x[4 * q4 + 3] *= f.w * rs;
                                }
                                if (!is_a) {  // warp-uniform: the P^ rows are warps 2, 3 of the group
#pragma unroll
                                    for (int e2 = 0; e2 < 16; ++e2) x[e2] = s0 + e2 <= t ? x[e2] : 0.f;
                                }
                            } else {
#pragma unroll
                                for (int e2 = 0; e2 < 16; ++e2)
                                    x[e2] = (tok && s0 + e2 < lim) ? x[e2] * bsc * __expf(gtt - gt[kGg + s0 + e2]) : 0.f;
                            }
                            if (is_a) {
                                float* Ar = AF + t * kTriLd + s0;
#pragma unroll
                                for (int q4 = 0; q4 < 4; ++q4)
                                    *reinterpret_cast<float4*>(Ar + 4 * q4) =
                                        make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
                            } else {
#pragma unroll
                                for (int h2 = 0; h2 < 2; ++h2)
                                    tc::st_shared_v4(tc::sw128(pst, t, 2 * part + h2),
                                                     tc::pack_bf16(x[8 * h2], x[8 * h2 + 1]),
                                                     tc::pack_bf16(x[8 * h2 + 2], x[8 * h2 + 3]),
                                                     tc::pack_bf16(x[8 * h2 + 4], x[8 * h2 + 5]),
                                                     tc::pack_bf16(x[8 * h2 + 6], x[8 * h2 + 7]));
                            }
                        }
                    }
                }
                tc::tc_fence_before();
                tc::named_bar(nb, 128);  // DP1[group] read, A and P^ rows stored
                if (gissuer) tc::mbar_arrive(bar(F_P1F + grp));
                __syncwarp();
                if (GDN) tri_inverse_64(AF, scr, pw, lane, nb, MAXD);
                // T' = R T diag(beta e^g) (bf16, K-major) for w^T = k^T T'^T on this SM
                // (rows 0..63), and T'' = R T diag(beta) for the state CTA's u MMA (rows
                // 64..127), both into the stage's dead q tile, 16 columns at a time.  T is
                // the inverse (GDN) or the identity.  R = diag(e^{g_last - g}) when the
                // decay range is moderate (else I): it makes the state CTA's u - S w^T
                // come out as v^ = e^{g_last - g} v_new directly.
                {
                    const float* cs = gt + (row < 64 ? kGbeg : kGbb);
                    const float rf = safe ? gt[kGkdec + t] : 1.f;
                    const uint32_t dst = stg + (row < 64 ? kFT1 : kFT2);
#pragma unroll 1
                    for (int jb = 0; jb < 4; ++jb) {
                        float v[16];
                        if (GDN && jb <= (t >> 4) && (t >> 4) - jb <= MAXD) {
                            const float* Tr = tri_block_row(AF, t, jb);
#pragma unroll
                            for (int e4 = 0; e4 < 16; e4 += 4) {
                                const float4 tv = *reinterpret_cast<const float4*>(Tr + e4);
                                const float4 sv = *reinterpret_cast<const float4*>(cs + 16 * jb + e4);
                                v[e4] = tv.x * sv.x * rf;
                                v[e4 + 1] = tv.y * sv.y * rf;
                                v[e4 + 2] = tv.z * sv.z * rf;
                                v[e4 + 3] = tv.w * sv.w * rf;
                            }
                        } else {
#pragma unroll
                            for (int e4 = 0; e4 < 16; ++e4) v[e4] = (!GDN && 16 * jb + e4 == t) ? cs[t] * rf : 0.f;
                        }
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2)
                            tc::st_shared_v4(tc::sw128(dst, t, 2 * jb + h2), tc::pack_bf16(v[8 * h2], v[8 * h2 + 1]),
                                             tc::pack_bf16(v[8 * h2 + 2], v[8 * h2 + 3]),
                                             tc::pack_bf16(v[8 * h2 + 4], v[8 * h2 + 5]),
                                             tc::pack_bf16(v[8 * h2 + 6], v[8 * h2 + 7]));
                    }
                }
                tc::fence_proxy_async();
                tc::tc_fence_before();
                tc::named_bar(nb, 128);  // T' and T'' staged; AF (T) is dead
                if (GDN) {
                    if (pw == 3 && !*abort_flag) {
                        tc::tc_fence_after();
                        tc::mma_ss_n<4>(tmem + kFColW + 64 * grp, tc::sdesc(stg + kFK0, kFBlk, 1024), 128,
                                        tc::sdesc(stg + kFT1, 16, 1024), 2, kIdWU, false);
                        tc::commit_e(bar(F_WD + grp));
                    }
                    __syncwarp();
                    // -w row i = row, as [i][t] (the MN-major B operand of the state CTA's
                    // w MMA), staged in AF
                    wait(bar(F_WD + grp), uf & 1);
                    __syncwarp();
                    tc::tc_fence_after();
                    const uint32_t wst = sbase + kFAF + grp * 64 * kTriLd * 4;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        float x[32];
                        tc::tmem_ld32(tmem + lane_off + kFColW + 64 * grp + 32 * half, x);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tc::st_shared_v4(tc::sw128(wst, row, 4 * half + j), tc::pack_bf16(-x[8 * j], -x[8 * j + 1]),
                                             tc::pack_bf16(-x[8 * j + 2], -x[8 * j + 3]),
                                             tc::pack_bf16(-x[8 * j + 4], -x[8 * j + 5]),
                                             tc::pack_bf16(-x[8 * j + 6], -x[8 * j + 7]));
                    }
                    tc::fence_proxy_async();
                }
                tc::tc_fence_before();
                tc::named_bar(nb, 128);  // P^, T'' and -w staged for the store warp
                if (gissuer) tc::mbar_arrive(bar(F_STAGED + grp));
                __syncwarp();
            }
            if (pw == 3) tc::commit_e(bar(F_FIN));  // once its last w MMA is done
            __syncwarp();
        } else if (warp == 13) {
            // ---- [k; q] k^T into DP1[c % 3] and the chunk's gate values, as each
            // chunk lands
            for (int u = 0; u < nu && !dead; ++u) {
                const int c = fr + FR * u;
                const int f = u % kFStages, g = u % kFGroups, ug = u / kFGroups;
                const uint32_t st = sbase + f * kFStage;
                wait(bar(F_FULL + f), (u / kFStages) & 1);
                if (u >= kFGroups) wait(bar(F_P1F + g), (ug - 1) & 1);
                __syncwarp();
                if (!*abort_flag) {
                    tc::tc_fence_after();
                    const uint64_t d0 = tc::sdesc(st + kFK0, 16, 1024), d1 = tc::sdesc(st + kFK0 + kFBlk, 16, 1024);
                    tc::mma_ss_n<4>(tmem + kFColP1 + g * 64, d0, 2, d0, 2, kIdP1, false);
                    tc::mma_ss_n<4>(tmem + kFColP1 + g * 64, d1, 2, d1, 2, kIdP1, true);
                    tc::commit_e(bar(F_P1D + g));
                }
                const float* la_raw = reinterpret_cast<const float*>(sptr + f * kFStage + kFGRaw);
                derive_gates<GDN>(la_raw, la_raw + 256, head & 3, min(kChunk, len - c * kChunk),
                                  reinterpret_cast<float*>(sptr + f * kFStage + kFGate), lane);
                if (lane == 0) tc::mbar_arrive(bar(F_GREADY + g));
                __syncwarp();
            }
            tc::commit_e(bar(F_FIN));  // once its last MMA is done
            __syncwarp();
        } else if (warp >= 14) {
            // ---- store warps (14: even u, 15: odd u): each chunk's P^, T'' and
            // -w go from the group's staging to this unit's global scratch slot c % 6
            // (bulk copies through L2; the state CTA loads them from there) and are
            // announced once written.  A slot is rewritten only after the state CTA has
            // read the chunk it held before.
            char* const slot0 = scratch + (size_t)unit * kScratchUnit;
            for (int u = warp - 14; u < nu && !dead; u += 2) {
                const int c = fr + FR * u;
                const int grp = u % kFGroups, uf = u / kFGroups, sl = c % kSlots;
                wait(bar(F_STAGED + grp), uf & 1);
                if (c >= kSlots) wait.remote(bar(F_ARMED + sl), (c / kSlots - 1) & 1);
                __syncwarp();
                if (lane == 0) {
                    const bool go = !*abort_flag;
                    if (go) {
                        char* const slot = slot0 + sl * kScratchSlot;
                        tc::bulk_store(slot, sbase + kFPst + grp * 8192, 8192);
                        tc::bulk_store(slot + 8192, sbase + (u % kFStages) * kFStage + kFT2, 8192);
                        if (GDN) tc::bulk_store(slot + 16384, sbase + kFAF + grp * 64 * kTriLd * 4, 16384);
                        tc::bulk_commit();
                        tc::bulk_wait_read0();
                    }
                    tc::mbar_arrive(bar(F_SFREE + grp));  // the staging and the stage may be reused
                    tc::mbar_arrive(bar(F_EMPTY + u % kFStages));
                    if (go) {  // the slot's writes are done: tell the state CTA
                        tc::bulk_wait0();
                        tc::fence_proxy_async_global();
                        tc::fence_acq_rel_gpu();
                        tc::mbar_arrive_remote(peer_bar_b + 8u * (B_STORED + sl));
                    }
                }
                __syncwarp();
            }
        }
    } else {
        // ============================================================ BACK
        if (warp == 0) {
            // ---- TMA into both rings (issue only; warp 14 derives the gate values,
            // warp 15 loads the solve CTA's tiles)
            int issued = 0;
            for (int c = 0; c < nch && !dead; ++c) {
                const int e = c % 3, a = c & 1;
                const uint32_t ce = sbase + e * kCEntry, ae = sbase + kARing + a * kAEntry;
                if (c >= 3) wait(bar(B_CFREE + e), (c / 3 - 1) & 1);
                if (c >= 2) {
                    wait(bar(B_AFREE + a), ((c >> 1) - 1) & 1);
                    // chunk c - 2's raw log-decay in this apply entry has been read
                    wait(bar(B_GREADY + (c - 2) % 3), ((c - 2) / 3) & 1);
                }
                const int t0 = start + c * kChunk;
                if (lane == 0 && !*abort_flag) {
                    tc::mbar_arrive_expect_tx(bar(B_FULLC + e), 4 * 8192);
                    tc::tma_load_3d(ce + kCQ, &tm_q, 0, head, t0, bar(B_FULLC + e));
                    tc::tma_load_3d(ce + kCQ + kBBox, &tm_q, 64, head, t0, bar(B_FULLC + e));
                    tc::tma_load_3d(ce + kCK, &tm_k, 0, head, t0, bar(B_FULLC + e));
                    tc::tma_load_3d(ce + kCK + kBBox, &tm_k, 64, head, t0, bar(B_FULLC + e));
                    tc::mbar_arrive_expect_tx(bar(B_FULLA + a), (vzero ? 0 : 2 * 8192) + (GDN ? 1024 : 0));
                    if (!vzero) {
                        tc::tma_load_3d(ae + kAV, &tm_v, 0, head, t0, bar(B_FULLA + a));
                        tc::tma_load_3d(ae + kAV + kBBox, &tm_v, 64, head, t0, bar(B_FULLA + a));
                    }
                    if (GDN) tc::tma_load_2d(ae + kALa, &tm_la, head & ~3, t0, bar(B_FULLA + a));
                    issued = c + 1;
                    if (c + 2 < nch && !vzero) {
                        const int tp = t0 + 2 * kChunk;
                        tc::tma_prefetch_3d(&tm_v, 0, head, tp);
                        tc::tma_prefetch_3d(&tm_v, 64, head, tp);
                    }
                }
                __syncwarp();
            }
            // after an abort, let the loads already issued land before the CTA exits
            // (up to three chain entries and two apply entries can be in flight)
            if (lane == 0 && *abort_flag)
                for (int c = max(0, issued - 3); c < issued; ++c) {
                    tc::mbar_wait(bar(B_FULLC + c % 3), (c / 3) & 1);
                    if (c >= issued - 2) tc::mbar_wait(bar(B_FULLA + (c & 1)), (c >> 1) & 1);
                }
            __syncwarp();
        } else if (warp <= 4) {
            // ---- output: o = e^g D1o (or D1o), thread = TMEM lane j (an o column)
            const int j = row;
            const bool ostore = (warp == 1 && lane == 0);
            for (int c = 0; c < nch && !dead; ++c) {
                const int e = c % 3, b = c & 1;
                const uint32_t ce = sbase + e * kCEntry;
                const float* gt = reinterpret_cast<const float*>(sptr + e * kCEntry + kCGate);
                wait(bar(B_M3 + b), (c >> 1) & 1);
                wait(bar(B_GREADY + e), (c / 3) & 1);
                __syncwarp();  // lanes may leave the waits apart; tcgen05.ld is warp-collective
                tc::tc_fence_after();
                const bool fold = gt[kGscal + 1] != 0.f;
                const int n = min(kChunk, len - c * kChunk);
                const int t0 = start + c * kChunk;
                const bool full = n == kChunk;
                // o = e^g D1o (or D1o) in four parts of 16 tokens: a full chunk is staged
                // as two [64 t][64 j] SW128 boxes in the k tile (k is dead once D1o is
                // complete) for two TMA stores; the last, partial chunk of a sequence goes
                // through fp32 scratch in the same dead entry and plain stores.
                // Row t = 8u + r of a swizzled box sits at u * 1024 + off[r].
                const uint32_t box = ce + kCK + (uint32_t)(j >> 6) * kBBox;
                const uint32_t ch = (uint32_t)(j & 63) >> 3, jj = (uint32_t)(j & 7) * 2;
                uint32_t off[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) off[r] = box + r * 128 + ((ch ^ r) << 4) + jj;
                float* xs = reinterpret_cast<float*>(sptr + e * kCEntry + kCK) + j * 65;
#pragma unroll 1
                for (int part = 0; part < 4; ++part) {
                    float x[16];
                    tc::tmem_ld16(tmem + lane_off + kTD1o + 64 * b + 16 * part, x);
                    tc::tmem_wait_ld();
                    if (opaque(fold)) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const float4 eg = *reinterpret_cast<const float4*>(gt + kGeg + 16 * part + 4 * q4);
                            x[4 * q4] *= eg.x;
                            x[4 * q4 + 1] *= eg.y;
                            x[4 * q4 + 2] *= eg.z;
                            x[4 * q4 + 3] *= eg.w;
                        }
                    }
                    if (opaque(full)) {
#pragma unroll
                        for (int e2 = 0; e2 < 16; ++e2)
                            st_shared_u16(off[e2 & 7] + (2 * part + (e2 >> 3)) * 1024,
                                          __bfloat16_as_ushort(__float2bfloat16_rn(x[e2])));
                    } else {
#pragma unroll
                        for (int e2 = 0; e2 < 16; ++e2) xs[16 * part + e2] = x[e2];
                    }
                }
                tc::fence_proxy_async();
                tc::tc_fence_before();
                tc::named_bar(1, 128);
                if (ostore) {
                    tc::mbar_arrive(bar(B_D1OF + b));
                    if (full) {
                        if (!*abort_flag && !no_o) {
                            tc::tma_store_3d(&tm_o, ce + kCK, 0, head, t0);
                            tc::tma_store_3d(&tm_o, ce + kCK + kBBox, 64, head, t0);
                            tc::bulk_commit();
                        }
                        tc::bulk_wait_read0();
                        tc::mbar_arrive(bar(B_CFREE + e));
                    }
                }
                __syncwarp();
                if (!full) {
                    if (!*abort_flag && !no_o) {
#pragma unroll 1
                        for (int t = 0; t < n; ++t)
                            o[((size_t)(t0 + t) * H + head) * kD + j] = __float2bfloat16_rn(xs[t]);
                    }
                    tc::named_bar(1, 128);
                    if (ostore) tc::mbar_arrive(bar(B_CFREE + e));
                    __syncwarp();
                }
            }
            if (ostore) tc::bulk_wait0();
            __syncwarp();
        } else if (warp <= 12) {
            // ---- the state chain: 8 warps; thread = (state row j = TMEM lane, half hh).
            // S = h^T (dv x dk) lives in TMEM: fp32 in D2 (the MMA accumulates the
            // chunk update onto it) and bf16 in TS (the A operand of the MMAs with q
            // and -w).
            const int hh = (warp - 5) >> 2;
            const int j = row;
            const int ct = tid - 160;  // 0..255
            const bool cl = (warp == 5 && lane == 0);  // signals the MMA warp
            const size_t hbase = ((size_t)seq * H + head) * kD * kD;  // h[i][j] at hbase + i * kD + j
            const uint32_t d2 = tmem + lane_off + kTD2 + 64 * hh;
            const uint32_t ts = tmem + lane_off + kTS + 32 * hh;
            // S (bf16) <- S (fp32)
            // (both halves loaded before one wait: this step is on the state chain's
            // critical path)
            auto snapshot = [&]() {
                float d[32], d1[32];
                tc::tmem_ld32(d2, d);
                tc::tmem_ld32(d2 + 32, d1);
                tc::tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) pk[e2] = tc::pack_bf16(d[2 * e2], d[2 * e2 + 1]);
                tc::tmem_st16(ts, pk);
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) pk[e2] = tc::pack_bf16(d1[2 * e2], d1[2 * e2 + 1]);
                tc::tmem_st16(ts + 16, pk);
                tc::tmem_wait_st();
            };
            // S (fp32) *= f
            auto decay = [&](float f) {
#pragma unroll 1
                for (int part = 0; part < 4; ++part) {
                    float d[16];
                    tc::tmem_ld16(d2 + 16 * part, d);
                    tc::tmem_wait_ld();
                    uint32_t r[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) r[e2] = __float_as_uint(d[e2] * f);
                    tc::tmem_st16(d2 + 16 * part, r);
                }
                tc::tmem_wait_st();
            };
            // strong-decay chunk: q~ = e^g q and k~ = e^{g_last - g} k in place
            auto prescale = [&](int c) {
                const int e = c % 3;
                wait(bar(B_FULLC + e), (c / 3) & 1);
                wait(bar(B_GREADY + e), (c / 3) & 1);
                __syncwarp();
                const float* gt = reinterpret_cast<const float*>(sptr + e * kCEntry + kCGate);
                if (gt[kGscal + 1] == 0.f) {
                    const int which = ct >> 7, t = (ct >> 1) & 63, bx = ct & 1;
                    const uint32_t rowbox = sbase + e * kCEntry + (which ? kCK : kCQ) + bx * kBBox;
                    const float f = which ? gt[kGkdec + t] : gt[kGeg + t];
                    const __nv_bfloat162 f2 = __float2bfloat162_rn(f);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const uint32_t ad = tc::sw128(rowbox, t, jj);
                        uint4 v4 = tc::ld_shared_v4(ad);
                        __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&v4);
                        p2[0] = __hmul2(p2[0], f2);
                        p2[1] = __hmul2(p2[1], f2);
                        p2[2] = __hmul2(p2[2], f2);
                        p2[3] = __hmul2(p2[3], f2);
                        tc::st_shared_v4(ad, v4.x, v4.y, v4.z, v4.w);
                    }
                    tc::fence_proxy_async();
                }
                return gt[kGscal + 0];  // e^{g_last} of chunk c
            };
            {  // S from h0 (h0[i][j], i = 64 hh + x)
#pragma unroll 1
                for (int part = 0; part < 4; ++part) {
                    uint32_t r[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x)
                        r[x] = __float_as_uint(h0eye ? (64 * hh + 16 * part + x == j ? 1.f : 0.f)
                                               : (h0 && !dead) ? h0[hbase + (size_t)(64 * hh + 16 * part + x) * kD + j] : 0.f);
                    tc::tmem_st16(d2 + 16 * part, r);
                }
                tc::tmem_wait_st();
            }
            // c = -1 only prepares chunk 0: S (bf16) from h0, the gates of chunk 0, the
            // decay of S (fp32) for chunk 0; every later pass first finishes chunk c.
            // (One copy of each step keeps this warp's instruction footprint small.)
            for (int c = -1; c < nch && !dead; ++c) {
                if (c >= 0) {
                    const int b = c & 1;
                    // (1) v^ = e^{g_last - g} v_new (or v_new) to bf16 in TMEM: the solve CTA
                    // folded the factor into the rows of T' and T'', so D1v already holds it
                    wait(bar(B_M1W), c & 1);
                    __syncwarp();
                    tc::tc_fence_after();
                    {
                        float x[32];
                        tc::tmem_ld32(tmem + lane_off + kTD1v + 64 * b + 32 * hh, x);
                        tc::tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int e2 = 0; e2 < 16; ++e2) pk[e2] = tc::pack_bf16(x[2 * e2], x[2 * e2 + 1]);
                        tc::tmem_st16(tmem + lane_off + kTVN + 16 * hh, pk);
                        tc::tmem_wait_st();
                    }
                    tc::tc_fence_before();
                    tc::named_bar(2, 256);
                    if (cl) tc::mbar_arrive(bar(B_VREADY));
                    __syncwarp();
                }
                // (2) q, k of a strong-decay next chunk, while S += v^^T k runs
                const float egl_next = c + 1 < nch ? prescale(c + 1) : 1.f;
                if (c >= 0) {  // S is now the state after chunk c
                    wait(bar(B_M2), c & 1);
                    __syncwarp();
                    tc::tc_fence_after();
                }
                // (3) S (bf16) for the next chunk's MMAs
                if (c + 1 < nch) snapshot();
                tc::tc_fence_before();
                tc::named_bar(2, 256);
                if (cl && c + 1 < nch) tc::mbar_arrive(bar(B_SREADY));
                __syncwarp();
                // (4) while the next MMAs run: S (fp32) <- e^{g_last} S for the next chunk;
                // the named barrier after the next v^ orders it before the next S += v^^T k
                if (GDN && c + 1 < nch) decay(egl_next);
            }
            if (h_T && !*abort_flag && !dead) {
                tc::tc_fence_after();
#pragma unroll 1
                for (int part = 0; part < 4; ++part) {
                    float d[16];
                    tc::tmem_ld16(d2 + 16 * part, d);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 16; ++x) h_T[hbase + (size_t)(64 * hh + 16 * part + x) * kD + j] = d[x];
                }
            }
        } else if (warp == 14) {
            // ---- the gate values of each chunk, as its log-decay lands
            for (int c = 0; c < nch && !dead; ++c) {
                const int e = c % 3, a = c & 1;
                wait(bar(B_FULLA + a), (c >> 1) & 1);
                __syncwarp();
                const float* la_raw = reinterpret_cast<const float*>(sptr + kARing + a * kAEntry + kALa);
                derive_gates<GDN>(la_raw, la_raw, head & 3, min(kChunk, len - c * kChunk),
                                  reinterpret_cast<float*>(sptr + e * kCEntry + kCGate), lane);
                if (lane == 0) tc::mbar_arrive(bar(B_GREADY + e));
                __syncwarp();
            }
        } else if (warp == 15) {
            // ---- the solve CTA's P^, -w (chain entry c % 3) and T'' (apply entry c % 2),
            // loaded from its global scratch slot c % 3 once it is stored there and the
            // entries are free
            const char* const slot0 = scratch + (size_t)unit * kScratchUnit;
            int issued = 0;
            for (int c = 0; c < nch && !dead; ++c) {
                const int e = c % 3, a = c & 1, sl = c % kSlots;
                wait.remote(bar(B_STORED + sl), (c / kSlots) & 1);
                if (c >= 3) wait(bar(B_CFREE + e), (c / 3 - 1) & 1);
                if (c >= 2) wait(bar(B_AFREE + a), ((c >> 1) - 1) & 1);
                __syncwarp();
                if (lane == 0 && !*abort_flag) {
                    const char* const slot = slot0 + sl * kScratchSlot;
                    const uint32_t ce = sbase + e * kCEntry, ae = sbase + kARing + a * kAEntry;
                    tc::fence_proxy_async_global();
                    tc::mbar_arrive_expect_tx(bar(B_FULLP + e), GDN ? 4 * 8192 : 2 * 8192);
                    tc::bulk_load(ce + kCP, slot, 8192, bar(B_FULLP + e));
                    tc::bulk_load(ae + kAT2, slot + 8192, 8192, bar(B_FULLP + e));
                    if (GDN) tc::bulk_load(ce + kCW, slot + 16384, 16384, bar(B_FULLP + e));
                    issued = c + 1;
                }
                __syncwarp();
            }
            // after an abort, let the loads already issued land before the CTA exits
            if (lane == 0 && *abort_flag)
                for (int c = max(0, issued - 3); c < issued; ++c) tc::mbar_wait(bar(B_FULLP + c % 3), (c / 3) & 1);
            __syncwarp();
        } else {
            // ---- the MMA warp: every MMA of the back, in chunk order
            for (int c = 0; c < nch && !dead; ++c) {
                const int e = c % 3, a = c & 1, b = c & 1;
                const uint32_t ce = sbase + e * kCEntry, ae = sbase + kARing + a * kAEntry;
                // D1v[b] = u^T = v^T T''^T
                wait(bar(B_FULLA + a), (c >> 1) & 1);
                wait(bar(B_FULLP + e), (c / 3) & 1);
                if (lane == 0)  // slot read: the solve CTA of chunk c may rewrite it
                    tc::mbar_arrive_remote_relaxed((c % FR == 0 ? peer_bar_f0 : peer_bar_f1) + 8u * (F_ARMED + c % kSlots));
                __syncwarp();
                if (!*abort_flag) {
                    tc::tc_fence_after();
                    tc::mma_ss_n<4>(tmem + kTD1v + 64 * b, tc::sdesc(ae + kAV, kBBox, 1024), 128,
                                    tc::sdesc(ae + kAT2, 16, 1024), 2, kIdWU, false);
                    tc::commit_e(bar(B_AFREE + a));
                }
                // D1v[b] += S (-w)^T once S(c) is in TMEM
                wait(bar(B_SREADY), c & 1);
                wait(bar(B_FULLC + e), (c / 3) & 1);
                if (!*abort_flag) {
                    tc::tc_fence_after();
                    if (GDN)
                        tc::mma_ts_n<8>(tmem + kTD1v + 64 * b, tmem + kTS, 8, tc::sdesc(ce + kCW, kBBox, 1024), 128,
                                        kId1w, true);
                    tc::commit_e(bar(B_M1W));
                }
                // D1o[b] = S q^T once the output warps have read D1o[b]
                if (c >= 2) wait(bar(B_D1OF + b), ((c >> 1) - 1) & 1);
                if (!*abort_flag) {
                    tc::tc_fence_after();
                    tc::mma_ts_n<4>(tmem + kTD1o + 64 * b, tmem + kTS, 8, tc::sdesc(ce + kCQ, 16, 1024), 2, kId1q, false);
                    tc::mma_ts_n<4>(tmem + kTD1o + 64 * b, tmem + kTS + 32, 8, tc::sdesc(ce + kCQ + kBBox, 16, 1024), 2,
                                    kId1q, true);
                }
                // S += v^^T k; D1o[b] += v^^T P^^T
                wait(bar(B_VREADY), c & 1);
                if (!*abort_flag) {
                    tc::tc_fence_after();
                    tc::mma_ts_n<4>(tmem + kTD2, tmem + kTVN, 8, tc::sdesc(ce + kCK, kBBox, 1024), 128, kId2, true);
                    tc::commit_e(bar(B_M2));
                    tc::mma_ts_n<4>(tmem + kTD1o + 64 * b, tmem + kTVN, 8, tc::sdesc(ce + kCP, 16, 1024), 2, kId3, true);
                    tc::commit_e(bar(B_M3 + b));
                }
            }
            tc::commit_e(bar(B_FIN));
        }
    }

    // drain this CTA's MMAs, then release TMEM; the cluster barrier keeps
    // either CTA from exiting while the other may still touch its memory
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) tc::mbar_wait(bar(front ? F_FIN : B_FIN), 0);
    __syncwarp();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, front ? kFTmemCols : kBTmemCols);
    tc::cluster_sync();
}

}  // namespace pair

// Workspace of the cluster kernel: the plan, then the per-(sequence, head)
// global scratch slots at the next 1 KB boundary.
static size_t pair_scratch_offset(int n_seqs) { return (PlanLayout(n_seqs).end + 1023) & ~(size_t)1023; }
size_t pair_workspace_bytes(int n_seqs, int H) {
    return pair_scratch_offset(n_seqs) + (size_t)n_seqs * (size_t)H * pair::kScratchUnit;
}

bool pair_shape_ok(const PrefillArgs& a) {
    return a.io == GDN_BF16 && a.dk == 128 && a.dv == 128 && (!a.delta_rule || a.H % 4 == 0);
}

bool pair_supported(const PrefillArgs& a) {
    auto al = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
    if (a.io != GDN_BF16 || a.dk != 128 || a.dv != 128) return false;
    if (a.delta_rule) {
        if (a.H % 4 != 0) return false;
        if (!al(a.log_alpha, 16) || !al(a.beta, 16)) return false;
    }
    return al(a.q, 16) && al(a.k, 16) && al(a.v, 16) && tensor_map_encoder() != nullptr;
}

// The instantiation for a call: the ordinary prefill (exact or block-adjacent
// solve, GDN or linear attention), or one of the runs of the two-level state
// scan (transition maps: no o, v = 0, h0 = I; offsets: no o).
using PairKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                            const float*, __nv_bfloat16*, float*, char*, char*, int);
template <int FR>
static PairKernel pick_fr(const PrefillArgs& a) {
    using namespace pair;
    constexpr int kMaps = kModeNoOutput | kModeZeroV | kModeIdentityH0;
    if (!a.delta_rule) {
        if (a.mode == 0) return pair_kernel<false, FR, 3, 0>;
        if (a.mode == kModeNoOutput) return pair_kernel<false, FR, 3, kModeNoOutput>;
        return nullptr;
    }
    if (a.mode == 0) return a.max_block_dist == 1 ? pair_kernel<true, FR, 1, 0> : pair_kernel<true, FR, 3, 0>;
    if (a.max_block_dist != 3) return nullptr;
    if (a.mode == kModeNoOutput) return pair_kernel<true, FR, 3, kModeNoOutput>;
    if (a.mode == kMaps) return pair_kernel<true, FR, 3, kMaps>;
    return nullptr;
}
static PairKernel pick_kernel(const PrefillArgs& a, int fronts) {
    return fronts == 2 ? pick_fr<2>(a) : pick_fr<1>(a);
}

cudaError_t launch_pair(const PrefillArgs& a, int fronts, cudaStream_t st) {
    using namespace pair;
    const long long units = (long long)a.n_seqs * a.H;
    if (units == 0) return cudaSuccess;
    if (fronts != 1 && fronts != 2) return cudaErrorInvalidValue;
    if ((fronts + 1) * units > 0x7fffffffLL) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mla, mb, mo;
    const int64_t T = a.T_total > 0 ? a.T_total : 1;
    const void* base = a.q ? a.q : a.ws;
    if (!encode_token_map(&mq, a.q ? a.q : base, T, a.H) || !encode_token_map(&mk, a.k ? a.k : base, T, a.H) ||
        !encode_token_map(&mv, a.v ? a.v : base, T, a.H) || !encode_token_map(&mo, a.o ? a.o : base, T, a.H))
        return cudaErrorInvalidValue;
    if (a.delta_rule) {
        if (!encode_gate_map(&mla, a.log_alpha ? a.log_alpha : (const float*)base, T, a.H) ||
            !encode_gate_map(&mb, a.beta ? a.beta : (const float*)base, T, a.H))
            return cudaErrorInvalidValue;
    } else {
        mla = mq;
        mb = mq;
    }
    auto kern = pick_kernel(a, fronts);
    if (kern == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((fronts + 1) * units), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = fronts + 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mla, mb, mo, a.h0, (__nv_bfloat16*)a.o, a.h_T, a.ws,
                           a.ws + pair_scratch_offset(a.n_seqs), a.H);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn
