// linear_variants.cu -- linear attention with the causal mask optional and the
// normaliser optional (bf16, dk = dv = 128):
//     o_t = sum_s (q_t . k_s) v_s  [/ sum_s (q_t . k_s)],
// s over all tokens of the sequence (bidirectional) or s <= t (causal).
// The normalised, bidirectional form is the listing of "За пределами
// self-attention…" (section "Линейное внимание…"): K^T V and the summed keys
// first, then q times each; the bidirectional mode and the causal restriction
// are those of the ai-vestnik.ru item on linear attention.
//
// Bidirectional: kv_reduce_kernel streams k and v of a group of chunks through
// a TMA ring and forms K^T V (tcgen05, fp32 in TMEM) and the summed keys per
// sequence and head, adding each group's partial sums to the workspace;
// kv_apply_kernel streams q through a TMA ring and computes q [K^T V | z]
// (tcgen05; K^T V and z rounded once to bf16 as the B operand, z as an extra
// column so q . z comes out of the same MMA), divides by q . z when
// normalised, and stores o with TMA.
// Causal (normalised or not): the sequences are cut into groups of chunks; the
// groups' K^T V and key sums give every group's starting state and key sum by
// a prefix, and every group then runs its chunks from there, all groups side
// by side (the causal normaliser q_t . (sum of k_s, s <= t) comes out of the
// same pass).
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"

namespace gdn {

int sm_count();
bool encode_token_map(CUtensorMap* m, const void* ptr, int64_t T, int H);

namespace linvar {

constexpr int kD = 128;
constexpr int kMinGroup = kGroupMinChunks;  // chunks per reduce / apply CTA, at least

struct ChunkRef {
    int seq, t0, n;
};
__device__ __forceinline__ ChunkRef chunk_ref(const int* cu, const int* chunk_off, int n_seqs, int gc) {
    ChunkRef r;
    r.seq = seq_of_chunk(chunk_off, n_seqs, gc);
    r.t0 = cu[r.seq] + (gc - chunk_off[r.seq]) * kChunk;
    r.n = min(kChunk, cu[r.seq + 1] - r.t0);
    return r;
}

// Bounded wait by one thread.  A wait that runs out records GDN_ERR_TIMEOUT
// (and the site) in the status word and sets the CTA's abort flag; a wait
// that finds the flag set returns false at once.
__device__ __noinline__ bool lv_wait(uint32_t bar, uint32_t parity, char* ws, volatile int* abort_flag, int site) {
    if (*abort_flag) return false;
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (tc::mbar_wait(bar, parity, abort_flag[1])) return true;
    WsHeader* h = reinterpret_cast<WsHeader*>(ws);
    atomicExch(&h->status, GDN_ERR_TIMEOUT);
    atomicCAS(&h->timeout_site, 0, site);
    *abort_flag = 1;
    return false;
}
// The same wait taken once for a whole warp (lane 0 waits) or a whole
// 128-thread group (its leader waits), the outcome shared by all of them, so
// that no member leaves a loop the others stay in.  The warp form reads the
// abort flag after the warp has converged, one load of one address for all
// 32 lanes (a shuffle of lane 0's result instead made the MMA warps of these
// kernels measurably slower); the group form reduces the leader's result over
// the group's named barrier.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, char* ws, volatile int* abort_flag, int site) {
    if ((threadIdx.x & 31) == 0) lv_wait(bar, parity, ws, abort_flag, site);
    __syncwarp();
    return *abort_flag == 0;
}
__device__ __forceinline__ bool group_wait(bool leader, int bar_id, uint32_t bar, uint32_t parity, char* ws,
                                           volatile int* abort_flag, int site) {
    bool ok = true;
    if (leader) ok = lv_wait(bar, parity, ws, abort_flag, site);
    return tc::named_bar_and(bar_id, 128, ok);
}

// Sum of column f (0..127) of a 64-row bf16 k tile in two SW128 boxes, rows
// 0..n-1 (the key sums; four running sums for a short dependent chain).
__device__ __forceinline__ float key_column_sum(uint32_t k0, int f, int n) {
    const uint32_t col = k0 + (uint32_t)(f >> 6) * 8192 + (uint32_t)((f & 7) * 2);
    const uint32_t c16 = (uint32_t)((f & 63) >> 3);
    auto at = [&](int t) {
        uint16_t h;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h)
                     : "r"(col + (uint32_t)t * 128 + (((c16 ^ (uint32_t)t) & 7u) << 4)));
        return __bfloat162float(__ushort_as_bfloat16(h));
    };
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int t = 0;
#pragma unroll 4
    for (; t + 4 <= n; t += 4) {
        a0 += at(t);
        a1 += at(t + 1);
        a2 += at(t + 2);
        a3 += at(t + 3);
    }
    for (; t < n; ++t) a0 += at(t);
    return (a0 + a1) + (a2 + a3);
}

constexpr int kLvThreads = 256;  // warp 0 TMA, warp 1 MMA, warps 4..7 the 128-thread worker group

// ---------------------------------------------------------------- reduce
// A ring of kRStages stages, each [k box0 | k box1 | v box0 | v box1] (64
// tokens x 64 features, SW128, straight from the tensor maps), then the
// barriers, the abort flag and bound, the TMEM slot.
constexpr int kRStages = 3;
constexpr uint32_t kRStage = 32768;
constexpr uint32_t kRBarOff = kRStages * kRStage;
enum { R_FULL = 0, R_READY = 3, R_EMPTY = 6, R_RUNDONE = 9, R_TFREE = 10, R_FIN = 11, R_COUNT = 12 };
constexpr uint32_t kRSmem = kRBarOff + 128 + 1024;
constexpr uint32_t kIdKV = tc::idesc_bf16(128, 128, true, true);  // A = k^T, B = v, both MN-major

// Sequence and chunk range of group g when every sequence is cut into groups
// of `group` consecutive chunks (group_off[s] = first group of sequence s).
__device__ __forceinline__ void group_range(const int* group_off, const int* chunk_off, int n_seqs, int group,
                                            int g, int& seq, int& c0, int& nc) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (group_off[mid] <= g) lo = mid; else hi = mid - 1;
    }
    seq = lo;
    c0 = chunk_off[seq] + (g - group_off[seq]) * group;
    nc = max(0, min(chunk_off[seq + 1], c0 + group) - c0);
}

// GROUPED = false: bidirectional sums; CTA (x, head) takes the global chunks
//   [x group, (x + 1) group) and adds each sequence's part of K^T V and of the
//   key sums to kv[seq][head], z[seq][head].
// GROUPED = true: the causal path's group sums in two halves; CTA (2 g + p,
//   head) takes half p of group g (group_off, the group size in
//   group_off[n_seqs + 1]) and writes its K^T V and key sums to
//   kv[2 g + p][head], z[2 g + p][head].
template <bool GROUPED>
__global__ void __launch_bounds__(kLvThreads, 2)  // two CTAs per SM (registers <= 128)
kv_reduce_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, int H,
                 int group, char* __restrict__ ws, const int* __restrict__ group_off, float* __restrict__ kv,
                 float* __restrict__ z) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sbase = raw + pad;
    char* const sptr = reinterpret_cast<char*>(smem_raw) + pad;
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;
    const int total = hdr->total_chunks, n_seqs = hdr->n_seqs;
    const int head = blockIdx.y;
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* chunk_off = reinterpret_cast<const int*>(ws + L.chunk_off);
    int g0, nc, gseq = 0;
    if (GROUPED) {  // CTA x = 2 g + part takes the first or the second half of group g
        const int gg = blockIdx.x >> 1, part = blockIdx.x & 1;
        if (gg >= group_off[n_seqs]) return;
        int c0g, ncg;
        group_range(group_off, chunk_off, n_seqs, group_off[n_seqs + 1], gg, gseq, c0g, ncg);
        const int first = (ncg + 1) >> 1;
        g0 = part ? c0g + first : c0g;
        nc = part ? ncg - first : first;
        if (nc == 0) {  // an empty half: its partial sums are zero
            float* dst = kv + ((size_t)blockIdx.x * H + head) * kD * kD;
            for (int x = threadIdx.x; x < kD * kD; x += blockDim.x) dst[x] = 0.f;
            if (threadIdx.x < kD) z[((size_t)blockIdx.x * H + head) * kD + threadIdx.x] = 0.f;
            return;
        }
    } else {
        g0 = blockIdx.x * group;
        if (g0 >= total) return;
        nc = min(total, g0 + group) - g0;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) { return sbase + kRBarOff + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + kRBarOff + 96);

    if (tid == 0) {
        for (int b = 0; b < R_COUNT; ++b) tc::mbar_init(bar(b), (b >= R_EMPTY && b < R_EMPTY + kRStages) ? 2 : 1);
        tc::fence_mbar_init();
        abort_flag[0] = 0;
        abort_flag[1] = hdr->wait_limit;
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
    }
    __syncwarp();
    if (warp == 0) tc::tmem_alloc(sbase + kRBarOff + 104, 128);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t*>(sptr + kRBarOff + 104), 0);

    if (warp == 0) {
        // ---- TMA: k and v of each chunk into stage i % kRStages
        int issued = 0;
        if (lane == 0) {
            for (int i = 0; i < nc; ++i) {
                const int s = i % kRStages;
                if (i >= kRStages && !lv_wait(bar(R_EMPTY + s), ((i / kRStages) - 1) & 1, ws, abort_flag, 4100)) break;
                const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, g0 + i);
                const uint32_t st = sbase + s * kRStage;
                tc::mbar_arrive_expect_tx(bar(R_FULL + s), kRStage);
                tc::tma_load_3d(st, &tm_k, 0, head, r.t0, bar(R_FULL + s));
                tc::tma_load_3d(st + 8192, &tm_k, 64, head, r.t0, bar(R_FULL + s));
                tc::tma_load_3d(st + 16384, &tm_v, 0, head, r.t0, bar(R_FULL + s));
                tc::tma_load_3d(st + 24576, &tm_v, 64, head, r.t0, bar(R_FULL + s));
                issued = i + 1;
            }
            if (*abort_flag)  // let the copies already issued land before the CTA exits
                for (int i = max(0, issued - kRStages); i < issued; ++i)
                    tc::mbar_wait(bar(R_FULL + i % kRStages), (i / kRStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA: D (TMEM, 128 x 128 fp32) += k^T v per chunk; one run per sequence
        int run_seq = -1, runs = 0;
        bool fresh = true, ok = true;
        for (int i = 0; i < nc && ok; ++i) {
            const int s = i % kRStages;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, g0 + i);
            if (r.seq != run_seq) {
                if (run_seq >= 0) {
                    tc::commit_e(bar(R_RUNDONE));  // the run's MMAs are done: the workers may read D
                    if (!(ok = warp_wait(bar(R_TFREE), (runs - 1) & 1, ws, abort_flag, 4101))) break;
                }
                run_seq = r.seq;
                ++runs;
                fresh = true;
            }
            if (!(ok = warp_wait(bar(R_READY + s), (i / kRStages) & 1, ws, abort_flag, 4102))) break;
            tc::tc_fence_after();
            const uint32_t st = sbase + s * kRStage;
            tc::mma_ss_n<4>(tmem, tc::sdesc(st, 8192, 1024), 128, tc::sdesc(st + 16384, 8192, 1024), 128, kIdKV, !fresh);
            tc::commit_e(bar(R_EMPTY + s));
            fresh = false;
        }
        if (ok && run_seq >= 0) tc::commit_e(bar(R_RUNDONE));
        tc::commit_e(bar(R_FIN));
        __syncwarp();
    } else if (warp >= 4) {
        // ---- workers: feature f = TMEM row f; zero v rows past a partial chunk's
        // end, sum the keys, and add each run's D and key sums to the totals
        const int f = tid - 128;
        const bool leader = f == 0;
        int run_seq = -1, runs = 0;
        float zsum = 0.f;
        auto flush = [&](int seq) -> bool {
            if (!group_wait(leader, 1, bar(R_RUNDONE), (runs - 1) & 1, ws, abort_flag, 4103)) return false;
            tc::tc_fence_after();
            const size_t slot = GROUPED ? (size_t)blockIdx.x : (size_t)seq;
            float* dst = kv + ((slot * H + head) * kD + f) * kD;
            float d[32];
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * c, d);
                tc::tmem_wait_ld();
                if (GROUPED) {  // this CTA alone owns the group's slot
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        *reinterpret_cast<float4*>(dst + 32 * c + x) = make_float4(d[x], d[x + 1], d[x + 2], d[x + 3]);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; x += 4)
                        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 32 * c + x),
                                     "f"(d[x]), "f"(d[x + 1]), "f"(d[x + 2]), "f"(d[x + 3])
                                     : "memory");
                }
            }
            if (GROUPED) z[(slot * H + head) * kD + f] = zsum;
            else atomicAdd(z + (slot * H + head) * kD + f, zsum);
            zsum = 0.f;
            tc::tc_fence_before();
            tc::named_bar(1, 128);
            return true;
        };
        bool ok = true;
        for (int i = 0; i < nc; ++i) {
            const int s = i % kRStages;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, g0 + i);
            if (!(ok = group_wait(leader, 1, bar(R_FULL + s), (i / kRStages) & 1, ws, abort_flag, 4104))) break;
            if (r.seq != run_seq) {
                if (run_seq >= 0) {
                    if (!(ok = flush(run_seq))) break;
                    if (leader) tc::mbar_arrive(bar(R_TFREE));
                }
                run_seq = r.seq;
                ++runs;
            }
            const uint32_t st = sbase + s * kRStage;
            if (r.n < kChunk) {  // rows past the sequence's end belong to the next one: zero them in v
                for (int x = f; x < (kChunk - r.n) * 16; x += 128) {
                    const int t = r.n + (x >> 4), c16 = x & 15;
                    tc::st_shared_v4(tc::sw128(st + 16384 + (uint32_t)(c16 >> 3) * 8192, t, c16 & 7), 0u, 0u, 0u, 0u);
                }
                tc::fence_proxy_async();
                tc::named_bar(1, 128);
            }
            if (leader) tc::mbar_arrive(bar(R_READY + s));  // the MMA may take the stage
            zsum += key_column_sum(st, f, r.n);
            tc::named_bar(1, 128);
            if (leader) tc::mbar_arrive(bar(R_EMPTY + s));
        }
        if (ok && run_seq >= 0) flush(run_seq);
    }
    __syncthreads();
    if (tid == 0) tc::mbar_wait(bar(R_FIN), 0);
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------- apply
// B operand [K^T V | z] (rows i, three 64-column SW128 boxes: columns
// 0..63, 64..127, and z in column 128 with zeros after it), a two-stage ring
// of q tiles, one o staging tile, the barriers: ~97 KB, and 256 TMEM columns
// with D = q [K^T V | z] (M = 64, N = 136: columns 0..127 the numerator, 128
// the normaliser q . z) single-buffered, so that two CTAs share an SM and
// one's epilogue overlaps the other's loads and MMAs.
constexpr int kAStages = 2;
constexpr uint32_t kAKVZ = 0, kAQ = 49152, kAO = kAQ + kAStages * 16384, kABarOff = kAO + 16384;
enum { A_FULL = 0, A_EMPTY = 3, A_MMAD = 6, A_EPID = 8, A_KVR = 10, A_FIN = 11, A_COUNT = 12 };
constexpr uint32_t kASmem = kABarOff + 128 + 1024;
constexpr int kAN = 136;
constexpr uint32_t kIdQ = tc::idesc_bf16(64, kAN, false, true);  // A = q (K-major), B = [K^T V | z] (MN-major)

__global__ void __launch_bounds__(kLvThreads, 2)
kv_apply_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o, int H,
                int group, char* __restrict__ ws, const float* __restrict__ kv, const float* __restrict__ z,
                int normalize, __nv_bfloat16* __restrict__ o) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sbase = raw + pad;
    char* const sptr = reinterpret_cast<char*>(smem_raw) + pad;
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;
    const int total = hdr->total_chunks, n_seqs = hdr->n_seqs;
    const int g0 = blockIdx.x * group, head = blockIdx.y;
    if (g0 >= total) return;
    const int nc = min(total, g0 + group) - g0;
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* chunk_off = reinterpret_cast<const int*>(ws + L.chunk_off);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) { return sbase + kABarOff + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + kABarOff + 96);

    if (tid == 0) {
        for (int b = 0; b < A_COUNT; ++b) tc::mbar_init(bar(b), 1);
        tc::fence_mbar_init();
        abort_flag[0] = 0;
        abort_flag[1] = hdr->wait_limit;
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_o);
    }
    __syncwarp();
    if (warp == 0) tc::tmem_alloc(sbase + kABarOff + 104, 256);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t*>(sptr + kABarOff + 104), 0);

    if (warp == 0) {
        // ---- TMA: q of each chunk into stage i % kAStages
        int issued = 0;
        if (lane == 0) {
            for (int i = 0; i < nc; ++i) {
                const int s = i % kAStages;
                if (i >= kAStages && !lv_wait(bar(A_EMPTY + s), ((i / kAStages) - 1) & 1, ws, abort_flag, 4200)) break;
                const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, g0 + i);
                const uint32_t st = sbase + kAQ + s * 16384;
                tc::mbar_arrive_expect_tx(bar(A_FULL + s), 16384);
                tc::tma_load_3d(st, &tm_q, 0, head, r.t0, bar(A_FULL + s));
                tc::tma_load_3d(st + 8192, &tm_q, 64, head, r.t0, bar(A_FULL + s));
                issued = i + 1;
            }
            if (*abort_flag)
                for (int i = max(0, issued - kAStages); i < issued; ++i)
                    tc::mbar_wait(bar(A_FULL + i % kAStages), (i / kAStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA: D[b] = q [K^T V | z] per chunk (b = chunk % 2)
        int run_seq = -1, runs = 0;
        for (int i = 0; i < nc; ++i) {
            const int s = i % kAStages, b = i & 1;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, g0 + i);
            if (r.seq != run_seq) {  // the workers load this sequence's K^T V first
                if (!warp_wait(bar(A_KVR), runs & 1, ws, abort_flag, 4201)) break;
                run_seq = r.seq;
                ++runs;
            }
            if (!warp_wait(bar(A_FULL + s), (i / kAStages) & 1, ws, abort_flag, 4202)) break;
            if (i >= 1 && !warp_wait(bar(A_EPID + ((i - 1) & 1)), ((i - 1) >> 1) & 1, ws, abort_flag, 4203)) break;
            tc::tc_fence_after();
            const uint32_t st = sbase + kAQ + s * 16384, d = tmem;
            tc::mma_ss_n<4>(d, tc::sdesc(st, 16, 1024), 2, tc::sdesc(sbase + kAKVZ, 16384, 1024), 128, kIdQ, false);
            tc::mma_ss_n<4>(d, tc::sdesc(st + 8192, 16, 1024), 2, tc::sdesc(sbase + kAKVZ + 64 * 128, 16384, 1024), 128,
                            kIdQ, true);
            tc::commit_e(bar(A_MMAD + b));
            tc::commit_e(bar(A_EMPTY + s));
        }
        tc::commit_e(bar(A_FIN));
        __syncwarp();
    } else if (warp >= 4) {
        // ---- workers: load [K^T V | z] per sequence; o = D / (q . z) (or D) per
        // chunk.  With M = 64, token t sits in TMEM lane 32 (t / 16) + t % 16: lanes
        // 0..15 of each worker warp (quadrant warp % 4) hold tokens 16 (warp % 4) ..
        const int f = tid - 128;
        const bool leader = f == 0;
        const int t = 16 * (warp & 3) + lane;  // this lane's token (lanes < 16)
        int run_seq = -1;
        for (int i = 0; i < nc; ++i) {
            const int b = i & 1;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, g0 + i);
            if (r.seq != run_seq) {
                // every MMA on the previous sequence's operand is done (its chunks' D were
                // waited for below); row f of [K^T V | z] in bf16
                const float* src = kv + (((size_t)r.seq * H + head) * kD + f) * kD;
                const float zf = z[((size_t)r.seq * H + head) * kD + f];
#pragma unroll 1
                for (int c16 = 0; c16 < 24; ++c16) {
                    uint32_t w[4] = {0u, 0u, 0u, 0u};
                    if (c16 < 16) {
                        const float4 a = *reinterpret_cast<const float4*>(src + 8 * c16);
                        const float4 e = *reinterpret_cast<const float4*>(src + 8 * c16 + 4);
                        w[0] = tc::pack_bf16(a.x, a.y);
                        w[1] = tc::pack_bf16(a.z, a.w);
                        w[2] = tc::pack_bf16(e.x, e.y);
                        w[3] = tc::pack_bf16(e.z, e.w);
                    } else if (c16 == 16) {
                        w[0] = tc::pack_bf16(zf, 0.f);
                    }
                    tc::st_shared_v4(tc::sw128(sbase + kAKVZ + (uint32_t)(c16 >> 3) * 16384, f, c16 & 7), w[0], w[1],
                                     w[2], w[3]);
                }
                tc::fence_proxy_async();
                tc::named_bar(1, 128);
                if (leader) tc::mbar_arrive(bar(A_KVR));
                run_seq = r.seq;
            }
            if (!group_wait(leader, 1, bar(A_MMAD + b), (i >> 1) & 1, ws, abort_flag, 4204)) break;
            tc::tc_fence_after();
            const bool full = r.n == kChunk;
            const uint32_t ob = sbase + kAO;
            if (full) {  // the previous store is done reading the staging tile
                if (leader) tc::bulk_wait_read0();
                tc::named_bar(1, 128);
            }
            float e[16];
            tc::tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 128, e);
            tc::tmem_wait_ld();
            const float inv = normalize ? 1.f / e[0] : 1.f;
            // o in four parts of 32 columns, each staged (or stored) as soon as it is packed
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float d[32];
                tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * c, d);
                tc::tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) pk[x] = tc::pack_bf16(d[2 * x] * inv, d[2 * x + 1] * inv);
                if (full) {
                    if (lane < 16) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const int c16 = 4 * c + q4;
                            tc::st_shared_v4(tc::sw128(ob + (uint32_t)(c16 >> 3) * 8192, t, c16 & 7), pk[4 * q4],
                                             pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                        }
                    }
                } else if (lane < 16 && t < r.n) {  // the last, partial chunk of a sequence
                    uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(r.t0 + t) * H + head) * kD) + 4 * c;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        dst[q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                }
            }
            tc::fence_proxy_async();
            tc::tc_fence_before();
            tc::named_bar(1, 128);
            if (leader) {
                tc::mbar_arrive(bar(A_EPID + b));  // D may be overwritten
                if (full) {
                    tc::tma_store_3d(&tm_o, ob, 0, head, r.t0);
                    tc::tma_store_3d(&tm_o, ob + 8192, 64, head, r.t0);
                    tc::bulk_commit();
                }
            }
        }
        if (leader) tc::bulk_wait0();
    }
    __syncthreads();
    if (tid == 0) tc::mbar_wait(bar(A_FIN), 0);
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------- causal, grouped
// Causal linear attention without a per-chunk chain across the whole
// sequence: every sequence is cut into groups of chunks (the size is picked by
// the call's plan kernel); the groups' K^T V (kv_reduce_kernel<true>) give
// each group's starting state by a prefix (group_scan_kernel), and every group
// then runs its own chunks in order from that state (group_apply_kernel<false>),
// all groups side by side.  Small problems do all three in one cooperative
// launch (group_apply_kernel<true>).

// Per (sequence, head, 8 state columns): each group's starting state
// hs[g] = h0 + the K^T V of the sequence's earlier groups (fp32; group g's
// sum is the two halves Sg[2 g] + Sg[2 g + 1]), the final state h_T, and
// (slab 0) each group's starting key sum zs[g] and the sequence's total z_T.
// The groups go four at a time, every load of the four issued before the
// running sum takes them.
constexpr int kScanCols = 8, kScanBatch = 4;
__global__ void __launch_bounds__(kD)
group_scan_kernel(const char* __restrict__ ws, const int* __restrict__ group_off, int H,
                  const float* __restrict__ h0, const float* __restrict__ Sg, const float* __restrict__ zg,
                  float* __restrict__ hs, float* __restrict__ zs, float* __restrict__ h_T,
                  float* __restrict__ z_T) {
    if (reinterpret_cast<const WsHeader*>(ws)->status != GDN_OK) return;
    const int seq = blockIdx.x, head = blockIdx.y, j0 = kScanCols * blockIdx.z, i = threadIdx.x;
    const bool zslab = blockIdx.z == 0;
    auto row = [&](int slot) { return (((size_t)slot * H + head) * kD + i) * kD + j0; };
    float h[kScanCols];
#pragma unroll
    for (int x = 0; x < kScanCols; ++x) h[x] = h0 ? h0[row(seq) + x] : 0.f;
    float zacc = 0.f;
    const int gb = group_off[seq], ge = group_off[seq + 1];
    for (int g = gb; g < ge; g += kScanBatch) {
        float d[kScanBatch][kScanCols], dz[kScanBatch];
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
            const bool on = g + u < ge;
#pragma unroll
            for (int x = 0; x < kScanCols; x += 4) {
                float4 p = make_float4(0.f, 0.f, 0.f, 0.f), q = p;
                if (on) {
                    p = *reinterpret_cast<const float4*>(Sg + row(2 * (g + u)) + x);
                    q = *reinterpret_cast<const float4*>(Sg + row(2 * (g + u) + 1) + x);
                }
                d[u][x] = p.x + q.x;
                d[u][x + 1] = p.y + q.y;
                d[u][x + 2] = p.z + q.z;
                d[u][x + 3] = p.w + q.w;
            }
            dz[u] = (on && zslab) ? zg[((size_t)(2 * (g + u)) * H + head) * kD + i] +
                                        zg[((size_t)(2 * (g + u) + 1) * H + head) * kD + i]
                                  : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
            if (g + u >= ge) break;
            float* dst = hs + row(g + u);
#pragma unroll
            for (int x = 0; x < kScanCols; x += 4) {
                *reinterpret_cast<float4*>(dst + x) = make_float4(h[x], h[x + 1], h[x + 2], h[x + 3]);
#pragma unroll
                for (int e = 0; e < 4; ++e) h[x + e] += d[u][x + e];
            }
            if (zslab) {
                zs[((size_t)(g + u) * H + head) * kD + i] = zacc;
                zacc += dz[u];
            }
        }
    }
    if (h_T) {
#pragma unroll
        for (int x = 0; x < kScanCols; x += 4)
            *reinterpret_cast<float4*>(h_T + row(seq) + x) = make_float4(h[x], h[x + 1], h[x + 2], h[x + 3]);
    }
    if (z_T && zslab) z_T[((size_t)seq * H + head) * kD + i] = zacc;
}

// Group apply, CTA (g, head), 448 threads: warp 0 TMA, warp 1 MMA, and three
// 128-thread groups (warps 2..5 the state, 6..9 the P mask, 10..13 the
// output; warp w reads TMEM lanes 32 (w % 4) ..).  The state S = h^T (lane j
// = v feature, column i = k feature) accumulates in TMEM in fp32.  Per chunk:
//   P  = q k^T               (M = 64, N = 64; the P group masks s <= t, s < n
//                              and stores P in bf16)
//   S += v^T k               (M = 128, N = 128, fp32)
//   O  = q [h_c | z_c] + P [v | 1]   (M = 64 over tokens, N = 136, two TMEM buffers)
// where the state group copies S (the state at the chunk's start) to shared
// memory in bf16 before the chunk's S update, as a K-major [j][i] tile whose
// rows 128 and 129 hold the running key sum z_c split into a bf16 high and low
// part, and P times a fixed column of ones (O[t][128] += sum_s P[t][s]) adds the
// row sums of P.  So O[t][0..127] is the numerator and
// O[t][128] + O[t][129] the normaliser q_t . z_c + sum_{s <= t} q_t . k_s.  The
// output group divides (when normalised) and stores o.  Shared memory holds
// either (the one-launch form, whose small groups are bound by load latency) a
// three-stage ring for q, k, v with one state copy and one o staging tile (the
// next copy waits for the MMA that reads the current one) and the ones in a
// separate 64 x 8 tile (its own N = 8 MMA), or (the large problems of the
// separate-kernel form, bound by HBM) two stages, each with the ones as a third
// box after v (one N = 136 MMA), and the state copy and the staging tile
// double-buffered.  Token t of an M = 64 result sits in TMEM lane
// 32 (t / 16) + t % 16: lanes 0..15 of each warp of the P and output groups.
constexpr int kGThreads = 448;
constexpr uint32_t kGSnapBox = 17408;  // 136 rows x 128 B: one 64-column half of [h_c^T ; z_c]
template <bool ONE_LAUNCH>
struct GLayout {
    static constexpr int kStages = ONE_LAUNCH ? 3 : 2;
    static constexpr int kCopies = ONE_LAUNCH ? 1 : 2;  // state copies (two halves each)
    static constexpr int kOTiles = ONE_LAUNCH ? 1 : 2;  // o staging tiles
    static constexpr bool kOnesInStage = !ONE_LAUNCH;   // the ones as a third box after v in each stage
    // stage: q box0 | q box1 | k box0 | k box1 | v box0 | v box1 [| ones]
    static constexpr uint32_t kStage = kOnesInStage ? 57344 : 49152;
    static constexpr uint32_t kSnap = kStages * kStage;
    static constexpr uint32_t kP = kSnap + kCopies * 2 * kGSnapBox;  // P, bf16 [t][s]
    static constexpr uint32_t kOnes = kP + 8192;                     // [s][8], ones in column 0 (one SW128 box)
    static constexpr uint32_t kO = kOnes + (kOnesInStage ? 0 : 8192);  // o staging, [t][j], two boxes per tile
    static constexpr uint32_t kBarOff = kO + kOTiles * 16384;
    static constexpr uint32_t kSmem = kBarOff + 256 + 1024;
};
static_assert(GLayout<true>::kSmem <= 232448 && GLayout<false>::kSmem <= 232448, "group apply shared memory");
// barriers (room for three stages); G_SD: the state copy may be rewritten (S
// updated, and with one copy also read by the output MMA)
enum {
    G_FULL = 0, G_EMPTY = 3, G_ZREADY = 6, G_PD = 7, G_PREADY = 8, G_SNAP = 9, G_SD = 10, G_OD = 11, G_OFREE = 13,
    G_FIN = 15, G_COUNT = 16
};
constexpr uint32_t kGFlag = 128, kGSlot = 136;  // abort flag and bound; TMEM address (offsets from kBarOff)
static_assert(8 * G_COUNT <= kGFlag, "group apply barriers");
// TMEM columns: S fp32 0..127 (M = 128), P 128..191 (M = 64), O[0] 192..327, O[1] 352..487 (M = 64)
constexpr uint32_t kTS32 = 0, kTP = 128, kTO0 = 192, kTO1 = 352;
constexpr int kGN = 136;
constexpr uint32_t kGIdP = tc::idesc_bf16(64, 64, false, false);    // A = q, B = k (both K-major)
constexpr uint32_t kGIdS = tc::idesc_bf16(128, 128, true, true);    // A = v^T, B = k (both MN-major)
constexpr uint32_t kGIdQ = tc::idesc_bf16(64, kGN, false, false);   // A = q, B = [h_c^T ; z_c] (both K-major)
constexpr uint32_t kGIdV = tc::idesc_bf16(64, 128, false, true);   // A = P (K-major), B = v (MN-major)
constexpr uint32_t kGIdV1 = tc::idesc_bf16(64, kGN, false, true);   // A = P, B = [v | ones] (MN-major, three boxes)
constexpr uint32_t kGId1 = tc::idesc_bf16(64, 8, false, true);      // A = P (K-major), B = the ones tile (MN-major)

// Cross-CTA counters of the fused form (gpu scope).
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void add_release_gpu(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Bounded wait of one thread until *p >= target (the fused form's hand-offs
// between the CTAs of one (sequence, head); all of them are resident at once).
__device__ __noinline__ bool wait_count(const int* p, int target, char* ws, volatile int* abort_flag, int site) {
    const int limit = abort_flag[1];
    for (int it = 0;; ++it) {
        if (*abort_flag) return false;
        if (ld_acquire_gpu(p) >= target) return true;
        if (it >= limit) break;
        __nanosleep(128);
    }
    WsHeader* h = reinterpret_cast<WsHeader*>(ws);
    atomicExch(&h->status, GDN_ERR_TIMEOUT);
    atomicCAS(&h->timeout_site, 0, site);
    *abort_flag = 1;
    return false;
}

// FUSED = false: CTA (g, head) applies group g from hs[g], zs[g] (kv_reduce_kernel<true>
//   and group_scan_kernel ran before).
// FUSED = true: one cooperative launch of `sms` CTAs, CTA b taking group b / H of
//   head b % H, when every (sequence, head) has its groups resident at once.
//   Phase 1: the group's K^T V (in S) and key sums, published to Sg[g][head],
//   zg[g][head]; phase 2: once every group of the (sequence, head) has published,
//   CTA j of them forms the prefix over the groups for its slice of the 128 x 128
//   entries (hs, and h_T from the total; CTA 0 the key sums zs, z_T); phase 3:
//   once every slice is done, the apply as above, its loads already in flight
//   (the TMA warp streams the phase-1 k, v and then the phase-3 q, k, v through
//   the same ring).  Idle CTAs first copy h0 to h_T for empty sequences.
template <bool FUSED>
__global__ void __launch_bounds__(kGThreads, 1)
group_apply_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, int H,
                   char* __restrict__ ws, const int* __restrict__ group_off, float* __restrict__ hs,
                   float* __restrict__ zs, int normalize, __nv_bfloat16* __restrict__ o, int* __restrict__ counters,
                   float* __restrict__ Sg, float* __restrict__ zg, const float* __restrict__ h0,
                   float* __restrict__ h_T, float* __restrict__ z_T) {
    using GL = GLayout<FUSED>;
    constexpr int kGStages = GL::kStages;
    constexpr uint32_t kGStage = GL::kStage, kGSnap = GL::kSnap, kGP = GL::kP, kGOnes = GL::kOnes, kGO = GL::kO,
                       kGBarOff = GL::kBarOff;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sbase = raw + pad;
    char* const sptr = reinterpret_cast<char*>(smem_raw) + pad;
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;
    const int n_seqs = hdr->n_seqs;
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* chunk_off = reinterpret_cast<const int*>(ws + L.chunk_off);
    int head, g;
    if (FUSED) {
        // empty sequences have no group: their final state is h0, their key sum zero
        for (int u = blockIdx.x; u < n_seqs * H; u += gridDim.x) {
            const int sq = u / H;
            if (chunk_off[sq + 1] != chunk_off[sq]) continue;
            if (h_T)
                for (int x = threadIdx.x; x < kD * kD; x += blockDim.x)
                    h_T[(size_t)u * kD * kD + x] = h0 ? h0[(size_t)u * kD * kD + x] : 0.f;
            if (z_T && threadIdx.x < kD) z_T[(size_t)u * kD + threadIdx.x] = 0.f;
        }
        if ((int)blockIdx.x >= group_off[n_seqs] * H) return;
        head = blockIdx.x % H;
        g = blockIdx.x / H;
    } else {
        head = blockIdx.y;
        g = blockIdx.x;
        if (g >= group_off[n_seqs]) return;
    }
    int gseq, c0, nc;
    group_range(group_off, chunk_off, n_seqs, group_off[n_seqs + 1], g, gseq, c0, nc);
    if (nc == 0) return;
    const int n1 = FUSED ? nc : 0;  // phase-1 loads before the apply's
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) { return sbase + kGBarOff + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sptr + kGBarOff + kGFlag);
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane quadrant

    if (tid == 0) {
        for (int b = 0; b < G_COUNT; ++b) tc::mbar_init(bar(b), (b >= G_EMPTY && b < G_EMPTY + kGStages) ? 2 : 1);
        tc::fence_mbar_init();
        abort_flag[0] = 0;
        abort_flag[1] = hdr->wait_limit;
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
        tc::prefetch_tmap(&tm_o);
    }
    __syncwarp();
    if (warp == 0) tc::tmem_alloc(sbase + kGBarOff + kGSlot, 512);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t*>(sptr + kGBarOff + kGSlot), 0);

    if (warp == 0) {
        // ---- TMA: load l (phase-1 k, v for l < n1, then q, k, v of chunk l - n1) into stage l % kGStages
        int issued = 0;
        if (lane == 0) {
            for (int l = 0; l < n1 + nc; ++l) {
                const int s = l % kGStages;
                if (l >= kGStages && !lv_wait(bar(G_EMPTY + s), ((l / kGStages) - 1) & 1, ws, abort_flag, 4300)) break;
                const bool apply = l >= n1;
                const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, c0 + (apply ? l - n1 : l));
                const uint32_t st = sbase + s * kGStage;
                tc::mbar_arrive_expect_tx(bar(G_FULL + s), apply ? 49152 : 32768);
                if (apply) {
                    tc::tma_load_3d(st, &tm_q, 0, head, r.t0, bar(G_FULL + s));
                    tc::tma_load_3d(st + 8192, &tm_q, 64, head, r.t0, bar(G_FULL + s));
                }
                tc::tma_load_3d(st + 16384, &tm_k, 0, head, r.t0, bar(G_FULL + s));
                tc::tma_load_3d(st + 24576, &tm_k, 64, head, r.t0, bar(G_FULL + s));
                tc::tma_load_3d(st + 32768, &tm_v, 0, head, r.t0, bar(G_FULL + s));
                tc::tma_load_3d(st + 40960, &tm_v, 64, head, r.t0, bar(G_FULL + s));
                issued = l + 1;
            }
            if (*abort_flag)
                for (int l = max(0, issued - kGStages); l < issued; ++l)
                    tc::mbar_wait(bar(G_FULL + l % kGStages), (l / kGStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA
        int npart = 0;
        // phase 1: S = sum over the group's chunks of v^T k
        for (int l = 0; l < n1; ++l) {
            const int s = l % kGStages;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, c0 + l);
            const uint32_t st = sbase + s * kGStage, k0 = st + 16384, v0 = st + 32768;
            if (!warp_wait(bar(G_FULL + s), (l / kGStages) & 1, ws, abort_flag, 4310)) break;
            if (r.n < kChunk) {
                if (!warp_wait(bar(G_ZREADY), npart & 1, ws, abort_flag, 4311)) break;
                ++npart;
            }
            tc::tc_fence_after();
            tc::mma_ss_n<4>(tmem + kTS32, tc::sdesc(v0, 8192, 1024), 128, tc::sdesc(k0, 8192, 1024), 128, kGIdS, l > 0);
            tc::commit_e(bar(G_EMPTY + s));
        }
        if (FUSED) tc::commit_e(bar(G_SD));  // phase 1 done: the state group may read S (phase 0 of G_SD)
        // the apply, chunk by chunk
        for (int i = 0; i < nc; ++i) {
            const int l = n1 + i, s = l % kGStages, b = i & 1;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, c0 + i);
            const uint32_t st = sbase + s * kGStage, q0 = st, k0 = st + 16384, v0 = st + 32768;
            const uint32_t snap = sbase + kGSnap + (GL::kCopies == 2 ? 2 * kGSnapBox * (uint32_t)b : 0u);
            const uint32_t dO = tmem + (b ? kTO1 : kTO0);
            if (!warp_wait(bar(G_FULL + s), (l / kGStages) & 1, ws, abort_flag, 4301)) break;
            if (r.n < kChunk) {  // the state group first zeroes the rows past the sequence's end
                if (!warp_wait(bar(G_ZREADY), npart & 1, ws, abort_flag, 4302)) break;
                ++npart;
            }
            tc::tc_fence_after();
            // P = q k^T
            tc::mma_ss_n<4>(tmem + kTP, tc::sdesc(q0, 16, 1024), 2, tc::sdesc(k0, 16, 1024), 2, kGIdP, false);
            tc::mma_ss_n<4>(tmem + kTP, tc::sdesc(q0 + 8192, 16, 1024), 2, tc::sdesc(k0 + 8192, 16, 1024), 2, kGIdP,
                            true);
            tc::commit_e(bar(G_PD));
            // S += v^T k once the state at this chunk's start has been copied out
            if (!warp_wait(bar(G_SNAP), i & 1, ws, abort_flag, 4303)) break;
            tc::tc_fence_after();
            tc::mma_ss_n<4>(tmem + kTS32, tc::sdesc(v0, 8192, 1024), 128, tc::sdesc(k0, 8192, 1024), 128, kGIdS, true);
            if (GL::kCopies == 2) tc::commit_e(bar(G_SD));  // S updated; the other copy was read by chunk i - 1
            // O[b] = q [h_c | z_c] once chunk i - 2's O[b] has been read
            if (i >= 2 && !warp_wait(bar(G_OFREE + b), ((i >> 1) - 1) & 1, ws, abort_flag, 4304)) break;
            tc::tc_fence_after();
            tc::mma_ss_n<4>(dO, tc::sdesc(q0, 16, 1024), 2, tc::sdesc(snap, 16, 1024), 2, kGIdQ, false);
            tc::mma_ss_n<4>(dO, tc::sdesc(q0 + 8192, 16, 1024), 2, tc::sdesc(snap + kGSnapBox, 16, 1024), 2, kGIdQ,
                            true);
            if (GL::kCopies == 1) tc::commit_e(bar(G_SD));  // S updated and the one copy read
            // O[b] += P v, O[b][128..135] += P 1 once P is masked and stored
            if (!warp_wait(bar(G_PREADY), i & 1, ws, abort_flag, 4305)) break;
            tc::tc_fence_after();
            if (GL::kOnesInStage) {
                tc::mma_ss_n<4>(dO, tc::sdesc(sbase + kGP, 16, 1024), 2, tc::sdesc(v0, 8192, 1024), 128, kGIdV1, true);
            } else {
                tc::mma_ss_n<4>(dO, tc::sdesc(sbase + kGP, 16, 1024), 2, tc::sdesc(v0, 8192, 1024), 128, kGIdV, true);
                tc::mma_ss_n<4>(dO + 128, tc::sdesc(sbase + kGP, 16, 1024), 2, tc::sdesc(sbase + kGOnes, 8192, 1024),
                                128, kGId1, true);
            }
            tc::commit_e(bar(G_OD + b));
            tc::commit_e(bar(G_EMPTY + s));
        }
        tc::commit_e(bar(G_FIN));
        __syncwarp();
    } else if (warp < 6) {
        // ---- state group: thread f owns state row j = f (a TMEM lane) and key-sum entry z[f]
        const int f = 32 * (warp & 3) + lane;
        const bool leader = warp == 2 && lane == 0;
        const int sd0 = FUSED ? 1 : 0;  // G_SD phases taken before the apply's
        // row f of a snapshot half from 64 fp32 values (columns 64 half .. 64 half + 63)
        auto snap_half = [&](uint32_t snap, int half, const float (&x)[64]) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                tc::st_shared_v4(tc::sw128(snap + (uint32_t)half * kGSnapBox, f, c), tc::pack_bf16(x[8 * c], x[8 * c + 1]),
                                 tc::pack_bf16(x[8 * c + 2], x[8 * c + 3]), tc::pack_bf16(x[8 * c + 4], x[8 * c + 5]),
                                 tc::pack_bf16(x[8 * c + 6], x[8 * c + 7]));
        };
        // entry f of the key sum, high and low bf16 parts, into rows 128 and 129
        auto snap_z = [&](uint32_t snap, float zf) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(zf);
            const __nv_bfloat16 lo = __float2bfloat16_rn(zf - __bfloat162float(hi));
            const uint32_t box = snap + (uint32_t)(f >> 6) * kGSnapBox, c = (uint32_t)((f & 63) >> 3);
            const uint32_t e = (uint32_t)(f & 7) * 2;
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(tc::sw128(box, 128, c) + e), "h"(__bfloat16_as_ushort(hi)) : "memory");
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(tc::sw128(box, 129, c) + e), "h"(__bfloat16_as_ushort(lo)) : "memory");
        };
        // rows past a partial chunk's end belong to the next sequence: zero them in k and v
        auto zero_tail = [&](uint32_t st, int n) {
            for (int x = f; x < (kChunk - n) * 32; x += 128) {
                const int t = n + (x >> 5), c32 = x & 31;  // 16-byte chunk c32 of k (0..15) or v (16..31)
                const uint32_t base = st + 16384 + (c32 < 16 ? 0u : 16384u) + (uint32_t)((c32 & 15) >> 3) * 8192;
                tc::st_shared_v4(tc::sw128(base, t, c32 & 7), 0u, 0u, 0u, 0u);
            }
            tc::fence_proxy_async();
            tc::named_bar(1, 128);
            if (leader) tc::mbar_arrive(bar(G_ZREADY));
        };
        // fixed parts: the ones (row s: 1 in column 0, the first element of its logical
        // 16-byte chunk 0) in the ones tile or after v in every stage, rows 128..135 of
        // the state copies zero
        for (int x = f; x < (GL::kOnesInStage ? kGStages : 1) * 64 * 8; x += 128) {
            const int box = x >> 9, row = (x >> 3) & 63, c = x & 7;
            const uint32_t base = GL::kOnesInStage ? sbase + (uint32_t)box * kGStage + 49152 : sbase + kGOnes;
            tc::st_shared_v4(base + (uint32_t)row * 128 + (uint32_t)c * 16, c == (row & 7) ? 0x3F80u : 0u, 0u, 0u, 0u);
        }
        for (int x = f; x < GL::kCopies * 2 * 8 * 8; x += 128) {
            const int box = x >> 6, row = 128 + ((x >> 3) & 7), c = x & 7;
            tc::st_shared_v4(sbase + kGSnap + (uint32_t)box * kGSnapBox + (uint32_t)row * 128 + (uint32_t)c * 16, 0u,
                             0u, 0u, 0u);
        }
        bool ok = true;
        if (FUSED) {
            // ---- phase 1: the group's key sums (the MMA warp sums v^T k into S)
            const bool need_z = normalize || z_T != nullptr;
            float zred = 0.f;
            for (int l = 0; l < n1 && ok; ++l) {
                const int s = l % kGStages;
                const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, c0 + l);
                const uint32_t st = sbase + s * kGStage;
                if (!(ok = group_wait(leader, 1, bar(G_FULL + s), (l / kGStages) & 1, ws, abort_flag, 4312))) break;
                if (r.n < kChunk) zero_tail(st, r.n);
                if (need_z) zred += key_column_sum(st + 16384, f, r.n);
                tc::named_bar(1, 128);
                if (leader) tc::mbar_arrive(bar(G_EMPTY + s));
            }
            const int u = gseq * H + head, jg = g - group_off[gseq], ng = group_off[gseq + 1] - group_off[gseq];
            const size_t gb = (size_t)group_off[gseq];
            if (ok) ok = group_wait(leader, 1, bar(G_SD), 0, ws, abort_flag, 4313);
            if (ok) {
                // publish this group's sum (h layout [i][j]: row i, entry j = f) and key sums
                tc::tc_fence_after();
                float* dst = Sg + ((size_t)g * H + head) * kD * kD + f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float x[32];
                    tc::tmem_ld32(tmem + lane_off + kTS32 + 32 * c, x);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) dst[(size_t)(32 * c + e) * kD] = x[e];
                }
                zg[((size_t)g * H + head) * kD + f] = zred;
                __threadfence();
                tc::tc_fence_before();
                tc::named_bar(1, 128);
                if (leader) add_release_gpu(counters + u, 1);
                // ---- phase 2: once all groups of (sequence, head) published, this CTA's slice of the prefix
                bool got = true;
                if (leader) got = wait_count(counters + u, ng, ws, abort_flag, 4314);
                ok = tc::named_bar_and(1, 128, got);
            }
            if (ok) {
                const int per = ((kD * kD / ng) + 3) & ~3;
                const int e0 = min(kD * kD, jg * per), e1 = min(kD * kD, e0 + per);
                const size_t ub = (size_t)u * kD * kD;
                // two float4 positions per thread and four groups at a time, all eight loads
                // issued before the running sums take them (L2 loads: other CTAs of this
                // launch wrote Sg)
                const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
                auto add4 = [](float4& a, const float4& d) {
                    a.x += d.x;
                    a.y += d.y;
                    a.z += d.z;
                    a.w += d.w;
                };
                for (int e = e0 + 4 * f; e < e1; e += 2 * 4 * 128) {
                    const bool two = e + 4 * 128 < e1;
                    float4 a0 = h0 ? *reinterpret_cast<const float4*>(h0 + ub + e) : zero4;
                    float4 a1 = (h0 && two) ? *reinterpret_cast<const float4*>(h0 + ub + e + 512) : zero4;
                    for (int gg = 0; gg < ng; gg += 4) {
                        float4 d0[4], d1[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const bool on = gg + u < ng;
                            const size_t at = ((gb + gg + u) * H + head) * kD * kD + e;
                            d0[u] = on ? __ldcg(reinterpret_cast<const float4*>(Sg + at)) : zero4;
                            d1[u] = (on && two) ? __ldcg(reinterpret_cast<const float4*>(Sg + at + 512)) : zero4;
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (gg + u >= ng) break;
                            const size_t at = ((gb + gg + u) * H + head) * kD * kD + e;
                            *reinterpret_cast<float4*>(hs + at) = a0;
                            add4(a0, d0[u]);
                            if (two) {
                                *reinterpret_cast<float4*>(hs + at + 512) = a1;
                                add4(a1, d1[u]);
                            }
                        }
                    }
                    if (h_T) {
                        *reinterpret_cast<float4*>(h_T + ub + e) = a0;
                        if (two) *reinterpret_cast<float4*>(h_T + ub + e + 512) = a1;
                    }
                }
                if (jg == 0) {
                    float zacc = 0.f;
                    for (int gg = 0; gg < ng; ++gg) {
                        const size_t at = ((gb + gg) * H + head) * kD + f;
                        const float d = __ldcg(zg + at);
                        zs[at] = zacc;
                        zacc += d;
                    }
                    if (z_T) z_T[(size_t)u * kD + f] = zacc;
                }
                __threadfence();
                tc::named_bar(1, 128);
                if (leader) add_release_gpu(counters + n_seqs * H + u, 1);
                bool got = true;
                if (leader) got = wait_count(counters + n_seqs * H + u, ng, ws, abort_flag, 4315);
                ok = tc::named_bar_and(1, 128, got);
            }
        }
        if (ok) {  // S and the first snapshot from the group's starting state (h[i][j] -> S[j][i])
            float zf = 0.f;
            const float* hsrc = hs + ((size_t)g * H + head) * kD * kD;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float x[64];
#pragma unroll
                for (int i2 = 0; i2 < 64; ++i2) x[i2] = __ldcg(hsrc + (size_t)(64 * half + i2) * kD + f);
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    uint32_t r[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) r[e2] = __float_as_uint(x[16 * part + e2]);
                    tc::tmem_st16(tmem + lane_off + kTS32 + 64 * half + 16 * part, r);
                }
                snap_half(sbase + kGSnap, half, x);
            }
            tc::tmem_wait_st();
            tc::named_bar(1, 128);  // rows 128..135 were zeroed by other threads: the z rows come after
            if (normalize) {
                zf = __ldcg(zs + ((size_t)g * H + head) * kD + f);
                snap_z(sbase + kGSnap, zf);
            }
            tc::fence_proxy_async();
            tc::tc_fence_before();
            tc::named_bar(1, 128);
            if (leader) tc::mbar_arrive(bar(G_SNAP));
            for (int i = 0; i < nc; ++i) {
                const int l = n1 + i, s = l % kGStages;
                const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, c0 + i);
                const uint32_t st = sbase + s * kGStage, k0 = st + 16384;
                if (!group_wait(leader, 1, bar(G_FULL + s), (l / kGStages) & 1, ws, abort_flag, 4306)) break;
                if (r.n < kChunk) zero_tail(st, r.n);
                const float zc = normalize ? key_column_sum(k0, f, r.n) : 0.f;
                if (i + 1 < nc) {
                    // the state after this chunk, for the next one
                    if (!group_wait(leader, 1, bar(G_SD), (sd0 + i) & 1, ws, abort_flag, 4307)) break;
                    tc::tc_fence_after();
                    const uint32_t snap = sbase + kGSnap + (GL::kCopies == 2 ? 2 * kGSnapBox * (uint32_t)((i + 1) & 1) : 0u);
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        float x[64], y[32];
                        tc::tmem_ld32(tmem + lane_off + kTS32 + 64 * half, y);
                        tc::tmem_ld32(tmem + lane_off + kTS32 + 64 * half + 32, *reinterpret_cast<float(*)[32]>(x + 32));
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e2 = 0; e2 < 32; ++e2) x[e2] = y[e2];
                        snap_half(snap, half, x);
                    }
                    if (normalize) {
                        zf += zc;
                        snap_z(snap, zf);
                    }
                    tc::fence_proxy_async();
                    tc::tc_fence_before();
                    tc::named_bar(1, 128);
                    if (leader) {
                        tc::mbar_arrive(bar(G_SNAP));
                        tc::mbar_arrive(bar(G_EMPTY + s));
                    }
                } else {
                    tc::named_bar(1, 128);
                    if (leader) tc::mbar_arrive(bar(G_EMPTY + s));
                }
            }
        }
    } else if (warp < 10) {
        // ---- P group: mask s <= t, s < n; bf16 tile for the P [v | 1] MMA
        const bool leader = warp == 6 && lane == 0;
        const int tP = 16 * (warp & 3) + lane;  // this lane's token (lanes < 16)
        for (int i = 0; i < nc; ++i) {
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, c0 + i);
            if (!group_wait(leader, 2, bar(G_PD), i & 1, ws, abort_flag, 4308)) break;
            tc::tc_fence_after();
            float p[32], p2[32];
            tc::tmem_ld32(tmem + lane_off + kTP, p);
            tc::tmem_ld32(tmem + lane_off + kTP + 32, p2);
            tc::tmem_wait_ld();
            if (lane < 16) {
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    float w[8];
#pragma unroll
                    for (int e2 = 0; e2 < 8; ++e2) {
                        const int sc = 8 * c8 + e2;
                        const float pv = c8 < 4 ? p[sc] : p2[sc - 32];
                        w[e2] = (sc <= tP && sc < r.n) ? pv : 0.f;
                    }
                    tc::st_shared_v4(tc::sw128(sbase + kGP, tP, c8), tc::pack_bf16(w[0], w[1]), tc::pack_bf16(w[2], w[3]),
                                     tc::pack_bf16(w[4], w[5]), tc::pack_bf16(w[6], w[7]));
                }
            }
            tc::fence_proxy_async();
            tc::tc_fence_before();
            tc::named_bar(2, 128);
            if (leader) tc::mbar_arrive(bar(G_PREADY));
        }
    } else {
        // ---- output group: o = O / den, staged and stored with TMA (a partial chunk directly)
        const bool leader = warp == 10 && lane == 0;
        const int tP = 16 * (warp & 3) + lane;
        for (int i = 0; i < nc; ++i) {
            const int b = i & 1;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, c0 + i);
            const uint32_t tO = tmem + lane_off + (b ? kTO1 : kTO0);
            const uint32_t stage_o = sbase + kGO + (GL::kOTiles == 2 ? 16384u * (uint32_t)b : 0u);
            if (leader) {  // the store that last read this staging tile is done reading it
                if (GL::kOTiles == 2) tc::bulk_wait_read1();
                else tc::bulk_wait_read0();
            }
            if (!group_wait(leader, 3, bar(G_OD + b), (i >> 1) & 1, ws, abort_flag, 4309)) break;
            tc::tc_fence_after();
            float inv = 1.f;
            if (normalize) {
                float dz[16];
                tc::tmem_ld16(tO + 128, dz);
                tc::tmem_wait_ld();
                inv = 1.f / (dz[0] + dz[1]);
            }
            const bool full = r.n == kChunk;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float y[32], y2[32];
                tc::tmem_ld32(tO + 64 * half, y);
                tc::tmem_ld32(tO + 64 * half + 32, y2);
                tc::tmem_wait_ld();
                uint32_t pk[32];
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) {
                    pk[e2] = tc::pack_bf16(y[2 * e2] * inv, y[2 * e2 + 1] * inv);
                    pk[16 + e2] = tc::pack_bf16(y2[2 * e2] * inv, y2[2 * e2 + 1] * inv);
                }
                if (full) {
                    if (lane < 16) {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            tc::st_shared_v4(tc::sw128(stage_o + (uint32_t)half * 8192, tP, c), pk[4 * c], pk[4 * c + 1],
                                             pk[4 * c + 2], pk[4 * c + 3]);
                    }
                } else if (lane < 16 && tP < r.n) {  // the last, partial chunk of a sequence
                    uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(r.t0 + tP) * H + head) * kD + 64 * half);
#pragma unroll
                    for (int c = 0; c < 8; ++c) dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                }
            }
            tc::fence_proxy_async();
            tc::tc_fence_before();
            tc::named_bar(3, 128);
            if (leader) {
                tc::mbar_arrive(bar(G_OFREE + b));
                if (full) {
                    tc::tma_store_3d(&tm_o, stage_o, 0, head, r.t0);
                    tc::tma_store_3d(&tm_o, stage_o + 8192, 64, head, r.t0);
                    tc::bulk_commit();
                }
            }
        }
        if (leader) tc::bulk_wait0();
    }
    __syncthreads();
    if (tid == 0) tc::mbar_wait(bar(G_FIN), 0);
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace linvar

// ---------------------------------------------------------------- host side
bool linear_variant_shape_ok(const PrefillArgs& a) { return a.io == GDN_BF16 && a.dk == 128 && a.dv == 128; }

size_t linear_variant_extra_bytes(int64_t T, int H, int n_seqs, bool causal) {
    const size_t nch = (size_t)max_chunks(T, n_seqs);
    (void)nch;
    if (causal) return linear_grouped_extra_bytes(T, H, n_seqs);
    return align256(sizeof(float) * (size_t)n_seqs * H * linvar::kD * linvar::kD) +
           align256(sizeof(float) * (size_t)n_seqs * H * linvar::kD);  // K^T V, summed keys
}

cudaError_t launch_linear_bidirectional(const PrefillArgs& a, char* plan_ws, char* extra, bool normalize,
                                        float* kv_out, float* z_out, cudaStream_t st) {
    using namespace linvar;
    float* kv = reinterpret_cast<float*>(extra);
    float* z = reinterpret_cast<float*>(extra + align256(sizeof(float) * (size_t)a.n_seqs * a.H * kD * kD));
    const size_t kv_bytes = sizeof(float) * (size_t)a.n_seqs * a.H * kD * kD;
    const size_t z_bytes = sizeof(float) * (size_t)a.n_seqs * a.H * kD;
    cudaError_t e = cudaMemsetAsync(kv, 0, kv_bytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(z, 0, z_bytes, st);
    // chunks per CTA: at least kMinGroup, and few enough CTAs per head that all of
    // them fit one wave of two CTAs per SM when that is possible (a partly filled
    // second wave would leave most SMs idle while it runs)
    const long long nch = max_chunks(a.T_total, a.n_seqs);
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    const long long per_head = max(1LL, (2 * sms) / a.H);
    const int group = (int)max((long long)kMinGroup, (nch + per_head - 1) / per_head);
    const unsigned groups = (unsigned)((nch + group - 1) / group);
    if (e == cudaSuccess && groups > 0 && a.T_total > 0) {
        CUtensorMap mq, mk, mv, mo;
        if (!encode_token_map(&mq, a.q, a.T_total, a.H) || !encode_token_map(&mk, a.k, a.T_total, a.H) ||
            !encode_token_map(&mv, a.v, a.T_total, a.H) || !encode_token_map(&mo, a.o, a.T_total, a.H))
            return cudaErrorInvalidValue;
        e = cudaFuncSetAttribute(kv_reduce_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmem);
        if (e == cudaSuccess) {
            kv_reduce_kernel<false><<<dim3(groups, a.H), kLvThreads, kRSmem, st>>>(mk, mv, a.H, group, plan_ws,
                                                                                   nullptr, kv, z);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kv_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem);
        if (e == cudaSuccess) {
            kv_apply_kernel<<<dim3(groups, a.H), kLvThreads, kASmem, st>>>(mq, mo, a.H, group, plan_ws, kv, z,
                                                                           normalize ? 1 : 0, (__nv_bfloat16*)a.o);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess && kv_out) e = cudaMemcpyAsync(kv_out, kv, kv_bytes, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && z_out) e = cudaMemcpyAsync(z_out, z, z_bytes, cudaMemcpyDeviceToDevice, st);
    return e;
}

// Groups of the causal path: the plan kernel picks the size on the device,
// with at most floor(sms / H) + n_seqs groups in all.
static long long max_groups(int H, int n_seqs) {
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    return sms / (H > 0 ? H : 1) + n_seqs;
}

// The one-launch form needs every group resident at once: true when even one
// group per (sequence, head) fits the SMs, which the group size search then
// guarantees for all of them.  It pays for small problems (measured on B300:
// ahead up to ~30 chunks of 64 tokens per SM and head, behind from ~55, where
// the separate sum kernel's two CTAs per SM win), so it is taken up to 40.
// GDN_LINEAR_GROUPED_FORM=fused or =unfused overrides the size rule (fused
// still only where it can run).
static bool grouped_fused(const PrefillArgs& a) {
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    if (a.T_total <= 0 || (long long)a.H * a.n_seqs > sms) return false;
    const char* f = getenv("GDN_LINEAR_GROUPED_FORM");
    if (f != nullptr && strcmp(f, "fused") == 0) return true;
    if (f != nullptr && strcmp(f, "unfused") == 0) return false;
    return (long long)max_chunks(a.T_total, a.n_seqs) * a.H <= 40 * sms;
}

size_t linear_grouped_extra_bytes(int64_t T, int H, int n_seqs) {
    (void)T;
    const size_t ng = (size_t)max_groups(H, n_seqs);
    // group_off, the half-group sums Sg (2 per group), the starting states hs,
    // the half-group key sums zg (2 per group), the starting key sums zs, the
    // fused form's two counters per (sequence, head)
    return align256(sizeof(int) * (size_t)(n_seqs + 2)) + align256(sizeof(float) * 2 * ng * H * linvar::kD * linvar::kD) +
           align256(sizeof(float) * ng * H * linvar::kD * linvar::kD) + align256(sizeof(float) * 2 * ng * H * linvar::kD) +
           align256(sizeof(float) * ng * H * linvar::kD) + align256(sizeof(int) * 2 * (size_t)n_seqs * H);
}

cudaError_t launch_linear_grouped(const PrefillArgs& a, char* plan_ws, char* extra, bool normalize, float* h_T,
                                  float* z_T, int wait_limit, cudaStream_t st) {
    using namespace linvar;
    const size_t ng = (size_t)max_groups(a.H, a.n_seqs);
    const int sms = sm_count() > 0 ? sm_count() : 148;
    int* group_off = reinterpret_cast<int*>(extra);
    char* p = extra + align256(sizeof(int) * (size_t)(a.n_seqs + 2));
    float* Sg = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * 2 * ng * a.H * kD * kD);
    float* hs = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * ng * a.H * kD * kD);
    float* zg = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * 2 * ng * a.H * kD);
    float* zs = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * ng * a.H * kD);
    int* counters = reinterpret_cast<int*>(p);
    const bool fused = grouped_fused(a);
    const GroupPlan gp{sms, a.H, group_off, counters, fused ? 2 * a.n_seqs * a.H : 0};
    cudaError_t e = launch_plan(a.cu_seqlens, a.n_seqs, a.T_total, wait_limit, plan_ws, st, nullptr, &gp);
    if (e != cudaSuccess || a.n_seqs == 0) return e;
    if (a.T_total > 0) {
        CUtensorMap mq, mk, mv, mo;
        if (!encode_token_map(&mq, a.q, a.T_total, a.H) || !encode_token_map(&mk, a.k, a.T_total, a.H) ||
            !encode_token_map(&mv, a.v, a.T_total, a.H) || !encode_token_map(&mo, a.o, a.T_total, a.H))
            return cudaErrorInvalidValue;
        __nv_bfloat16* o = (__nv_bfloat16*)a.o;
        const int nrm = normalize ? 1 : 0;
        if (fused) {
            e = cudaFuncSetAttribute(group_apply_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)GLayout<true>::kSmem);
            if (e != cudaSuccess) return e;
            int H = a.H;
            char* ws = plan_ws;
            const float* h0 = a.h0;
            void* args[] = {&mq, &mk, &mv, &mo, &H, &ws, &group_off, &hs, &zs, (void*)&nrm, &o, &counters, &Sg, &zg,
                            (void*)&h0, &h_T, &z_T};
            e = cudaLaunchCooperativeKernel((const void*)group_apply_kernel<true>, dim3((unsigned)sms),
                                            dim3(kGThreads), args, GLayout<true>::kSmem, st);
            if (e != cudaErrorCooperativeLaunchTooLarge && e != cudaErrorNotSupported) return e;
            // cooperative launches refused here (e.g. a shared device): the same groups
            // through the separate kernels below
            (void)cudaGetLastError();
        }
        e = cudaFuncSetAttribute(kv_reduce_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmem);
        if (e != cudaSuccess) return e;
        kv_reduce_kernel<true><<<dim3((unsigned)(2 * ng), a.H), kLvThreads, kRSmem, st>>>(mk, mv, a.H, 0, plan_ws,
                                                                                         group_off, Sg, zg);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        group_scan_kernel<<<dim3((unsigned)a.n_seqs, a.H, kD / kScanCols), kD, 0, st>>>(plan_ws, group_off, a.H, a.h0,
                                                                                       Sg, zg, hs, zs, h_T, z_T);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        e = cudaFuncSetAttribute(group_apply_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)GLayout<false>::kSmem);
        if (e != cudaSuccess) return e;
        group_apply_kernel<false><<<dim3((unsigned)ng, a.H), kGThreads, GLayout<false>::kSmem, st>>>(
            mq, mk, mv, mo, a.H, plan_ws, group_off, hs, zs, nrm, o, nullptr, nullptr, nullptr, nullptr, nullptr,
            nullptr);
        return cudaGetLastError();
    }
    // no tokens: every final state is its initial state, every key sum zero
    group_scan_kernel<<<dim3((unsigned)a.n_seqs, a.H, kD / kScanCols), kD, 0, st>>>(plan_ws, group_off, a.H, a.h0, Sg,
                                                                                   zg, hs, zs, h_T, z_T);
    return cudaGetLastError();
}

}  // namespace gdn
