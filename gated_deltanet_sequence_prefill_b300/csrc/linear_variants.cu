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
// Causal normalised: the numerator is the causal linear attention of the
// library's prefill; the normaliser q_t . (sum of k_s, s <= t) comes from
// per-chunk key sums, their prefix over the chunks of each sequence, and a
// per-chunk pass that divides o.
#include <cuda_runtime.h>

#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"

namespace gdn {

int sm_count();
bool encode_token_map(CUtensorMap* m, const void* ptr, int64_t T, int H);

namespace linvar {

constexpr int kD = 128;
constexpr int kThreads = 128;  // the causal normaliser's kernels
constexpr int kMinGroup = 4;   // chunks per reduce / apply CTA, at least

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
// (and the site) in the status word and sets the CTA's abort flag; every role
// reads the flag after its group synchronises, so each group stops together.
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

__global__ void __launch_bounds__(kLvThreads, 1)
kv_reduce_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, int H,
                 int group, char* __restrict__ ws, float* __restrict__ kv, float* __restrict__ z) {
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
        bool fresh = true;
        for (int i = 0; i < nc; ++i) {
            const int s = i % kRStages;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, g0 + i);
            if (r.seq != run_seq) {
                if (run_seq >= 0) {
                    tc::commit_e(bar(R_RUNDONE));  // the run's MMAs are done: the workers may read D
                    if (lane == 0) lv_wait(bar(R_TFREE), (runs - 1) & 1, ws, abort_flag, 4101);
                    __syncwarp();
                    if (*abort_flag) break;
                }
                run_seq = r.seq;
                ++runs;
                fresh = true;
            }
            if (lane == 0) lv_wait(bar(R_READY + s), (i / kRStages) & 1, ws, abort_flag, 4102);
            __syncwarp();
            if (*abort_flag) break;
            tc::tc_fence_after();
            const uint32_t st = sbase + s * kRStage;
            tc::mma_ss_n<4>(tmem, tc::sdesc(st, 8192, 1024), 128, tc::sdesc(st + 16384, 8192, 1024), 128, kIdKV, !fresh);
            tc::commit_e(bar(R_EMPTY + s));
            fresh = false;
        }
        if (!*abort_flag && run_seq >= 0) tc::commit_e(bar(R_RUNDONE));
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
            if (leader) lv_wait(bar(R_RUNDONE), (runs - 1) & 1, ws, abort_flag, 4103);
            tc::named_bar(1, 128);
            if (*abort_flag) return false;
            tc::tc_fence_after();
            float* dst = kv + (((size_t)seq * H + head) * kD + f) * kD;
            float d[32];
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * c, d);
                tc::tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 32; ++x) atomicAdd(dst + 32 * c + x, d[x]);
            }
            atomicAdd(z + ((size_t)seq * H + head) * kD + f, zsum);
            zsum = 0.f;
            tc::tc_fence_before();
            tc::named_bar(1, 128);
            return true;
        };
        const uint32_t kcol = (uint32_t)(f >> 6) * 8192 + (uint32_t)((f & 7) * 2);
        const uint32_t kchunk = (uint32_t)((f & 63) >> 3);
        for (int i = 0; i < nc; ++i) {
            const int s = i % kRStages;
            const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, g0 + i);
            if (leader) lv_wait(bar(R_FULL + s), (i / kRStages) & 1, ws, abort_flag, 4104);
            tc::named_bar(1, 128);
            if (*abort_flag) break;
            if (r.seq != run_seq) {
                if (run_seq >= 0) {
                    if (!flush(run_seq)) break;
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
            }
            float acc = 0.f;
            for (int t = 0; t < r.n; ++t) {
                uint16_t h;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h)
                             : "r"(st + kcol + (uint32_t)t * 128 + (((kchunk ^ (uint32_t)t) & 7u) << 4)));
                acc += __bfloat162float(__ushort_as_bfloat16(h));
            }
            zsum += acc;
            tc::named_bar(1, 128);
            if (leader) {
                tc::mbar_arrive(bar(R_READY + s));
                tc::mbar_arrive(bar(R_EMPTY + s));
            }
        }
        if (!*abort_flag && run_seq >= 0) flush(run_seq);
    }
    __syncthreads();
    if (tid == 0) tc::mbar_wait(bar(R_FIN), 0);
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------- apply
// B operand [K^T V | z] (rows i, three 64-column SW128 boxes: columns
// 0..63, 64..127, and z in column 128 with zeros after it), a ring of q
// tiles, two o staging tiles, the barriers.  D = q [K^T V | z] (M = 64,
// N = 136) in one of two TMEM buffers: columns 0..127 the numerator, 128
// the normaliser q . z.
constexpr int kAStages = 3;
constexpr uint32_t kAKVZ = 0, kAQ = 49152, kAO = kAQ + kAStages * 16384, kABarOff = kAO + 2 * 16384;
enum { A_FULL = 0, A_EMPTY = 3, A_MMAD = 6, A_EPID = 8, A_KVR = 10, A_FIN = 11, A_COUNT = 12 };
constexpr uint32_t kASmem = kABarOff + 128 + 1024;
constexpr int kAN = 136;
constexpr uint32_t kIdQ = tc::idesc_bf16(64, kAN, false, true);  // A = q (K-major), B = [K^T V | z] (MN-major)

__global__ void __launch_bounds__(kLvThreads, 1)
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
    if (warp == 0) tc::tmem_alloc(sbase + kABarOff + 104, 512);
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
                if (lane == 0) lv_wait(bar(A_KVR), runs & 1, ws, abort_flag, 4201);
                run_seq = r.seq;
                ++runs;
            }
            if (lane == 0) {
                lv_wait(bar(A_FULL + s), (i / kAStages) & 1, ws, abort_flag, 4202);
                if (i >= 2) lv_wait(bar(A_EPID + b), ((i >> 1) - 1) & 1, ws, abort_flag, 4203);
            }
            __syncwarp();
            if (*abort_flag) break;
            tc::tc_fence_after();
            const uint32_t st = sbase + kAQ + s * 16384, d = tmem + 256u * b;
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
            if (leader) lv_wait(bar(A_MMAD + b), (i >> 1) & 1, ws, abort_flag, 4204);
            tc::named_bar(1, 128);
            if (*abort_flag) break;
            tc::tc_fence_after();
            float d[32], e[16];
            uint32_t pk[64];
            tc::tmem_ld16(tmem + 256u * b + ((uint32_t)(32 * (warp & 3)) << 16) + 128, e);
            tc::tmem_wait_ld();
            const float inv = normalize ? 1.f / e[0] : 1.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                tc::tmem_ld32(tmem + 256u * b + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * c, d);
                tc::tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 16; ++x) pk[16 * c + x] = tc::pack_bf16(d[2 * x] * inv, d[2 * x + 1] * inv);
            }
            tc::tc_fence_before();
            tc::named_bar(1, 128);
            if (leader) tc::mbar_arrive(bar(A_EPID + b));  // D[b] may be overwritten
            if (r.n == kChunk) {
                // stage o in SW128 boxes and store it with the tensor map
                const uint32_t ob = sbase + kAO + (uint32_t)b * 16384;
                if (leader) tc::bulk_wait_read0();  // earlier stores are done reading the staging tiles
                tc::named_bar(1, 128);
                if (lane < 16) {
#pragma unroll
                    for (int c16 = 0; c16 < 16; ++c16)
                        tc::st_shared_v4(tc::sw128(ob + (uint32_t)(c16 >> 3) * 8192, t, c16 & 7), pk[4 * c16],
                                         pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
                }
                tc::fence_proxy_async();
                tc::named_bar(1, 128);
                if (leader) {
                    tc::tma_store_3d(&tm_o, ob, 0, head, r.t0);
                    tc::tma_store_3d(&tm_o, ob + 8192, 64, head, r.t0);
                    tc::bulk_commit();
                }
            } else if (lane < 16 && t < r.n) {  // the last, partial chunk of a sequence
                uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(r.t0 + t) * H + head) * kD);
#pragma unroll
                for (int c16 = 0; c16 < 16; ++c16)
                    dst[c16] = make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
            }
        }
        if (leader) tc::bulk_wait0();
    }
    __syncthreads();
    if (tid == 0) tc::mbar_wait(bar(A_FIN), 0);
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- causal normaliser
// Sum of the keys of each chunk.
__global__ void __launch_bounds__(kThreads)
chunk_key_sum_kernel(const __nv_bfloat16* __restrict__ k, int H, const char* __restrict__ ws,
                     float* __restrict__ ks) {
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK || (int)blockIdx.x >= hdr->total_chunks) return;
    PlanLayout L(hdr->n_seqs);
    const ChunkRef r = chunk_ref(reinterpret_cast<const int*>(ws + L.cu),
                                 reinterpret_cast<const int*>(ws + L.chunk_off), hdr->n_seqs, blockIdx.x);
    const int i = threadIdx.x, head = blockIdx.y;
    float s = 0.f;
    for (int t = 0; t < r.n; ++t) s += __bfloat162float(k[((size_t)(r.t0 + t) * H + head) * kD + i]);
    ks[((size_t)blockIdx.x * H + head) * kD + i] = s;
}

// Exclusive prefix of the chunk key sums over each sequence's chunks, and the
// sequence's total (the summed keys z, when asked for).  One block per
// (sequence, head, 16 features): each of its 256 threads takes a contiguous
// run of the sequence's chunks for those 16 features, the runs' totals are
// scanned in shared memory, and each thread then writes its run's prefixes.
constexpr int kPrefixThreads = 256, kPrefixFeat = 16;
__global__ void __launch_bounds__(kPrefixThreads)
key_prefix_kernel(int H, const char* __restrict__ ws, const float* __restrict__ ks,
                  float* __restrict__ zstart, float* __restrict__ z) {
    __shared__ float part[kPrefixThreads][kPrefixFeat + 1];
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;
    PlanLayout L(hdr->n_seqs);
    const int* chunk_off = reinterpret_cast<const int*>(ws + L.chunk_off);
    const int seq = blockIdx.x, head = blockIdx.y, f0 = blockIdx.z * kPrefixFeat, tid = threadIdx.x;
    const int c0 = chunk_off[seq], nch = chunk_off[seq + 1] - c0;
    const int per = (nch + kPrefixThreads - 1) / kPrefixThreads;
    const int a = c0 + min(nch, tid * per), e = c0 + min(nch, (tid + 1) * per);
    float run[kPrefixFeat];
#pragma unroll
    for (int x = 0; x < kPrefixFeat; ++x) run[x] = 0.f;
    for (int c = a; c < e; ++c) {
        const float* src = ks + ((size_t)c * H + head) * kD + f0;
#pragma unroll
        for (int x = 0; x < kPrefixFeat; ++x) run[x] += src[x];
    }
#pragma unroll
    for (int x = 0; x < kPrefixFeat; ++x) part[tid][x] = run[x];
    __syncthreads();
    // inclusive scan of the runs' totals, per feature (Hillis-Steele over 256 entries)
    for (int off = 1; off < kPrefixThreads; off <<= 1) {
        float add[kPrefixFeat];
#pragma unroll
        for (int x = 0; x < kPrefixFeat; ++x) add[x] = tid >= off ? part[tid - off][x] : 0.f;
        __syncthreads();
#pragma unroll
        for (int x = 0; x < kPrefixFeat; ++x) part[tid][x] += add[x];
        __syncthreads();
    }
#pragma unroll
    for (int x = 0; x < kPrefixFeat; ++x) run[x] = tid > 0 ? part[tid - 1][x] : 0.f;  // before this run
    for (int c = a; c < e; ++c) {
        const size_t at = ((size_t)c * H + head) * kD + f0;
#pragma unroll
        for (int x = 0; x < kPrefixFeat; ++x) {
            zstart[at + x] = run[x];
            run[x] += ks[at + x];
        }
    }
    if (z && tid == kPrefixThreads - 1) {
#pragma unroll
        for (int x = 0; x < kPrefixFeat; ++x) z[((size_t)seq * H + head) * kD + f0 + x] = part[tid][x];
    }
}

// o_t /= q_t . (z_start + sum of k_s over s <= t in the chunk), per chunk.
__global__ void __launch_bounds__(kThreads)
causal_normalise_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int H,
                        const char* __restrict__ ws, const float* __restrict__ zstart,
                        __nv_bfloat16* __restrict__ o) {
    __shared__ float part[kChunk][kD + 1];
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK || (int)blockIdx.x >= hdr->total_chunks) return;
    PlanLayout L(hdr->n_seqs);
    const ChunkRef r = chunk_ref(reinterpret_cast<const int*>(ws + L.cu),
                                 reinterpret_cast<const int*>(ws + L.chunk_off), hdr->n_seqs, blockIdx.x);
    const int i = threadIdx.x, head = blockIdx.y;
    float zi = zstart[((size_t)blockIdx.x * H + head) * kD + i];
    for (int t = 0; t < r.n; ++t) {
        const size_t row = ((size_t)(r.t0 + t) * H + head) * kD;
        zi += __bfloat162float(k[row + i]);
        part[t][i] = __bfloat162float(q[row + i]) * zi;
    }
    __syncthreads();
    // two threads per token: features 0..63 and 64..127
    const int t = i >> 1, half = i & 1;
    float den = 0.f;
    if (t < r.n)
        for (int x = 0; x < 64; ++x) den += part[t][64 * half + x];
    den += __shfl_xor_sync(0xffffffffu, den, 1);
    if (t < r.n) {
        __nv_bfloat16* row = o + ((size_t)(r.t0 + t) * H + head) * kD + 64 * half;
        const float inv = 1.f / den;
        for (int x = 0; x < 64; x += 8) {
            uint4 w = *reinterpret_cast<uint4*>(row + x);
            uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const float2 f = tc::unpack_bf16(u[y]);
                u[y] = tc::pack_bf16(f.x * inv, f.y * inv);
            }
            *reinterpret_cast<uint4*>(row + x) = make_uint4(u[0], u[1], u[2], u[3]);
        }
    }
}

}  // namespace linvar

// ---------------------------------------------------------------- host side
bool linear_variant_shape_ok(const PrefillArgs& a) { return a.io == GDN_BF16 && a.dk == 128 && a.dv == 128; }

size_t linear_variant_extra_bytes(int64_t T, int H, int n_seqs, bool causal) {
    const size_t nch = (size_t)max_chunks(T, n_seqs);
    if (causal) return 2 * align256(sizeof(float) * nch * H * linvar::kD);  // chunk key sums, prefixes
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
    // chunks per CTA: about two CTAs per SM in all, at least kMinGroup chunks each,
    // so that each (sequence, head) gets few partial sums of K^T V to add up
    const long long nch = max_chunks(a.T_total, a.n_seqs);
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    const int group = (int)max((long long)kMinGroup, (nch * a.H + 2 * sms - 1) / (2 * sms));
    const unsigned groups = (unsigned)((nch + group - 1) / group);
    if (e == cudaSuccess && groups > 0 && a.T_total > 0) {
        CUtensorMap mq, mk, mv, mo;
        if (!encode_token_map(&mq, a.q, a.T_total, a.H) || !encode_token_map(&mk, a.k, a.T_total, a.H) ||
            !encode_token_map(&mv, a.v, a.T_total, a.H) || !encode_token_map(&mo, a.o, a.T_total, a.H))
            return cudaErrorInvalidValue;
        e = cudaFuncSetAttribute(kv_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmem);
        if (e == cudaSuccess) {
            kv_reduce_kernel<<<dim3(groups, a.H), kLvThreads, kRSmem, st>>>(mk, mv, a.H, group, plan_ws, kv, z);
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

cudaError_t launch_linear_causal_normaliser(const PrefillArgs& a, char* plan_ws, char* extra, bool divide,
                                            float* z_out, cudaStream_t st) {
    using namespace linvar;
    const size_t nch = (size_t)max_chunks(a.T_total, a.n_seqs);
    if (nch == 0) return cudaSuccess;
    float* ks = reinterpret_cast<float*>(extra);
    float* zstart = reinterpret_cast<float*>(extra + align256(sizeof(float) * nch * a.H * kD));
    chunk_key_sum_kernel<<<dim3((unsigned)nch, a.H), kThreads, 0, st>>>((const __nv_bfloat16*)a.k, a.H, plan_ws, ks);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && a.n_seqs > 0) {
        key_prefix_kernel<<<dim3((unsigned)a.n_seqs, a.H, kD / kPrefixFeat), kPrefixThreads, 0, st>>>(
            a.H, plan_ws, ks, zstart, z_out);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && divide) {
        causal_normalise_kernel<<<dim3((unsigned)nch, a.H), kThreads, 0, st>>>(
            (const __nv_bfloat16*)a.q, (const __nv_bfloat16*)a.k, a.H, plan_ws, zstart, (__nv_bfloat16*)a.o);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace gdn
