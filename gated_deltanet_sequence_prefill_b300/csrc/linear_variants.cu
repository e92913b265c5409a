// linear_variants.cu -- linear attention with the causal mask optional and the
// normaliser optional (bf16, dk = dv = 128):
//     o_t = sum_s (q_t . k_s) v_s  [/ sum_s (q_t . k_s)],
// s over all tokens of the sequence (bidirectional) or s <= t (causal).
// The normalised, bidirectional form is the listing of "За пределами
// self-attention…" (section "Линейное внимание…"): K^T V and the summed keys
// first, then q times each; the bidirectional mode and the causal restriction
// are those of the ai-vestnik.ru item on linear attention.
//
// Bidirectional: kv_reduce_kernel forms K^T V (tcgen05, fp32 in TMEM) and the
// summed keys per sequence and head from groups of chunks, adding the partial
// sums of each group to the workspace; kv_apply_kernel then computes q (K^T V)
// (tcgen05, K^T V rounded once to bf16 as the B operand) and divides by
// q . z when normalised.
// Causal normalised: the numerator is the causal linear attention of the
// library's prefill; the normaliser q_t . (sum of k_s, s <= t) comes from
// per-chunk key sums, their prefix over the chunks of each sequence, and a
// per-chunk pass that divides o.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "tc_util.cuh"

namespace gdn {

int sm_count();

namespace linvar {

constexpr int kD = 128;
constexpr int kThreads = 128;
constexpr int kMinGroup = 8;  // chunks per reduce / apply CTA, at least

// 64 tokens x 128 features of one head, bf16, as two 64-column SW128 boxes
// (row t of box b holds features 64 b .. 64 b + 63): 16 KB.  Rows t >= n are
// zero.  Plain 16-byte loads, 128 threads.
__device__ __forceinline__ void load_rows(uint32_t sbase, uint32_t box_stride, const __nv_bfloat16* src,
                                          int t0, int n, int H, int head, int tid) {
#pragma unroll 2
    for (int x = tid; x < 64 * 16; x += kThreads) {
        const int t = x >> 4, c16 = x & 15;  // row, 16-byte chunk of the 256-byte row
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t < n) v = *reinterpret_cast<const uint4*>(src + ((size_t)(t0 + t) * H + head) * kD + c16 * 8);
        tc::st_shared_v4(tc::sw128(sbase + (uint32_t)(c16 >> 3) * box_stride, t, c16 & 7), v.x, v.y, v.z, v.w);
    }
}

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

// Bounded wait on an mbarrier phase; a wait that runs out records
// GDN_ERR_TIMEOUT in the status word (the kernel then stops issuing work).
// Every thread of the block polls; the callers combine the outcomes with
// __syncthreads_and so that the whole block takes the same branch.
__device__ __forceinline__ bool wait_or_fail(uint32_t bar, uint32_t parity, char* ws, int limit) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (tc::mbar_wait(bar, parity, limit)) return true;
    WsHeader* h = reinterpret_cast<WsHeader*>(ws);
    atomicExch(&h->status, GDN_ERR_TIMEOUT);
    atomicCAS(&h->timeout_site, 0, 4000);
    return false;
}

// ---------------------------------------------------------------- reduce
// smem: two buffers of [k (16 KB) | v (16 KB)], two mbarriers, TMEM slot
constexpr uint32_t kRBuf = 32768;
constexpr uint32_t kRBar = 2 * kRBuf;
constexpr uint32_t kRSmem = kRBar + 64 + 1024;
constexpr uint32_t kIdKV = tc::idesc_bf16(128, 128, true, true);  // A = k^T, B = v, both MN-major

__global__ void __launch_bounds__(kThreads, 1)
kv_reduce_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v, int H, int group,
                 char* __restrict__ ws, float* __restrict__ kv, float* __restrict__ z) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t sbase = raw + ((1024u - (raw & 1023u)) & 1023u);
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;
    const int total = hdr->total_chunks, n_seqs = hdr->n_seqs, limit = hdr->wait_limit;
    const int g0 = blockIdx.x * group, head = blockIdx.y;
    if (g0 >= total) return;
    const int g1 = min(total, g0 + group);
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* chunk_off = reinterpret_cast<const int*>(ws + L.chunk_off);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar0 = sbase + kRBar, tslot = sbase + kRBar + 16;

    if (tid == 0) {
        tc::mbar_init(bar0, 1);
        tc::mbar_init(bar0 + 8, 1);
        tc::fence_mbar_init();
    }
    __syncwarp();
    if (warp == 0) tc::tmem_alloc(tslot, 128);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem_raw + (sbase - raw) + kRBar + 16);

    // this thread's share of the summed keys: features 8 (tid % 16) .. + 7
    float zs[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) zs[x] = 0.f;
    uint32_t phase[2] = {0u, 0u};
    bool ok = true;
    int run_seq = -1;
    bool fresh = true;  // next MMA starts the accumulator
    int issued_on[2] = {0, 0};

    auto flush = [&](int seq) {
        // wait for every MMA of this run, then add D and the key sums to the sequence's totals
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
        float d[32];
        float* dst = kv + (((size_t)seq * H + head) * kD + (size_t)(32 * warp + lane)) * kD;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * c, d);
            tc::tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) atomicAdd(dst + 32 * c + x, d[x]);
        }
        float* zd = z + ((size_t)seq * H + head) * kD + 8 * (tid & 15);
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            atomicAdd(zd + x, zs[x]);
            zs[x] = 0.f;
        }
        tc::tc_fence_before();
        __syncthreads();
        tc::tc_fence_after();
    };

    for (int gc = g0; gc < g1 && ok; ++gc) {
        const int i = gc - g0, b = i & 1;
        const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, gc);
        if (r.seq != run_seq) {
            if (run_seq >= 0) {
                // the run's last MMAs: each buffer's latest commit
                for (int bb = 0; bb < 2 && ok; ++bb)
                    if (issued_on[bb]) {
                        ok = __syncthreads_and(wait_or_fail(bar0 + 8 * bb, phase[bb], ws, limit));
                        if (ok) {  // a commit that was not seen stays pending for the drain below
                            phase[bb] ^= 1u;
                            issued_on[bb] = 0;
                        }
                    }
                if (!ok) break;
                flush(run_seq);
            }
            run_seq = r.seq;
            fresh = true;
        }
        // buffer b is free once the MMAs that read it (two chunks ago) are done
        if (issued_on[b]) {
            ok = __syncthreads_and(wait_or_fail(bar0 + 8 * b, phase[b], ws, limit));
            if (!ok) break;
            phase[b] ^= 1u;
            issued_on[b] = 0;
        }
        const uint32_t kb = sbase + b * kRBuf, vb = kb + 16384;
        load_rows(kb, 8192, k, r.t0, r.n, H, head, tid);
        load_rows(vb, 8192, v, r.t0, r.n, H, head, tid);
        // key sums: this thread's 8 features over its rows (from global, already in L1/L2)
        for (int t = tid >> 4; t < r.n; t += kThreads / 16) {
            const uint4 kk = *reinterpret_cast<const uint4*>(k + ((size_t)(r.t0 + t) * H + head) * kD + 8 * (tid & 15));
            const uint32_t w[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float2 f = tc::unpack_bf16(w[x]);
                zs[2 * x] += f.x;
                zs[2 * x + 1] += f.y;
            }
        }
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc::tc_fence_after();
            tc::mma_ss_n<4>(tmem, tc::sdesc(kb, 8192, 1024), 128, tc::sdesc(vb, 8192, 1024), 128, kIdKV, !fresh);
            tc::commit_e(bar0 + 8 * b);
        }
        __syncwarp();
        issued_on[b] = 1;
        fresh = false;
    }
    if (ok && run_seq >= 0) {
        for (int bb = 0; bb < 2 && ok; ++bb)
            if (issued_on[bb]) {
                ok = __syncthreads_and(wait_or_fail(bar0 + 8 * bb, phase[bb], ws, limit));
                if (ok) {
                    phase[bb] ^= 1u;
                    issued_on[bb] = 0;
                }
            }
        if (ok) flush(run_seq);
    }
    // drain anything still in flight before TMEM is released (unbounded only
    // for MMAs that were issued: they complete on their own)
    for (int bb = 0; bb < 2; ++bb)
        if (issued_on[bb]) tc::mbar_wait(bar0 + 8 * bb, phase[bb]);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------- apply
// smem: K^T V as bf16 B operand (rows = feature i, two 64-column boxes of
// 128 rows: 32 KB), q as A operand (128 rows, the last 64 zero: 32 KB), the
// summed keys (512 B), mbarrier, TMEM slot
constexpr uint32_t kAKV = 0, kAQ = 32768, kAZ = 65536, kABar = kAZ + 512;
constexpr uint32_t kASmem = kABar + 64 + 1024;
constexpr uint32_t kIdQKV = tc::idesc_bf16(128, 128, false, true);  // A = q (K-major), B = K^T V (MN-major)

__global__ void __launch_bounds__(kThreads, 1)
kv_apply_kernel(const __nv_bfloat16* __restrict__ q, int H, int group, char* __restrict__ ws,
                const float* __restrict__ kv, const float* __restrict__ z, int normalize,
                __nv_bfloat16* __restrict__ o) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = tc::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sbase = raw + pad;
    char* const sptr = reinterpret_cast<char*>(smem_raw) + pad;
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;
    const int total = hdr->total_chunks, n_seqs = hdr->n_seqs, limit = hdr->wait_limit;
    const int g0 = blockIdx.x * group, head = blockIdx.y;
    if (g0 >= total) return;
    const int g1 = min(total, g0 + group);
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* chunk_off = reinterpret_cast<const int*>(ws + L.chunk_off);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar = sbase + kABar, tslot = sbase + kABar + 16;
    float* zsm = reinterpret_cast<float*>(sptr + kAZ);

    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::fence_mbar_init();
    }
    // rows 64 .. 127 of the q operand stay zero
    for (int x = tid; x < 2 * 64 * 8; x += kThreads) {
        const int bx = x >> 9, t = 64 + ((x >> 3) & 63), c = x & 7;
        tc::st_shared_v4(tc::sw128(sbase + kAQ + bx * 16384, t, c), 0u, 0u, 0u, 0u);
    }
    __syncwarp();
    if (warp == 0) tc::tmem_alloc(tslot, 128);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sptr + kABar + 16);

    uint32_t phase = 0;
    int cur_seq = -1;
    bool ok = true, pending = false;
    for (int gc = g0; gc < g1 && ok; ++gc) {
        const ChunkRef r = chunk_ref(cu, chunk_off, n_seqs, gc);
        if (r.seq != cur_seq) {
            // K^T V of this sequence and head, rounded to bf16: row i (the K
            // dimension) holds features j = 64 box .. + 63 of each box
            const float* src = kv + ((size_t)r.seq * H + head) * kD * kD;
            for (int x = tid; x < kD * 16; x += kThreads) {
                const int i = x >> 4, c16 = x & 15;
                const float4 a = *reinterpret_cast<const float4*>(src + (size_t)i * kD + 8 * c16);
                const float4 bq = *reinterpret_cast<const float4*>(src + (size_t)i * kD + 8 * c16 + 4);
                tc::st_shared_v4(tc::sw128(sbase + kAKV + (uint32_t)(c16 >> 3) * 16384, i, c16 & 7),
                                 tc::pack_bf16(a.x, a.y), tc::pack_bf16(a.z, a.w), tc::pack_bf16(bq.x, bq.y),
                                 tc::pack_bf16(bq.z, bq.w));
            }
            zsm[tid] = normalize ? z[((size_t)r.seq * H + head) * kD + tid] : 0.f;
            cur_seq = r.seq;
        }
        load_rows(sbase + kAQ, 16384, q, r.t0, r.n, H, head, tid);
        tc::fence_proxy_async();
        tc::tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc::tc_fence_after();
            // D = q (K^T V): features 0..63 of q from box 0, 64..127 from box 1
            tc::mma_ss_n<4>(tmem, tc::sdesc(sbase + kAQ, 16, 1024), 2, tc::sdesc(sbase + kAKV, 16384, 1024), 128,
                            kIdQKV, false);
            tc::mma_ss_n<4>(tmem, tc::sdesc(sbase + kAQ + 16384, 16, 1024), 2,
                            tc::sdesc(sbase + kAKV + 64 * 128, 16384, 1024), 128, kIdQKV, true);
            tc::commit_e(bar);
        }
        __syncwarp();
        pending = true;
        ok = __syncthreads_and(wait_or_fail(bar, phase, ws, limit));
        if (!ok) break;  // the commit stays pending for the drain below
        phase ^= 1u;
        pending = false;
        tc::tc_fence_after();
        if (warp < 2) {  // rows (tokens) 0 .. 63 live in the lanes of warps 0 and 1
            const int t = 32 * warp + lane;
            float den = 1.f;
            if (normalize) {
                // q_t . z from the swizzled q tile
                den = 0.f;
#pragma unroll 1
                for (int c16 = 0; c16 < 16; ++c16) {
                    const uint4 qq = tc::ld_shared_v4(tc::sw128(sbase + kAQ + (uint32_t)(c16 >> 3) * 16384, t, c16 & 7));
                    const uint32_t w[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float2 f = tc::unpack_bf16(w[x]);
                        den = fmaf(f.x, zsm[8 * c16 + 2 * x], den);
                        den = fmaf(f.y, zsm[8 * c16 + 2 * x + 1], den);
                    }
                }
            }
            const float inv = 1.f / den;
            float d[32];
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * c, d);
                tc::tmem_wait_ld();
                if (t < r.n) {
                    uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(r.t0 + t) * H + head) * kD + 32 * c);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        dst[x] = make_uint4(tc::pack_bf16(d[8 * x] * inv, d[8 * x + 1] * inv),
                                            tc::pack_bf16(d[8 * x + 2] * inv, d[8 * x + 3] * inv),
                                            tc::pack_bf16(d[8 * x + 4] * inv, d[8 * x + 5] * inv),
                                            tc::pack_bf16(d[8 * x + 6] * inv, d[8 * x + 7] * inv));
                }
            }
        }
        tc::tc_fence_before();
        __syncthreads();  // the q tile, K^T V and D may be rewritten
        tc::tc_fence_after();
    }
    if (pending) tc::mbar_wait(bar, phase);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
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
// sequence's total (the summed keys z, when asked for).
__global__ void __launch_bounds__(kThreads)
key_prefix_kernel(int H, const char* __restrict__ ws, const float* __restrict__ ks,
                  float* __restrict__ zstart, float* __restrict__ z) {
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;
    PlanLayout L(hdr->n_seqs);
    const int* chunk_off = reinterpret_cast<const int*>(ws + L.chunk_off);
    const int seq = blockIdx.x, head = blockIdx.y, i = threadIdx.x;
    float run = 0.f;
    for (int c = chunk_off[seq]; c < chunk_off[seq + 1]; ++c) {
        const size_t at = ((size_t)c * H + head) * kD + i;
        zstart[at] = run;
        run += ks[at];
    }
    if (z) z[((size_t)seq * H + head) * kD + i] = run;
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
    // chunks per CTA: enough CTAs for about eight per SM, and no more, so that
    // each (sequence, head) gets few partial sums of K^T V to add up
    const long long nch = max_chunks(a.T_total, a.n_seqs);
    const long long sms = sm_count() > 0 ? sm_count() : 148;
    const int group = (int)max((long long)kMinGroup, (nch * a.H + 8 * sms - 1) / (8 * sms));
    const unsigned groups = (unsigned)((nch + group - 1) / group);
    if (e == cudaSuccess && groups > 0) {
        e = cudaFuncSetAttribute(kv_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmem);
        if (e == cudaSuccess) {
            kv_reduce_kernel<<<dim3(groups, a.H), kThreads, kRSmem, st>>>(
                (const __nv_bfloat16*)a.k, (const __nv_bfloat16*)a.v, a.H, group, plan_ws, kv, z);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kv_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem);
        if (e == cudaSuccess) {
            kv_apply_kernel<<<dim3(groups, a.H), kThreads, kASmem, st>>>(
                (const __nv_bfloat16*)a.q, a.H, group, plan_ws, kv, z, normalize ? 1 : 0, (__nv_bfloat16*)a.o);
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
        key_prefix_kernel<<<dim3((unsigned)a.n_seqs, a.H), kThreads, 0, st>>>(a.H, plan_ws, ks, zstart, z_out);
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
