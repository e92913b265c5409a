// plan.cu -- per-call plan kernel: validates cu_seqlens on the device and
// writes the chunk offsets and the longest-first sequence order that the
// prefill kernels read.  One block; runs first on the call's stream, so
// every later kernel of the call sees its status word.
#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr int kPlanThreads = 1024;
constexpr int kOrderQuadraticMax = 4096;  // above this, keep the natural order

// The group plan of the grouped causal linear attention, by the plan's block
// once chunk_off is complete.  The size is the smallest g >= kGroupMinChunks
// for which all (sequence, head) pairs together have at most `sms` groups (one
// wave of one-CTA-per-SM launches), or, when even one group per sequence is
// more than that, g = max(kGroupMinChunks, ceil(H total / sms)).  Either way
// the group count is at most floor(sms / H) + n_seqs.  group_off[s] = first
// group of sequence s, group_off[n_seqs] = the number of groups,
// group_off[n_seqs + 1] = the group size.
__device__ void plan_groups(const int* chunk_off, int n_seqs, const GroupPlan& gp, int* s_scan) {
    __shared__ int s_red[2][32];
    __shared__ int s_gcarry;
    int* const s_carry = &s_gcarry;
    const int tid = threadIdx.x, H = gp.H, sms = gp.sms;
    for (int x = tid; x < gp.n_counters; x += kPlanThreads) gp.counters[x] = 0;
    // this thread's sequences' chunk counts (the first 8 x 1024 kept in registers;
    // only the entries that exist are divided below)
    constexpr int kKeep = 8;
    int cnt[kKeep];
    const int mine = tid < n_seqs ? (n_seqs - 1 - tid) / kPlanThreads + 1 : 0;
#pragma unroll
    for (int k = 0; k < kKeep; ++k) {
        const int i = tid + kPlanThreads * k;
        cnt[k] = i < n_seqs ? chunk_off[i + 1] - chunk_off[i] : 0;
    }
    // number of groups of size g over all sequences (every thread gets it; at most
    // the number of chunks, which fits an int)
    int flip = 0;
    auto groups_of = [&](int g) -> int {
        int c = 0;
#pragma unroll
        for (int k = 0; k < kKeep; ++k)
            if (k < mine) c += (cnt[k] + g - 1) / g;
        for (int i = tid + kPlanThreads * kKeep; i < n_seqs; i += kPlanThreads)
            c += (chunk_off[i + 1] - chunk_off[i] + g - 1) / g;
        c = __reduce_add_sync(0xffffffffu, c);
        if ((tid & 31) == 0) s_red[flip][tid >> 5] = c;
        __syncthreads();  // alternate buffers: one barrier per evaluation
        int t = 0;
#pragma unroll
        for (int w = 0; w < kPlanThreads / 32; ++w) t += s_red[flip][w];
        flip ^= 1;
        return t;
    };
    const int total = chunk_off[n_seqs];
    int lo = kGroupMinChunks, hi = max(kGroupMinChunks, total);
    int group;
    if ((long long)H * groups_of(hi) <= sms) {
        while (lo < hi) {  // groups_of is non-increasing in g
            const int mid = (lo + hi) >> 1;
            if ((long long)H * groups_of(mid) <= sms) hi = mid; else lo = mid + 1;
        }
        group = lo;
    } else {
        group = (int)max((long long)kGroupMinChunks, ((long long)H * total + sms - 1) / sms);
    }
    if (tid == 0) *s_carry = 0;
    __syncthreads();
    for (int base = 0; base < n_seqs; base += kPlanThreads) {
        const int i = base + tid;
        const int ng = i < n_seqs ? (chunk_off[i + 1] - chunk_off[i] + group - 1) / group : 0;
        s_scan[tid] = ng;
        __syncthreads();
        for (int off = 1; off < kPlanThreads; off <<= 1) {
            const int x = tid >= off ? s_scan[tid - off] : 0;
            __syncthreads();
            s_scan[tid] += x;
            __syncthreads();
        }
        if (i < n_seqs) gp.group_off[i] = *s_carry + s_scan[tid] - ng;
        __syncthreads();
        if (tid == kPlanThreads - 1) *s_carry += s_scan[kPlanThreads - 1];
        __syncthreads();
    }
    if (tid == 0) {
        gp.group_off[n_seqs] = *s_carry;
        gp.group_off[n_seqs + 1] = group;
    }
}

// The whole plan (and group plan) by one warp, for calls of at most 32
// sequences: the same results as the block-wide path below, with shuffles and
// warp reductions in place of block barriers.
__device__ void plan_small(const int32_t* __restrict__ cu_in, int n_seqs, long long T_total, int wait_limit, char* ws,
                           const int* __restrict__ upstream, const GroupPlan& gp) {
    constexpr unsigned kAll = 0xffffffffu;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    PlanLayout L(n_seqs);
    int* cu = reinterpret_cast<int*>(ws + L.cu);
    int* chunk_off = reinterpret_cast<int*>(ws + L.chunk_off);
    int* order = reinterpret_cast<int*>(ws + L.order);
    const int lane = threadIdx.x;
    // copy + validate: cu[0] = 0, non-decreasing, cu[n] = T_total
    bool bad = false;
    for (int i = lane; i <= n_seqs; i += 32) {
        const long long c = cu_in ? (long long)cu_in[i] : (i == 0 ? 0 : T_total);
        cu[i] = (int)c;
        bool b = (i == 0 && c != 0) || (i == n_seqs && c != T_total) || c < 0 || c > T_total;
        if (i > 0 && cu_in) b |= cu_in[i] < cu_in[i - 1];
        bad |= b;
    }
    if (__any_sync(kAll, bad)) {
        if (lane == 0) {
            hdr->status = GDN_ERR_SEQLENS;
            hdr->counter = 0;
            hdr->timeout_site = 0;
            hdr->wait_limit = wait_limit;
            hdr->n_seqs = n_seqs;
            hdr->total_chunks = 0;
            hdr->max_len = 0;
        }
        return;
    }
    __syncwarp();
    const int len = lane < n_seqs ? cu[lane + 1] - cu[lane] : 0;
    const int maxlen = __reduce_max_sync(kAll, len);
    const int nch = (len + kChunk - 1) / kChunk;
    int incl = nch;  // inclusive scan of the chunk counts
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(kAll, incl, o);
        if (lane >= o) incl += x;
    }
    const int total = __shfl_sync(kAll, incl, 31);
    if (lane < n_seqs) chunk_off[lane] = incl - nch;
    if (lane == 0) chunk_off[n_seqs] = total;
    // longest-first order (ties by index)
    int rank = 0;
    for (int j = 0; j < n_seqs; ++j) {
        const int lj = __shfl_sync(kAll, len, j);
        rank += (lj > len) || (lj == len && j < lane);
    }
    if (lane < n_seqs) order[rank] = lane;
    if (gp.group_off != nullptr) {
        for (int x = lane; x < gp.n_counters; x += 32) gp.counters[x] = 0;
        auto groups_of = [&](int g) { return __reduce_add_sync(kAll, lane < n_seqs ? (nch + g - 1) / g : 0); };
        int lo = kGroupMinChunks, hi = max(kGroupMinChunks, total), group;
        if ((long long)gp.H * groups_of(hi) <= gp.sms) {
            while (lo < hi) {  // groups_of is non-increasing in g
                const int mid = (lo + hi) >> 1;
                if ((long long)gp.H * groups_of(mid) <= gp.sms) hi = mid; else lo = mid + 1;
            }
            group = lo;
        } else {
            group = (int)max((long long)kGroupMinChunks, ((long long)gp.H * total + gp.sms - 1) / gp.sms);
        }
        const int ng = lane < n_seqs ? (nch + group - 1) / group : 0;
        int gincl = ng;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(kAll, gincl, o);
            if (lane >= o) gincl += x;
        }
        const int gtotal = __shfl_sync(kAll, gincl, 31);
        if (lane < n_seqs) gp.group_off[lane] = gincl - ng;
        if (lane == 0) {
            gp.group_off[n_seqs] = gtotal;
            gp.group_off[n_seqs + 1] = group;
        }
    }
    if (lane == 0) {
        // a call whose own inputs were already found bad upstream does nothing
        hdr->status = (upstream != nullptr && *upstream != GDN_OK) ? *upstream : GDN_OK;
        hdr->counter = 0;
        hdr->timeout_site = 0;
        hdr->wait_limit = wait_limit;
        hdr->n_seqs = n_seqs;
        hdr->total_chunks = total;
        hdr->max_len = maxlen;
    }
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ cu_in, int n_seqs, long long T_total, int wait_limit, char* ws,
            const int* __restrict__ upstream, GroupPlan gp) {
    if (n_seqs <= 32) {
        if (threadIdx.x < 32) plan_small(cu_in, n_seqs, T_total, wait_limit, ws, upstream, gp);
        return;
    }
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    PlanLayout L(n_seqs);
    int* cu = reinterpret_cast<int*>(ws + L.cu);
    int* chunk_off = reinterpret_cast<int*>(ws + L.chunk_off);
    int* order = reinterpret_cast<int*>(ws + L.order);

    __shared__ int s_bad;
    __shared__ int s_maxlen;
    __shared__ int s_scan[kPlanThreads];
    __shared__ int s_carry;
    const int tid = threadIdx.x;
    if (tid == 0) { s_bad = 0; s_maxlen = 0; s_carry = 0; }
    __syncthreads();

    // copy + validate: cu[0] = 0, non-decreasing, cu[n] = T_total
    for (int i = tid; i <= n_seqs; i += kPlanThreads) {
        long long c = cu_in ? (long long)cu_in[i] : (i == 0 ? 0 : T_total);
        cu[i] = (int)c;
        bool bad = (i == 0 && c != 0) || (i == n_seqs && c != T_total) || c < 0 || c > T_total;
        if (i > 0 && cu_in) bad |= cu_in[i] < cu_in[i - 1];
        if (bad) atomicOr(&s_bad, 1);
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            hdr->status = GDN_ERR_SEQLENS;
            hdr->counter = 0;
            hdr->timeout_site = 0;
            hdr->wait_limit = wait_limit;
            hdr->n_seqs = n_seqs;
            hdr->total_chunks = 0;
            hdr->max_len = 0;
        }
        return;
    }

    // chunk offsets: exclusive scan of ceil(L_s / 64), tile by tile
    for (int base = 0; base < n_seqs; base += kPlanThreads) {
        int i = base + tid;
        int len = i < n_seqs ? cu[i + 1] - cu[i] : 0;
        if (i < n_seqs) atomicMax(&s_maxlen, len);
        int nch = (len + kChunk - 1) / kChunk;
        s_scan[tid] = nch;
        __syncthreads();
        for (int off = 1; off < kPlanThreads; off <<= 1) {
            int x = tid >= off ? s_scan[tid - off] : 0;
            __syncthreads();
            s_scan[tid] += x;
            __syncthreads();
        }
        if (i < n_seqs) chunk_off[i] = s_carry + s_scan[tid] - nch;
        __syncthreads();
        if (tid == kPlanThreads - 1) s_carry += s_scan[tid];
        __syncthreads();
    }
    if (tid == 0) chunk_off[n_seqs] = s_carry;
    if (gp.group_off != nullptr) {
        __syncthreads();  // chunk_off (global, this block's writes) is complete
        plan_groups(chunk_off, n_seqs, gp, s_scan);
    }

    // longest-first order (ties by index), so long chains start first
    for (int i = tid; i < n_seqs; i += kPlanThreads) {
        if (n_seqs > kOrderQuadraticMax) { order[i] = i; continue; }
        int li = cu[i + 1] - cu[i];
        int rank = 0;
        for (int j = 0; j < n_seqs; ++j) {
            int lj = cu[j + 1] - cu[j];
            rank += (lj > li) || (lj == li && j < i);
        }
        order[rank] = i;
    }
    if (tid == 0) {
        // a call whose own inputs were already found bad upstream does nothing
        hdr->status = (upstream != nullptr && *upstream != GDN_OK) ? *upstream : GDN_OK;
        hdr->counter = 0;
        hdr->timeout_site = 0;
        hdr->wait_limit = wait_limit;
        hdr->n_seqs = n_seqs;
        hdr->total_chunks = s_carry;
        hdr->max_len = s_maxlen;
    }
}

cudaError_t launch_plan(const int32_t* cu, int n_seqs, int64_t T_total, int wait_limit, void* ws,
                        cudaStream_t st, const int* upstream, const GroupPlan* gp) {
    const GroupPlan none{0, 0, nullptr, nullptr, 0};
    plan_kernel<<<1, kPlanThreads, 0, st>>>(cu, n_seqs, (long long)T_total, wait_limit, (char*)ws, upstream,
                                            gp ? *gp : none);
    return cudaGetLastError();
}

}  // namespace gdn
