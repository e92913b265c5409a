// plan.cu -- per-call plan kernel: validates cu_seqlens on the device and
// writes the chunk offsets and the longest-first sequence order that the
// prefill kernels read.  One block; runs first on the call's stream, so
// every later kernel of the call sees its status word.
#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr int kPlanThreads = 1024;
constexpr int kOrderQuadraticMax = 4096;  // above this, keep the natural order

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ cu_in, int n_seqs, long long T_total, int wait_limit, char* ws,
            const int* __restrict__ upstream) {
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
                        cudaStream_t st, const int* upstream) {
    plan_kernel<<<1, kPlanThreads, 0, st>>>(cu, n_seqs, (long long)T_total, wait_limit, (char*)ws, upstream);
    return cudaGetLastError();
}

}  // namespace gdn
