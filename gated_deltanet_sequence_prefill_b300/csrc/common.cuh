// common.cuh -- shared device helpers and the workspace header layout.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;  // tokens per chunk on every path

// Workspace header (device memory, 256-byte aligned, written by the plan
// kernel at the start of every call and read by every later kernel).
struct WsHeader {
    int status;        // GDN_OK or a negative gdn_status found on the device
    int counter;       // work counter of the persistent prefill kernel
    int n_seqs;
    int total_chunks;  // sum over sequences of ceil(L_s / 64)
    int max_len;       // longest sequence
    int timeout_site;  // first barrier a timed-out wait gave up on (0: none)
    int wait_limit;    // polls a bounded device wait makes before it gives up
    int pad[57];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Offsets of the plan arrays after the header (all int32).
struct PlanLayout {
    size_t cu;         // [n_seqs + 1] copy of cu_seqlens (or {0, T})
    size_t chunk_off;  // [n_seqs + 1] first global chunk of each sequence
    size_t order;      // [n_seqs] sequences by decreasing length
    size_t end;
    __host__ __device__ explicit PlanLayout(int n_seqs) {
        cu = align256(sizeof(WsHeader));
        chunk_off = cu + align256(sizeof(int) * (size_t)(n_seqs + 1));
        order = chunk_off + align256(sizeof(int) * (size_t)(n_seqs + 1));
        end = order + align256(sizeof(int) * (size_t)n_seqs);
    }
};

// Upper bound on the number of chunks: sum ceil(L_s/64) <= floor(T/64) + n_seqs.
__host__ __device__ inline int64_t max_chunks(int64_t T, int n_seqs) { return T / kChunk + n_seqs; }

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Sequence that owns global chunk `gc`: the largest s with chunk_off[s] <= gc
// (zero-length sequences own no chunk and are skipped by the search).
__device__ __forceinline__ int seq_of_chunk(const int* chunk_off, int n_seqs, int gc) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= gc) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace gdn
