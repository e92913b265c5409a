// launch.h -- host-side launchers of the kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Arguments common to the prefill paths (device pointers; see gdn.h).
struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* log_alpha;
    const float* beta;
    const float* h0;
    const int32_t* cu_seqlens;
    int n_seqs;
    int64_t T_total;
    int H, dk, dv;
    gdn_dtype io;
    bool delta_rule;  // false: plain linear attention (no gates, no delta term)
    // Farthest 16-token block below the diagonal at which the inverse of the
    // delta system is kept: 3 = the exact solve (a 64-token chunk has four
    // blocks), 1 = the block-adjacent solver.
    int max_block_dist;
    // Runs of the two-level state scan use the cluster kernel with these bits
    // (0 for an ordinary call): 1 = o is not stored; 2 = v is taken as zero;
    // 4 = h0 is taken as the identity (dk = dv).
    int mode;
    void* o;
    float* h_T;
    char* ws;
};

// Intermediates of the staged path (fp32, all in the workspace unless the
// caller supplies its own buffers).
struct StagedBuffers {
    float* g;  // [T][H]
    float* A;  // [max_chunks][H][64][64]
    float* w;  // [T][H][dk]
    float* u;  // [T][H][dv]
};

size_t staged_intermediate_bytes(int64_t T, int H, int dk, int dv, int n_seqs);
StagedBuffers staged_buffers(char* ws, int64_t T, int H, int dk, int dv, int n_seqs);

// wait_limit: polls a bounded device wait of the call's kernels makes before
// it reports GDN_ERR_TIMEOUT (recorded in the workspace header).  upstream
// (device, may be NULL): a status word found earlier in the same call; if it
// is not GDN_OK the plan carries it, and the kernels reading the plan skip
// their work.
// The grouped causal linear attention's part of the plan (group_off NULL: none):
// the group size and numbering, written to group_off (n_seqs + 2 ints), and
// n_counters hand-off counters zeroed.
struct GroupPlan {
    int sms, H;
    int* group_off;
    int* counters;
    int n_counters;
};
constexpr int kGroupMinChunks = 4;  // chunks per group, at least
cudaError_t launch_plan(const int32_t* cu, int n_seqs, int64_t T_total, int wait_limit, void* ws,
                        cudaStream_t st, const int* upstream = nullptr, const GroupPlan* gp = nullptr);
cudaError_t launch_kkt(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st);
cudaError_t launch_wy(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st);
cudaError_t launch_state_ffma(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st);
cudaError_t launch_decode(const void* q, const void* k, const void* v, const void* log_alpha,
                          const void* beta, float* state, void* o, int B, int H, int dk, int dv,
                          cudaStream_t st);

// Fused single-kernel prefill (bf16, dk = dv = 128): tcgen05 + TMA, one SM
// per (sequence, head, 64-column half of the state).
bool fused_supported(const PrefillArgs& a);
cudaError_t launch_fused(const PrefillArgs& a, cudaStream_t st);

// Fused prefill on a 2-CTA cluster per (sequence, head): solve on one SM,
// state pass on the other (bf16, dk = dv = 128).
bool pair_shape_ok(const PrefillArgs& a);  // sizes and dtype only
bool pair_supported(const PrefillArgs& a);
size_t pair_workspace_bytes(int n_seqs, int H);  // plan + global scratch
// fronts: solve CTAs per cluster (1 or 2), next to the one state CTA.
cudaError_t launch_pair(const PrefillArgs& a, int fronts, cudaStream_t st);
// Solve CTAs per cluster the cluster kernel takes for these arguments.
int pair_fronts(const PrefillArgs& a);

// Two-level state scan (long sequences with few (sequence, head) chains):
// segments per sequence the call takes (1: none), its workspace, its launch.
int two_level_segments(const PrefillArgs& a);
size_t two_level_workspace_bytes(int n_seqs, int H, int G);
cudaError_t launch_two_level(const PrefillArgs& a, int G, int wait_limit, cudaStream_t st);

// Linear attention (bf16, dk = dv = 128) without the cluster kernel:
// bidirectional via K^T V, and causal through groups of chunks (normalised or
// not).  plan_ws holds a plan of the call's sequences; extra holds
// linear_variant_extra_bytes() (bidirectional) or
// linear_grouped_extra_bytes() (causal).
bool linear_variant_shape_ok(const PrefillArgs& a);
size_t linear_variant_extra_bytes(int64_t T, int H, int n_seqs, bool causal);
cudaError_t launch_linear_bidirectional(const PrefillArgs& a, char* plan_ws, char* extra, bool normalize,
                                        float* kv_out, float* z_out, cudaStream_t st);
size_t linear_grouped_extra_bytes(int64_t T, int H, int n_seqs);
// Runs its own plan (with the group plan) at plan_ws.
cudaError_t launch_linear_grouped(const PrefillArgs& a, char* plan_ws, char* extra, bool normalize, float* h_T,
                                  float* z_T, int wait_limit, cudaStream_t st);

}  // namespace gdn
