// api.cu -- the extern "C" entry points of libgdn_b300.so (declared in gdn.h):
// host-side argument checks, workspace carving and kernel launches.
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"
#include "gdn.h"
#include "launch.h"

using namespace gdn;

namespace gdn {

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

// Solve CTAs per cluster for the cluster kernel: two (a 3-SM cluster) when
// every (sequence, head) then still has its cluster at once, else one (more
// clusters side by side pay off more than a faster solve).
// GDN_PREFILL_FRONTS=1 or 2 in the environment forces the choice.
int pair_fronts(const PrefillArgs& a) {
    const char* e = getenv("GDN_PREFILL_FRONTS");
    if (e != nullptr && (e[0] == '1' || e[0] == '2')) return e[0] - '0';
    return 3LL * a.n_seqs * a.H <= (long long)sm_count() ? 2 : 1;
}

}  // namespace gdn

namespace {

// Polls per bounded device wait, for the calls launched from now on.
constexpr int kDefaultWaitLimit = 1 << 22;
std::atomic<int> g_wait_limit{kDefaultWaitLimit};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool head_ok(int d) { return d == 64 || d == 128; }

size_t plan_bytes(int n_seqs) { return PlanLayout(n_seqs).end; }

bool sizes_ok(int64_t T, int H, int dk, int dv, int n_seqs) {
    return T >= 0 && T < (int64_t(1) << 31) - kChunk && H >= 1 && n_seqs >= 0 &&
           n_seqs < (1 << 28) && head_ok(dk) && head_ok(dv);
}

// Checks shared by the prefill entry points; `need` is the workspace size.
gdn_status check_prefill(const PrefillArgs& a, size_t ws_bytes, size_t need, bool need_outputs) {
    if (a.io != GDN_BF16 && a.io != GDN_FP32) return GDN_ERR_DTYPE;
    if (a.T_total < 0 || a.H < 1 || a.n_seqs < 0 || a.T_total >= (int64_t(1) << 31) - kChunk)
        return GDN_ERR_SHAPE;
    if (!head_ok(a.dk) || !head_ok(a.dv)) return GDN_ERR_UNSUPPORTED;
    if (a.cu_seqlens == nullptr && a.n_seqs != 1) return GDN_ERR_SHAPE;
    if (a.n_seqs == 0 && a.T_total != 0) return GDN_ERR_SHAPE;
    if (a.T_total > 0) {
        if (!a.k || !a.v) return GDN_ERR_NULL;
        if (need_outputs && (!a.q || !a.o)) return GDN_ERR_NULL;
        if (a.delta_rule && (!a.log_alpha || !a.beta)) return GDN_ERR_NULL;
    }
    if (!a.ws) return GDN_ERR_WORKSPACE;
    if (ws_bytes < need) return GDN_ERR_WORKSPACE;
    if (!aligned(a.ws, 256)) return GDN_ERR_ALIGN;
    if (!aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.o, 16) ||
        !aligned(a.h0, 16) || !aligned(a.h_T, 16) || !aligned(a.log_alpha, 4) ||
        !aligned(a.beta, 4) || !aligned(a.cu_seqlens, 4))
        return GDN_ERR_ALIGN;
    return GDN_OK;
}

gdn_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    cudaGetLastError();  // clear a non-sticky error so later calls are not blamed
    return GDN_ERR_CUDA;
}

gdn_status run_staged(const PrefillArgs& a, cudaStream_t st, float* g_out, float* A_out,
                      float* w_out, float* u_out, bool state_pass) {
    StagedBuffers b = staged_buffers(a.ws, a.T_total, a.H, a.dk, a.dv, a.n_seqs);
    if (g_out) b.g = g_out;
    if (A_out) b.A = A_out;
    if (w_out) b.w = w_out;
    if (u_out) b.u = u_out;
    cudaError_t e = launch_plan(a.cu_seqlens, a.n_seqs, a.T_total, g_wait_limit.load(), a.ws, st);
    if (e == cudaSuccess && a.delta_rule && a.T_total > 0) e = launch_kkt(a, b, st);
    if (e == cudaSuccess && a.delta_rule && a.T_total > 0) e = launch_wy(a, b, st);
    if (e == cudaSuccess && state_pass) e = launch_state_ffma(a, b, st);
    return cuda_status(e);
}

PrefillArgs make_args(const void* q, const void* k, const void* v, const float* la,
                      const float* beta, const float* h0, const int32_t* cu, int n_seqs,
                      int64_t T, int H, int dk, int dv, gdn_dtype io, bool delta, void* o,
                      float* h_T, void* ws) {
    PrefillArgs a;
    a.q = q; a.k = k; a.v = v; a.log_alpha = la; a.beta = beta; a.h0 = h0;
    a.cu_seqlens = cu; a.n_seqs = n_seqs; a.T_total = T; a.H = H; a.dk = dk; a.dv = dv;
    a.io = io; a.delta_rule = delta; a.o = o; a.h_T = h_T; a.ws = (char*)ws;
    a.max_block_dist = 3;
    a.mode = 0;
    return a;
}

// Which fused kernel: the 2-SM cluster kernel (solve and state pass on
// separate SMs) unless GDN_PREFILL_PAIR=0 in the environment selects the
// single-SM kernel (one CTA per sequence, head and 64-column half of the
// state).
bool use_pair(const PrefillArgs& a) {
    if (!pair_supported(a)) return false;
    const char* e = getenv("GDN_PREFILL_PAIR");
    return !(e != nullptr && e[0] == '0');
}

// Causal linear attention (bf16, dk = dv = 128) runs through groups of chunks
// (linear_variants.cu) unless the environment picks another path:
// GDN_LINEAR_PATH=cluster or GDN_PREFILL_PAIR=0 (the fused prefill kernels)
// or GDN_TWO_LEVEL (the two-level scan over the cluster kernel).
bool use_grouped_linear(const PrefillArgs& a) {
    if (a.delta_rule || a.io != GDN_BF16 || a.dk != 128 || a.dv != 128) return false;
    const char* e = getenv("GDN_LINEAR_PATH");
    if (e != nullptr && strcmp(e, "cluster") == 0) return false;
    const char* p = getenv("GDN_PREFILL_PAIR");
    if (p != nullptr && p[0] == '0') return false;
    const char* t = getenv("GDN_TWO_LEVEL");
    return !(t != nullptr && t[0] != '\0');
}

size_t grouped_linear_bytes(int64_t T, int H, int n_seqs) {
    return align256(plan_bytes(n_seqs)) + linear_grouped_extra_bytes(T, H, n_seqs);
}

gdn_status prefill(const PrefillArgs& a, size_t ws_bytes, cudaStream_t st) {
    if (use_grouped_linear(a)) {
        gdn_status s = check_prefill(a, ws_bytes, grouped_linear_bytes(a.T_total, a.H, a.n_seqs), true);
        if (s != GDN_OK) return s;
        cudaError_t e = launch_linear_grouped(a, a.ws, a.ws + align256(plan_bytes(a.n_seqs)), false, a.h_T, nullptr,
                                              g_wait_limit.load(), st);
        return cuda_status(e);
    }
    const bool pair = use_pair(a);
    if (pair) {
        const int G = two_level_segments(a);
        if (G >= 2) {
            gdn_status s = check_prefill(a, ws_bytes, two_level_workspace_bytes(a.n_seqs, a.H, G), true);
            if (s != GDN_OK) return s;
            return cuda_status(launch_two_level(a, G, g_wait_limit.load(), st));
        }
    }
    const bool fused = pair || fused_supported(a);
    size_t need = pair ? pair_workspace_bytes(a.n_seqs, a.H) : plan_bytes(a.n_seqs);
    if (!fused) need += staged_intermediate_bytes(a.T_total, a.H, a.dk, a.dv, a.n_seqs);
    gdn_status s = check_prefill(a, ws_bytes, need, true);
    if (s != GDN_OK) return s;
    if (!fused) return run_staged(a, st, nullptr, nullptr, nullptr, nullptr, true);
    cudaError_t e = launch_plan(a.cu_seqlens, a.n_seqs, a.T_total, g_wait_limit.load(), a.ws, st);
    if (e == cudaSuccess) e = pair ? launch_pair(a, pair_fronts(a), st) : launch_fused(a, st);
    return cuda_status(e);
}

}  // namespace

extern "C" {

const char* gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL: return "a required pointer is NULL";
        case GDN_ERR_ALIGN: return "a pointer is not aligned as required";
        case GDN_ERR_SHAPE: return "invalid or inconsistent sizes";
        case GDN_ERR_SEQLENS: return "cu_seqlens is malformed";
        case GDN_ERR_DTYPE: return "unknown io dtype";
        case GDN_ERR_UNSUPPORTED: return "unsupported head size or dtype combination";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_CUDA: return "CUDA runtime or launch error";
        case GDN_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        default: return "unknown status";
    }
}

const char* gdn_version(void) { return "gdn_b300 0.2 sm_103a"; }

int gdn_set_wait_limit(int polls) {
    return g_wait_limit.exchange(polls < 0 ? kDefaultWaitLimit : polls);
}

gdn_status gdn_workspace_timeout_site(const void* workspace, void* stream, int* site) {
    if (!workspace || !site) return GDN_ERR_NULL;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemcpy(site, (const char*)workspace + offsetof(WsHeader, timeout_site), sizeof(int),
                       cudaMemcpyDeviceToHost);
    return cuda_status(e);
}

size_t gdn_staged_workspace_size(int64_t T, int H, int dk, int dv, int n_seqs, gdn_dtype io) {
    if (!sizes_ok(T, H, dk, dv, n_seqs) || (io != GDN_BF16 && io != GDN_FP32)) return 0;
    return plan_bytes(n_seqs) + staged_intermediate_bytes(T, H, dk, dv, n_seqs);
}

size_t gdn_chunk_fwd_workspace_size(int64_t T, int H, int dk, int dv, int n_seqs, gdn_dtype io) {
    if (!sizes_ok(T, H, dk, dv, n_seqs) || (io != GDN_BF16 && io != GDN_FP32)) return 0;
    PrefillArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, n_seqs,
                              T, H, dk, dv, io, true, nullptr, nullptr, nullptr);
    if (pair_shape_ok(a)) {
        const int G = two_level_segments(a);
        return G >= 2 ? two_level_workspace_bytes(n_seqs, H, G) : pair_workspace_bytes(n_seqs, H);
    }
    if (fused_supported(a)) return plan_bytes(n_seqs);
    return gdn_staged_workspace_size(T, H, dk, dv, n_seqs, io);
}

size_t linear_attn_fwd_workspace_size(int64_t T, int H, int dk, int dv, int n_seqs, gdn_dtype io) {
    if (!sizes_ok(T, H, dk, dv, n_seqs) || (io != GDN_BF16 && io != GDN_FP32)) return 0;
    PrefillArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, n_seqs,
                              T, H, dk, dv, io, false, nullptr, nullptr, nullptr);
    if (use_grouped_linear(a)) return grouped_linear_bytes(T, H, n_seqs);
    if (pair_shape_ok(a)) {
        const int G = two_level_segments(a);
        return G >= 2 ? two_level_workspace_bytes(n_seqs, H, G) : pair_workspace_bytes(n_seqs, H);
    }
    if (fused_supported(a)) return plan_bytes(n_seqs);
    return gdn_staged_workspace_size(T, H, dk, dv, n_seqs, io);
}

int gdn_prefill_segments(int64_t T, int H, int dk, int dv, int n_seqs, gdn_dtype io, int delta_rule) {
    if (!sizes_ok(T, H, dk, dv, n_seqs) || (io != GDN_BF16 && io != GDN_FP32)) return 0;
    PrefillArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, n_seqs,
                              T, H, dk, dv, io, delta_rule != 0, nullptr, nullptr, nullptr);
    return two_level_segments(a);
}

gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* log_alpha,
                         const float* beta, const float* h0, const int32_t* cu_seqlens, int n_seqs,
                         int64_t T_total, int H, int dk, int dv, gdn_dtype io_dtype, void* o,
                         float* h_T, void* workspace, size_t ws_bytes, void* stream) {
    PrefillArgs a = make_args(q, k, v, log_alpha, beta, h0, cu_seqlens, n_seqs, T_total, H, dk, dv,
                              io_dtype, true, o, h_T, workspace);
    return prefill(a, ws_bytes, (cudaStream_t)stream);
}

gdn_status gdn_chunk_fwd_block_adjacent(const void* q, const void* k, const void* v,
                                        const float* log_alpha, const float* beta, const float* h0,
                                        const int32_t* cu_seqlens, int n_seqs, int64_t T_total,
                                        int H, int dk, int dv, gdn_dtype io_dtype, void* o,
                                        float* h_T, void* workspace, size_t ws_bytes,
                                        void* stream) {
    PrefillArgs a = make_args(q, k, v, log_alpha, beta, h0, cu_seqlens, n_seqs, T_total, H, dk, dv,
                              io_dtype, true, o, h_T, workspace);
    a.max_block_dist = 1;
    return prefill(a, ws_bytes, (cudaStream_t)stream);
}

gdn_status linear_attn_fwd(const void* q, const void* k, const void* v, const float* h0,
                           const int32_t* cu_seqlens, int n_seqs, int64_t T_total, int H, int dk,
                           int dv, gdn_dtype io_dtype, void* o, float* h_T, void* workspace,
                           size_t ws_bytes, void* stream) {
    PrefillArgs a = make_args(q, k, v, nullptr, nullptr, h0, cu_seqlens, n_seqs, T_total, H, dk, dv,
                              io_dtype, false, o, h_T, workspace);
    return prefill(a, ws_bytes, (cudaStream_t)stream);
}

size_t linear_attn_variant_workspace_size(int64_t T, int H, int dk, int dv, int n_seqs, gdn_dtype io,
                                          int causal, int normalize) {
    (void)normalize;
    if (!sizes_ok(T, H, dk, dv, n_seqs) || io != GDN_BF16 || dk != 128 || dv != 128) return 0;
    return align256(plan_bytes(n_seqs)) + linear_variant_extra_bytes(T, H, n_seqs, causal != 0);
}

gdn_status linear_attn_variant_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                                   int n_seqs, int64_t T_total, int H, int dk, int dv, gdn_dtype io_dtype,
                                   int causal, int normalize, void* o, float* kv, float* z, void* workspace,
                                   size_t ws_bytes, void* stream) {
    PrefillArgs a = make_args(q, k, v, nullptr, nullptr, nullptr, cu_seqlens, n_seqs, T_total, H, dk, dv,
                              io_dtype, false, o, kv, workspace);
    const size_t need = linear_attn_variant_workspace_size(T_total, H, dk, dv, n_seqs, io_dtype, causal, normalize);
    gdn_status s = check_prefill(a, ws_bytes, need, true);
    if (s != GDN_OK) return s;
    if (!linear_variant_shape_ok(a) || need == 0) return GDN_ERR_UNSUPPORTED;
    if (!aligned(z, 16)) return GDN_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    const int wl = g_wait_limit.load();
    char* plan = a.ws;
    char* extra = a.ws + align256(plan_bytes(n_seqs));
    cudaError_t e;
    if (causal) {
        e = launch_linear_grouped(a, plan, extra, normalize != 0, kv, z, wl, st);
    } else {
        e = launch_plan(cu_seqlens, n_seqs, T_total, wl, plan, st);
        if (e == cudaSuccess) e = launch_linear_bidirectional(a, plan, extra, normalize != 0, kv, z, st);
    }
    return cuda_status(e);
}

gdn_status gdn_chunk_fwd_staged(const void* q, const void* k, const void* v,
                                const float* log_alpha, const float* beta, const float* h0,
                                const int32_t* cu_seqlens, int n_seqs, int64_t T_total, int H,
                                int dk, int dv, gdn_dtype io_dtype, int delta_rule, void* o,
                                float* h_T, void* workspace, size_t ws_bytes, void* stream) {
    PrefillArgs a = make_args(q, k, v, delta_rule ? log_alpha : nullptr, delta_rule ? beta : nullptr,
                              h0, cu_seqlens, n_seqs, T_total, H, dk, dv, io_dtype, delta_rule != 0,
                              o, h_T, workspace);
    size_t need = plan_bytes(n_seqs) + staged_intermediate_bytes(T_total, H, dk, dv, n_seqs);
    gdn_status s = check_prefill(a, ws_bytes, need, true);
    if (s != GDN_OK) return s;
    return run_staged(a, (cudaStream_t)stream, nullptr, nullptr, nullptr, nullptr, true);
}

gdn_status gdn_chunk_prepare(const void* k, const void* v, const float* log_alpha,
                             const float* beta, const int32_t* cu_seqlens, int n_seqs,
                             int64_t T_total, int H, int dk, int dv, gdn_dtype io_dtype, float* g,
                             float* A, float* w, float* u, void* workspace, size_t ws_bytes,
                             void* stream) {
    PrefillArgs a = make_args(nullptr, k, v, log_alpha, beta, nullptr, cu_seqlens, n_seqs, T_total,
                              H, dk, dv, io_dtype, true, nullptr, nullptr, workspace);
    size_t need = plan_bytes(n_seqs) + staged_intermediate_bytes(T_total, H, dk, dv, n_seqs);
    gdn_status s = check_prefill(a, ws_bytes, need, false);
    if (s != GDN_OK) return s;
    if (T_total > 0 && (!w || !u)) return GDN_ERR_NULL;
    if (!aligned(g, 4) || !aligned(A, 4) || !aligned(w, 4) || !aligned(u, 4)) return GDN_ERR_ALIGN;
    return run_staged(a, (cudaStream_t)stream, g, A, w, u, false);
}

gdn_status gdn_recurrent_step(const void* q, const void* k, const void* v, const void* log_alpha,
                              const void* beta, float* state, void* o, int B, int H, int dk, int dv,
                              void* stream) {
    if (B < 0 || H < 1) return GDN_ERR_SHAPE;
    if (!head_ok(dk) || !head_ok(dv)) return GDN_ERR_UNSUPPORTED;
    if (B == 0) return GDN_OK;
    if (!q || !k || !v || !log_alpha || !beta || !state || !o) return GDN_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(state, 16) ||
        !aligned(o, 16) || !aligned(log_alpha, 2) || !aligned(beta, 2))
        return GDN_ERR_ALIGN;
    return cuda_status(launch_decode(q, k, v, log_alpha, beta, state, o, B, H, dk, dv,
                                     (cudaStream_t)stream));
}

gdn_status gdn_workspace_status(const void* workspace, void* stream, int* status) {
    if (!workspace || !status) return GDN_ERR_NULL;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaMemcpy(status, workspace, sizeof(int), cudaMemcpyDeviceToHost);
    return cuda_status(e);
}

}  // extern "C"
