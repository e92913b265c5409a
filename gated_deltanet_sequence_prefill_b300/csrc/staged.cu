// staged.cu -- the chunked prefill as three separate CUDA-core (FFMA) kernels
// with fp32 intermediates in the workspace.  This is the general path (fp32
// or bf16 I/O, dk, dv in {64, 128}) and the per-stage reference on the GPU.
//
// Stages (SparseGDN article, "Чем дорог префилл в Gated Delta Networks…"):
//   1. kkt_kernel:   g = running sum of log_alpha inside the chunk and the
//                    beta-scaled, decay-masked K K^T (A, strictly lower)
//   2. wy_kernel:    T = (I + A)^-1 by forward substitution in shared memory,
//                    w = T (beta * exp(g) * K), u = T (beta * V)
//   3. state_kernel: per (sequence, head, 32-column slice of the state), the
//                    sequential pass over chunks: v_new = u - w h,
//                    o = (q * exp(g)) h + ((q k^T) * Gamma) v_new,
//                    h <- exp(g_last) h + (k * exp(g_last - g))^T v_new
// with Gamma[i][j] = exp(g_i - g_j) for j <= i.  All decays are formed from
// differences g_i - g_j <= 0, never as exp(g_i) * exp(-g_j).
#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr int kStagedThreads = 256;
constexpr int kSlice = 32;  // state columns per block in the state pass

size_t staged_intermediate_bytes(int64_t T, int H, int dk, int dv, int n_seqs) {
    size_t g = align256(sizeof(float) * (size_t)T * H);
    size_t A = align256(sizeof(float) * (size_t)max_chunks(T, n_seqs) * H * kChunk * kChunk);
    size_t w = align256(sizeof(float) * (size_t)T * H * dk);
    size_t u = align256(sizeof(float) * (size_t)T * H * dv);
    return g + A + w + u;
}

StagedBuffers staged_buffers(char* ws, int64_t T, int H, int dk, int dv, int n_seqs) {
    char* p = ws + PlanLayout(n_seqs).end;
    StagedBuffers b;
    b.g = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * (size_t)T * H);
    b.A = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * (size_t)max_chunks(T, n_seqs) * H * kChunk * kChunk);
    b.w = reinterpret_cast<float*>(p);
    p += align256(sizeof(float) * (size_t)T * H * dk);
    b.u = reinterpret_cast<float*>(p);
    return b;
}

// Locate chunk `gc` of the plan: returns false when gc is past the last chunk.
struct ChunkPos { int seq, t0, n; };
__device__ __forceinline__ bool locate_chunk(const char* ws, int gc, ChunkPos& c) {
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return false;
    const int n_seqs = hdr->n_seqs;
    if (gc >= hdr->total_chunks) return false;
    PlanLayout L(n_seqs);
    const int* cu = reinterpret_cast<const int*>(ws + L.cu);
    const int* chunk_off = reinterpret_cast<const int*>(ws + L.chunk_off);
    c.seq = seq_of_chunk(chunk_off, n_seqs, gc);
    c.t0 = cu[c.seq] + (gc - chunk_off[c.seq]) * kChunk;
    c.n = min(kChunk, cu[c.seq + 1] - c.t0);
    return true;
}

// ---------------------------------------------------------------- stage 1
template <typename IO, int DK>
__global__ void __launch_bounds__(kStagedThreads)
kkt_kernel(const IO* __restrict__ k, const float* __restrict__ log_alpha,
           const float* __restrict__ beta, int H, const char* __restrict__ ws,
           float* __restrict__ g_out, float* __restrict__ A_out) {
    __shared__ float ks[kChunk][DK + 1];
    __shared__ float gs[kChunk];
    __shared__ float bs[kChunk];
    ChunkPos c;
    if (!locate_chunk(ws, blockIdx.x, c)) return;
    const int h = blockIdx.y, tid = threadIdx.x;

    for (int e = tid; e < kChunk * DK; e += kStagedThreads) {
        int t = e / DK, x = e % DK;
        ks[t][x] = t < c.n ? to_f32(k[((size_t)(c.t0 + t) * H + h) * DK + x]) : 0.f;
    }
    if (tid < kChunk) {
        bool ok = tid < c.n;
        gs[tid] = ok ? log_alpha[(size_t)(c.t0 + tid) * H + h] : 0.f;
        bs[tid] = ok ? beta[(size_t)(c.t0 + tid) * H + h] : 0.f;
    }
    __syncthreads();
    if (tid < 32) {  // inclusive running sum of the 64 log-gates by one warp
        float a = gs[tid], b = gs[tid + 32];
        for (int off = 1; off < 32; off <<= 1) {
            float xa = __shfl_up_sync(0xffffffffu, a, off);
            float xb = __shfl_up_sync(0xffffffffu, b, off);
            if (tid >= off) { a += xa; b += xb; }
        }
        b += __shfl_sync(0xffffffffu, a, 31);
        gs[tid] = a;
        gs[tid + 32] = b;
    }
    __syncthreads();
    if (g_out && tid < c.n) g_out[(size_t)(c.t0 + tid) * H + h] = gs[tid];

    float* A = A_out + ((size_t)blockIdx.x * H + h) * kChunk * kChunk;
    for (int e = tid; e < kChunk * kChunk; e += kStagedThreads) {
        int i = e / kChunk, j = e % kChunk;
        float val = 0.f;
        if (j < i && i < c.n) {
            float dot = 0.f;
#pragma unroll 8
            for (int x = 0; x < DK; ++x) dot = fmaf(ks[i][x], ks[j][x], dot);
            val = bs[i] * __expf(gs[i] - gs[j]) * dot;
        }
        A[e] = val;
    }
}

// ---------------------------------------------------------------- stage 2
template <typename IO, int DK, int DV>
struct WySmem {
    float A[kChunk][kChunk + 1];
    float T[kChunk][kChunk + 1];
    float kh[kChunk][DK];
    float vh[kChunk][DV];
};

template <typename IO, int DK, int DV>
__global__ void __launch_bounds__(kStagedThreads)
wy_kernel(const IO* __restrict__ k, const IO* __restrict__ v, const float* __restrict__ beta,
          int H, const char* __restrict__ ws, const float* __restrict__ g_in,
          const float* __restrict__ A_in, float* __restrict__ w_out, float* __restrict__ u_out,
          int maxd) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    WySmem<IO, DK, DV>& s = *reinterpret_cast<WySmem<IO, DK, DV>*>(smem_raw);
    ChunkPos c;
    if (!locate_chunk(ws, blockIdx.x, c)) return;
    const int h = blockIdx.y, tid = threadIdx.x;

    const float* A = A_in + ((size_t)blockIdx.x * H + h) * kChunk * kChunk;
    for (int e = tid; e < kChunk * kChunk; e += kStagedThreads) s.A[e / kChunk][e % kChunk] = A[e];
    for (int e = tid; e < kChunk * DK; e += kStagedThreads) {
        int t = e / DK, x = e % DK;
        float sc = 0.f, val = 0.f;
        if (t < c.n) {
            size_t row = (size_t)(c.t0 + t) * H + h;
            sc = beta[row] * __expf(g_in[row]);
            val = to_f32(k[row * DK + x]);
        }
        s.kh[t][x] = sc * val;
    }
    for (int e = tid; e < kChunk * DV; e += kStagedThreads) {
        int t = e / DV, y = e % DV;
        float sc = 0.f, val = 0.f;
        if (t < c.n) {
            size_t row = (size_t)(c.t0 + t) * H + h;
            sc = beta[row];
            val = to_f32(v[row * DV + y]);
        }
        s.vh[t][y] = sc * val;
    }
    __syncthreads();

    // forward substitution, one column per thread:
    // T[i][col] = [i == col] - sum_{j < i} A[i][j] T[j][col]
    if (tid < kChunk) {
        const int col = tid;
        for (int i = 0; i < kChunk; ++i) {
            float x = (i == col) ? 1.f : 0.f;
            for (int j = 0; j < i; ++j) x = fmaf(-s.A[i][j], s.T[j][col], x);
            s.T[i][col] = x;
        }
    }
    __syncthreads();

    // T[i][j] for j at most maxd 16-token blocks before row i's block (all of
    // them for the exact solve; the block-adjacent solver drops the rest)
    for (int e = tid; e < kChunk * DK; e += kStagedThreads) {
        int i = e / DK, x = e % DK;
        if (i >= c.n) continue;
        float acc = 0.f;
        for (int j = max(0, (i >> 4) - maxd) << 4; j <= i; ++j) acc = fmaf(s.T[i][j], s.kh[j][x], acc);
        w_out[((size_t)(c.t0 + i) * H + h) * DK + x] = acc;
    }
    for (int e = tid; e < kChunk * DV; e += kStagedThreads) {
        int i = e / DV, y = e % DV;
        if (i >= c.n) continue;
        float acc = 0.f;
        for (int j = max(0, (i >> 4) - maxd) << 4; j <= i; ++j) acc = fmaf(s.T[i][j], s.vh[j][y], acc);
        u_out[((size_t)(c.t0 + i) * H + h) * DV + y] = acc;
    }
}

// ---------------------------------------------------------------- stage 3
template <int DK>
struct StateSmem {
    float h[DK][kSlice];
    float q[kChunk][DK + 1];
    float k[kChunk][DK + 1];
    float w[kChunk][DK + 1];
    float P[kChunk][kChunk + 1];
    float u[kChunk][kSlice + 1];
    float vn[kChunk][kSlice + 1];
    float g[kChunk];
    float dec[kChunk];
};

template <typename IO, int DK, int DV, bool GDN>
__global__ void __launch_bounds__(kStagedThreads)
state_kernel(const IO* __restrict__ q, const IO* __restrict__ k, const IO* __restrict__ v,
             const float* __restrict__ h0, int H, const char* __restrict__ ws,
             const float* __restrict__ g_in, const float* __restrict__ w_in,
             const float* __restrict__ u_in, IO* __restrict__ o, float* __restrict__ h_T) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    StateSmem<DK>& s = *reinterpret_cast<StateSmem<DK>*>(smem_raw);
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(ws);
    if (hdr->status != GDN_OK) return;
    const int seq = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * kSlice, tid = threadIdx.x;
    const int* cu = reinterpret_cast<const int*>(ws + PlanLayout(hdr->n_seqs).cu);
    const int start = cu[seq], end = cu[seq + 1];
    const size_t hoff = ((size_t)seq * H + h) * DK * DV;

    for (int e = tid; e < DK * kSlice; e += kStagedThreads) {
        int x = e / kSlice, j = e % kSlice;
        s.h[x][j] = h0 ? h0[hoff + (size_t)x * DV + j0 + j] : 0.f;
    }

    for (int t0 = start; t0 < end; t0 += kChunk) {
        const int n = min(kChunk, end - t0);
        __syncthreads();  // previous chunk fully consumed
        for (int e = tid; e < kChunk * DK; e += kStagedThreads) {
            int t = e / DK, x = e % DK;
            bool ok = t < n;
            size_t idx = ((size_t)(t0 + t) * H + h) * DK + x;
            s.q[t][x] = ok ? to_f32(q[idx]) : 0.f;
            s.k[t][x] = ok ? to_f32(k[idx]) : 0.f;
            if (GDN) s.w[t][x] = ok ? w_in[idx] : 0.f;
        }
        for (int e = tid; e < kChunk * kSlice; e += kStagedThreads) {
            int t = e / kSlice, j = e % kSlice;
            bool ok = t < n;
            size_t idx = ((size_t)(t0 + t) * H + h) * DV + j0 + j;
            s.u[t][j] = ok ? (GDN ? u_in[idx] : to_f32(v[idx])) : 0.f;
        }
        if (tid < kChunk) s.g[tid] = (GDN && tid < n) ? g_in[(size_t)(t0 + tid) * H + h] : 0.f;
        __syncthreads();

        // P = (q k^T) * Gamma (causal, diagonal included)
        for (int e = tid; e < kChunk * kChunk; e += kStagedThreads) {
            int t = e / kChunk, r = e % kChunk;
            float val = 0.f;
            if (r <= t && t < n) {
                float dot = 0.f;
#pragma unroll 8
                for (int x = 0; x < DK; ++x) dot = fmaf(s.q[t][x], s.k[r][x], dot);
                val = GDN ? dot * __expf(s.g[t] - s.g[r]) : dot;
            }
            s.P[t][r] = val;
        }
        // v_new = u - w h   (plain linear attention: v_new = v)
        for (int e = tid; e < kChunk * kSlice; e += kStagedThreads) {
            int t = e / kSlice, j = e % kSlice;
            float acc = s.u[t][j];
            if (GDN) {
#pragma unroll 8
                for (int x = 0; x < DK; ++x) acc = fmaf(-s.w[t][x], s.h[x][j], acc);
            }
            s.vn[t][j] = t < n ? acc : 0.f;
        }
        __syncthreads();

        // o = exp(g) * (q h) + P v_new
        for (int e = tid; e < kChunk * kSlice; e += kStagedThreads) {
            int t = e / kSlice, j = e % kSlice;
            if (t >= n) continue;
            float inter = 0.f;
#pragma unroll 8
            for (int x = 0; x < DK; ++x) inter = fmaf(s.q[t][x], s.h[x][j], inter);
            float intra = 0.f;
            for (int r = 0; r <= t; ++r) intra = fmaf(s.P[t][r], s.vn[r][j], intra);
            float out = (GDN ? __expf(s.g[t]) : 1.f) * inter + intra;
            o[((size_t)(t0 + t) * H + h) * DV + j0 + j] = from_f32<IO>(out);
        }
        __syncthreads();

        // h <- exp(g_last) h + (k * exp(g_last - g))^T v_new
        const float gl = s.g[n - 1];
        if (tid < kChunk) s.dec[tid] = (GDN && tid < n) ? __expf(gl - s.g[tid]) : 1.f;
        __syncthreads();
        for (int e = tid; e < DK * kSlice; e += kStagedThreads) {
            int x = e / kSlice, j = e % kSlice;
            float acc = (GDN ? __expf(gl) : 1.f) * s.h[x][j];
            for (int r = 0; r < n; ++r) acc = fmaf(s.k[r][x] * s.dec[r], s.vn[r][j], acc);
            s.h[x][j] = acc;
        }
    }
    __syncthreads();
    if (h_T)
        for (int e = tid; e < DK * kSlice; e += kStagedThreads) {
            int x = e / kSlice, j = e % kSlice;
            h_T[hoff + (size_t)x * DV + j0 + j] = s.h[x][j];
        }
}

// ---------------------------------------------------------------- launchers
template <typename F>
static cudaError_t set_smem(F* f, size_t bytes) {
    return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename IO, int DK>
static cudaError_t kkt_t(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st) {
    dim3 grid((unsigned)max_chunks(a.T_total, a.n_seqs), a.H);
    if (grid.x == 0) return cudaSuccess;
    kkt_kernel<IO, DK><<<grid, kStagedThreads, 0, st>>>((const IO*)a.k, a.log_alpha, a.beta, a.H,
                                                        a.ws, b.g, b.A);
    return cudaGetLastError();
}

cudaError_t launch_kkt(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st) {
    if (a.io == GDN_BF16) return a.dk == 64 ? kkt_t<__nv_bfloat16, 64>(a, b, st) : kkt_t<__nv_bfloat16, 128>(a, b, st);
    return a.dk == 64 ? kkt_t<float, 64>(a, b, st) : kkt_t<float, 128>(a, b, st);
}

template <typename IO, int DK, int DV>
static cudaError_t wy_t(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st) {
    dim3 grid((unsigned)max_chunks(a.T_total, a.n_seqs), a.H);
    if (grid.x == 0) return cudaSuccess;
    size_t sm = sizeof(WySmem<IO, DK, DV>);
    cudaError_t e = set_smem(wy_kernel<IO, DK, DV>, sm);
    if (e != cudaSuccess) return e;
    wy_kernel<IO, DK, DV><<<grid, kStagedThreads, sm, st>>>((const IO*)a.k, (const IO*)a.v, a.beta,
                                                            a.H, a.ws, b.g, b.A, b.w, b.u,
                                                            a.max_block_dist);
    return cudaGetLastError();
}

template <typename IO>
static cudaError_t wy_io(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st) {
    if (a.dk == 64) return a.dv == 64 ? wy_t<IO, 64, 64>(a, b, st) : wy_t<IO, 64, 128>(a, b, st);
    return a.dv == 64 ? wy_t<IO, 128, 64>(a, b, st) : wy_t<IO, 128, 128>(a, b, st);
}

cudaError_t launch_wy(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st) {
    return a.io == GDN_BF16 ? wy_io<__nv_bfloat16>(a, b, st) : wy_io<float>(a, b, st);
}

template <typename IO, int DK, int DV, bool GDN>
static cudaError_t state_t(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st) {
    dim3 grid(a.n_seqs, a.H, DV / kSlice);
    size_t sm = sizeof(StateSmem<DK>);
    cudaError_t e = set_smem(state_kernel<IO, DK, DV, GDN>, sm);
    if (e != cudaSuccess) return e;
    state_kernel<IO, DK, DV, GDN><<<grid, kStagedThreads, sm, st>>>(
        (const IO*)a.q, (const IO*)a.k, (const IO*)a.v, a.h0, a.H, a.ws, b.g, b.w, b.u, (IO*)a.o,
        a.h_T);
    return cudaGetLastError();
}

template <typename IO, bool GDN>
static cudaError_t state_io(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st) {
    if (a.dk == 64) return a.dv == 64 ? state_t<IO, 64, 64, GDN>(a, b, st) : state_t<IO, 64, 128, GDN>(a, b, st);
    return a.dv == 64 ? state_t<IO, 128, 64, GDN>(a, b, st) : state_t<IO, 128, 128, GDN>(a, b, st);
}

cudaError_t launch_state_ffma(const PrefillArgs& a, const StagedBuffers& b, cudaStream_t st) {
    if (a.n_seqs == 0) return cudaSuccess;
    if (a.io == GDN_BF16)
        return a.delta_rule ? state_io<__nv_bfloat16, true>(a, b, st) : state_io<__nv_bfloat16, false>(a, b, st);
    return a.delta_rule ? state_io<float, true>(a, b, st) : state_io<float, false>(a, b, st);
}

}  // namespace gdn
