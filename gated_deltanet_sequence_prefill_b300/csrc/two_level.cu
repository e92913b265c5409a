// two_level.cu -- the two-level state scan for long sequences with few
// (sequence, head) chains.
//
// A chunk acts on the state as an affine map, h -> M_c h + B_c (SparseGDN
// article, "Схема встраивания селектора…": the chunk update S -> A_c S + B_c),
// so a run of chunks is one such map too, and a long sequence can be cut into
// G segments that are handled side by side:
//   1. plan:   every sequence is cut into G segments of whole chunks; the
//              segments become the "sequences" of the runs below;
//   2. maps:   the cluster prefill kernel runs over all segments twice without
//              storing o: with v = 0 and h0 = I its final state is the
//              segment's M (dk x dk), with h0 = 0 it is the segment's B
//              (dk x dv) (linear attention has M = I and skips this run);
//   3. scan:   per (sequence, head), in segment order,
//                  h_start(0) = h0,  h_start(s + 1) = M_s h_start(s) + B_s,
//              and the sequence's final state h_T = h_start(G);
//   4. output: the cluster kernel runs over all segments once more from
//              h_start, storing o.
// The per-chunk work is done three times (twice for linear attention) instead
// of once, in exchange for G-fold shorter chains; the host takes this path
// only when the ordinary call would leave most SMs idle (see
// two_level_segments).  Everything stays in the caller's workspace.
#include <stdlib.h>

#include "common.cuh"
#include "launch.h"

namespace gdn {

int sm_count();

namespace {

constexpr int kD = 128;            // dk = dv of the cluster kernel
constexpr int kScanCols = 16;      // state columns per scan block
constexpr int kScanThreads = 256;
constexpr size_t kStateBytes = sizeof(float) * kD * kD;

size_t up1k(size_t x) { return (x + 1023) & ~(size_t)1023; }

// Workspace: [main header | segment cu_seqlens | inner workspace of the runs
// (plan and cluster scratch) | M | B | h_start], each part at a 1 KB boundary.
struct TwoLevelLayout {
    size_t seg_cu, inner, M, B, hstart, end;
    TwoLevelLayout(int n_seqs, int H, int G) {
        const size_t n_seg = (size_t)n_seqs * G;
        seg_cu = up1k(sizeof(WsHeader));
        inner = seg_cu + up1k(sizeof(int) * (n_seg + 1));
        M = inner + up1k(pair_workspace_bytes((int)n_seg, H));
        B = M + n_seg * H * kStateBytes;
        hstart = B + n_seg * H * kStateBytes;
        end = hstart + n_seg * H * kStateBytes;
    }
};

// Validates the caller's cu_seqlens (as the plan kernel does) into the main
// header and cuts every sequence into G segments of whole chunks: segment s
// of a sequence of n chunks takes chunks [s n / G, (s + 1) n / G).
__global__ void __launch_bounds__(1024)
segment_plan_kernel(const int32_t* __restrict__ cu_in, int n_seqs, long long T_total, int G,
                    char* __restrict__ ws, int* __restrict__ seg_cu) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    __shared__ int s_bad;
    const int tid = threadIdx.x;
    if (tid == 0) s_bad = 0;
    __syncthreads();
    for (int i = tid; i <= n_seqs; i += blockDim.x) {
        const long long c = cu_in ? (long long)cu_in[i] : (i == 0 ? 0 : T_total);
        bool bad = (i == 0 && c != 0) || (i == n_seqs && c != T_total) || c < 0 || c > T_total;
        if (i > 0 && cu_in) bad |= cu_in[i] < cu_in[i - 1];
        if (bad) atomicOr(&s_bad, 1);
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    for (int i = tid; i < n_seqs; i += blockDim.x) {
        const int a = bad ? 0 : (cu_in ? cu_in[i] : 0);
        const int e = bad ? 0 : (cu_in ? cu_in[i + 1] : (int)T_total);
        const int nch = (e - a + kChunk - 1) / kChunk;
        for (int s = 0; s < G; ++s) {
            const long long c0 = (long long)s * nch / G;
            seg_cu[(size_t)i * G + s] = (int)min((long long)e, a + c0 * kChunk);
        }
    }
    if (tid == 0) {
        seg_cu[(size_t)n_seqs * G] = bad ? 0 : (int)T_total;
        hdr->status = bad ? GDN_ERR_SEQLENS : GDN_OK;
        hdr->counter = 0;
        hdr->n_seqs = n_seqs;
        hdr->timeout_site = 0;
    }
}

// h_start(s) for every segment and the final state, per (sequence, head, 16
// state columns): h <- M_s h + B_s in fp32, segment by segment (M = I when
// M is NULL).  Skipped when the runs so far have failed.
__global__ void __launch_bounds__(kScanThreads)
segment_scan_kernel(const char* __restrict__ inner_ws, int G, int H, const float* __restrict__ h0,
                    const float* __restrict__ M, const float* __restrict__ B,
                    float* __restrict__ hstart, float* __restrict__ h_T) {
    if (reinterpret_cast<const WsHeader*>(inner_ws)->status != GDN_OK) return;
    __shared__ __align__(16) float Ms[kD][kD / 2 + 4];  // half of M's columns at a time
    __shared__ float hs[kD][kScanCols];
    const int unit = blockIdx.x, seq = unit / H, head = unit % H;
    const int col0 = blockIdx.y * kScanCols;
    const int tid = threadIdx.x;
    const int r = tid >> 1, c0 = (tid & 1) * 8;  // this thread: row r, columns c0 .. c0 + 7
    for (int x = tid; x < kD * kScanCols; x += kScanThreads) {
        const int i = x / kScanCols, j = x % kScanCols;
        hs[i][j] = h0 ? h0[((size_t)seq * H + head) * kD * kD + (size_t)i * kD + col0 + j] : 0.f;
    }
    __syncthreads();
    for (int s = 0; s < G; ++s) {
        const size_t base = (((size_t)seq * G + s) * H + head) * kD * kD;
        for (int x = tid; x < kD * kScanCols; x += kScanThreads) {
            const int i = x / kScanCols, j = x % kScanCols;
            hstart[base + (size_t)i * kD + col0 + j] = hs[i][j];
        }
        __syncthreads();
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = B[base + (size_t)r * kD + col0 + c0 + j];
        if (M) {
#pragma unroll 1
            for (int kh = 0; kh < 2; ++kh) {
                for (int x = tid; x < kD * kD / 8; x += kScanThreads) {
                    const int i = x / (kD / 8), j4 = x % (kD / 8);
                    *reinterpret_cast<float4*>(&Ms[i][4 * j4]) =
                        *reinterpret_cast<const float4*>(M + base + (size_t)i * kD + kh * (kD / 2) + 4 * j4);
                }
                __syncthreads();
#pragma unroll 4
                for (int k = 0; k < kD / 2; ++k) {
                    const float m = Ms[r][k];
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = fmaf(m, hs[kh * (kD / 2) + k][c0 + j], acc[j]);
                }
                __syncthreads();
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += hs[r][c0 + j];
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 8; ++j) hs[r][c0 + j] = acc[j];
        __syncthreads();
    }
    if (h_T) {
        for (int x = tid; x < kD * kScanCols; x += kScanThreads) {
            const int i = x / kScanCols, j = x % kScanCols;
            h_T[((size_t)seq * H + head) * kD * kD + (size_t)i * kD + col0 + j] = hs[i][j];
        }
    }
}

// The call's status: the caller's cu_seqlens check, else whatever the runs
// reported (a wait that ran out), with the barrier it gave up on.
__global__ void finalize_status_kernel(char* ws, const char* inner_ws) {
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    const WsHeader* in = reinterpret_cast<const WsHeader*>(inner_ws);
    if (hdr->status == GDN_OK && in->status != GDN_OK) {
        hdr->status = in->status;
        hdr->timeout_site = in->timeout_site;
    }
}

}  // namespace

// Segments per sequence: G is about 37 / chains + 1, capped at 16 (so that each
// run of the scan has roughly 37 to 74 clusters of two SMs), lowered until the
// sequences average at least 32 chunks per segment; the two-level path is
// taken for the cluster kernel's shapes (exact solve) only when that leaves
// G >= 5.  The scan does each chunk's work three times, so with fewer
// segments it cannot win (measured on B300: 16 chains of 32768 tokens took
// 1.69 ms cut in 3 segments against 0.84 ms in one pass, while 4 chains of
// 131072 tokens took 1.16 ms in 10 segments against 3.24 ms).
// GDN_TWO_LEVEL=0 in the environment disables the path; GDN_TWO_LEVEL=G
// (2 .. 64) forces G segments whenever the shapes allow it.
int two_level_segments(const PrefillArgs& a) {
    if (!pair_shape_ok(a) || a.max_block_dist != 3 || a.n_seqs <= 0 || a.T_total <= 0) return 1;
    const char* e = getenv("GDN_TWO_LEVEL");
    if (e != nullptr && e[0] != '\0') {
        const int g = atoi(e);
        return (g >= 2 && g <= 64) ? g : 1;
    }
    const long long units = (long long)a.n_seqs * a.H;
    if (units > 37) return 1;
    const long long avg_chunks = a.T_total / a.n_seqs / kChunk;
    int G = (int)(37 / units) + 1;
    if (G > 16) G = 16;
    while (G >= 5 && avg_chunks < 32LL * G) --G;
    return G >= 5 ? G : 1;
}

size_t two_level_workspace_bytes(int n_seqs, int H, int G) {
    return TwoLevelLayout(n_seqs, H, G).end;
}

cudaError_t launch_two_level(const PrefillArgs& a, int G, int wait_limit, cudaStream_t st) {
    const TwoLevelLayout L(a.n_seqs, a.H, G);
    int* seg_cu = reinterpret_cast<int*>(a.ws + L.seg_cu);
    char* inner = a.ws + L.inner;
    float* Mb = reinterpret_cast<float*>(a.ws + L.M);
    float* Bb = reinterpret_cast<float*>(a.ws + L.B);
    float* Hs = reinterpret_cast<float*>(a.ws + L.hstart);
    const int n_seg = a.n_seqs * G;

    segment_plan_kernel<<<1, 1024, 0, st>>>(a.cu_seqlens, a.n_seqs, (long long)a.T_total, G, a.ws, seg_cu);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        e = launch_plan(seg_cu, n_seg, a.T_total, wait_limit, inner, st, reinterpret_cast<const int*>(a.ws));

    PrefillArgs r = a;  // the runs: the segments are their sequences
    r.cu_seqlens = seg_cu;
    r.n_seqs = n_seg;
    r.ws = inner;
    const int fronts = pair_fronts(r);
    if (e == cudaSuccess && a.delta_rule) {  // transition maps M
        PrefillArgs m = r;
        m.v = a.v;  // only its tensor map is built; v is taken as zero
        m.h0 = nullptr;
        m.h_T = Mb;
        m.o = nullptr;
        m.mode = 1 | 2 | 4;
        e = launch_pair(m, fronts, st);
    }
    if (e == cudaSuccess) {  // offsets B
        PrefillArgs b = r;
        b.h0 = nullptr;
        b.h_T = Bb;
        b.o = nullptr;
        b.mode = 1;
        e = launch_pair(b, fronts, st);
    }
    if (e == cudaSuccess) {
        dim3 grid((unsigned)(a.n_seqs * a.H), kD / kScanCols);
        segment_scan_kernel<<<grid, kScanThreads, 0, st>>>(inner, G, a.H, a.h0, a.delta_rule ? Mb : nullptr,
                                                            Bb, Hs, a.h_T);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) {  // outputs from the segment starts
        PrefillArgs c = r;
        c.h0 = Hs;
        c.h_T = nullptr;
        c.mode = 0;
        e = launch_pair(c, fronts, st);
    }
    if (e == cudaSuccess) {
        finalize_status_kernel<<<1, 1, 0, st>>>(a.ws, inner);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace gdn
