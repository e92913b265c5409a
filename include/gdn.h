/*
 * gdn.h -- C ABI of the B300 (sm_103a) gated-delta-rule / linear-attention
 * library libgdn_b300.so.
 *
 * The operation (the gated delta rule, "GDN"), per sequence and head:
 *     S_t = a_t * S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t
 * with a_t = exp(log_alpha_t) and b_t = beta_t.  GatedDeltaNet is named among
 * the gated linear-attention variants in the forpes.ru survey of linear
 * attention (section "Введение"; its update table was lost in extraction);
 * the plain rule S_t = S_{t-1} + v_t k_t^T is printed in "Как ускорить LLM на
 * длинном контексте" (section "Linear attention").  Prefill is evaluated chunk
 * by chunk as the SparseGDN article describes ("Чем дорог префилл в Gated
 * Delta Networks…"): an intra-chunk delta-system solve, a sequential per-head
 * pass over chunks, and each chunk's outputs from the state at its start.
 *
 * Conventions shared by every entry point
 *  - Device pointers unless stated otherwise.  The caller owns every buffer;
 *    the library never allocates device memory (it only sets kernel
 *    attributes once per process).
 *  - Token-major packed layout: q, k [T_total][H][dk], v, o [T_total][H][dv],
 *    log_alpha, beta [T_total][H].  Sequences are delimited by cu_seqlens
 *    (int32, device, n_seqs + 1 entries, cu[0] = 0, non-decreasing,
 *    cu[n_seqs] = T_total).  cu_seqlens == NULL means one sequence of
 *    T_total tokens (n_seqs must then be 1).  Zero-length sequences are
 *    allowed: their final state is their initial state.
 *  - The state is stored transposed, h = S^T, as fp32 [n_seqs][H][dk][dv]
 *    row-major.  h0 == NULL means a zero initial state; h_T == NULL skips
 *    the final-state write.
 *  - o_t uses the state after token t's update.  q is not scaled by
 *    1/sqrt(dk): callers pre-scale it if they want that.
 *  - Supported head sizes: dk, dv in {64, 128}; anything else returns
 *    GDN_ERR_UNSUPPORTED.  There is no CPU fallback.
 *  - All calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  The returned status reports argument errors
 *    (checked on the host, nothing is launched then) and launch errors.
 *    Errors found on the device (a malformed cu_seqlens, a device wait that
 *    ran out) are written to a status word in the workspace, read with
 *    gdn_workspace_status() after the stream's work completes; when it is
 *    non-zero the outputs of that call are unspecified.
 *  - Alignment: q, k, v, o, h0, h_T, state must be 16-byte aligned;
 *    log_alpha, beta 4-byte; the workspace 256-byte.
 *  - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef GDN_B300_H
#define GDN_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL = -1,        /* a required pointer is NULL */
    GDN_ERR_ALIGN = -2,       /* a pointer is not aligned as required */
    GDN_ERR_SHAPE = -3,       /* negative or inconsistent sizes */
    GDN_ERR_SEQLENS = -4,     /* cu_seqlens malformed (device-detected) */
    GDN_ERR_DTYPE = -5,       /* unknown io dtype */
    GDN_ERR_UNSUPPORTED = -6, /* head size or dtype combination not built */
    GDN_ERR_WORKSPACE = -7,   /* workspace NULL or smaller than the query */
    GDN_ERR_CUDA = -8,        /* a CUDA runtime call or launch failed */
    GDN_ERR_TIMEOUT = -9      /* a bounded device-side wait ran out */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_FP32 = 1 } gdn_dtype;

/* Message for a status code (static string, never NULL). */
GDN_API const char *gdn_status_string(int status);

/* Library build identifier: "<version> sm_103a". */
GDN_API const char *gdn_version(void);

/*
 * Workspace bytes needed by gdn_chunk_fwd for these sizes (0 on bad sizes).
 * The bf16 path with dk = dv = 128 keeps every intermediate on-chip or in L2:
 * it needs a small scheduling area plus 192 KB per (sequence, head) through
 * which the solve SM of each cluster hands its per-chunk tiles to the state
 * SM (n_seqs * H * 196608 bytes, rounded up to a 1 KB boundary after the
 * scheduling area); other combinations run the staged path and need
 * gdn_staged_workspace_size() bytes.  The same holds for
 * linear_attn_fwd_workspace_size().
 */
GDN_API size_t gdn_chunk_fwd_workspace_size(int64_t T_total, int H, int dk, int dv, int n_seqs,
                                    gdn_dtype io_dtype);

/*
 * GDN prefill (forward).  Inputs q, k, v in io_dtype; log_alpha (<= 0) and
 * beta in fp32; outputs o in io_dtype and h_T fp32.  Sections of the
 * SparseGDN article: "Чем дорог префилл в Gated Delta Networks…" (three
 * cost sources: intra-chunk solve, sequential chunk pass, chunk-start states)
 * and "Селектор бюджета по парам голов и компактные снапшоты…" (outputs are
 * produced for every token).  Chunk size 64; chunks restart at every
 * sequence start and the last chunk of a sequence may be partial.
 * For bf16 with dk = dv = 128 the call runs one fused kernel that puts each
 * (sequence, head) on a cluster of one or two solve SMs and one state SM (two
 * when 3 x n_seqs x H <= the SM count; GDN_PREFILL_FRONTS=1 or =2 in the
 * environment forces it); GDN_PREFILL_PAIR=0 selects the kernel with one CTA
 * per (sequence, head, 64-column half of the state) instead (same results up
 * to rounding).
 */
GDN_API gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *log_alpha, const float *beta, const float *h0,
                         const int32_t *cu_seqlens, int n_seqs, int64_t T_total, int H,
                         int dk, int dv, gdn_dtype io_dtype, void *o, float *h_T,
                         void *workspace, size_t ws_bytes, void *stream);

/*
 * Long sequences with few (sequence, head) chains: the two-level state scan.
 * A chunk acts on the state as an affine map h -> M h + B (SparseGDN
 * article, "Схема встраивания селектора…"), and so does a run of chunks.
 * When a gdn_chunk_fwd / linear_attn_fwd call of the cluster kernel's shapes
 * (bf16, dk = dv = 128) has few chains (at most 9) and sequences long
 * enough for at least 5 segments of 32 chunks, it
 * cuts every sequence into G segments of whole chunks, forms every segment's
 * map in parallel (two extra passes over the segments, without outputs; one
 * for linear attention, whose M is the identity), composes the maps in
 * segment order into each segment's starting state and the final state, and
 * then computes the outputs of all segments in parallel.  The result is the
 * same as the one-pass evaluation up to rounding; the workspace query
 * includes the extra space.  gdn_prefill_segments() returns the G a call of
 * these sizes takes (1: the one-pass evaluation; 0: bad sizes).  In the
 * environment, GDN_TWO_LEVEL=0 turns the scan off and GDN_TWO_LEVEL=G
 * (2..64) forces G segments for the shapes that support it.
 */
GDN_API int gdn_prefill_segments(int64_t T_total, int H, int dk, int dv, int n_seqs,
                                 gdn_dtype io_dtype, int delta_rule);

/*
 * GDN prefill with the block-adjacent solver of the SparseGDN article
 * ("Двухуровневая разреженность SparseGDN…", first observation: the
 * intra-chunk delta-system solve is restricted to links between
 * neighbouring blocks, a fixed, input-independent approximation).  Each
 * 64-token chunk is split into four blocks of 16 tokens; the inverse
 * (I + A)^-1 of the delta system is formed exactly on the diagonal blocks
 * and on the blocks right below them and taken as zero two or more blocks
 * away (the rest of the computation is unchanged).  The result is an
 * approximation of gdn_chunk_fwd's; its deviation depends on the input.
 * Same arguments, layouts, workspace query (gdn_chunk_fwd_workspace_size)
 * and error rules as gdn_chunk_fwd.
 */
GDN_API gdn_status gdn_chunk_fwd_block_adjacent(const void *q, const void *k, const void *v,
                                        const float *log_alpha, const float *beta,
                                        const float *h0, const int32_t *cu_seqlens, int n_seqs,
                                        int64_t T_total, int H, int dk, int dv,
                                        gdn_dtype io_dtype, void *o, float *h_T, void *workspace,
                                        size_t ws_bytes, void *stream);

/*
 * Plain causal linear attention S_t = S_{t-1} + v_t k_t^T, o_t = S_t q_t
 * ("Как ускорить LLM на длинном контексте", section "Linear attention"; the
 * reassociated evaluation order of "За пределами self-attention", section
 * "Линейное внимание…").  No gates, no delta term, no normaliser, causal.
 * Same layouts and rules as gdn_chunk_fwd.  For bf16 with dk = dv = 128 the
 * chain is cut into groups of chunks: each group's sum of k^T v, a prefix over
 * the groups (h0 first) for each group's starting state, then every group's
 * outputs from its own start, all groups side by side.  Small calls (every
 * (sequence, head) resident, at most 40 chunks per SM) do this in one
 * cooperative launch whose CTAs hand their sums to each other through
 * bounded waits on counters in the workspace.  The result equals the
 * sequential evaluation up to rounding.  GDN_LINEAR_GROUPED_FORM=fused or
 * =unfused overrides the size rule; GDN_LINEAR_PATH=cluster runs the
 * sequential kernels of gdn_chunk_fwd instead.
 */
GDN_API size_t linear_attn_fwd_workspace_size(int64_t T_total, int H, int dk, int dv, int n_seqs,
                                      gdn_dtype io_dtype);
GDN_API gdn_status linear_attn_fwd(const void *q, const void *k, const void *v, const float *h0,
                           const int32_t *cu_seqlens, int n_seqs, int64_t T_total, int H,
                           int dk, int dv, gdn_dtype io_dtype, void *o, float *h_T,
                           void *workspace, size_t ws_bytes, void *stream);

/*
 * Linear attention, causal or bidirectional, with or without the normaliser
 * (bf16 q, k, v, o; dk = dv = 128; other combinations return
 * GDN_ERR_UNSUPPORTED):
 *     o_t = sum_s (q_t . k_s) v_s  [ / sum_s (q_t . k_s) ],
 * s over all tokens of t's sequence (causal = 0) or over s <= t (causal = 1).
 * The bidirectional, normalised form is the listing of "За пределами
 * self-attention…" (section "Линейное внимание…": K^T V and the summed keys
 * first, then q_t times each); the bidirectional mode and the causal
 * restriction are the two modes of the ai-vestnik.ru item on linear
 * attention (HSE / VK students).  Feature maps (elu + 1 on the page) are the
 * caller's: q and k are used as given; no epsilon is added to the normaliser,
 * so normalised calls need q_t . sum k_s != 0 (positive features give that).
 * No initial state.  Optional fp32 outputs (NULL to skip, 16-byte aligned):
 * kv [n_seqs][H][dk][dv] = sum_t k_t v_t^T over each sequence (h = S^T of the
 * final state), z [n_seqs][H][dk] = sum_t k_t.  Bidirectional calls run a
 * tcgen05 reduction of K^T V over groups of chunks and a tcgen05 apply pass;
 * causal calls run the grouped evaluation of linear_attn_fwd, whose output
 * MMA also yields the normaliser q_t . (sum of k_s, s <= t) (the running key
 * sum rides as extra rows of the state operand, a column of ones after v).
 * kv and z of a causal call are the final state and key sum.  Workspace: the
 * query below; status word at its offset 0, as for the other calls.
 */
GDN_API size_t linear_attn_variant_workspace_size(int64_t T_total, int H, int dk, int dv, int n_seqs,
                                          gdn_dtype io_dtype, int causal, int normalize);
GDN_API gdn_status linear_attn_variant_fwd(const void *q, const void *k, const void *v,
                                   const int32_t *cu_seqlens, int n_seqs, int64_t T_total, int H,
                                   int dk, int dv, gdn_dtype io_dtype, int causal, int normalize,
                                   void *o, float *kv, float *z, void *workspace, size_t ws_bytes,
                                   void *stream);

/*
 * One decode token of the gated delta rule for B sequences x H heads, the
 * state updated in place: S <- a S + b (v - a S k) k^T, o = S q (the same
 * rule as above for a single t; O(1) state per step as in "Как ускорить LLM
 * на длинном контексте", section "Linear attention").
 * q, k [B][H][dk], v [B][H][dv], log_alpha, beta [B][H], o [B][H][dv] are
 * bf16; state is fp32 [B][H][dk][dv] (h = S^T), read and written once.
 * No workspace; errors are argument errors or launch errors only.
 */
GDN_API gdn_status gdn_recurrent_step(const void *q, const void *k, const void *v,
                              const void *log_alpha, const void *beta, float *state, void *o,
                              int B, int H, int dk, int dv, void *stream);

/*
 * Staged prefill: the three chunk stages as separate kernels with their
 * intermediates in the workspace (fp32 g, A, w, u) -- gate cumsum and
 * decay-masked K K^T; (I + A)^-1 by forward substitution and w, u; the
 * state pass with outputs.  Same contract as gdn_chunk_fwd /
 * linear_attn_fwd (delta_rule = 1 / 0; log_alpha and beta are ignored and
 * may be NULL when delta_rule = 0).  Any supported dtype and head size.
 */
GDN_API size_t gdn_staged_workspace_size(int64_t T_total, int H, int dk, int dv, int n_seqs,
                                 gdn_dtype io_dtype);
GDN_API gdn_status gdn_chunk_fwd_staged(const void *q, const void *k, const void *v,
                                const float *log_alpha, const float *beta, const float *h0,
                                const int32_t *cu_seqlens, int n_seqs, int64_t T_total, int H,
                                int dk, int dv, gdn_dtype io_dtype, int delta_rule, void *o,
                                float *h_T, void *workspace, size_t ws_bytes, void *stream);

/*
 * The intra-chunk stages alone (SparseGDN article, "Чем дорог префилл…": the
 * first cost source), writing their fp32 results to caller buffers:
 *   g  [T_total][H]        running sum of log_alpha within each chunk
 *   A  [n_chunks][H][64][64]  b_i exp(g_i - g_j) (k_i . k_j) for j < i, else 0
 *   w  [T_total][H][dk]    (I + A)^-1 (b * exp(g) * K)
 *   u  [T_total][H][dv]    (I + A)^-1 (b * V)
 * where chunks are numbered sequence by sequence (n_chunks = sum over
 * sequences of ceil(L_s / 64)); rows of A past a partial chunk's end are 0.
 * Any of g, A may be NULL; w and u may not.  Workspace: the staged query.
 */
GDN_API gdn_status gdn_chunk_prepare(const void *k, const void *v, const float *log_alpha,
                             const float *beta, const int32_t *cu_seqlens, int n_seqs,
                             int64_t T_total, int H, int dk, int dv, gdn_dtype io_dtype,
                             float *g, float *A, float *w, float *u, void *workspace,
                             size_t ws_bytes, void *stream);

/*
 * Staged prefill for callers that cannot allocate device memory (no paper
 * counterpart: this is a packaging variant of gdn_chunk_fwd_staged).  Some
 * callers cannot call cudaMalloc -- code running inside a stream capture or
 * a host callback, allocators that own all device memory, or plug-in hosts
 * that hand out only input and output buffers -- so this entry point takes
 * no workspace.  Its scratch is one fixed array of GDN_STATIC_SCRATCH_BYTES
 * in the library's device memory; every GPU that loads the library holds it
 * until the process exits.  The caller still passes inputs and outputs.
 *  - Same arguments and results as gdn_chunk_fwd_staged, without workspace.
 *  - Returns GDN_ERR_WORKSPACE, launching nothing, when the problem needs
 *    more scratch than that (gdn_staged_workspace_size(...) bytes).
 *  - The first call on each device looks up the array's device address
 *    (with that device current), and so does the first call after a
 *    cudaDeviceReset (which recreates the context and the array); make that
 *    first call before any stream capture.
 *  - Every call shares the one array, which keeps the last call's contents;
 *    the call re-initialises what it reads before reading it.  Calls that
 *    overlap on the GPU (two streams, two threads) race on the array.
 *  - device_status (device pointer, may be NULL) receives the call's device
 *    status word (GDN_OK or GDN_ERR_SEQLENS) once the stream reaches it.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define GDN_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
GDN_API gdn_status gdn_chunk_fwd_staged_static(const void *q, const void *k, const void *v,
                                       const float *log_alpha, const float *beta,
                                       const float *h0, const int32_t *cu_seqlens, int n_seqs,
                                       int64_t T_total, int H, int dk, int dv,
                                       gdn_dtype io_dtype, int delta_rule, void *o, float *h_T,
                                       int *device_status, void *stream);

/*
 * Waits for `stream`, then reads the device status word of a workspace used
 * by one of the calls above into *status (GDN_OK or a negative gdn_status).
 */
GDN_API gdn_status gdn_workspace_status(const void *workspace, void *stream, int *status);

/*
 * Failure detection (no paper counterpart).  Every wait inside the fused
 * prefill kernels (one SM waiting for another's copy, MMA or hand-off) is
 * bounded: after `polls` unsuccessful polls of its barrier it gives up, the
 * call's status word becomes GDN_ERR_TIMEOUT, and every CTA of the call
 * skips its remaining work (still completing the copies it already issued
 * and releasing its tensor memory) and exits, leaving the context usable.
 *  - gdn_set_wait_limit(polls) sets the bound for calls launched afterwards,
 *    process-wide, and returns the previous one.  The default is 4194304
 *    (1 << 22); polls < 0 restores it; polls = 0 makes every bounded wait
 *    that finds its barrier incomplete at its first poll give up at once
 *    (used by the tests to exercise the timeout path).  The outputs of a
 *    call that timed out are unspecified.
 *  - gdn_workspace_timeout_site() waits for `stream`, then reads which
 *    barrier the first timed-out wait of the call gave up on (0: none;
 *    1000 + index on a solve CTA, 2000 + index on a state CTA of the cluster
 *    kernel, 3000 in the single-SM kernel), for diagnosis.
 */
GDN_API int gdn_set_wait_limit(int polls);
GDN_API gdn_status gdn_workspace_timeout_site(const void *workspace, void *stream, int *site);

#ifdef __cplusplus
}
#endif

#endif /* GDN_B300_H */
