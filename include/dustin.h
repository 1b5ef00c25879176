/*
 * dustin.h -- C-ABI of the GB300 (sm_103a) library for Dustin's
 * draft-augmented sparse verification hot path.
 *
 * Sources of the operations (cited by page title and section):
 *   [Paper]  "Dustin: Draft-Augmented Sparse Verification for Efficient
 *            Long-Context Generation with Speculative Decoding"
 *            (arXiv 2606.24957, HTML translation), section 3.1 Eq. (1)-(4).
 *   [Notes]  "dustin-long-context" paper notes: section 2.2 (S_Draft,
 *            S_Target, one global index set, Fig. 5), section 2.3
 *            (I_verify = sink + window + draft top-m + target rest),
 *            section 2.4 (SRH: scoring on a few (layer, head) pairs, Fig. 6),
 *            section 3 (Fig. 7 self-attention speedup against full cache).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library keeps no reference after the call returns and allocates
 *     no device memory.  Scratch space, where a call needs it, is passed by
 *     the caller as (ws, ws_bytes), sized by the matching *_workspace_size
 *     query for the current device.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (uint16), row-major, with
 *     the innermost (head-dim) axis contiguous.  Base pointers and row
 *     strides must be 16-byte aligned.
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL
 *     is the legacy default stream) and returns a dustin_status.  Arguments
 *     are validated on the host before anything is launched: an invalid call
 *     launches nothing.  A failed launch returns DUSTIN_ERR_CUDA with the
 *     CUDA error text in dustin_last_error().  Nothing is thrown across the
 *     ABI and no kernel traps.
 *   - Device-side checks (an index >= n, a page id outside the pool) never
 *     fault: the offending position is left out of the attention and a flag
 *     is raised, read with dustin_device_status().  Every wait inside a
 *     kernel is bounded (about one second); one that gives up raises
 *     DUSTIN_DEVFLAG_WAIT_TIMEOUT and the kernel returns.
 *   - Grouped-query attention: query head h reads kv head h / (h_q / h_kv).
 */
#ifndef DUSTIN_H_
#define DUSTIN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dustin_status {
  DUSTIN_OK = 0,
  DUSTIN_ERR_INVALID_ARG = 1, /* NULL pointer where one is needed, bad enum */
  DUSTIN_ERR_SHAPE = 2,       /* sizes inconsistent or out of range         */
  DUSTIN_ERR_UNSUPPORTED = 3, /* valid but not built (e.g. d not 64 / 128)  */
  DUSTIN_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than required    */
  DUSTIN_ERR_ALIGNMENT = 5,   /* pointer or stride not 16-byte aligned      */
  DUSTIN_ERR_CUDA = 6,        /* a CUDA runtime call failed                 */
  DUSTIN_ERR_DEVICE = 7       /* a device-side check raised a flag          */
} dustin_status;

/* Device-side flags reported by dustin_device_status(). */
#define DUSTIN_DEVFLAG_INDEX_RANGE 0x1u /* idx[b][i] < 0 or >= n            */
#define DUSTIN_DEVFLAG_PAGE_RANGE 0x2u  /* page id < 0 or >= num_pages      */
#define DUSTIN_DEVFLAG_WAIT_TIMEOUT 0x4u /* a pipeline wait gave up (~1 s);
                                            the outputs of that call are void */

#define DUSTIN_NORM_NONE 0 /* hybrid mix of the raw score vectors          */
#define DUSTIN_NORM_L1 1   /* each score vector divided by its own sum     */

/*
 * One layer's KV cache for one (layer) of the target or the draft.
 *
 * Contiguous layout (page_table == NULL): element (b, kv head h, position
 * j, dim c) is at  base + b*stride_b + h*stride_h + j*stride_n + c.
 * Paged layout (page_table != NULL): a pool of pages [page][h_kv][page_size]
 * [d]; position j of sequence b lives in page
 * p = page_table[b*pages_per_seq + j/page_size] at
 * base + p*stride_b + h*stride_h + (j % page_size)*stride_n + c, so stride_b
 * is then the stride between pages.  page_table is a device int32 array.
 * page_size is a positive multiple of 16 (scoring reads pages of 16, 32 or
 * 64 positions as one TMA box each; other sizes take a cp.async path).
 * v may be NULL for calls that read keys only (scoring).
 * Strides are in elements; every stride must be a multiple of 8 (16 bytes).
 */
typedef struct dustin_kv {
  const void* k;
  const void* v;
  int64_t stride_b;
  int64_t stride_h;
  int64_t stride_n;
  const int32_t* page_table;
  int32_t page_size;
  int32_t pages_per_seq;
  int32_t num_pages;
} dustin_kv;

/* Text for a status code (static storage, never NULL). */
const char* dustin_status_string(int status);

/* Detail of the last failing call on this host thread ("" if none). */
const char* dustin_last_error(void);

/* Library ABI version: major*10000 + minor*100 + patch. */
int dustin_version(void);

/* Number of kernels this library has launched in this process. */
uint64_t dustin_launch_count(void);

/*
 * Reads and clears the device-side flags (DUSTIN_DEVFLAG_*) of the current
 * device.  Synchronises the device.  Returns DUSTIN_ERR_DEVICE if any flag
 * was set, DUSTIN_OK otherwise; *flags (may be NULL) receives the flags.
 */
int dustin_device_status(uint32_t* flags);

/*
 * Self-test of the bounded wait that every pipeline wait of the library
 * uses: launches one CTA of 32 threads on `stream` that waits on an
 * mbarrier no thread ever arrives at, with a limit of `limit_cycles` SM
 * clock cycles (1 .. 2^31; about 2 * 10^9 inside the compute calls).  The
 * wait gives up, raises DUSTIN_DEVFLAG_WAIT_TIMEOUT and the kernel returns:
 * the context stays usable.  Returns DUSTIN_ERR_SHAPE for a limit outside
 * that range, DUSTIN_ERR_CUDA if the launch fails, DUSTIN_OK otherwise.
 */
int dustin_wait_selftest(int64_t limit_cycles, void* stream);

/* ------------------------------------------------------------------------
 * Importance scoring on the scored (layer, head) pairs.
 *
 * [Notes] section 2.2: S_Draft sums the draft's attention over its heads,
 * layers and Gamma lookahead queries; S_Target sums the target's attention
 * of its latest token over its heads and layers.  [Notes] section 2.4
 * (Fig. 6): only the selected (layer, head) pairs are recomputed.
 *
 *   s_out[b][j] = sum_{p < n_pairs} sum_{r < rows}
 *                 softmax_j( scale * q[p][b][r] . K_p[b][kv_head[p]][j] )
 * over history positions j in [0, n); fp32 out, fp32 accumulation.
 *
 *   q        bf16 [n_pairs][b][rows][d], device
 *   kv       host array [n_pairs]: the key cache of pair p's layer (v unused)
 *   kv_head  host array [n_pairs]: kv head of pair p (q_head / group)
 *   s_out    fp32 [b][n], device, fully overwritten
 *   ws       device scratch of dustin_score_heads_workspace_size() bytes
 * Called once for the target (rows = 1) and once for the draft
 * (rows = Gamma).  Limits: d in {64, 128}; 1 <= rows <= 16;
 * 1 <= n_pairs <= 64; n_pairs * rows <= 1024.
 * b == 0 or n == 0 is a no-op.
 */
size_t dustin_score_heads_workspace_size(int b, int n, int n_pairs, int rows);
int dustin_score_heads(int b, int n, int d, int n_pairs, int rows,
                       const void* q, const dustin_kv* kv,
                       const int32_t* kv_head, float scale, float* s_out,
                       void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Scoring without a caller-provided workspace.  The paper has no
 * counterpart: this is a convenience of this library.
 *
 * For callers that cannot allocate device memory when they score -- for
 * example a serving loop that has given all of HBM to the KV cache (a
 * cudaMalloc there fails or stalls the step), or a plugin whose framework
 * owns the allocator and hands over only inputs and outputs.  Same inputs,
 * outputs and limits as dustin_score_heads, but the scratch lives in a fixed
 * array of DUSTIN_NOALLOC_SCRATCH_BYTES compiled into the library (every GPU
 * that loads the library keeps it until the process exits).  The call
 * allocates nothing.
 *   - A call whose scratch (dustin_score_heads_workspace_size) exceeds the
 *     array is rejected with DUSTIN_ERR_WORKSPACE before anything runs.
 *   - The argument checks of dustin_score_heads run first (same statuses);
 *     then a call whose scratch (dustin_score_heads_workspace_size) exceeds
 *     the array is rejected with DUSTIN_ERR_WORKSPACE before anything runs.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is remembered per device and
 *     CUDA context: after cudaDeviceReset the next call looks it up again
 *     (again outside any capture).
 *   - All calls share the one array, which keeps the last call's contents.
 *     Each call overwrites every scratch byte it reads, so nothing needs
 *     clearing, but calls that overlap on the GPU (other streams, other
 *     threads) race on the array: serialise them.
 */
#define DUSTIN_NOALLOC_SCRATCH_BYTES (64u << 20)
int dustin_score_heads_noalloc(int b, int n, int d, int n_pairs, int rows,
                               const void* q, const dustin_kv* kv,
                               const int32_t* kv_head, float scale,
                               float* s_out, void* stream);
/* Size in bytes of that built-in array (DUSTIN_NOALLOC_SCRATCH_BYTES of the
 * library as built), for callers that plan around it at run time. */
size_t dustin_score_heads_noalloc_capacity(void);

/* ------------------------------------------------------------------------
 * Hybrid combination and global per-sequence Top-K ([Notes] sections 2.2
 * and 2.3).  One index set per sequence, shared by all layers and heads.
 *
 * Protected positions [0, n_sink) and [n - n_recent, n) are always kept;
 * k counts them.  The remaining budget r = k - |protected| is filled from
 * the other positions:
 *   m < 0  (alpha mode): top-r of c_j = a_D*S_D[j] + a_T*S_T[j], where
 *          a_D = alpha / sum(S_D) and a_T = (1 - alpha) / sum(S_T) under
 *          DUSTIN_NORM_L1 (alpha and 1 - alpha under DUSTIN_NORM_NONE).
 *          Sums in fp64, coefficients rounded once to fp32, then
 *          c_j = fl(fl(a_D*S_D[j]) + fl(a_T*S_T[j])) in fp32 round-to-nearest.
 *          A term with weight 0 or a NULL vector is left out.  A sum that is
 *          not positive and finite leaves that vector unscaled.
 *   m >= 0 (budget split): top-min(m, r) of S_D, then the top of S_T for the
 *          rest of the budget over the positions not yet taken.
 * Order: higher score first, ties to the lower position; -0 equals +0; NaN
 * ranks below every number.  idx rows come out strictly ascending.
 * k >= n keeps all n positions (idx row length n).
 *
 *   s_draft, s_target  fp32 [b][n], device; either may be NULL (not both)
 *   idx                int32 [b][min(k, n)], device, fully overwritten
 * Errors: |protected| > k with k < n is DUSTIN_ERR_SHAPE.  n <= 2^20.
 */
int dustin_hybrid_topk(int b, int n, int k, int n_sink, int n_recent,
                       double alpha, int m, int norm, const float* s_draft,
                       const float* s_target, int32_t* idx, void* stream);

/* ------------------------------------------------------------------------
 * Sparse verification attention ([Notes] section 2.2 Fig. 5, Stage 2: the
 * target verifies its w window rows over the selected KV only).
 *
 * For each sequence b, query head h and window row t (no causal mask: all
 * selected history precedes the window; the window's own causal block is
 * merged by the caller through lse):
 *   o[b][h][t]   = softmax_i(scale * q[b][h][t] . K[b][g][idx[b][i]]) V[..]
 *   lse[b][h][t] = log sum_i exp(scale * q[b][h][t] . K[b][g][idx[b][i]])
 * with g = h / (h_q / h_kv).  k == 0 gives o = 0, lse = -inf.
 *
 *   q    bf16 [b][h_q][w][d], device (contiguous)
 *   kv   host pointer to one dustin_kv (k and v both required)
 *   idx  int32 [b][k], device, each entry in [0, n); ascending order is
 *        fastest but not required
 *   o    bf16 [b][h_q][w][d], device;  lse fp32 [b][h_q][w] (natural log)
 *   ws   device scratch of dustin_sparse_verify_attn_workspace_size() bytes
 *        (may be 0 bytes; ws may then be NULL)
 *   flags  0, or DUSTIN_ATTN_KV_READY (below)
 * Limits: d in {64, 128}; h_q a multiple of h_kv; k <= n; scale finite and
 * > 0; flags has no other bit set (DUSTIN_ERR_INVALID_ARG).
 */
size_t dustin_sparse_verify_attn_workspace_size(int b, int h_q, int h_kv,
                                                int d, int w, int k);
int dustin_sparse_verify_attn(int b, int h_q, int h_kv, int d, int w, int n,
                              int k, const void* q, const dustin_kv* kv,
                              const int32_t* idx, float scale, void* o,
                              float* lse, void* ws, size_t ws_bytes,
                              unsigned flags, void* stream);

/* The same with the window's own causal block merged in (the w window
 * tokens follow the history, so window row t also attends to window
 * positions 0..t, as in ordinary causal decoding):
 *   o[b][h][t] = softmax over [idx[b][0..k), window 0..t] of scale * q . K
 *   lse        = log sum exp over the same positions
 * where the window part reads win (k and v both required, contiguous, no
 * page table): bf16 [b][h_kv][w][d] through win->stride_b/h/n.  Same
 * workspace as dustin_sparse_verify_attn.  With DUSTIN_ATTN_KV_READY the
 * window rows, like q, are read only after the preceding kernel finished.
 * (The sparse call's LSE lets a caller merge this block itself; this entry
 * point does it inside the same launch, as one more tile of w rows.) */
int dustin_sparse_verify_attn_window(int b, int h_q, int h_kv, int d, int w,
                                     int n, int k, const void* q,
                                     const dustin_kv* kv, const int32_t* idx,
                                     const dustin_kv* win, float scale, void* o,
                                     float* lse, void* ws, size_t ws_bytes,
                                     unsigned flags, void* stream);

/* Sparse verification attention of n_layers layers in one persistent
 * launch: for each layer l, the call dustin_sparse_verify_attn(b, h_q, h_kv,
 * d, w, n, k, q[l], &kv[l], idx, scale, o[l], lse[l]) with one index set
 * for all layers.  For callers that hold several layers' queries at once
 * (the layers of one model run one after another, so within a single
 * forward pass only one layer is ready at a time).  The (layer, sequence,
 * kv head, row block) units are dealt round-robin to one CTA per SM, which
 * streams them back to back without draining its pipeline.
 *   q, o, lse  host arrays [n_layers] of device pointers (as in the sparse
 *              call); kv host array [n_layers] of descriptors, all paged or
 *              all contiguous
 *   flags      0 or DUSTIN_ATTN_KV_READY (accepted, no effect)
 * No workspace.  Limits as the sparse call, and k <= 2048
 * (DUSTIN_ERR_UNSUPPORTED); any number of layers (launches of up to 128).
 * Not an API of the paper. */
int dustin_sparse_verify_attn_layers(int n_layers, int b, int h_q, int h_kv, int d,
                                     int w, int n, int k, const void* const* q,
                                     const dustin_kv* kv, const int32_t* idx,
                                     float scale, void* const* o, float* const* lse,
                                     unsigned flags, void* stream);

/* ------------------------------------------------------------------------
 * Quest page scoring: the page-level baseline selector of the comparison
 * ([Notes] section 1 and related work; "Quest-16" in Fig. 8).  Not part of
 * Dustin; for measurements beside it.
 *
 * dustin_quest_page_stats: per page of `page` consecutive positions (the
 * last may be short), the channel-wise minimum and maximum of the keys:
 *   stats bf16 [b][h_kv][P][2][d], P = ceil(n / page), minimum row first;
 *   dustin_quest_stats_size() bytes, 16-byte aligned.
 * kv: keys only (v unused), contiguous or paged.  In Quest the statistics
 * are kept up to date as tokens are appended, not rebuilt every step.
 *
 * dustin_quest_page_scores: for one query row per head, q bf16 [b][h_q][d],
 *   scores[b][h][p] = sum_c max(q[b][h][c] * min_c, q[b][h][c] * max_c)
 * with the stats of kv head h / (h_q / h_kv): the largest q . k over the
 * page's channel box.  scores fp32 [b][h_q][P].  The top pages per (b, h)
 * come from dustin_hybrid_topk on scores viewed as b*h_q rows of P (alpha
 * 1, s_target NULL, norm NONE, no protected positions).
 * At most 64 query heads per kv head. */
size_t dustin_quest_stats_size(int b, int h_kv, int d, int n, int page);
int dustin_quest_page_stats(int b, int h_kv, int d, int n, int page,
                            const dustin_kv* kv, void* stats, void* stream);
int dustin_quest_page_scores(int b, int h_q, int h_kv, int d, int n, int page,
                             const void* q, const void* stats, float* scores,
                             void* stream);

/* DUSTIN_ATTN_KV_READY: the caller guarantees that idx, the page table and
 * the K/V cache were complete before the kernel enqueued just before this
 * call on `stream` started (that kernel does not write them; q may be its
 * output).  The attention kernels are launched with programmatic dependent
 * launch and may then gather their first K/V tiles while that kernel is
 * still running; q is read, and o, lse and ws are written, only after it
 * has finished.  This holds, for example, for consecutive layers'
 * verification attention over one index set whose K/V were appended
 * before the step.  Without the flag nothing is read early.  A wrong
 * promise gives stale rows, never a fault.  Not an API of the paper: a
 * launch-overlap hint. */
#define DUSTIN_ATTN_KV_READY 1u

/* ------------------------------------------------------------------------
 * Full-cache verification attention: the dense in-run baseline ([Notes]
 * section 3, Fig. 7 "Full Cache").  The sparse call over idx = 0..n-1;
 * flags as there (DUSTIN_ATTN_KV_READY: the page table and K/V).
 */
size_t dustin_full_verify_attn_workspace_size(int b, int h_q, int h_kv,
                                              int d, int w, int n);
int dustin_full_verify_attn(int b, int h_q, int h_kv, int d, int w, int n,
                            const void* q, const dustin_kv* kv, float scale,
                            void* o, float* lse, void* ws, size_t ws_bytes,
                            unsigned flags, void* stream);
/* The full-cache call with the window's causal block merged in, as
 * dustin_sparse_verify_attn_window.  dustin_full_verify_attn_workspace_size
 * covers both. */
int dustin_full_verify_attn_window(int b, int h_q, int h_kv, int d, int w, int n,
                                   const void* q, const dustin_kv* kv,
                                   const dustin_kv* win, float scale, void* o,
                                   float* lse, void* ws, size_t ws_bytes,
                                   unsigned flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DUSTIN_H_ */
