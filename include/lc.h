/*
 * lc.h -- attention-matching compaction of one layer's KV cache on one GPU.
 *
 * For each KV head the library runs five steps over the reference queries Q
 * of every query head that shares that KV head (context-prefill queries):
 *
 *  1. full statistics: S = scale * Q K^T, row max m, log mass lse and output
 *     O = softmax(S) V  ("Latent Compaction with Test-Time Training", §3
 *     Preliminaries, Eq. (1));
 *  2. key score: u_j = max_i (S_ij - lse_i), the log of the largest attention
 *     probability key j receives (same paper, §3.2, Eq. (6));
 *  3. selection: the t keys with the highest score, ties to the lower index,
 *     returned in ascending order ("KV compaction" blog, section "Fast KV
 *     Compaction via Attention Matching": C_k is the set of keys with the
 *     highest attention and is a subset of K);
 *  4. biases: w = exp(beta) >= 0 minimising
 *     sum_i (sum_j exp(s q_i.C_kj + beta_j - m_i) - exp(lse_i - m_i))^2,
 *     the mass-matching equation of the same blog section solved as
 *     non-negative least squares in per-query max-shifted form;
 *  5. values: C_v minimising sum_i || softmax_j(s q_i.C_kj + beta_j) C_v - O_i ||^2,
 *     the output-matching equation solved as ordinary least squares (biased
 *     compact attention as in "Latent Compaction ...", §3.1 Eq. (2)-(3)).
 *
 * Conventions shared by every entry point
 *  - Tensors are device pointers owned by the caller; the library never
 *    allocates or frees caller memory.  Scratch memory is a caller-provided
 *    device workspace of at least lc_workspace_bytes() bytes (256-byte
 *    aligned).  Host-side state lives in an lc_handle.
 *  - Layouts are row-major and dense: Q [H][n_q][d], K and V [H][T][d],
 *    rowmax and lse [H][n_q], O [H][n_q][d], u [H][T], idx [H][t],
 *    w and beta [H][t], Cv [H][t][d].  Row g*T + p of a head's Q is query
 *    head g of the group at position p (any order works: queries are a set).
 *  - Q, K, V are bfloat16 (in_dtype LC_BF16, d = 64 or 128) or float32
 *    (LC_FP32, d = 64 only).  All other floating-point tensors are float32;
 *    idx is int32.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.  An error found on the host is
 *    returned at once and nothing is enqueued.  Outcomes found on the device
 *    (an NNLS or solver iteration cap, a singular system, a timed-out wait)
 *    are recorded per head and read back with lc_get_report().
 *  - Outputs are finite except beta_j = -inf where w_j = 0 (key j keeps a
 *    zero weight, so it never receives attention).
 *  - Two kept keys with equal vectors (value for value, -0 = +0) give equal
 *    columns of the mass system, whose minimiser is then not unique: the
 *    copy at the later position of idx gets w = 0 and keeps its own value
 *    row, the minimiser an active-set method reaches when ties in its choice
 *    of index go to the lower index.
 *  - A handle may be used by one host thread at a time; calls that share a
 *    workspace must not overlap on the device.
 */
#ifndef LC_H_
#define LC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LC_OK = 0,
  LC_ERR_INVALID_ARG = 1,    /* bad pointer, size or shape */
  LC_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. d = 96) */
  LC_ERR_WORKSPACE = 3,      /* workspace too small or misaligned */
  LC_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
  LC_ERR_NOT_CONVERGED = 5,  /* NNLS hit its iteration cap (outputs finite) */
  LC_ERR_SINGULAR = 6,       /* a Cholesky factorisation of an n x n system
                                broke down (a pivot that is not positive); a
                                ridge of n * 2^-20 * mean(diag) was added once
                                and the outputs are that ridge solution's */
  LC_ERR_TIMEOUT = 7         /* a device-side wait gave up (internal error) */
} lc_status;

typedef enum { LC_BF16 = 0, LC_FP32 = 1 } lc_dtype;

typedef struct {
  int n_kv_heads;     /* H >= 1 */
  int n_q;            /* reference queries per KV head (G*T for context prefill), >= 1 */
  int T;              /* cached keys per head, >= 1 */
  int d;              /* head dimension: 64 or 128 */
  int t;              /* keys kept per head, 1 <= t <= min(T, 1024) */
  int in_dtype;       /* lc_dtype of Q, K and V */
  float scale;        /* softmax scale; 0 selects 1/sqrt(d) */
  int nnls_max_iter;  /* NNLS iteration cap; 0 selects 3*t */
} lc_shape;

typedef struct lc_context* lc_handle;

/* Create a handle bound to CUDA device `device`.  Allocates the handle's own
 * per-head report buffers (a few KB) on that device. */
lc_status lc_create(lc_handle* out, int device);
lc_status lc_destroy(lc_handle h);

/* Workspace bytes that lc_compact_layer / lc_full_attn_stats / lc_key_scores
 * / lc_fit_only need for `shape` (the largest of the four). */
lc_status lc_workspace_bytes(const lc_shape* shape, size_t* bytes);

/* Step 1.  rowmax, lse: [H][n_q] (natural-log units, scale applied);
 * O: [H][n_q][d].  Any of the three outputs may be NULL to skip it. */
lc_status lc_full_attn_stats(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                             const void* V, float* rowmax, float* lse, float* O, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Step 2 given the log masses: u [H][T] = max_i (scale*q_i.k_j - lse_i). */
lc_status lc_key_scores(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                        const float* lse, float* u, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Step 3 on given scores: idx [n_heads][t], ascending; the t largest of each
 * row of u [n_heads][T]; equal scores go to the lower index; -0 == +0.
 * Scores must not be NaN. */
lc_status lc_select_topt(lc_handle h, int n_heads, int T, int t, const float* u, int32_t* idx,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Step 3 for callers that cannot allocate device memory or pass a workspace
 * (for example code under a memory planner that forbids allocation on the
 * serving path).  No counterpart on the pages: this is a deployment variant
 * of lc_select_topt with identical results.  Its scratch is a fixed array of
 * LC_NOALLOC_MAX_SCORES 32-bit codes (4 MiB) compiled into the library, held
 * on every GPU that loads it until the process exits.  Works on the current
 * CUDA device; the first call on a device looks up the array's address and
 * should come before any stream capture.  The address is kept per device
 * with the ID of the context it belongs to; after the device's context is
 * reset (cudaDeviceReset) the next call looks it up again, and that call too
 * belongs before any capture.  n_heads*T above
 * LC_NOALLOC_MAX_SCORES returns LC_ERR_UNSUPPORTED and enqueues nothing.
 * Calls that overlap on the GPU share the array and race: serialise them.
 * No cudaMalloc, cudaFree or allocating library call is made. */
#define LC_NOALLOC_MAX_SCORES (1 << 20)
lc_status lc_select_topt_noalloc(int n_heads, int T, int t, const float* u, int32_t* idx,
                                 void* stream);

/* Steps 4-5 for given selected keys and full statistics (rowmax, lse, O as
 * produced by lc_full_attn_stats).  idx entries must be distinct and in
 * [0, T).  Outputs w, beta [H][t] and Cv [H][t][d]. */
lc_status lc_fit_only(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                      const void* V, const int32_t* idx, const float* rowmax, const float* lse,
                      const float* O, float* w, float* beta, float* Cv, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Steps 1-5.  Outputs idx [H][t], w, beta [H][t], Cv [H][t][d]. */
lc_status lc_compact_layer(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                           const void* V, int32_t* idx, float* w, float* beta, float* Cv,
                           void* workspace, size_t workspace_bytes, void* stream);

/* lc_compact_layer on HOST buffers: copies Q, K, V to the device workspace,
 * runs the five steps, copies idx, w, beta, Cv back, and synchronises
 * `stream`.  Host buffers should be page-locked for full copy bandwidth.
 * Needs lc_host_workspace_bytes() bytes of device workspace. */
lc_status lc_host_workspace_bytes(const lc_shape* shape, size_t* bytes);
lc_status lc_compact_layer_host(lc_handle h, const lc_shape* shape, const void* Q_host,
                                const void* K_host, const void* V_host, int32_t* idx_host,
                                float* w_host, float* beta_host, float* Cv_host,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Fast compaction of one layer without the full score matrix ("KV
 * compaction" blog: "Attempt #3: Two-Pass", "Choosing beta" -- uniform
 * redistribution -- and "Choosing C_v" -- direct selection).
 *   1. the query subset Q' (qsel[h][0..n_sub), row indices 0 <= r < n_q of
 *      head h; the random draw is the caller's) scores every key under full
 *      attention, u'_j = max_{i in Q'} (s q_i.k_j - lse_i);
 *   2. the min(k t, T) best keys form the shortlist K';
 *   3. every query scores the shortlist normalised over the shortlist,
 *      u_j = max_i (s q_i.k'_j - lse'_i), lse'_i = log sum_{l in K'} e^{s q_i.k'_l};
 *      the t best are C_k (idx, ascending; ties to the lower index);
 *   4. beta_j = log((m_j + Delta/t) / m_j) with m_j = mean_i e^{s q_i.c_j} and
 *      Delta = mean_i (sum_{K'} e^{s q_i.k'} - sum_{C_k} e^{s q_i.c}) over all
 *      n_q queries (no fit);
 *   5. Cv = V[idx] (fp32).
 * bf16 inputs only (LC_ERR_UNSUPPORTED otherwise); 1 <= n_sub <= n_q, k >= 1.
 * short_out [H][min(k t, T)] receives the shortlist if not NULL.  All
 * pointers are device pointers; the workspace has
 * lc_fast_workspace_bytes(shape, n_sub, k) bytes, 256-byte aligned. */
lc_status lc_fast_workspace_bytes(const lc_shape* shape, int n_sub, int k, size_t* bytes);
lc_status lc_compact_layer_fast(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                                const void* V, const int32_t* qsel, int n_sub, int k,
                                int32_t* idx, float* beta, float* Cv, int32_t* short_out,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Attention of queries over a compacted cache plus tokens appended after it
 * ("Latent Compaction with Test-Time Training", §3.1 "Handling Subsequent
 * Tokens", Eq. (4)-(5), and Appendix A.2): per KV head h and query row r,
 *   A = (Z_cmp A_cmp + Z_new A_new) / (Z_cmp + Z_new),
 * the compacted branch with logits scale q.Ck_j + beta_j over the entries
 * with finite beta_j, the appended branch with logits scale q.Knew_m over
 * m < n_vis[h][r] (no bias); log_z = log(Z_cmp + Z_new) (-inf and A = 0 for
 * a row that sees nothing).
 *   q [H][n][d], Ck [H][t][d], Knew, Vnew [H][n_new][d]: bfloat16;
 *   beta [H][t], Cv [H][t][d]: float32; n_vis [H][n] int32 (NULL: every row
 *   sees all n_new appended tokens); outputs A [H][n][d] and log_z [H][n]
 *   (NULL allowed) float32.  d = 64 or 128; scale <= 0 means 1/sqrt(d).
 *   Knew and Vnew may be NULL when n_new = 0.  Device pointers; no
 *   workspace. */
lc_status lc_compact_attention(lc_handle h, int n_heads, int n, int t, int n_new, int d,
                               float scale, const void* q, const void* Ck, const float* beta,
                               const float* Cv, const void* Knew, const void* Vnew,
                               const int32_t* n_vis, float* A, float* log_z, void* stream);

/* Quality of a compaction on held-out queries ("KV compaction" blog,
 * "Choosing beta" and "Choosing C_v": mass and attention-output
 * reconstruction errors).  shape->n_q is the number of held-out query rows
 * Qh [H][n_q][d] (bfloat16 only), shape->t the compacted size; the compacted
 * cache is (K[idx], beta, Cv) as lc_compact_layer returns it.  Per head:
 *   mass_err[h] = mean_r |log Z_cmp(q_r) - log Z_full(q_r)|,
 *   out_err[h]  = mean_r ||A_cmp(q_r) - A_full(q_r)||_2,
 * the full-cache side from step 1 over all T keys, the compacted side from
 * lc_compact_attention with no appended tokens.  Outputs are device float32
 * [H]; the workspace has lc_heldout_workspace_bytes(shape) bytes. */
lc_status lc_heldout_workspace_bytes(const lc_shape* shape, size_t* bytes);
lc_status lc_heldout_errors(lc_handle h, const lc_shape* shape, const void* Qh, const void* K,
                            const void* V, const int32_t* idx, const float* beta,
                            const float* Cv, float* mass_err, float* out_err, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Diversifier selection by farthest-first traversal ("Latent Compaction with
 * Test-Time Training", §3.2 Eq. (7), after Gonzalez 1985): per head, starting
 * from the seed set S (seeds[h][0..n_seed), e.g. the anchors), repeatedly add
 *   i* = argmax_{i not in S} min_{j in S} ||k_i - k_j||^2
 * until |S| = M; ties go to the lower index.  K [H][T][d] bfloat16 (d = 64 or
 * 128), seeds int32 (valid, distinct; an index outside [0, T) is ignored),
 * out [H][M - n_seed] int32: the added keys in the order chosen (-1 past the
 * point where no key is left).  1 <= n_seed <= M <= T.  Distances are fp32.
 * Device pointers; no workspace. */
lc_status lc_farthest_first(lc_handle h, int n_heads, int T, int d, const void* K,
                            const int32_t* seeds, int n_seed, int M, int32_t* out, void* stream);

/* The Attention Matching baseline variant ("Latent Compaction with Test-Time
 * Training", Appendix A.3): steps 1-5 with
 *  - step 2 as RMS attention: u_j = log sqrt((1/n_q) sum_i p_ij^2),
 *    p_ij = exp(S_ij - lse_i), top t as in step 3;
 *  - step 4 as bounded least squares, w in [e^-3, e^3]: each iteration
 *    solves the mass system over the free weights with the pinned ones at
 *    their bounds, then pins every free weight outside the box at the bound
 *    it crossed; shape->nnls_max_iter iterations (0 = two, the page's
 *    setting), from all-free, stopping early when nothing is pinned;
 *  - step 5 unchanged (every w_j > 0, so every key takes part).
 * bfloat16 inputs only.  Outputs and report as lc_compact_layer; the
 * workspace has lc_baseline_workspace_bytes(shape) bytes.
 * lc_key_scores_rms is the RMS step alone (lse [H][n_q] given, u [H][T]). */
lc_status lc_baseline_workspace_bytes(const lc_shape* shape, size_t* bytes);
lc_status lc_compact_layer_baseline(lc_handle h, const lc_shape* shape, const void* Q,
                                    const void* K, const void* V, int32_t* idx, float* w,
                                    float* beta, float* Cv, void* workspace,
                                    size_t workspace_bytes, void* stream);
lc_status lc_key_scores_rms(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                            const float* lse, float* u, void* workspace, size_t workspace_bytes,
                            void* stream);

/* lc_compact_layer for n_layers layers stored one after another (Q
 * [L][H][n_q][d], K and V [L][H][T][d], idx [L][H][t], w and beta [L][H][t],
 * Cv [L][H][t][d]) in one call, pipelined across layers: the latency-bound
 * solves of layer l (steps 4-5, a CTA per head) run on a second stream of
 * the handle while steps 1-3 and the mass system of layer l + 1 fill the
 * rest of the GPU.  Two workspaces alternate between layers
 * (lc_layers_workspace_bytes).  Results equal separate lc_compact_layer
 * calls; the report (lc_get_report with n_heads = L*H, L*H <= 4096) holds
 * every layer's per-head outcome in layer order.  Returns once the work is
 * enqueued; `stream` waits for all of it. */
lc_status lc_layers_workspace_bytes(const lc_shape* shape, int n_layers, size_t* bytes);
lc_status lc_compact_layers(lc_handle h, const lc_shape* shape, int n_layers, const void* Q,
                            const void* K, const void* V, int32_t* idx, float* w, float* beta,
                            float* Cv, void* workspace, size_t workspace_bytes, void* stream);

/* Per-head outcome of the last lc_fit_only / lc_compact_layer on this handle:
 * head_status[H] (lc_status values), nnls_iters[H] and device error bits.
 * Synchronises `stream`.  Any pointer may be NULL. */
lc_status lc_get_report(lc_handle h, int n_heads, int32_t* head_status, int32_t* nnls_iters,
                        uint32_t* device_error_bits, void* stream);

/* Per-kernel timing of this handle's own launches: with profiling on, every
 * launch is bracketed by CUDA events on the call's stream (a few
 * microseconds each).  lc_profile_read() waits for the recorded events, fills
 * up to max_kernels entries -- names (32 chars each, NUL-terminated),
 * total milliseconds and launch counts, grouped by kernel name -- sets
 * *n_kernels to the number of distinct names, and clears the totals. */
lc_status lc_profile_enable(lc_handle h, int on);
lc_status lc_profile_read(lc_handle h, int max_kernels, char* names, double* total_ms,
                          int32_t* launches, int* n_kernels);

const char* lc_status_string(lc_status s);

#ifdef __cplusplus
}
#endif

#endif /* LC_H_ */
