// Kernel parameter blocks and host-side launch entry points.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace lc {

// Which operand encoding the tensor-core passes use.
//  kBF16d128 / kBF16d64: Q, K bf16 with d_qk = d; V converted to fp16 (exact
//      for bf16 values in the fp16 range) and P rounded to fp16: one P.V
//      product (moves C_v by ~1e-5..1e-4 relative at 2x or more compression);
//      below 2x compression P is split into fp16 hi + lo (two products).
//  kSplitF16d64: fp32 inputs; Q = [Qhi|Qlo|Qhi], K = [Khi|Khi|Klo] as fp16
//      (d_qk = 3d = 192) so S keeps fp32 accuracy; V = Vhi + Vlo.
enum OperandMode { kBF16d128 = 0, kBF16d64 = 1, kSplitF16d64 = 2 };

struct AttnStatsParams {
  int n_q, T, n_q_pad;
  float scale_log2;        // softmax scale * log2(e)
  float* rowmax;           // [H][n_q], natural-log units; may be null
  float* lse;              // [H][n_q]; may be null
  float* rowmax_pad;       // [H][n_q_pad], +inf in padded rows; may be null
  float* lse_pad;          // [H][n_q_pad], +inf in padded rows; may be null
  float* O;                // [H][n_q][d_v] fp32; may be null
  __half* O_hi;            // [H][n_q][d_v] fp16 hi/lo pair; may be null
  __half* O_lo;
  uint32_t* err;
};

struct KeyScoreParams {
  int n_q_pad, T;
  int tiles_per_split;     // query tiles handled by one CTA (blockIdx.z range)
  float scale;             // softmax scale (natural-log units)
  const float* lse_pad;    // [H][n_q_pad], +inf padding
  uint32_t* u_code;        // [H][T] order codes, atomicMax-merged (pre-zeroed)
  int n_rows;              // mass mode: real query rows (later rows carry no mass)
  float2* part;            // mass mode: [nsplit][H][T] base-2 (max, sum) per split
  uint32_t* err;
};

// Gram builder: for key blocks (bi, bj), bi <= bj, of 128 selected keys, over
// the query rows r of the CTA's split:
//   E_jr = 2^(s2 * S_jr + colb2_j - rowsh2_r),  S = Kc q^T (scores)
//   G[bi,bj] += E_bi E_bj^T   (hi/lo split, three products)
//   c[bi]    += E_bi b         (diagonal blocks, when row_b != null)
//   R[bi]    += E_bi O         (diagonal blocks, when O maps given)
//
// The tensor core adds each product into its fp32 accumulator with
// truncation, so a long chain of additions drifts low: about 2.6e-7 of the
// sum per query slab summed (three products of four k-steps each), 2e-4
// after 2048 slabs.  One accumulator therefore sums at most kGramChain
// slabs.  The per-block kernels hold two in tensor memory: the first
// chunk's becomes the CTA's running sum, and each later chunk, summed in
// the second, is added into it (fp32, round to nearest, tensor memory to
// registers and back) before the next chunk starts.  The launches whose
// tensor memory has no room for the second take at least
// gram_min_split(slabs) query splits, reduced afterwards in fp32.
constexpr int kGramChain = 64;  // power of two
inline int gram_min_split(int slabs) { return (slabs + kGramChain - 1) / kGramChain; }

struct GramParams {
  int n_q_pad, n_q;
  int t_pad;
  int nblk;                // t_pad / 128
  int slabs_per_split;     // 64-row query slabs per CTA
  float scale_log2;
  const float* rowsh2;     // [H][n_q_pad]; +inf padding zeroes the row
  const float* row_b;      // [H][n_q_pad] or null
  const float* colb2;      // [H][t_pad]; -inf for unused keys
  float* Gpart;            // [nsplit][H][t_pad][t_pad]
  float* cpart;            // [nsplit][H][t_pad] or null
  float* Rpart;            // [nsplit][H][t_pad][d_v] or null
  int d_v;
  int r_only;              // launch holds only the R CTAs (blockIdx.x = key block)
  uint32_t* err;
};

// Compact log mass per query: lc2_r = log2 sum_j 2^(s2 * S_rj + colb2_j).
// Key splits (blockIdx.z): with key_stride > t_pad, CTA z takes keys
// [z t_pad, (z + 1) t_pad) of key_stride padded keys (colb2 rows have
// key_stride entries) and writes its base-2 (max, sum) per query to part
// instead of lc2_pad; merge_row_lse combines the splits.
struct CompactLseParams {
  int n_q, n_q_pad, t_pad;
  float scale_log2;
  const float* colb2;      // [H][key_stride or t_pad]
  float* lc2_pad;          // [H][n_q_pad], +inf padding
  uint32_t* err;
  int key_stride;          // 0: t_pad (no split)
  float2* part;            // [nsplit][H][n_q_pad] or null
};

// Launchers (return cudaGetLastError()).
// split_p: P.V as fp16 hi + lo products (bf16 inputs; fp32 inputs always
// split).  Needed when more than half of the keys are kept: the output fit
// is then close to an interpolation and amplifies P's fp16 rounding.
cudaError_t launch_attn_stats(OperandMode mode, bool split_p, const CUtensorMap& mQ,
                              const CUtensorMap& mK, const CUtensorMap& mV,
                              const CUtensorMap& mVlo, const AttnStatsParams& p, int H,
                              cudaStream_t st);
cudaError_t launch_key_scores(OperandMode mode, const CUtensorMap& mK, const CUtensorMap& mQ,
                              const KeyScoreParams& p, int H, int nsplit, cudaStream_t st);
// Key scores plus each key's column log mass in the same pass (bf16 modes):
// per query split, p.part = (max_i b_ij, sum_i 2^(b_ij - max)) with
// b_ij = s log2e q_i.k_j over the rows i < p.n_rows.
cudaError_t launch_key_scores_mass(OperandMode mode, const CUtensorMap& mK,
                                   const CUtensorMap& mQ, const KeyScoreParams& p, int H,
                                   int nsplit, cudaStream_t st);
// RMS key scores (bf16 modes): per query split, p.part = (max_i b_ij,
// sum_i 2^(b_ij - max)), b_ij = 2 log2e (s q_i.k_j - lse_pad_i).
cudaError_t launch_key_scores_rms(OperandMode mode, const CUtensorMap& mK,
                                  const CUtensorMap& mQ, const KeyScoreParams& p, int H,
                                  int nsplit, cudaStream_t st);
// From the merged L2 of the RMS pass over n_rows queries: u = log RMS
// probability, as order codes (and floats when u is not null).
cudaError_t launch_rms_finish(const float* L2, int n_rows, uint32_t* code, float* u, size_t n,
                              cudaStream_t st);
cudaError_t launch_gram(OperandMode mode, bool with_r, const CUtensorMap& mKc,
                        const CUtensorMap& mQ, const CUtensorMap& mOhi, const CUtensorMap& mOlo,
                        const GramParams& p, int H, int nsplit, cudaStream_t st);
// Both key blocks of a 256-key system in one CTA per (head, split) (bf16
// operand modes, nblk == 2): all three Gram blocks (and c) ...
cudaError_t launch_gram_all_pairs(OperandMode mode, const CUtensorMap& mKc, const CUtensorMap& mQ,
                                  const CUtensorMap& mOhi, const CUtensorMap& mOlo,
                                  const GramParams& p, int H, int nsplit, cudaStream_t st);
// ... or R for both blocks.
cudaError_t launch_gram_r(OperandMode mode, const CUtensorMap& mKc, const CUtensorMap& mQ,
                          const CUtensorMap& mOhi, const CUtensorMap& mOlo, const GramParams& p,
                          int H, int nsplit, cudaStream_t st);
cudaError_t launch_compact_lse(OperandMode mode, const CUtensorMap& mQ, const CUtensorMap& mKc,
                               const CompactLseParams& p, int H, cudaStream_t st);
// bf16 operand modes with t_pad <= 256: C_k resident, persistent over query
// tiles (grid nsplit x H).
cudaError_t launch_compact_lse_resident(OperandMode mode, const CUtensorMap& mQ,
                                        const CUtensorMap& mKc, const CompactLseParams& p, int H,
                                        int nsplit, cudaStream_t st);

// Kernel shared-memory sizes (for the host's capability check).
int attn_stats_smem(OperandMode mode);
int key_scores_smem(OperandMode mode);
int gram_smem(OperandMode mode);
int compact_lse_smem(OperandMode mode);

// ----------------------------------------------------------- SIMT kernels
cudaError_t launch_convert_bf16_to_f16(const __nv_bfloat16* in, __half* out, size_t n,
                                       cudaStream_t st);
cudaError_t launch_split_f32(const float* in, __half* hi, __half* lo, size_t n, cudaStream_t st);
// rows of d floats -> rows of 3d halves: qk_order 0 = [hi|lo|hi] (queries),
// 1 = [hi|hi|lo] (keys)
cudaError_t launch_split_rows3(const float* in, __half* out, size_t rows, int d, int qk_order,
                               cudaStream_t st);
cudaError_t launch_fill_f32(float* p, size_t n, float v, cudaStream_t st);
cudaError_t launch_pad_rows(const float* in, float* out, int H, int n, int n_pad, float pad,
                            cudaStream_t st);
cudaError_t launch_decode_scores(const uint32_t* code, float* u, size_t n, cudaStream_t st);
cudaError_t launch_encode_scores(const float* u, uint32_t* code, size_t n, cudaStream_t st);
cudaError_t launch_select_topt(const uint32_t* code, int H, int T, int t, int32_t* idx,
                               cudaStream_t st);

// Step 3 for long heads (T >= kWideMinT, T % 4 == 0, 16-byte aligned input,
// t <= 1024): sampled threshold, a streaming filter over all SMs and an exact
// selection among the candidates, with the single-CTA selection over the
// whole head as fallback; same result as launch_select_topt.  The scratch
// (select_wide_bytes) holds a threshold, a count and a candidate list per
// head.  _codes reads order codes, _scores fp32 scores.  `stage` 0, 1, 2
// launches the sample, the filter and the final selection; all three, in
// order, make one selection.
struct WideScratch {
  uint32_t* theta;
  int* count;
  uint32_t* cand_code;
  int32_t* cand_idx;
  uint32_t* err;  // error word of the handle (a timed-out wait sets a bit)
};
constexpr int kWideMinT = 65536;
bool select_wide_applies(int T, int t);
size_t select_wide_bytes(int H);
cudaError_t launch_select_wide_codes(const uint32_t* code, int H, int T, int t, int32_t* idx,
                                     void* scratch, int sm_count, uint32_t* err, int stage,
                                     cudaStream_t st);
cudaError_t launch_select_wide_scores(const float* u, int H, int T, int t, int32_t* idx,
                                      void* scratch, int sm_count, uint32_t* err, int stage,
                                      cudaStream_t st);
// Row r of head h of dst = row idx[h][r] of src (zero rows past t); with
// `hash`, also a hash of each gathered row into hash[h * t_pad + r].
cudaError_t launch_gather_rows(const void* src, void* dst, const int32_t* idx, int H, int T,
                               int t, int t_pad, int row_bytes, cudaStream_t st,
                               uint32_t* hash = nullptr);
cudaError_t launch_gather_v(const void* V, int in_dtype, const int32_t* idx, float* Vc, int H,
                            int T, int t, int t_pad, int d, cudaStream_t st);
cudaError_t launch_reduce_partials(const float* part, float* out, int nsplit, size_t n,
                                   cudaStream_t st);
cudaError_t launch_symmetrize(float* G, int H, int t_pad, cudaStream_t st);
// Split-partial sum of a symmetric system built as its upper block triangle,
// written symmetric (fused sum and transpose); with cpart, the same launch
// also sums the right-hand side's partials ([nsplit][H][t_pad]) into cout.
cudaError_t launch_reduce_gram(const float* part, float* out, int nsplit, int H, int t_pad,
                               cudaStream_t st, const float* cpart = nullptr,
                               float* cout = nullptr);
// Per-query shift and mass rows of the mass system; with colb2, the same
// launch also fills the per-key biases as launch_fill_colb2 does.
cudaError_t launch_mass_rows(const float* rowmax_pad, const float* lse_pad, float* rowsh2,
                             float* row_b, int H, int n_q, int n_q_pad, cudaStream_t st,
                             float* colb2 = nullptr, int t = 0, int t_pad = 0);
cudaError_t launch_fill_colb2(float* colb2, int H, int t, int t_pad, cudaStream_t st);
// lc2_pad[h][r] = log2 sum_z part_z.sum 2^(part_z.max) for r < n, +inf for
// the padding rows n <= r < n_pad.
cudaError_t launch_merge_row_lse(const float2* part, float* lc2_pad, int nsplit, int H, int n,
                                 int n_pad, cudaStream_t st);
// L2[h][j] = log2 sum_z part_z.sum 2^(part_z.max) over the nsplit partials.
cudaError_t launch_merge_key_lse(const float2* part, float* L2, int nsplit, int H, int T,
                                 cudaStream_t st);
// out[i] = in[i] * mul (padding values +-inf stay infinite).
cudaError_t launch_scale_f32(const float* in, float* out, size_t n, float mul, cudaStream_t st);
// idx[h][r] = short[h][pos[h][r]]; chosen[h][pos[h][r]] = 1 (pre-zeroed).
cudaError_t launch_compose_idx(const int32_t* short_idx, const int32_t* pos, int32_t* idx,
                               uint8_t* chosen, int H, int kt, int t, cudaStream_t st);
// Uniform redistribution of the missing mass over the chosen shortlist keys:
// beta[h][r] = ln(1 + Delta_h / (t m_j)), j = pos[h][r], with log2 m_j =
// L2[h][j] and Delta_h the mass of the shortlist keys not chosen.
cudaError_t launch_redistribute_beta(const float* L2, const uint8_t* chosen, const int32_t* pos,
                                     float* beta, int H, int kt, int t, cudaStream_t st);

// Attention over a compacted cache plus appended tokens (decode consumer).
struct CompactAttnParams {
  int n, t, n_new;
  float scale;                 // softmax scale (natural-log units)
  const __nv_bfloat16* q;      // [H][n][d]
  const __nv_bfloat16* Ck;     // [H][t][d]
  const float* beta;           // [H][t]; -inf excludes the entry
  const float* Cv;             // [H][t][d]
  const __nv_bfloat16* Knew;   // [H][n_new][d]
  const __nv_bfloat16* Vnew;   // [H][n_new][d]
  const int32_t* n_vis;        // [H][n] appended tokens visible to each row, or null (all)
  float* A;                    // [H][n][d]
  float* log_z;                // [H][n] or null
};
cudaError_t launch_compact_attention(int d, const CompactAttnParams& p, int H, cudaStream_t st);
// mass_err[h] = mean_i |lz - lse|, out_err[h] = mean_i ||A_i - O_i|| over n rows.
cudaError_t launch_heldout_reduce(int d, const float* A, const float* lz, const float* O,
                                  const float* lse, int H, int n, float* mass_err, float* out_err,
                                  cudaStream_t st);

// Farthest-first traversal per head (one thread-block cluster per head):
// out[h][0..n_add) = the keys added after the n_seed seeds, in order.
cudaError_t launch_farthest_first(int d, const __nv_bfloat16* K, int H, int T,
                                  const int32_t* seeds, int n_seed, int n_add, int32_t* out,
                                  cudaStream_t st);

struct SolveParams {
  int H, t, t_pad, d_v, max_iter;
  const float* G;          // [H][t_pad][t_pad]
  const float* c;          // [H][t_pad]
  float* w;                // [H][t]
  float* beta;             // [H][t]
  float* colb2;            // [H][t_pad]: beta * log2(e), -inf for w = 0 and padding
  float* mat;              // [H][t_pad][t_pad] scratch
  float* vec;              // [H][8][t_pad] scratch
  float* wbuf;             // [H][t_pad][64] scratch (L^-1 E_D of the active set D)
  int32_t* head_status;    // [H]
  int32_t* head_iters;     // [H]
  uint32_t* err;
  // Kept-key rows for the duplicate check of the NNLS (null: no check): the
  // gathered key operand [H][t_pad][k_row_bytes / 2] (16-bit elements) and
  // the hash of each row (launch_gather_rows).
  const void* krows;
  const uint32_t* khash;   // [H][t_pad]
  int k_row_bytes;
};
cudaError_t launch_nnls(const SolveParams& p, cudaStream_t st);
// Bounded least squares w in [lo, hi], p.max_iter iterations (see the kernel).
cudaError_t launch_bounded_ls(const SolveParams& p, float lo, float hi, cudaStream_t st);
size_t solver_smem(int t);  // dynamic shared memory of the solver kernels

struct OlsParams {
  int H, t, t_pad, d_v;
  const float* Hm;         // [H][t_pad][t_pad]
  float* R;                // [H][t_pad][d_v]; overwritten (solved in place)
  const float* Vc;         // [H][t_pad][d_v] original values of the selected keys
  const float* w;          // [H][t]
  float* mat;              // [H][t_pad][t_pad] scratch (factor, packed blocks)
  float* dinv;             // [H][t_pad] scratch (reciprocal diagonal of the factor)
  float* Cv;               // [H][t][d_v]
  int32_t* head_status;
  uint32_t* err;
};
cudaError_t launch_ols(const OlsParams& p, cudaStream_t st);
// The two halves of launch_ols: the factor needs Hm and w only; the solve
// also needs R and Vc (it substitutes the original values for the rows of
// zero-weight keys).
cudaError_t launch_ols_factor(const OlsParams& p, cudaStream_t st);
cudaError_t launch_ols_solve(const OlsParams& p, cudaStream_t st);

}  // namespace lc
