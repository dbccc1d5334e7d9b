// Per-head dense solves of attention-matching compaction.
//
// Step 4 ("KV compaction" blog, section "Fast KV Compaction via Attention
// Matching": beta from the mass equation by NNLS): min_{w >= 0} ||A w - b||^2
// given G = A^T A and c = A^T b, by block principal pivoting (Kim & Park,
// "Fast nonnegative matrix factorization: an active-set-like method and
// comparisons", SIAM J. Sci. Comput. 2011).  Like Lawson-Hanson it is an
// active-set method and reaches the same minimiser (unique when G is positive
// definite), but it exchanges every infeasible index at once, so it needs a
// handful of full solves instead of one solve per index -- the right shape for
// a GPU.  Start: every index passive.  Each step solves G_FF x_F = c_F,
// sets y = G x - c, and flips the indices with x_j < 0 (passive) or y_j < -tol
// (active); if the number of infeasible indices stops falling for three steps
// only the largest such index flips (Murty's rule), which guarantees
// termination.  A fixed iteration cap bounds the loop.  G is factored once;
// each step's passive solve then goes through the capacitance (Schur
// complement) form of the active set D (at most 64 indices), see
// nnls_bpp_kernel.
//
// Step 5 (C_v from the output equation by OLS): C = H^-1 R by Cholesky, with
// the rows of keys whose weight is zero replaced by identity rows and their
// original value vectors, so those keys keep V[idx] and the rest of the system
// is untouched.
//
// One CTA (512 threads) per head.  Matrices are stored as packed
// lower-triangular 32x32 blocks (row stride 33), in shared memory when the
// system has at most 256 unknowns, in the L2-resident workspace otherwise.
// Cholesky is blocked right-looking with one block of look-ahead: the
// diagonal block is factored in registers by one warp with shuffles, the
// panel rows are solved by substitution against it (reciprocal diagonal
// kept; explicit block inverses lost accuracy at kappa ~ 1e6), and the
// trailing update is a register-tiled 32x32x32 warp product.
#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBS = 32;            // block size
constexpr int kLD = 33;            // row stride inside a block
constexpr int kBlk = kBS * kLD;    // floats per block
constexpr int kResidentMax = 256;  // unknowns kept in shared memory
constexpr int kMaxRhs = 128;       // right-hand sides solved in one pass
constexpr int kMaxD = 64;          // active indices handled in capacitance form
constexpr int kPL = 64;            // row stride of the tile staging buffers
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float* blk(float* base, int I, int J) {
  return base + static_cast<size_t>(I * (I + 1) / 2 + J) * kBlk;
}

// One elimination step of the register Cholesky below; the step index is a
// template parameter so that every register index is a compile-time constant.
template <int K>
__device__ __forceinline__ void chol32_step(float (&a)[kBS], int lane, bool& ok) {
  const float piv = __shfl_sync(kFull, a[K], K);
  const bool good = piv > 0.f;
  ok = ok && good;
  // 1/sqrt(pivot) from the hardware approximation (relative error ~2^-22)
  const float rs = rsqrtf(good ? piv : 1.f);
  const float l = (lane == K) ? (good ? piv : 1.f) * rs : a[K] * rs;
  if (lane >= K) a[K] = l;
#pragma unroll
  for (int c = K + 1; c < kBS; ++c) {
    const float lc = __shfl_sync(kFull, l, c);
    if (lane > K) a[c] = fmaf(-l, lc, a[c]);
  }
  if constexpr (K + 1 < kBS) chol32_step<K + 1>(a, lane, ok);
}

// Cholesky of a 32x32 SPD block held by rows in registers (lane r: row r).
// On return lane r holds row r of L in a[0..r].  Returns false if a pivot
// was not positive (the pivot is then replaced by 1).
__device__ __forceinline__ bool warp_chol32(float (&a)[kBS]) {
  bool ok = true;
  chol32_step<0>(a, lane_id(), ok);
  return ok;
}

// Register-tiled 32x32x32 product for one warp: lane = 4*rg + cg owns rows
// 4rg..4rg+3 and columns 8cg..8cg+7 of the output tile, and
//   acc[i][j] += sum_k A(4rg+i, k) * B(k, 8cg+j)
// with A(r, k) = A[r*lda + k] (or A[k*lda + r] when A_T) and B(k, c) =
// B[k*ldb + c] (or B[c*ldb + k] when B_T).  With the stride-33 blocks every
// access pattern is free of bank conflicts (equal addresses broadcast).
template <bool A_T, bool B_T>
__device__ __forceinline__ void warp_mm32(const float* A, int lda, const float* B, int ldb,
                                          float (&acc)[4][8]) {
  const int lane = lane_id(), rg = lane >> 2, cg = lane & 3;
#pragma unroll 4
  for (int k = 0; k < kBS; ++k) {
    float a[4], b[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = A_T ? A[k * lda + 4 * rg + i] : A[(4 * rg + i) * lda + k];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = B_T ? B[(8 * cg + j) * ldb + k] : B[k * ldb + 8 * cg + j];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
}

__device__ __forceinline__ void zero_acc(float (&acc)[4][8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
}

// Factor diagonal block K (one warp) in place and store the reciprocals of
// its diagonal in dinv[32K..32K+31].
__device__ __forceinline__ void diag_factor(float* S, float* dinv, int K, int* bad) {
  const int lane = lane_id();
  float* Akk = blk(S, K, K);
  float a[kBS];
#pragma unroll
  for (int c = 0; c < kBS; ++c) a[c] = Akk[lane * kLD + c];
  if (!warp_chol32(a) && lane == 0) *bad = 1;
#pragma unroll
  for (int c = 0; c < kBS; ++c)
    if (c <= lane) Akk[lane * kLD + c] = a[c];
  float dl = a[0];
#pragma unroll
  for (int c = 1; c < kBS; ++c)
    if (c == lane) dl = a[c];
  dinv[K * kBS + lane] = __frcp_rn(dl);
  __syncwarp();
}

// A_IJ -= L_IK L_JK^T (one warp).
__device__ __forceinline__ void tile_update(float* S, int I, int J, int K) {
  float acc[4][8];
  zero_acc(acc);
  warp_mm32<false, true>(blk(S, I, K), kLD, blk(S, J, K), kLD, acc);
  float* C = blk(S, I, J);
  const int lane = lane_id(), rg = lane >> 2, cg = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) C[(4 * rg + i) * kLD + 8 * cg + j] -= acc[i][j];
}

// Factor the packed block matrix S (NB x NB blocks) in place; dinv receives
// the reciprocal diagonal of L.  Right-looking with one block of look-ahead:
// warp 0 updates and factors the next diagonal block while the other warps
// finish the trailing update.  Panels are solved row by row (one thread per
// row, substitution against the factored diagonal block).  Every pivot that
// is not positive is replaced by 1 and reported.
__device__ __noinline__ bool cta_cholesky(float* S, float* dinv, int NB, int* bad) {
  const int tid = threadIdx.x, warp = warp_id();
  if (tid == 0) *bad = 0;
  __syncthreads();
  if (warp == 0) diag_factor(S, dinv, 0, bad);
  __syncthreads();
  for (int K = 0; K < NB; ++K) {
    // panel: rows of L_IK solve x L_KK^T = a
    const float* Lkk = blk(S, K, K);
    const float* di = dinv + K * kBS;
    for (int g = tid; g < (NB - K - 1) * kBS; g += kThreads) {
      const int I = K + 1 + g / kBS, r = g % kBS;
      float* row = blk(S, I, K) + r * kLD;
      float x[kBS];
#pragma unroll
      for (int c = 0; c < kBS; ++c) {
        float v = row[c];
#pragma unroll
        for (int k = 0; k < c; ++k) v = fmaf(-x[k], Lkk[c * kLD + k], v);
        x[c] = v * di[c];
      }
#pragma unroll
      for (int c = 0; c < kBS; ++c) row[c] = x[c];
    }
    __syncthreads();
    // trailing update; warp 0 takes the next diagonal block and factors it
    const int m = NB - K - 1;
    if (m > 0) {
      if (warp == 0) {
        tile_update(S, K + 1, K + 1, K);
        __syncwarp();
        diag_factor(S, dinv, K + 1, bad);
      } else if (warp % 4 != 0) {
        // warps 4, 8, 12 share a scheduler with warp 0 and stay idle, so
        // the diagonal factorisation -- the critical path -- issues alone
        const int wi = warp - warp / 4 - 1;
        for (int task = wi; task < m * (m + 1) / 2 - 1; task += kWarps - kWarps / 4) {
          // tasks enumerate the lower tiles (i >= j) except (0, 0)
          int i = 0, rem = task + 1;
          while (rem > i) {
            rem -= i + 1;
            ++i;
          }
          tile_update(S, K + 1 + i, K + 1 + rem, K);
        }
      }
    }
    __syncthreads();
  }
  const bool ok = *bad == 0;
  __syncthreads();
  return ok;
}

// Solve L L^T X = B for the factor (S, dinv) and nc columns of B (row-major,
// stride ldb, NB*32 rows; shared or global memory) in place.  Each 32-row
// block of B is staged in shared memory (T), solved against the diagonal
// block by substitution (one thread per column) into T2, written back, and
// used for the update of the remaining rows -- through the register-tiled
// warp product when nc is a multiple of 32, element-wise otherwise.  T and T2
// hold 32 * max(nc, 32) floats.  passes: 1 = forward only (L Y = B),
// 2 = backward only (L^T X = B), 3 = both.
__device__ __noinline__ void cta_chol_solve(const float* S, const float* dinv, int NB, float* B, int ldb,
                               int nc, float* T, float* T2, int passes = 3) {
  const int tid = threadIdx.x, warp = warp_id(), lane = lane_id();
  const int rg = lane >> 2, cg = lane & 3;
  const int n_out = kBS * nc;
  const bool wide = (nc % kBS) == 0;
  const int ntc = nc / kBS;
  float* Sm = const_cast<float*>(S);
  for (int pass = 0; pass < 2; ++pass) {
    if (!(passes & (1 << pass))) continue;
    const bool fwd = pass == 0;
    for (int step = 0; step < NB; ++step) {
      const int K = fwd ? step : NB - 1 - step;
      const float* Lkk = blk(Sm, K, K);
      const float* di = dinv + K * kBS;
      float* BK = B + static_cast<size_t>(K) * kBS * ldb;
      for (int e = tid; e < n_out; e += kThreads) T[e] = BK[(e / nc) * ldb + e % nc];
      __syncthreads();
      for (int j = tid; j < nc; j += kThreads) {
        float x[kBS];
        if (fwd) {
#pragma unroll
          for (int r = 0; r < kBS; ++r) {
            float v = T[r * nc + j];
#pragma unroll
            for (int k = 0; k < r; ++k) v = fmaf(-Lkk[r * kLD + k], x[k], v);
            x[r] = v * di[r];
          }
        } else {
#pragma unroll
          for (int r = kBS - 1; r >= 0; --r) {
            float v = T[r * nc + j];
#pragma unroll
            for (int k = r + 1; k < kBS; ++k) v = fmaf(-Lkk[k * kLD + r], x[k], v);
            x[r] = v * di[r];
          }
        }
#pragma unroll
        for (int r = 0; r < kBS; ++r) {
          T2[r * nc + j] = x[r];
          BK[r * ldb + j] = x[r];
        }
      }
      __syncthreads();
      // remaining rows: forward Y_I -= L_IK X_K (I > K); backward Y_I -= L_KI^T X_K (I < K)
      const int i0 = fwd ? K + 1 : 0, i1 = fwd ? NB : K;
      if (wide) {
        for (int task = warp; task < (i1 - i0) * ntc; task += kWarps) {
          const int I = i0 + task / ntc, ct = task % ntc;
          float acc[4][8];
          zero_acc(acc);
          if (fwd) warp_mm32<false, false>(blk(Sm, I, K), kLD, T2 + ct * kBS, nc, acc);
          else warp_mm32<true, false>(blk(Sm, K, I), kLD, T2 + ct * kBS, nc, acc);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float* row = B + (static_cast<size_t>(I) * kBS + 4 * rg + i) * ldb + ct * kBS + 8 * cg;
#pragma unroll
            for (int j = 0; j < 8; ++j) row[j] -= acc[i][j];
          }
        }
      } else {
        for (int e = tid; e < (i1 - i0) * kBS * nc; e += kThreads) {
          const int gi = e / nc, j = e % nc;
          const int I = i0 + gi / kBS, r = gi % kBS;
          float acc = 0.f;
          if (fwd) {
            const float* Lik = blk(Sm, I, K) + r * kLD;
#pragma unroll
            for (int k = 0; k < kBS; ++k) acc = fmaf(Lik[k], T2[k * nc + j], acc);
          } else {
            const float* Lki = blk(Sm, K, I);
#pragma unroll
            for (int k = 0; k < kBS; ++k) acc = fmaf(Lki[k * kLD + r], T2[k * nc + j], acc);
          }
          B[(static_cast<size_t>(I) * kBS + r) * ldb + j] -= acc;
        }
      }
      __syncthreads();
    }
  }
}

// Solve L L^T x = v (passes as in cta_chol_solve) for one right-hand side v
// in shared memory (NB*32 entries).  Step K: warp 0 solves block K with one
// lane per row (x_k broadcast by shuffle, the row updates run in parallel),
// then one warp per remaining block applies its 32 x 32 product.
__device__ __noinline__ void cta_solve1(const float* S, const float* dinv, int NB, float* v,
                                        int passes = 3) {
  const int warp = warp_id(), lane = lane_id();
  float* Sm = const_cast<float*>(S);
  __syncthreads();
  for (int pass = 0; pass < 2; ++pass) {
    if (!(passes & (1 << pass))) continue;
    const bool fwd = pass == 0;
    for (int step = 0; step < NB; ++step) {
      const int K = fwd ? step : NB - 1 - step;
      if (warp == 0) {
        const float* Lkk = blk(Sm, K, K);
        const float* di = dinv + K * kBS;
        float y = v[K * kBS + lane], xr = 0.f;
        if (fwd) {
#pragma unroll
          for (int k = 0; k < kBS; ++k) {
            const float xk = __shfl_sync(kFull, y, k) * di[k];
            if (lane == k) xr = xk;
            if (lane > k) y = fmaf(-Lkk[lane * kLD + k], xk, y);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < kBS; ++kk) {
            const int k = kBS - 1 - kk;
            const float xk = __shfl_sync(kFull, y, k) * di[k];
            if (lane == k) xr = xk;
            if (lane < k) y = fmaf(-Lkk[k * kLD + lane], xk, y);
          }
        }
        v[K * kBS + lane] = xr;
      }
      __syncthreads();
      const int i0 = fwd ? K + 1 : 0, i1 = fwd ? NB : K;
      for (int I = i0 + warp; I < i1; I += kWarps) {
        const float* xK = v + K * kBS;
        float a0 = 0.f, a1 = 0.f;
        if (fwd) {
          const float* Lr = blk(Sm, I, K) + lane * kLD;
#pragma unroll
          for (int k = 0; k < kBS; k += 2) {
            a0 = fmaf(Lr[k], xK[k], a0);
            a1 = fmaf(Lr[k + 1], xK[k + 1], a1);
          }
        } else {
          const float* Lc = blk(Sm, K, I) + lane;
#pragma unroll
          for (int k = 0; k < kBS; k += 2) {
            a0 = fmaf(Lc[k * kLD], xK[k], a0);
            a1 = fmaf(Lc[(k + 1) * kLD], xK[k + 1], a1);
          }
        }
        v[I * kBS + lane] -= a0 + a1;
      }
      __syncthreads();
    }
  }
}

// Blocked substitution with the resident factor (NB <= 8 blocks) for up to
// two 32-column tiles of right-hand sides that stay in registers: warp w owns
// row block I = w / nct, column tile ct = w % nct (when I < NB), in the
// fragment layout of warp_mm32, holding the NEGATED right-hand side on entry
// and the negated solution on exit (so the block updates accumulate in place).
// Step K: the owners of block K stage their tile in P, solve it against the
// diagonal block by substitution (one lane per column) and reload it; after one
// CTA barrier every warp below (forward) or above (backward) subtracts its
// product with the solved block.  P holds two 32 x kPL buffers, used in turn.
template <bool FWD>
__device__ void reg_tri_solve(const float* S, const float* dinv, int NB, int nct,
                              float (&nb)[4][8], float* P) {
  constexpr bool fwd = FWD;
  const int warp = warp_id(), lane = lane_id(), rg = lane >> 2, cg = lane & 3;
  const int I = warp / nct, ct = warp % nct;
  const bool owns = I < NB;
  float* Sm = const_cast<float*>(S);
  for (int step = 0; step < NB; ++step) {
    const int K = fwd ? step : NB - 1 - step;
    float* Pk = P + (step & 1) * kBS * kPL;
    if (owns && I == K) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float4* row = reinterpret_cast<float4*>(Pk + (4 * rg + i) * kPL + ct * kBS + 8 * cg);
        row[0] = make_float4(-nb[i][0], -nb[i][1], -nb[i][2], -nb[i][3]);
        row[1] = make_float4(-nb[i][4], -nb[i][5], -nb[i][6], -nb[i][7]);
      }
      __syncwarp();
      const float* Lkk = blk(Sm, K, K);
      const float* di = dinv + K * kBS;
      float* col = Pk + ct * kBS + lane;
      float x[kBS];
      if constexpr (FWD) {
#pragma unroll
        for (int r = 0; r < kBS; ++r) {
          float v0 = col[r * kPL], v1 = 0.f;
#pragma unroll
          for (int k = 0; k < r; ++k) {
            if (k & 1) v1 = fmaf(-Lkk[r * kLD + k], x[k], v1);
            else v0 = fmaf(-Lkk[r * kLD + k], x[k], v0);
          }
          x[r] = (v0 + v1) * di[r];
        }
      } else {
#pragma unroll
        for (int rr = 0; rr < kBS; ++rr) {
          const int r = kBS - 1 - rr;
          float v0 = col[r * kPL], v1 = 0.f;
#pragma unroll
          for (int kk = 0; kk < rr; ++kk) {
            const int k = kBS - 1 - kk;
            if (kk & 1) v1 = fmaf(-Lkk[k * kLD + r], x[k], v1);
            else v0 = fmaf(-Lkk[k * kLD + r], x[k], v0);
          }
          x[r] = (v0 + v1) * di[r];
        }
      }
#pragma unroll
      for (int r = 0; r < kBS; ++r) col[r * kPL] = x[r];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4* row =
            reinterpret_cast<const float4*>(Pk + (4 * rg + i) * kPL + ct * kBS + 8 * cg);
        const float4 u0 = row[0], u1 = row[1];
        nb[i][0] = -u0.x; nb[i][1] = -u0.y; nb[i][2] = -u0.z; nb[i][3] = -u0.w;
        nb[i][4] = -u1.x; nb[i][5] = -u1.y; nb[i][6] = -u1.z; nb[i][7] = -u1.w;
      }
    }
    __syncthreads();
    if (owns && (fwd ? I > K : I < K)) {
      if constexpr (FWD) warp_mm32<false, false>(blk(Sm, I, K), kLD, Pk + ct * kBS, kPL, nb);
      else warp_mm32<true, false>(blk(Sm, K, I), kLD, Pk + ct * kBS, kPL, nb);
    }
  }
  __syncthreads();
}

__device__ int block_sum_int(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  if (warp_id() == 0) {
    int x = lane_id() < kWarps ? red[lane_id()] : 0;
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    if (lane_id() == 0) red[32] = x;
  }
  __syncthreads();
  const int r = red[32];
  __syncthreads();
  return r;
}

__device__ int block_max_int(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  if (warp_id() == 0) {
    int x = lane_id() < kWarps ? red[lane_id()] : -1;
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(kFull, x, o));
    if (lane_id() == 0) red[32] = x;
  }
  __syncthreads();
  const int r = red[32];
  __syncthreads();
  return r;
}

__device__ float block_sum_f(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  if (warp_id() == 0) {
    float x = lane_id() < kWarps ? red[lane_id()] : 0.f;
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    if (lane_id() == 0) red[32] = x;
  }
  __syncthreads();
  const float r = red[32];
  __syncthreads();
  return r;
}

// Ascending list of the set flags into pos[]; returns the count.
__device__ int block_compact(const int* flag, int* pos, int n, int* red) {
  const int tid = threadIdx.x, lane = lane_id(), w = warp_id();
  const int chunk = (n + kThreads - 1) / kThreads;
  const int j0 = min(n, tid * chunk), j1 = min(n, j0 + chunk);
  int cnt = 0;
  for (int j = j0; j < j1; ++j) cnt += flag[j] != 0;
  int x = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < kWarps ? red[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, s, o);
      if (lane >= o) s += y;
    }
    red[lane] = s;
  }
  __syncthreads();
  int o = (w > 0 ? red[w - 1] : 0) + x - cnt;
  const int total = red[kWarps - 1];
  for (int j = j0; j < j1; ++j)
    if (flag[j]) pos[o++] = j;
  __syncthreads();
  return total;
}

// Shared-memory plan of the solver kernels.
struct SolverSmem {
  float* S;      // packed blocks (resident) or null
  float* dinv;   // reciprocal diagonal of L
  float* vec;    // 4 * n_pad floats
  int* ivec;     // 4 * n_pad ints
  float* T;      // 32 * kMaxRhs floats
  float* T2;     // 32 * kMaxRhs floats
};

__host__ __device__ inline size_t solver_smem_bytes(int n_pad) {
  const int NB = n_pad / kBS;
  const bool resident = n_pad <= kResidentMax;
  size_t b = 0;
  if (resident) b += static_cast<size_t>(NB * (NB + 1) / 2) * kBlk * 4;
  b += static_cast<size_t>(n_pad) * 4;
  b += 4ull * n_pad * 4 + 4ull * n_pad * 4;
  b += 2ull * kBS * kMaxRhs * 4;
  return b;
}

__device__ SolverSmem carve(float* dyn, int n_pad) {
  SolverSmem s;
  const int NB = n_pad / kBS;
  float* p = dyn;
  s.S = nullptr;
  if (n_pad <= kResidentMax) {
    s.S = p;
    p += static_cast<size_t>(NB * (NB + 1) / 2) * kBlk;
  }
  s.dinv = p;
  p += n_pad;
  s.vec = p;
  p += 4 * n_pad;
  s.ivec = reinterpret_cast<int*>(p);
  p += 4 * n_pad;
  s.T = p;
  s.T2 = p + kBS * kMaxRhs;
  return s;
}

// Packed lower blocks of M_ab = fix(a, b, src[map(a) * ld + map(b)]) for
// a, b < n and the identity beyond n (S in shared or global memory), one
// warp per matrix row, one lane per column.
template <class Map, class Fix>
__device__ void gather_packed(float* S, int NB, int n, const float* src, int ld, Map map,
                              Fix fix) {
  const int lane = lane_id();
  for (int a = warp_id(); a < NB * kBS; a += kWarps) {
    const int I = a / kBS, r = a % kBS;
    for (int J = 0; J <= I; ++J) {
      const int b = J * kBS + lane;
      blk(S, I, J)[r * kLD + lane] =
          (a < n && b < n) ? fix(a, b, src[static_cast<size_t>(map(a)) * ld + map(b)])
                           : (a == b ? 1.f : 0.f);
    }
  }
}

// The same for the unpermuted rows and columns of a system of at most 256
// unknowns (NB <= 8; ld a multiple of 4 and at least NB * 32).  The copy is
// bound by load latency and by the instructions per element, so a warp takes
// four rows at a time, each lane loading 16-byte pieces (columns 4l..4l+3 of
// the two 128-column halves), and applies fix as it stores.
template <class Fix>
__device__ void gather_packed_rows(float* S, int NB, int n, const float* src, int ld, Fix fix) {
  const int lane = lane_id();
  const int rows = NB * kBS;
  const int c0 = 4 * (lane % 8), Jl = lane / 8;  // column piece and block within a half
  for (int a0 = warp_id(); a0 < rows; a0 += 4 * kWarps) {
    float4 v[4][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int a = a0 + q * kWarps, I = a / kBS;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const bool need = a < n && a < rows && hf * 4 + Jl <= I && (hf * 4 + Jl) * kBS + c0 < n;
        v[q][hf] = need ? *reinterpret_cast<const float4*>(src + static_cast<size_t>(a) * ld +
                                                          hf * 128 + 4 * lane)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int a = a0 + q * kWarps, I = a / kBS, r = a % kBS;
      if (a >= rows) break;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int J = hf * 4 + Jl;
        if (J > I) continue;
        const float e4[4] = {v[q][hf].x, v[q][hf].y, v[q][hf].z, v[q][hf].w};
        float* dst = blk(S, I, J) + r * kLD + c0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int b = J * kBS + c0 + e;
          dst[e] = (a < n && b < n) ? fix(a, b, e4[e]) : (a == b ? 1.f : 0.f);
        }
      }
    }
  }
}

// Ridge added once to an n x n system whose factorisation broke down (a
// pivot that is not positive), from the sum of its diagonal: n * 2^-20 *
// mean(diag) = 2^-20 * diag_sum.  On a rank-deficient system the rounding
// errors of the factorisation add up coherently to about n unit roundoffs of
// the diagonal (all queries at q = 0 give a rank-one mass system whose
// leftover block after one elimination step is a constant of that size), so
// the ridge scales with n to stay above them.
__device__ __forceinline__ float ridge_of(float diag_sum, int n) {
  return n > 0 ? diag_sum * 9.5367431640625e-7f : 0.f;
}

// dup[j] = 1 for each kept key j whose operand row equals, value for value,
// the row of a kept key at an earlier position (dup must be zero on entry).
// Such a key's column of the mass system equals the earlier key's, so the
// NNLS minimiser is not unique; the later copy is held at w = 0, the
// minimiser Lawson-Hanson reaches with its argmax ties going to the lower
// index.  The gather of the kept keys hashed each row; each key's hash is
// compared with the earlier keys' and a match is confirmed on the full
// gathered rows.  hsh: t words of shared memory.
__device__ void mark_later_duplicates(const SolveParams& p, int h, int* dup, uint32_t* hsh) {
  const int t = p.t, warp = warp_id(), lane = lane_id();
  const int nw = p.k_row_bytes / 4;
  const uint32_t* K = static_cast<const uint32_t*>(p.krows) + static_cast<size_t>(h) * p.t_pad * nw;
  const uint32_t* hg = p.khash + static_cast<size_t>(h) * p.t_pad;
  for (int j = threadIdx.x; j < t; j += kThreads) hsh[j] = hg[j];
  __syncthreads();
  for (int j = 1 + warp; j < t; j += kWarps) {
    const uint32_t hj = hsh[j];
    bool found = false;
    for (int base = 0; base < j && !found; base += 32) {
      const int jp = base + lane;
      unsigned m = __ballot_sync(kFull, jp < j && hsh[jp] == hj);
      while (m != 0u && !found) {
        const int c = base + __ffs(m) - 1;
        m &= m - 1u;
        const uint32_t* a = K + static_cast<size_t>(j) * nw;
        const uint32_t* b = K + static_cast<size_t>(c) * nw;
        bool eq = true;
        for (int k = lane; k < nw; k += 32)
          eq = eq && row_word_mix(a[k], k) == row_word_mix(b[k], k);
        found = __all_sync(kFull, eq);
      }
    }
    if (lane == 0) dup[j] = found ? 1 : 0;
  }
  __syncthreads();
}

// Step 4 for one head (one CTA).
//
// G is factored once (L L^T = G) and z0 = G^-1 c.  For an active set D
// (w_D = 0, |D| <= 64) the passive solution is
//   x = z0 + G^-1 E_D mu,   (G^-1)_DD mu = -z0_D,
// which gives x_D = 0 and (G x - c) = E_D mu, i.e. (G x - c)_F = 0.  With
// Y = L^-1 E_D (one forward substitution with |D| unit right-hand sides, kept
// in registers), (G^-1)_DD = Y^T Y and G^-1 E_D mu = L^-T (Y mu), so a step
// costs one forward solve with |D| columns, a |D| x |D| Cholesky and one
// backward solve with a single column -- no refactorisation.  Systems with
// more than 256 unknowns, a G that is not positive definite in fp32 even with
// the ridge, or an active set larger than 64 factor G_FF directly at every
// step instead.  Later copies of a kept key (mark_later_duplicates) stay at
// w = 0: their rows and columns of the factored matrix are the identity's and
// they never enter the passive or the active index lists.  A factorisation
// that breaks down (a pivot that is not positive) is redone once with the
// ridge of ridge_of, and the head's status becomes LC_ERR_SINGULAR.
__global__ void __launch_bounds__(kThreads, 1) nnls_bpp_kernel(const SolveParams p) {
  extern __shared__ float dyn[];
  __shared__ int redi[33];
  __shared__ float redf[33];
  __shared__ int bad;
  const int h = blockIdx.x, tid = threadIdx.x, warp = warp_id(), lane = lane_id();
  const int rg = lane >> 2, cg = lane & 3;
  const int t = p.t, tp = p.t_pad;
  const int n_pad = (t + kBS - 1) / kBS * kBS;
  const int NB = n_pad / kBS;
  SolverSmem sm = carve(dyn, n_pad);
  float* S = sm.S ? sm.S : p.mat + static_cast<size_t>(h) * tp * tp;
  float* x = sm.vec;
  float* cv = x + n_pad;
  float* z0 = cv + n_pad;
  float* aux = z0 + n_pad;
  int* F = sm.ivec;
  int* Didx = F + n_pad;
  int* flip = Didx + n_pad;
  int* dup = flip + n_pad;
  float* Yg = p.wbuf + static_cast<size_t>(h) * tp * kMaxD;  // Y spilled for Y^T Y
  // small system in the first staging buffer
  float* Ms = sm.T;
  float* ds = Ms + 3 * kBlk;
  float* mu = ds + 2 * kBS;
  const float* G = p.G + static_cast<size_t>(h) * tp * tp;

  for (int j = tid; j < n_pad; j += kThreads) dup[j] = 0;
  __syncthreads();
  if (p.krows) mark_later_duplicates(p, h, dup, reinterpret_cast<uint32_t*>(aux));
  for (int j = tid; j < n_pad; j += kThreads) {
    const bool live = j < t && !dup[j];
    cv[j] = live ? p.c[static_cast<size_t>(h) * tp + j] : 0.f;
    F[j] = live;
    x[j] = 0.f;
  }
  __syncthreads();
  int status = LC_OK_STATUS;
  bool direct = sm.S == nullptr;
  if (!direct) {
    float ridge = 0.f;
    for (int attempt = 0; attempt < 2; ++attempt) {
      gather_packed_rows(S, NB, t, G, tp, [&](int a, int b, float v) {
        if (dup[a] || dup[b]) return (a == b) ? 1.f : 0.f;
        return v + (a == b ? ridge : 0.f);
      });
      __syncthreads();
      if (cta_cholesky(S, sm.dinv, NB, &bad)) break;
      if (attempt == 1) {
        direct = true;
        break;
      }
      status = LC_SINGULAR_STATUS;
      float dsum = 0.f;
      int cnt = 0;
      for (int a = tid; a < t; a += kThreads)
        if (!dup[a]) {
          dsum += G[static_cast<size_t>(a) * tp + a];
          ++cnt;
        }
      dsum = block_sum_f(dsum, redf);
      cnt = block_sum_int(cnt, redi);
      ridge = ridge_of(dsum, cnt);
    }
  }
  if (!direct) {
    for (int j = tid; j < n_pad; j += kThreads) z0[j] = cv[j];
    __syncthreads();
    cta_solve1(S, sm.dinv, NB, z0);
  }
  int ninf_best = t + 1, backup = 3, it = 0;
  bool converged = false;
  for (it = 0; it < p.max_iter; ++it) {
    for (int j = tid; j < n_pad; j += kThreads) flip[j] = (j < t) && !F[j] && !dup[j];
    __syncthreads();
    const int nD = block_compact(flip, Didx, t, redi);
    if (!direct && nD > kMaxD) direct = true;
    if (!direct) {
      if (nD == 0) {
        for (int j = tid; j < n_pad; j += kThreads) x[j] = z0[j];
        __syncthreads();
      } else {
        const int nct = nD > kBS ? 2 : 1;
        const int NBs = nct;
        for (int e = tid; e < 3 * kBlk; e += kThreads) Ms[e] = 0.f;
        // Y = L^-1 E_D, one warp per column: lane r keeps the running
        // right-hand side of row r of every block; block K is solved
        // lane-parallel (x_k broadcast by shuffle) and its product with the
        // blocks below applied at once.  Rows above the unit entry stay 0.
        for (int q = warp; q < nct * kBS; q += kWarps) {
          if (q >= nD) {  // padding columns of Y are zero
            for (int r = lane; r < n_pad; r += 32) Yg[static_cast<size_t>(r) * kMaxD + q] = 0.f;
            continue;
          }
          const int a = Didx[q], Ka = a / kBS;
          float acc[8];
#pragma unroll
          for (int I = 0; I < 8; ++I) acc[I] = (I == Ka && lane == a % kBS) ? 1.f : 0.f;
#pragma unroll
          for (int K = 0; K < 8; ++K) {
            if (K >= NB) break;
            float* ycol = Yg + static_cast<size_t>(K * kBS + lane) * kMaxD + q;
            if (K < Ka) {
              *ycol = 0.f;
              continue;
            }
            const float* Lkk = blk(S, K, K);
            const float* di = sm.dinv + K * kBS;
            float y = acc[K], xr = 0.f;
#pragma unroll
            for (int k = 0; k < kBS; ++k) {
              const float xk = __shfl_sync(kFull, y, k) * di[k];
              if (lane == k) xr = xk;
              if (lane > k) y = fmaf(-Lkk[lane * kLD + k], xk, y);
            }
            *ycol = xr;
#pragma unroll
            for (int k = 0; k < kBS; ++k) {
              const float xk = __shfl_sync(kFull, xr, k);
#pragma unroll
              for (int I = K + 1; I < 8; ++I)
                if (I < NB) acc[I] = fmaf(-blk(S, I, K)[lane * kLD + k], xk, acc[I]);
            }
          }
        }
        __syncthreads();
        // (G^-1)_DD = Y^T Y, lower tiles (0,0), (1,0), (1,1): one register-
        // tiled product per (tile, 32-row block of Y), written to the dense
        // scratch (unused here: the factor is in shared memory), then summed
        // over the row blocks in ascending order -- the same result on every
        // run, and exactly symmetric diagonal tiles.
        const int npair = nct == 2 ? 3 : 1;
        float* Mpart = p.mat + static_cast<size_t>(h) * tp * tp;
        for (int task = warp; task < npair * NB; task += kWarps) {
          const int pr = task / NB, Ib = task % NB;
          const int ta = pr == 0 ? 0 : 1, tb = pr == 2 ? 1 : 0;
          float acc[4][8];
          zero_acc(acc);
          const float* Yb = Yg + static_cast<size_t>(Ib) * kBS * kMaxD;
          warp_mm32<true, false>(Yb + ta * kBS, kMaxD, Yb + tb * kBS, kMaxD, acc);
          float* dst = Mpart + static_cast<size_t>(task) * kBS * kBS;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float4* d4 = reinterpret_cast<float4*>(dst + (4 * rg + i) * kBS + 8 * cg);
            d4[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            d4[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
          }
        }
        __syncthreads();
        for (int e = tid; e < npair * kBS * kBS; e += kThreads) {
          const int pr = e / (kBS * kBS), rc = e % (kBS * kBS);
          const float* src = Mpart + static_cast<size_t>(pr * NB) * kBS * kBS + rc;
          float sacc = 0.f;
          for (int Ib = 0; Ib < NB; ++Ib) sacc += src[static_cast<size_t>(Ib) * kBS * kBS];
          const int ta = pr == 0 ? 0 : 1, tb = pr == 2 ? 1 : 0;
          blk(Ms, ta, tb)[(rc / kBS) * kLD + rc % kBS] = sacc;
        }
        __syncthreads();
        for (int q = nD + tid; q < NBs * kBS; q += kThreads)
          blk(Ms, q / kBS, q / kBS)[(q % kBS) * kLD + q % kBS] = 1.f;
        for (int q = tid; q < NBs * kBS; q += kThreads) mu[q] = q < nD ? -z0[Didx[q]] : 0.f;
        __syncthreads();
        if (!cta_cholesky(Ms, ds, NBs, &bad)) status = LC_SINGULAR_STATUS;
        cta_solve1(Ms, ds, NBs, mu);
        // v = Y mu, then x = z0 + L^-T v
        for (int a = tid; a < n_pad; a += kThreads) {
          const float4* yr = reinterpret_cast<const float4*>(Yg + static_cast<size_t>(a) * kMaxD);
          float s0 = 0.f, s1 = 0.f;
          for (int q4 = 0; q4 < NBs * kBS / 4; ++q4) {
            const float4 y4 = yr[q4];
            s0 = fmaf(y4.x, mu[4 * q4], s0);
            s1 = fmaf(y4.y, mu[4 * q4 + 1], s1);
            s0 = fmaf(y4.z, mu[4 * q4 + 2], s0);
            s1 = fmaf(y4.w, mu[4 * q4 + 3], s1);
          }
          aux[a] = s0 + s1;
        }
        __syncthreads();
        cta_solve1(S, sm.dinv, NB, aux, 2);
        for (int a = tid; a < n_pad; a += kThreads)
          x[a] = (a < t && F[a]) ? z0[a] + aux[a] : 0.f;
        __syncthreads();
      }
    } else {
      // direct: factor G_FF
      const int nF = block_compact(F, Didx, t, redi);
      const int NBf = (nF + kBS - 1) / kBS;
      float ridge = 0.f;
      for (int attempt = 0; attempt < 2; ++attempt) {
        gather_packed(S, NBf, nF, G, tp, [&](int a) { return Didx[a]; },
                      [&](int a, int b, float v) { return v + (a == b ? ridge : 0.f); });
        __syncthreads();
        if (cta_cholesky(S, sm.dinv, NBf, &bad)) break;
        status = LC_SINGULAR_STATUS;
        if (attempt == 1) break;  // keep the factor with its non-positive pivots set to 1
        float dsum = 0.f;
        for (int a = tid; a < nF; a += kThreads) dsum += G[static_cast<size_t>(Didx[a]) * tp + Didx[a]];
        ridge = ridge_of(block_sum_f(dsum, redf), nF);
      }
      for (int a = tid; a < NBf * kBS; a += kThreads) aux[a] = a < nF ? cv[Didx[a]] : 0.f;
      __syncthreads();
      cta_solve1(S, sm.dinv, NBf, aux);
      for (int j = tid; j < n_pad; j += kThreads) x[j] = 0.f;
      __syncthreads();
      for (int a = tid; a < nF; a += kThreads) x[Didx[a]] = aux[a];
      __syncthreads();
      // the active rows for the dual check below
      for (int j = tid; j < n_pad; j += kThreads) flip[j] = (j < t) && !F[j] && !dup[j];
      __syncthreads();
      block_compact(flip, Didx, t, redi);
    }
    // infeasible set: x_j < 0 on F; on D, y_j = (G x - c)_j < -tol with tol a
    // few ulps of the terms of y_j
    for (int j = tid; j < n_pad; j += kThreads) flip[j] = (j < t) && F[j] && x[j] < 0.f;
    __syncthreads();
    for (int q = warp; q < nD; q += kWarps) {
      const int j = Didx[q];
      const float* g = G + static_cast<size_t>(j) * tp;
      float sacc = 0.f, sa = 0.f;
#pragma unroll 8
      for (int k = lane; k < t; k += 32) {
        const float v = g[k] * x[k];
        sacc += v;
        sa += fabsf(v);
      }
      for (int o = 16; o > 0; o >>= 1) {
        sacc += __shfl_xor_sync(kFull, sacc, o);
        sa += __shfl_xor_sync(kFull, sa, o);
      }
      if (lane == 0) {
        const float yj = sacc - cv[j];
        const float tol = 8.f * 1.1920929e-7f * (sa + fabsf(cv[j]));
        flip[j] = yj < -tol;
      }
    }
    __syncthreads();
    int cnt = 0, maxj = -1;
    for (int j = tid; j < t; j += kThreads)
      if (flip[j]) {
        ++cnt;
        maxj = j;
      }
    cnt = block_sum_int(cnt, redi);
    if (cnt == 0) {
      converged = true;
      break;
    }
    maxj = block_max_int(maxj, redi);
    bool all;
    if (cnt < ninf_best) {
      ninf_best = cnt;
      backup = 3;
      all = true;
    } else if (backup > 0) {
      --backup;
      all = true;
    } else {
      all = false;
    }
    for (int j = tid; j < t; j += kThreads)
      if (flip[j] && (all || j == maxj)) F[j] = !F[j];
    __syncthreads();
  }
  for (int j = tid; j < tp; j += kThreads) {
    float wj = 0.f;
    if (j < t) {
      wj = fmaxf(x[j], 0.f);
      p.w[static_cast<size_t>(h) * t + j] = wj;
      p.beta[static_cast<size_t>(h) * t + j] = wj > 0.f ? logf(wj) : -kInf;
    }
    p.colb2[static_cast<size_t>(h) * tp + j] = (j < t && wj > 0.f) ? log2f(wj) : -kInf;
  }
  if (tid == 0) {
    if (!converged && status == LC_OK_STATUS) status = LC_NOT_CONVERGED_STATUS;
    p.head_status[h] = status;
    p.head_iters[h] = it + (converged ? 1 : 0);
  }
}

// Bounded variant of step 4 ("Latent Compaction with Test-Time Training",
// Appendix A.3: the Attention Matching baseline's bounded NNLS iterations,
// bounds [lo, hi] = [e^-3, e^3]).  Each iteration solves G_FF w_F =
// c_F - G_FB w_B over the free set F with the pinned set B at its bounds
// (G_FF factored directly), then pins every free weight outside [lo, hi] at
// the bound it crossed; it starts with every weight free and stops after
// p.max_iter iterations or when an iteration pins nothing.  A factorisation
// that breaks down is redone once with the ridge of ridge_of (status
// LC_ERR_SINGULAR).
__global__ void __launch_bounds__(kThreads, 1)
    bounded_ls_kernel(const SolveParams p, float lo, float hi) {
  extern __shared__ float dyn[];
  __shared__ int redi[33];
  __shared__ float redf[33];
  __shared__ int bad;
  const int h = blockIdx.x, tid = threadIdx.x, warp = warp_id(), lane = lane_id();
  const int t = p.t, tp = p.t_pad;
  const int n_pad = (t + kBS - 1) / kBS * kBS;
  SolverSmem sm = carve(dyn, n_pad);
  float* S = sm.S ? sm.S : p.mat + static_cast<size_t>(h) * tp * tp;
  float* x = sm.vec;
  float* cv = x + n_pad;
  float* xb = cv + n_pad;   // pinned weights at their bounds, 0 elsewhere
  float* aux = xb + n_pad;
  int* freev = sm.ivec;
  int* Fidx = freev + n_pad;
  int* pin = Fidx + n_pad;
  const float* G = p.G + static_cast<size_t>(h) * tp * tp;

  for (int j = tid; j < n_pad; j += kThreads) {
    cv[j] = j < t ? p.c[static_cast<size_t>(h) * tp + j] : 0.f;
    freev[j] = j < t;
    x[j] = 0.f;
    xb[j] = 0.f;
  }
  __syncthreads();
  int status = LC_OK_STATUS, it = 0;
  while (it < p.max_iter) {
    const int nF = block_compact(freev, Fidx, t, redi);
    if (nF == 0) break;
    ++it;
    const int NBf = (nF + kBS - 1) / kBS;
    // right-hand side c_F - G_FB w_B, one warp per free row
    for (int a = warp; a < NBf * kBS; a += kWarps) {
      float acc = 0.f;
      if (a < nF) {
        const float* g = G + static_cast<size_t>(Fidx[a]) * tp;
        for (int k = lane; k < t; k += 32) acc = fmaf(g[k], xb[k], acc);
      }
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
      if (lane == 0) aux[a] = a < nF ? cv[Fidx[a]] - acc : 0.f;
    }
    float ridge = 0.f;
    for (int attempt = 0; attempt < 2; ++attempt) {
      gather_packed(S, NBf, nF, G, tp, [&](int a) { return Fidx[a]; },
                    [&](int a, int b, float v) { return v + (a == b ? ridge : 0.f); });
      __syncthreads();
      if (cta_cholesky(S, sm.dinv, NBf, &bad)) break;
      status = LC_SINGULAR_STATUS;
      if (attempt == 1) break;
      float dsum = 0.f;
      for (int a = tid; a < nF; a += kThreads) dsum += G[static_cast<size_t>(Fidx[a]) * tp + Fidx[a]];
      ridge = ridge_of(block_sum_f(dsum, redf), nF);
    }
    cta_solve1(S, sm.dinv, NBf, aux);
    for (int a = tid; a < nF; a += kThreads) x[Fidx[a]] = aux[a];
    __syncthreads();
    // pin the free weights that left the box
    int npin = 0;
    for (int j = tid; j < t; j += kThreads) {
      int f = 0;
      if (freev[j]) {
        if (x[j] < lo) {
          x[j] = lo;
          f = 1;
        } else if (x[j] > hi) {
          x[j] = hi;
          f = 1;
        }
      }
      pin[j] = f;
      npin += f;
    }
    npin = block_sum_int(npin, redi);
    if (npin == 0) break;
    for (int j = tid; j < t; j += kThreads)
      if (pin[j]) {
        freev[j] = 0;
        xb[j] = x[j];
      }
    __syncthreads();
  }
  for (int j = tid; j < tp; j += kThreads) {
    const float wj = j < t ? fminf(fmaxf(x[j], lo), hi) : 0.f;
    if (j < t) {
      p.w[static_cast<size_t>(h) * t + j] = wj;
      p.beta[static_cast<size_t>(h) * t + j] = logf(wj);
    }
    p.colb2[static_cast<size_t>(h) * tp + j] = j < t ? log2f(wj) : -kInf;
  }
  if (tid == 0) {
    p.head_status[h] = status;
    p.head_iters[h] = it;
  }
}

// Step 5, part 1: factor the output system (identity rows for zero-weight
// keys and padding) into the packed blocks in p.mat, reciprocal diagonal in
// p.dinv; the right-hand sides of those rows become the original values.
__global__ void __launch_bounds__(kThreads, 1) ols_factor_kernel(const OlsParams p) {
  extern __shared__ float dyn[];
  __shared__ float redf[33];
  __shared__ int redi[33];
  __shared__ int bad;
  const int h = blockIdx.x, tid = threadIdx.x;
  const int t = p.t, tp = p.t_pad, dv = p.d_v;
  const int n_pad = (t + kBS - 1) / kBS * kBS;
  const int NB = n_pad / kBS;
  SolverSmem sm = carve(dyn, n_pad);
  float* gS = p.mat + static_cast<size_t>(h) * tp * tp;
  float* S = sm.S ? sm.S : gS;
  const float* Hm = p.Hm + static_cast<size_t>(h) * tp * tp;
  const float* w = p.w + static_cast<size_t>(h) * t;
  // keys with w > 0 (the support), staged so that the gather's loads do not
  // wait on loads of w
  int* live = sm.ivec;
  for (int j = tid; j < n_pad; j += kThreads) live[j] = j < t && w[j] > 0.f;
  __syncthreads();
  float ridge = 0.f;
  int status = LC_OK_STATUS;
  for (int attempt = 0; attempt < 2; ++attempt) {
    auto fix = [&](int a, int b, float v) {
      if (!live[a] || !live[b]) return (a == b) ? 1.f : 0.f;
      return v + (a == b ? ridge : 0.f);
    };
    if (sm.S) gather_packed_rows(S, NB, t, Hm, tp, fix);
    else gather_packed(S, NB, t, Hm, tp, [](int a) { return a; }, fix);
    __syncthreads();
    if (cta_cholesky(S, sm.dinv, NB, &bad)) break;
    status = LC_SINGULAR_STATUS;
    float dsum = 0.f;
    int cnt = 0;
    for (int a = tid; a < t; a += kThreads)
      if (live[a]) {
        dsum += Hm[static_cast<size_t>(a) * tp + a];
        ++cnt;
      }
    dsum = block_sum_f(dsum, redf);
    cnt = block_sum_int(cnt, redi);
    ridge = ridge_of(dsum, cnt);
  }
  // publish the factor for the solve kernel
  if (sm.S) {
    const size_t nel = static_cast<size_t>(NB * (NB + 1) / 2) * kBlk;
    for (size_t e = tid; e < nel; e += kThreads) gS[e] = sm.S[e];
  }
  float* gd = p.dinv + static_cast<size_t>(h) * tp;
  for (int a = tid; a < n_pad; a += kThreads) gd[a] = sm.dinv[a];
  if (tid == 0 && status != LC_OK_STATUS && p.head_status[h] == LC_OK_STATUS)
    p.head_status[h] = status;
}

// Step 5, part 2: C_v columns [32*blockIdx.y, +32) by forward and backward

// Step 5, part 2: C_v columns [32*blockIdx.y, +32) by forward and backward
// substitution with the published factor -- held in registers when the system
// has at most 256 unknowns (reg_tri_solve), else staged through the workspace.
__global__ void __launch_bounds__(kThreads, 1) ols_solve_kernel(const OlsParams p) {
  extern __shared__ float dyn[];
  const int h = blockIdx.x, tid = threadIdx.x;
  const int t = p.t, tp = p.t_pad, dv = p.d_v;
  const int n_pad = (t + kBS - 1) / kBS * kBS;
  const int NB = n_pad / kBS;
  SolverSmem sm = carve(dyn, n_pad);
  const float* gS = p.mat + static_cast<size_t>(h) * tp * tp;
  const float* S = gS;
  if (sm.S) {
    // the published factor by asynchronous 16-byte copies, all in flight
    // at once (a copy loop of loads and stores waits on every load)
    const size_t nel = static_cast<size_t>(NB * (NB + 1) / 2) * kBlk;
    for (size_t e = tid; e < nel / 4; e += kThreads)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                       __cvta_generic_to_shared(sm.S + 4 * e))),
                   "l"(__cvta_generic_to_global(gS + 4 * e))
                   : "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
    S = sm.S;
  }
  const float* gd = p.dinv + static_cast<size_t>(h) * tp;
  for (int a = tid; a < n_pad; a += kThreads) sm.dinv[a] = gd[a];
  float* B = p.R + static_cast<size_t>(h) * tp * dv;
  float* Cv = p.Cv + static_cast<size_t>(h) * t * dv;
  const float* w = p.w + static_cast<size_t>(h) * t;
  const float* Vc = p.Vc + static_cast<size_t>(h) * tp * dv;
  // right-hand side of row a: R_a, the original value row where w_a = 0
  // (identity row of the factor), 0 in the padding
  auto rhs = [&](int a, int col) -> float {
    if (a >= t) return 0.f;
    const size_t e = static_cast<size_t>(a) * dv + col;
    return w[a] > 0.f ? B[e] : Vc[e];
  };
  if (sm.S) {
    const int warp = warp_id(), lane = lane_id(), rg = lane >> 2, cg = lane & 3;
    const int c0 = blockIdx.y * kBS;
    const int nc = min(kBS, dv - c0);
    const int nct = 1;
    const int I = warp / nct, ct = warp % nct;
    float nb[4][8];
    if (nc == kBS) {
      // every load first (w, R and the value rows, 16 bytes at a time), then
      // the choice between R and V[idx]: no load waits on another
      float wa[4];
      float4 rv[4][2], vv[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int a = I * kBS + 4 * rg + i;
        const bool in = I < NB && a < t;
        const size_t e = static_cast<size_t>(a) * dv + c0 + 8 * cg;
        wa[i] = in ? w[a] : 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          rv[i][hf] = in ? *reinterpret_cast<const float4*>(B + e + 4 * hf) : make_float4(0.f, 0.f, 0.f, 0.f);
          vv[i][hf] = in ? *reinterpret_cast<const float4*>(Vc + e + 4 * hf) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const float4 v4 = wa[i] > 0.f ? rv[i][hf] : vv[i][hf];
          nb[i][4 * hf] = -v4.x;
          nb[i][4 * hf + 1] = -v4.y;
          nb[i][4 * hf + 2] = -v4.z;
          nb[i][4 * hf + 3] = -v4.w;
        }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int a = I * kBS + 4 * rg + i, q = ct * kBS + 8 * cg + j;
          nb[i][j] = (I < NB && q < nc) ? -rhs(a, c0 + q) : 0.f;
        }
    }
    __syncthreads();
    reg_tri_solve<true>(S, sm.dinv, NB, nct, nb, sm.T2);
    reg_tri_solve<false>(S, sm.dinv, NB, nct, nb, sm.T2);
    if (I < NB) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int a = I * kBS + 4 * rg + i, q = ct * kBS + 8 * cg + j;
          if (a < t && q < nc) Cv[static_cast<size_t>(a) * dv + c0 + q] = -nb[i][j];
        }
    }
    return;
  }
  const int c0 = blockIdx.y * kBS;
  const int nc = min(kBS, dv - c0);
  for (int e = tid; e < n_pad * nc; e += kThreads) {
    const int a = e / nc, j = e % nc;
    if (a >= t || !(w[a] > 0.f)) B[static_cast<size_t>(a) * dv + c0 + j] = rhs(a, c0 + j);
  }
  __syncthreads();
  cta_chol_solve(S, sm.dinv, NB, B + c0, dv, nc, sm.T, sm.T2);
  for (int e = tid; e < t * nc; e += kThreads) {
    const int a = e / nc, j = e % nc;
    Cv[static_cast<size_t>(a) * dv + c0 + j] = B[static_cast<size_t>(a) * dv + c0 + j];
  }
}

}  // namespace

size_t solver_smem(int t) {
  const int n_pad = (t + kBS - 1) / kBS * kBS;
  return solver_smem_bytes(n_pad);
}

cudaError_t launch_nnls(const SolveParams& p, cudaStream_t st) {
  const size_t smem = solver_smem(p.t);
  cudaError_t e = cudaFuncSetAttribute(nnls_bpp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  nnls_bpp_kernel<<<p.H, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bounded_ls(const SolveParams& p, float lo, float hi, cudaStream_t st) {
  const size_t smem = solver_smem(p.t);
  cudaError_t e = cudaFuncSetAttribute(bounded_ls_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  bounded_ls_kernel<<<p.H, kThreads, smem, st>>>(p, lo, hi);
  return cudaGetLastError();
}

cudaError_t launch_ols_factor(const OlsParams& p, cudaStream_t st) {
  const size_t smem = solver_smem(p.t);
  cudaError_t e = cudaFuncSetAttribute(ols_factor_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  ols_factor_kernel<<<p.H, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_ols_solve(const OlsParams& p, cudaStream_t st) {
  const size_t smem = solver_smem(p.t);
  cudaError_t e = cudaFuncSetAttribute(ols_solve_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  ols_solve_kernel<<<dim3(p.H, (p.d_v + kBS - 1) / kBS), kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_ols(const OlsParams& p, cudaStream_t st) {
  cudaError_t e = launch_ols_factor(p, st);
  if (e != cudaSuccess) return e;
  return launch_ols_solve(p, st);
}

}  // namespace lc
