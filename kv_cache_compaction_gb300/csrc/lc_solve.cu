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
// termination.  A fixed iteration cap bounds the loop.
//
// Step 5 (C_v from the output equation by OLS): C = H^-1 R by Cholesky, with
// the rows of keys whose weight is zero replaced by identity rows and their
// original value vectors, so those keys keep V[idx] and the rest of the system
// is untouched.
//
// One CTA (512 threads) per head.  Matrices are stored as packed
// lower-triangular 32x32 blocks (row stride 33), in shared memory when the
// system has at most 256 unknowns, in the L2-resident workspace otherwise.
// Cholesky is blocked right-looking: the diagonal block is factored in
// registers by one warp with shuffles, its inverse is formed explicitly, and
// the panel, the trailing update and both triangular solves are small
// data-parallel products with those inverses -- no dependent chains through
// memory.
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
// Right-hand sides per pass: fewer when the factor lives in L2, so that the
// diagonal-block inverses and the chunk still fit in shared memory.
__host__ __device__ inline int rhs_chunk(int n_pad) { return n_pad <= 256 ? 16 : 8; }
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float* blk(float* base, int I, int J) {
  return base + static_cast<size_t>(I * (I + 1) / 2 + J) * kBlk;
}

// Cholesky of a 32x32 SPD block held by rows in registers (lane r: row r).
// On return lane r holds row r of L in a[0..r].  Returns false if a pivot
// was not positive (the pivot is then replaced by 1).
__device__ __forceinline__ bool warp_chol32(float (&a)[kBS]) {
  const int lane = lane_id();
  bool ok = true;
#pragma unroll
  for (int k = 0; k < kBS; ++k) {
    const float piv = __shfl_sync(kFull, a[k], k);
    const bool good = piv > 0.f;
    ok = ok && good;
    const float d = sqrtf(good ? piv : 1.f);
    const float l = (lane == k) ? d : a[k] / d;
    if (lane >= k) a[k] = l;
#pragma unroll
    for (int c = k + 1; c < kBS; ++c) {
      const float lc = __shfl_sync(kFull, l, c);
      if (lane > k) a[c] = fmaf(-l, lc, a[c]);
    }
  }
  return ok;
}

// Factor the packed block matrix S (NB x NB blocks) in place; Linv receives
// the inverses of the diagonal blocks (lower, stride 33).  Every diagonal
// pivot that is not positive is replaced by 1 and reported.
__device__ bool cta_cholesky(float* S, float* Linv, int NB, int* bad) {
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  if (tid == 0) *bad = 0;
  __syncthreads();
  for (int K = 0; K < NB; ++K) {
    float* Akk = blk(S, K, K);
    float* Li = Linv + static_cast<size_t>(K) * kBlk;
    if (warp == 0) {
      float a[kBS];
#pragma unroll
      for (int c = 0; c < kBS; ++c) a[c] = Akk[lane * kLD + c];
      if (!warp_chol32(a) && lane == 0) *bad = 1;
#pragma unroll
      for (int c = 0; c < kBS; ++c)
        if (c <= lane) Akk[lane * kLD + c] = a[c];
      __syncwarp();
      // column `lane` of L^-1: forward substitution with L read back
      float x[kBS];
#pragma unroll
      for (int r = 0; r < kBS; ++r) {
        float s = (r == lane) ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < r; ++k) s = fmaf(-Akk[r * kLD + k], x[k], s);
        x[r] = s / Akk[r * kLD + r];
      }
#pragma unroll
      for (int r = 0; r < kBS; ++r) Li[r * kLD + lane] = x[r];
    }
    __syncthreads();
    // panel: L_IK = A_IK L_KK^-T, one warp per block row, lane = column
    for (int task = warp; task < (NB - K - 1) * kBS; task += kWarps) {
      const int I = K + 1 + task / kBS, r = task % kBS;
      float* row = blk(S, I, K) + r * kLD;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < kBS; ++k) acc = fmaf(row[k], Li[lane * kLD + k], acc);
      __syncwarp();
      row[lane] = acc;
    }
    __syncthreads();
    // trailing update: A_IJ -= L_IK L_JK^T for K < J <= I, one warp per block
    const int m = NB - K - 1;
    for (int task = warp; task < m * (m + 1) / 2; task += kWarps) {
      int i = 0, rem = task;
      while (rem > i) {
        rem -= i + 1;
        ++i;
      }
      const int I = K + 1 + i, J = K + 1 + rem;
      const float* Lik = blk(S, I, K);
      const float* Ljk = blk(S, J, K);
      float* Aij = blk(S, I, J);
      float lj[kBS];
#pragma unroll
      for (int k = 0; k < kBS; ++k) lj[k] = Ljk[lane * kLD + k];
      for (int r = 0; r < kBS; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kBS; ++k) acc = fmaf(Lik[r * kLD + k], lj[k], acc);
        Aij[r * kLD + lane] -= acc;
      }
    }
    __syncthreads();
  }
  const bool ok = *bad == 0;
  __syncthreads();
  return ok;
}

// Solve L L^T X = B for the factor in (S, Linv) and nc columns of B
// (row-major, stride ldb, NB*32 rows) in place.  T: scratch of 32 * nc floats.
__device__ void cta_chol_solve(const float* S, const float* Linv, int NB, float* B, int ldb,
                               int nc, float* T) {
  const int tid = threadIdx.x;
  const int n_out = kBS * nc;
  // forward: L Y = B
  for (int K = 0; K < NB; ++K) {
    const float* Li = Linv + static_cast<size_t>(K) * kBlk;
    float* BK = B + static_cast<size_t>(K) * kBS * ldb;
    for (int e = tid; e < n_out; e += kThreads) {
      const int r = e / nc, j = e % nc;
      float acc = 0.f;
      for (int k = 0; k <= r; ++k) acc = fmaf(Li[r * kLD + k], BK[k * ldb + j], acc);
      T[e] = acc;
    }
    __syncthreads();
    for (int e = tid; e < n_out; e += kThreads) BK[(e / nc) * ldb + e % nc] = T[e];
    __syncthreads();
    const int rows = (NB - K - 1) * kBS;
    for (int e = tid; e < rows * nc; e += kThreads) {
      const int gi = e / nc, j = e % nc;
      const int I = K + 1 + gi / kBS, r = gi % kBS;
      const float* Lik = blk(const_cast<float*>(S), I, K) + r * kLD;
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < kBS; ++k) acc = fmaf(Lik[k], T[k * nc + j], acc);
      B[(static_cast<size_t>(I) * kBS + r) * ldb + j] -= acc;
    }
    __syncthreads();
  }
  // backward: L^T X = Y
  for (int K = NB - 1; K >= 0; --K) {
    const float* Li = Linv + static_cast<size_t>(K) * kBlk;
    float* BK = B + static_cast<size_t>(K) * kBS * ldb;
    for (int e = tid; e < n_out; e += kThreads) {
      const int r = e / nc, j = e % nc;
      float acc = 0.f;
      for (int k = r; k < kBS; ++k) acc = fmaf(Li[k * kLD + r], BK[k * ldb + j], acc);
      T[e] = acc;
    }
    __syncthreads();
    for (int e = tid; e < n_out; e += kThreads) BK[(e / nc) * ldb + e % nc] = T[e];
    __syncthreads();
    const int rows = K * kBS;
    for (int e = tid; e < rows * nc; e += kThreads) {
      const int gi = e / nc, j = e % nc;
      const int I = gi / kBS, r = gi % kBS;  // I < K: Y_I -= L_KI^T X_K
      const float* Lki = blk(const_cast<float*>(S), K, I);
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < kBS; ++k) acc = fmaf(Lki[k * kLD + r], T[k * nc + j], acc);
      B[(static_cast<size_t>(I) * kBS + r) * ldb + j] -= acc;
    }
    __syncthreads();
  }
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
  float* Linv;   // diagonal-block inverses
  float* vec;    // 4 * n_pad floats
  int* ivec;     // 3 * n_pad ints
  float* rhs;    // n_pad * kRhsChunk floats
  float* T;      // 32 * kRhsChunk floats
};

__host__ __device__ inline size_t solver_smem_bytes(int n_pad) {
  const int NB = n_pad / kBS;
  const bool resident = n_pad <= kResidentMax;
  size_t b = 0;
  if (resident) b += static_cast<size_t>(NB * (NB + 1) / 2) * kBlk * 4;
  b += static_cast<size_t>(NB) * kBlk * 4;
  b += 4ull * n_pad * 4 + 3ull * n_pad * 4;
  b += static_cast<size_t>(n_pad) * rhs_chunk(n_pad) * 4 + kBS * rhs_chunk(n_pad) * 4;
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
  s.Linv = p;
  p += static_cast<size_t>(NB) * kBlk;
  s.vec = p;
  p += 4 * n_pad;
  s.ivec = reinterpret_cast<int*>(p);
  p += 3 * n_pad;
  s.rhs = p;
  p += static_cast<size_t>(n_pad) * rhs_chunk(n_pad);
  s.T = p;
  return s;
}

__global__ void __launch_bounds__(kThreads, 1) nnls_bpp_kernel(const SolveParams p) {
  extern __shared__ float dyn[];
  __shared__ int redi[33];
  __shared__ int bad;
  const int h = blockIdx.x, tid = threadIdx.x;
  const int t = p.t, tp = p.t_pad;
  const int n_pad = (t + kBS - 1) / kBS * kBS;
  SolverSmem sm = carve(dyn, n_pad);
  float* S = sm.S ? sm.S : p.mat + static_cast<size_t>(h) * tp * tp;
  float* x = sm.vec;
  float* cv = x + n_pad;
  float* rhs = sm.rhs;
  int* F = sm.ivec;
  int* Fidx = F + n_pad;
  int* flip = Fidx + n_pad;
  const float* G = p.G + static_cast<size_t>(h) * tp * tp;

  for (int j = tid; j < n_pad; j += kThreads) {
    cv[j] = j < t ? p.c[static_cast<size_t>(h) * tp + j] : 0.f;
    F[j] = j < t;
    x[j] = 0.f;
  }
  __syncthreads();
  int ninf_best = t + 1, backup = 3, status = LC_OK_STATUS, it = 0;
  bool converged = false;
  for (it = 0; it < p.max_iter; ++it) {
    const int nF = block_compact(F, Fidx, t, redi);
    const int NB = (nF + kBS - 1) / kBS;
    // gather G_FF into packed blocks; identity beyond nF
    const int nb_el = NB * (NB + 1) / 2 * kBlk;
    for (int e = tid; e < nb_el; e += kThreads) {
      const int b = e / kBlk, o = e % kBlk;
      const int r = o / kLD, c = o % kLD;
      if (c >= kBS) continue;
      int I = 0, rem = b;
      while (rem > I) {
        rem -= I + 1;
        ++I;
      }
      const int a = I * kBS + r, bb = rem * kBS + c;
      float v;
      if (a < nF && bb < nF) v = G[static_cast<size_t>(Fidx[a]) * tp + Fidx[bb]];
      else v = (a == bb) ? 1.f : 0.f;
      S[static_cast<size_t>(b) * kBlk + o] = v;
    }
    for (int a = tid; a < NB * kBS; a += kThreads) rhs[a] = a < nF ? cv[Fidx[a]] : 0.f;
    __syncthreads();
    if (!cta_cholesky(S, sm.Linv, NB, &bad)) status = LC_SINGULAR_STATUS;
    cta_chol_solve(S, sm.Linv, NB, rhs, 1, 1, sm.T);
    for (int j = tid; j < n_pad; j += kThreads) x[j] = 0.f;
    __syncthreads();
    for (int a = tid; a < nF; a += kThreads) x[Fidx[a]] = rhs[a];
    __syncthreads();
    // y = G x - c and the infeasible set; tolerance a few ulps of the terms
    const int warp = warp_id(), lane = lane_id();
    for (int j = warp; j < t; j += kWarps) {
      const float* g = G + static_cast<size_t>(j) * tp;
      float s = 0.f, sa = 0.f;
      for (int k = lane; k < t; k += 32) {
        const float v = g[k] * x[k];
        s += v;
        sa += fabsf(v);
      }
      for (int o = 16; o > 0; o >>= 1) {
        s += __shfl_xor_sync(kFull, s, o);
        sa += __shfl_xor_sync(kFull, sa, o);
      }
      if (lane == 0) {
        const float yj = s - cv[j];
        const float tol = 8.f * 1.1920929e-7f * (sa + fabsf(cv[j]));
        flip[j] = F[j] ? (x[j] < 0.f) : (yj < -tol);
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

__global__ void __launch_bounds__(kThreads, 1) ols_kernel(const OlsParams p) {
  extern __shared__ float dyn[];
  __shared__ float redf[33];
  __shared__ int bad;
  const int h = blockIdx.x, tid = threadIdx.x;
  const int t = p.t, tp = p.t_pad, dv = p.d_v;
  const int n_pad = (t + kBS - 1) / kBS * kBS;
  const int NB = n_pad / kBS;
  SolverSmem sm = carve(dyn, n_pad);
  float* S = sm.S ? sm.S : p.mat + static_cast<size_t>(h) * tp * tp;
  const float* Hm = p.Hm + static_cast<size_t>(h) * tp * tp;
  const float* R = p.R + static_cast<size_t>(h) * tp * dv;
  const float* w = p.w + static_cast<size_t>(h) * t;
  const float* Vc = p.Vc + static_cast<size_t>(h) * tp * dv;
  float* Cv = p.Cv + static_cast<size_t>(h) * t * dv;

  // system with identity rows for zero-weight keys and padding
  float ridge = 0.f;
  int status = LC_OK_STATUS;
  for (int attempt = 0; attempt < 2; ++attempt) {
    const int nb_el = NB * (NB + 1) / 2 * kBlk;
    for (int e = tid; e < nb_el; e += kThreads) {
      const int b = e / kBlk, o = e % kBlk;
      const int r = o / kLD, c = o % kLD;
      if (c >= kBS) continue;
      int I = 0, rem = b;
      while (rem > I) {
        rem -= I + 1;
        ++I;
      }
      const int a = I * kBS + r, bb = rem * kBS + c;
      float v;
      const bool za = a >= t || !(w[a] > 0.f), zb = bb >= t || !(w[bb] > 0.f);
      if (za || zb) v = (a == bb) ? 1.f : 0.f;
      else v = Hm[static_cast<size_t>(a) * tp + bb] + (a == bb ? ridge : 0.f);
      S[static_cast<size_t>(b) * kBlk + o] = v;
    }
    __syncthreads();
    if (cta_cholesky(S, sm.Linv, NB, &bad)) break;
    status = LC_SINGULAR_STATUS;
    float dsum = 0.f;
    for (int a = tid; a < t; a += kThreads)
      dsum += (w[a] > 0.f) ? Hm[static_cast<size_t>(a) * tp + a] : 0.f;
    ridge = 1e-6f * block_sum_f(dsum, redf) / t;
  }
  // right-hand sides in chunks of rc columns
  const int rc = rhs_chunk(n_pad);
  for (int c0 = 0; c0 < dv; c0 += rc) {
    const int nc = min(rc, dv - c0);
    for (int e = tid; e < n_pad * nc; e += kThreads) {
      const int a = e / nc, j = e % nc;
      float v = 0.f;
      if (a < t)
        v = (w[a] > 0.f) ? R[static_cast<size_t>(a) * dv + c0 + j]
                         : Vc[static_cast<size_t>(a) * dv + c0 + j];
      sm.rhs[a * rc + j] = v;
    }
    __syncthreads();
    cta_chol_solve(S, sm.Linv, NB, sm.rhs, rc, nc, sm.T);
    for (int e = tid; e < t * nc; e += kThreads) {
      const int a = e / nc, j = e % nc;
      Cv[static_cast<size_t>(a) * dv + c0 + j] = sm.rhs[a * rc + j];
    }
    __syncthreads();
  }
  if (tid == 0 && status != LC_OK_STATUS && p.head_status[h] == LC_OK_STATUS)
    p.head_status[h] = status;
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

cudaError_t launch_ols(const OlsParams& p, cudaStream_t st) {
  const size_t smem = solver_smem(p.t);
  cudaError_t e = cudaFuncSetAttribute(ols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  ols_kernel<<<p.H, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace lc
