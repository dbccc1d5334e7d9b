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
// One CTA (1024 threads) per head.  The factorisation is blocked right-looking
// Cholesky with 32-wide panels on an L2-resident copy of the matrix.
#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kThreads = 1024;
constexpr int kNB = 32;

struct SolveSmem {
  float D[kNB * 33];  // diagonal block
  int bad;
};

// Blocked Cholesky of the leading n x n block of A (row-major, stride lda),
// lower triangle, in place.  P: shared buffer of at least n * 33 floats for
// the current panel.  Returns true if every pivot was positive.
__device__ bool cta_cholesky(float* A, int n, int lda, float* P, SolveSmem& sm) {
  const int tid = threadIdx.x, lane = lane_id(), warp = warp_id();
  if (tid == 0) sm.bad = 0;
  __syncthreads();
  for (int kb = 0; kb < n; kb += kNB) {
    const int nb = min(kNB, n - kb);
    for (int e = tid; e < kNB * kNB; e += kThreads) {
      const int r = e / kNB, c = e % kNB;
      sm.D[r * 33 + c] = (r < nb && c <= r) ? A[static_cast<size_t>(kb + r) * lda + kb + c] : 0.f;
    }
    __syncthreads();
    if (warp == 0) {
      for (int k = 0; k < nb; ++k) {
        float piv = sm.D[k * 33 + k];
        if (!(piv > 0.f)) {
          if (lane == 0) sm.bad = 1;
          piv = 1.f;
        }
        const float dk = sqrtf(piv);
        __syncwarp();
        if (lane == k) sm.D[k * 33 + k] = dk;
        if (lane > k && lane < nb) sm.D[lane * 33 + k] /= dk;
        __syncwarp();
        if (lane > k && lane < nb) {
          const float lrk = sm.D[lane * 33 + k];
          for (int c = k + 1; c <= lane; ++c) sm.D[lane * 33 + c] -= lrk * sm.D[c * 33 + k];
        }
        __syncwarp();
      }
    }
    __syncthreads();
    for (int e = tid; e < nb * nb; e += kThreads) {
      const int r = e / nb, c = e % nb;
      if (c <= r) A[static_cast<size_t>(kb + r) * lda + kb + c] = sm.D[r * 33 + c];
    }
    // panel: rows below the diagonal block, L_ik = A_ik L_kk^-T
    const int m = n - kb - nb;
    for (int i = tid; i < m; i += kThreads) {
      float* row = A + static_cast<size_t>(kb + nb + i) * lda + kb;
      float x[kNB];
#pragma unroll
      for (int c = 0; c < kNB; ++c) {
        if (c < nb) {
          float s = row[c];
          for (int c2 = 0; c2 < c; ++c2) s -= x[c2] * sm.D[c * 33 + c2];
          x[c] = s / sm.D[c * 33 + c];
        } else {
          x[c] = 0.f;
        }
      }
#pragma unroll
      for (int c = 0; c < kNB; ++c) {
        if (c < nb) row[c] = x[c];
        P[i * 33 + c] = x[c];
      }
    }
    __syncthreads();
    // trailing update of the lower triangle: A_ij -= sum_c P_ic P_jc
    const int mt = (m + 31) / 32;
    const int ntiles = mt * (mt + 1) / 2;
    for (int tile = warp; tile < ntiles; tile += kThreads / 32) {
      int ti = 0, rem = tile;
      while (rem > ti) {
        rem -= ti + 1;
        ++ti;
      }
      const int tj = rem;  // tj <= ti
      const int j = tj * 32 + lane;
      float pj[kNB];
#pragma unroll
      for (int c = 0; c < kNB; ++c) pj[c] = (j < m) ? P[j * 33 + c] : 0.f;
      for (int r = 0; r < 32; ++r) {
        const int i = ti * 32 + r;
        if (i >= m) break;
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < kNB; ++c) acc = fmaf(P[i * 33 + c], pj[c], acc);
        if (j < m && j <= i) A[static_cast<size_t>(kb + nb + i) * lda + kb + nb + j] -= acc;
      }
    }
    __syncthreads();
  }
  const bool ok = sm.bad == 0;
  __syncthreads();
  return ok;
}

// Solve L L^T X = B in place for the leading n x n factor L (stride lda) and
// nrhs right-hand sides B (row-major, stride ldb).
__device__ void cta_chol_solve(const float* A, int n, int lda, float* B, int ldb, int nrhs) {
  const int tid = threadIdx.x;
  // forward: L Y = B, block by block
  for (int kb = 0; kb < n; kb += kNB) {
    const int nb = min(kNB, n - kb);
    for (int col = tid; col < nrhs; col += kThreads) {
      for (int r = 0; r < nb; ++r) {
        const float* lr = A + static_cast<size_t>(kb + r) * lda + kb;
        float s = B[static_cast<size_t>(kb + r) * ldb + col];
        for (int c = 0; c < r; ++c) s -= lr[c] * B[static_cast<size_t>(kb + c) * ldb + col];
        B[static_cast<size_t>(kb + r) * ldb + col] = s / lr[r];
      }
    }
    __syncthreads();
    const int rows = n - kb - nb;
    for (int e = tid; e < rows * nrhs; e += kThreads) {
      const int i = kb + nb + e / nrhs, col = e % nrhs;
      const float* li = A + static_cast<size_t>(i) * lda + kb;
      float s = 0.f;
      for (int c = 0; c < nb; ++c) s = fmaf(li[c], B[static_cast<size_t>(kb + c) * ldb + col], s);
      B[static_cast<size_t>(i) * ldb + col] -= s;
    }
    __syncthreads();
  }
  // backward: L^T X = Y
  const int nblk = (n + kNB - 1) / kNB;
  for (int bk = nblk - 1; bk >= 0; --bk) {
    const int kb = bk * kNB, nb = min(kNB, n - kb);
    for (int col = tid; col < nrhs; col += kThreads) {
      for (int r = nb - 1; r >= 0; --r) {
        float s = B[static_cast<size_t>(kb + r) * ldb + col];
        for (int c = r + 1; c < nb; ++c)
          s -= A[static_cast<size_t>(kb + c) * lda + kb + r] * B[static_cast<size_t>(kb + c) * ldb + col];
        B[static_cast<size_t>(kb + r) * ldb + col] = s / A[static_cast<size_t>(kb + r) * lda + kb + r];
      }
    }
    __syncthreads();
    // rows above: Y_i -= sum_{c in block} L_ci X_c  for i < kb
    for (int e = tid; e < kb * nrhs; e += kThreads) {
      const int i = e / nrhs, col = e % nrhs;
      float s = 0.f;
      for (int c = 0; c < nb; ++c)
        s = fmaf(A[static_cast<size_t>(kb + c) * lda + i], B[static_cast<size_t>(kb + c) * ldb + col], s);
      B[static_cast<size_t>(i) * ldb + col] -= s;
    }
    __syncthreads();
  }
}

__device__ int block_sum_int(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  if (warp_id() == 0) {
    int x = red[lane_id()];
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane_id() == 0) red[32] = x;
  }
  __syncthreads();
  const int r = red[32];
  __syncthreads();
  return r;
}

__device__ int block_max_int(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane_id() == 0) red[warp_id()] = v;
  __syncthreads();
  if (warp_id() == 0) {
    int x = red[lane_id()];
    for (int o = 16; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane_id() == 0) red[32] = x;
  }
  __syncthreads();
  const int r = red[32];
  __syncthreads();
  return r;
}

// Exclusive prefix count of flags[0..n) into pos[], returns the total.
__device__ int block_compact(const int* flag, int* pos, int n, int* red) {
  // simple two-level scan: each thread a contiguous chunk
  const int tid = threadIdx.x;
  const int chunk = (n + kThreads - 1) / kThreads;
  const int j0 = min(n, tid * chunk), j1 = min(n, j0 + chunk);
  int cnt = 0;
  for (int j = j0; j < j1; ++j) cnt += flag[j] != 0;
  // warp scan
  int x = cnt;
  const int lane = lane_id(), w = warp_id();
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = red[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    red[lane] = s;
  }
  __syncthreads();
  int o = (w > 0 ? red[w - 1] : 0) + x - cnt;
  const int total = red[31];
  for (int j = j0; j < j1; ++j)
    if (flag[j]) pos[o++] = j;
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kThreads, 1) nnls_bpp_kernel(const SolveParams p) {
  extern __shared__ float dyn[];
  __shared__ SolveSmem sm;
  __shared__ float redf[33];
  __shared__ int redi[33];
  const int h = blockIdx.x, tid = threadIdx.x;
  const int t = p.t, tp = p.t_pad;
  // shared vectors
  float* P = dyn;                                   // [t_pad * 33] panel
  float* x = P + static_cast<size_t>(tp) * 33;      // [t_pad]
  float* y = x + tp;
  float* cv = y + tp;
  float* rhs = cv + tp;
  int* F = reinterpret_cast<int*>(rhs + tp);        // passive flags
  int* Fidx = F + tp;                               // compact passive list
  int* flip = Fidx + tp;

  const float* G = p.G + static_cast<size_t>(h) * tp * tp;
  float* M = p.mat + static_cast<size_t>(h) * tp * tp;
  for (int j = tid; j < t; j += kThreads) {
    cv[j] = p.c[static_cast<size_t>(h) * tp + j];
    F[j] = 1;
    x[j] = 0.f;
  }
  __syncthreads();
  int ninf_best = t + 1, backup = 3, status = LC_OK_STATUS, it = 0;
  bool converged = false;
  for (it = 0; it < p.max_iter; ++it) {
    const int nF = block_compact(F, Fidx, t, redi);
    // gather G_FF (lower) and c_F
    for (size_t e = tid; e < static_cast<size_t>(nF) * nF; e += kThreads) {
      const int a = static_cast<int>(e / nF), b = static_cast<int>(e % nF);
      if (b <= a) M[static_cast<size_t>(a) * tp + b] = G[static_cast<size_t>(Fidx[a]) * tp + Fidx[b]];
    }
    for (int a = tid; a < nF; a += kThreads) rhs[a] = cv[Fidx[a]];
    __syncthreads();
    bool ok = cta_cholesky(M, nF, tp, P, sm);
    if (!ok) {
      // ridge fallback: regather with 1e-6 * mean(diag) added
      status = LC_SINGULAR_STATUS;
      float dsum = 0.f;
      for (int a = tid; a < nF; a += kThreads) dsum += G[static_cast<size_t>(Fidx[a]) * tp + Fidx[a]];
      for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
      if (lane_id() == 0) redf[warp_id()] = dsum;
      __syncthreads();
      if (tid == 0) {
        float s = 0.f;
        for (int k = 0; k < 32; ++k) s += redf[k];
        redf[32] = 1e-6f * s / max(nF, 1);
      }
      __syncthreads();
      const float ridge = redf[32];
      for (size_t e = tid; e < static_cast<size_t>(nF) * nF; e += kThreads) {
        const int a = static_cast<int>(e / nF), b = static_cast<int>(e % nF);
        if (b <= a)
          M[static_cast<size_t>(a) * tp + b] =
              G[static_cast<size_t>(Fidx[a]) * tp + Fidx[b]] + (a == b ? ridge : 0.f);
      }
      __syncthreads();
      cta_cholesky(M, nF, tp, P, sm);
    }
    cta_chol_solve(M, nF, tp, rhs, 1, 1);
    for (int j = tid; j < t; j += kThreads) x[j] = 0.f;
    __syncthreads();
    for (int a = tid; a < nF; a += kThreads) x[Fidx[a]] = rhs[a];
    __syncthreads();
    // y = G x - c and the infeasible set
    const int warp = warp_id(), lane = lane_id();
    for (int j = warp; j < t; j += kThreads / 32) {
      const float* g = G + static_cast<size_t>(j) * tp;
      float s = 0.f, sa = 0.f;
      for (int k = lane; k < t; k += 32) {
        const float v = g[k] * x[k];
        s += v;
        sa += fabsf(v);
      }
      for (int o = 16; o > 0; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
      }
      if (lane == 0) {
        const float yj = s - cv[j];
        y[j] = yj;
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
  // outputs
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
  __shared__ SolveSmem sm;
  __shared__ float redf[33];
  const int h = blockIdx.x, tid = threadIdx.x;
  const int t = p.t, tp = p.t_pad, dv = p.d_v;
  float* P = dyn;
  const float* Hm = p.Hm + static_cast<size_t>(h) * tp * tp;
  float* M = p.mat + static_cast<size_t>(h) * tp * tp;
  float* B = const_cast<float*>(p.R) + static_cast<size_t>(h) * tp * dv;  // solved in place
  const float* w = p.w + static_cast<size_t>(h) * t;
  const float* Vc = p.Vc + static_cast<size_t>(h) * tp * dv;
  // system with identity rows for zero-weight keys
  for (size_t e = tid; e < static_cast<size_t>(t) * t; e += kThreads) {
    const int a = static_cast<int>(e / t), b = static_cast<int>(e % t);
    if (b <= a) {
      const bool za = !(w[a] > 0.f), zb = !(w[b] > 0.f);
      float v = Hm[static_cast<size_t>(a) * tp + b];
      if (za || zb) v = (a == b) ? 1.f : 0.f;
      M[static_cast<size_t>(a) * tp + b] = v;
    }
  }
  for (size_t e = tid; e < static_cast<size_t>(t) * dv; e += kThreads) {
    const int a = static_cast<int>(e / dv);
    if (!(w[a] > 0.f)) B[e] = Vc[e];
  }
  __syncthreads();
  int status = LC_OK_STATUS;
  if (!cta_cholesky(M, t, tp, P, sm)) {
    status = LC_SINGULAR_STATUS;
    float dsum = 0.f;
    for (int a = tid; a < t; a += kThreads)
      dsum += (w[a] > 0.f) ? Hm[static_cast<size_t>(a) * tp + a] : 1.f;
    for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
    if (lane_id() == 0) redf[warp_id()] = dsum;
    __syncthreads();
    if (tid == 0) {
      float s = 0.f;
      for (int k = 0; k < 32; ++k) s += redf[k];
      redf[32] = 1e-6f * s / t;
    }
    __syncthreads();
    const float ridge = redf[32];
    for (size_t e = tid; e < static_cast<size_t>(t) * t; e += kThreads) {
      const int a = static_cast<int>(e / t), b = static_cast<int>(e % t);
      if (b <= a) {
        const bool za = !(w[a] > 0.f), zb = !(w[b] > 0.f);
        float v = Hm[static_cast<size_t>(a) * tp + b];
        if (za || zb) v = (a == b) ? 1.f : 0.f;
        if (a == b) v += ridge;
        M[static_cast<size_t>(a) * tp + b] = v;
      }
    }
    __syncthreads();
    cta_cholesky(M, t, tp, P, sm);
  }
  cta_chol_solve(M, t, tp, B, dv, dv);
  for (size_t e = tid; e < static_cast<size_t>(t) * dv; e += kThreads)
    p.Cv[static_cast<size_t>(h) * t * dv + e] = B[e];
  if (tid == 0 && status != LC_OK_STATUS && p.head_status[h] == LC_OK_STATUS)
    p.head_status[h] = status;
}

}  // namespace

cudaError_t launch_nnls(const SolveParams& p, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(p.t_pad) * 33 * 4 + 4 * p.t_pad * 4 + 3 * p.t_pad * 4;
  cudaError_t e = cudaFuncSetAttribute(nnls_bpp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  nnls_bpp_kernel<<<p.H, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_ols(const OlsParams& p, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(p.t_pad) * 33 * 4;
  cudaError_t e = cudaFuncSetAttribute(ols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  ols_kernel<<<p.H, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace lc
