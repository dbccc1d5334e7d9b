// Decode-time consumer of a compacted cache and the held-out error metrics.
//
// Attention of a query over a compacted cache plus the tokens appended after
// it ("Latent Compaction with Test-Time Training", §3.1 "Handling Subsequent
// Tokens", Eq. (4)-(5), and Appendix A.2 "Normalizer Computation and
// Storage"): the compacted entries carry their biases beta_j (an entry with
// beta_j = -inf is excluded), the appended entries carry none and are visible
// to row r only below n_vis[r].  Eq. (5) is a single softmax over both sets,
// so one online softmax runs over the compacted keys and then the appended
// ones; the result is the combined output A and log Z = log(Z_cmp + Z_new).
//
// One CTA takes 32 query rows of one head (8 warps x 4 rows).  Key tiles of
// 32 entries are staged in shared memory as fp32 (key rows padded to D + 1
// words, so that lane j reading key j's column c hits bank (j + c) mod 32);
// lane j scores key j for the warp's four rows, and every lane then
// accumulates D/32 output columns for the four rows.  Scores, exponentials
// and sums are fp32 (base 2 internally).  The kernel is bound by shared-
// memory traffic and latency, not by HBM: the staged tiles come from L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kDecWarps = 8;
constexpr int kDecRows = kRowsPerWarp * kDecWarps;  // rows per CTA
constexpr int kKeyTile = 32;

template <int D>
struct DecLayout {
  static constexpr int KS = D + 1;                     // padded key row (floats)
  static constexpr int OFF_Q = 0;                      // [32 rows][D]
  static constexpr int OFF_K = OFF_Q + kDecRows * D;   // [32 keys][D + 1]
  static constexpr int OFF_V = OFF_K + kKeyTile * KS;  // [32 keys][D]
  static constexpr int OFF_B = OFF_V + kKeyTile * D;   // [32] bias (base 2), -inf = excluded
  static constexpr int FLOATS = OFF_B + kKeyTile;
  static constexpr int SMEM = FLOATS * 4;
};

__device__ __forceinline__ float bf16_at(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

template <int D>
__global__ void __launch_bounds__(256) compact_attention_kernel(const CompactAttnParams p) {
  using L = DecLayout<D>;
  constexpr int DPL = D / 32;  // output columns per lane
  extern __shared__ float sm[];
  float* sQ = sm + L::OFF_Q;
  float* sK = sm + L::OFF_K;
  float* sV = sm + L::OFF_V;
  float* sB = sm + L::OFF_B;
  const int h = blockIdx.y, r0 = blockIdx.x * kDecRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float s2 = p.scale * kLog2e;

  const __nv_bfloat16* q = p.q + (static_cast<size_t>(h) * p.n) * D;
  for (int i = tid; i < kDecRows * D; i += 256) {
    const int r = r0 + i / D;
    sQ[i] = r < p.n ? bf16_at(q, static_cast<size_t>(r) * D + i % D) : 0.f;
  }
  int vis[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int r = r0 + warp * kRowsPerWarp + k;
    vis[k] = r < p.n ? (p.n_vis ? p.n_vis[static_cast<size_t>(h) * p.n + r] : p.n_new) : 0;
  }
  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DPL];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    m[k] = -kInf;
    l[k] = 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) acc[k][c] = 0.f;
  }

  const int ndoc = (p.t + kKeyTile - 1) / kKeyTile;
  const int nnew = (p.n_new + kKeyTile - 1) / kKeyTile;
  for (int tile = 0; tile < ndoc + nnew; ++tile) {
    const bool doc = tile < ndoc;
    const int j0 = (doc ? tile : tile - ndoc) * kKeyTile;
    const int nk = doc ? p.t : p.n_new;
    __syncthreads();  // previous tile consumed (and sQ written, first time)
    for (int i = tid; i < kKeyTile * D; i += 256) {
      const int j = i / D, c = i % D, jj = j0 + j;
      float kv = 0.f, vv = 0.f;
      if (jj < nk) {
        const size_t row = static_cast<size_t>(h) * nk + jj;
        if (doc) {
          kv = bf16_at(p.Ck, row * D + c);
          vv = p.Cv[row * D + c];
        } else {
          kv = bf16_at(p.Knew, row * D + c);
          vv = bf16_at(p.Vnew, row * D + c);
        }
      }
      sK[j * L::KS + c] = kv;
      sV[j * D + c] = vv;
    }
    if (tid < kKeyTile) {
      const int jj = j0 + tid;
      float b = -kInf;
      if (jj < nk) {
        if (doc) {
          const float be = p.beta[static_cast<size_t>(h) * p.t + jj];
          b = isfinite(be) ? be * kLog2e : -kInf;
        } else {
          b = 0.f;
        }
      }
      sB[tid] = b;
    }
    __syncthreads();

    const float bias = sB[lane];
    const float* kr = sK + lane * L::KS;
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const float* qr = sQ + (warp * kRowsPerWarp + k) * D;
      float dot = 0.f;
#pragma unroll 16
      for (int c = 0; c < D; ++c) dot = fmaf(qr[c], kr[c], dot);
      const bool seen = doc ? bias > -kInf : (j0 + lane < vis[k]);
      const float sc = seen ? fmaf(dot, s2, bias) : -kInf;
      float tm = sc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
      const float mn = fmaxf(m[k], tm);
      if (mn == -kInf) continue;  // nothing visible so far for this row
      const float pj = ex2(sc - mn);
      const float corr = ex2(m[k] - mn);
      float ps = pj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l[k] = fmaf(l[k], corr, ps);
      m[k] = mn;
#pragma unroll
      for (int c = 0; c < DPL; ++c) acc[k][c] *= corr;
#pragma unroll 8
      for (int j = 0; j < kKeyTile; ++j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
        const float* vr = sV + j * D + lane * DPL;
#pragma unroll
        for (int c = 0; c < DPL; ++c) acc[k][c] = fmaf(pb, vr[c], acc[k][c]);
      }
    }
  }

#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int r = r0 + warp * kRowsPerWarp + k;
    if (r >= p.n) continue;
    const size_t row = static_cast<size_t>(h) * p.n + r;
    const bool any = l[k] > 0.f;
    const float inv = any ? 1.f / l[k] : 0.f;
#pragma unroll
    for (int c = 0; c < DPL; ++c) p.A[row * D + lane * DPL + c] = acc[k][c] * inv;
    if (p.log_z && lane == 0) p.log_z[row] = any ? (m[k] + log2f(l[k])) * kLn2 : -kInf;
  }
}

// Per head: mean_i |lz_i - lse_i| and mean_i ||A_i - O_i||_2 over n rows.
template <int D>
__global__ void __launch_bounds__(256) heldout_reduce_kernel(const float* A, const float* lz,
                                                             const float* O, const float* lse,
                                                             int n, float* mass_err,
                                                             float* out_err) {
  __shared__ float red[2][8];
  const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float me = 0.f, oe = 0.f;
  for (int r = warp; r < n; r += 8) {
    const size_t row = static_cast<size_t>(h) * n + r;
    float ss = 0.f;
#pragma unroll
    for (int c = lane; c < D; c += 32) {
      const float e = A[row * D + c] - O[row * D + c];
      ss = fmaf(e, e, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) {
      oe += sqrtf(ss);
      me += fabsf(lz[row] - lse[row]);
    }
  }
  if (lane == 0) {
    red[0][warp] = me;
    red[1][warp] = oe;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f, b = 0.f;
    for (int w = 0; w < 8; ++w) {
      a += red[0][w];
      b += red[1][w];
    }
    mass_err[h] = a / n;
    out_err[h] = b / n;
  }
}

template <int D>
cudaError_t launch_ca_t(const CompactAttnParams& p, int H, cudaStream_t st) {
  using L = DecLayout<D>;
  auto kern = compact_attention_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((p.n + kDecRows - 1) / kDecRows, H);
  kern<<<grid, 256, L::SMEM, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compact_attention(int d, const CompactAttnParams& p, int H, cudaStream_t st) {
  if (p.n < 1 || H < 1) return cudaSuccess;
  switch (d) {
    case 64: return launch_ca_t<64>(p, H, st);
    case 128: return launch_ca_t<128>(p, H, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_heldout_reduce(int d, const float* A, const float* lz, const float* O,
                                  const float* lse, int H, int n, float* mass_err, float* out_err,
                                  cudaStream_t st) {
  switch (d) {
    case 64: heldout_reduce_kernel<64><<<H, 256, 0, st>>>(A, lz, O, lse, n, mass_err, out_err); break;
    case 128: heldout_reduce_kernel<128><<<H, 256, 0, st>>>(A, lz, O, lse, n, mass_err, out_err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace lc
