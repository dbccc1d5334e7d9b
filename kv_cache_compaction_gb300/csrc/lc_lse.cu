// Per-query log mass over a set of keys with per-key biases:
//   lc2_r = log2 sum_j 2^(scale*log2e * S_rj + colb2_j)   (base-2 units)
// the log-normaliser of the biased compact attention ("Latent Compaction with
// Test-Time Training", §3.1 Eq. (2)-(4)), used by step 5 and, with all-zero
// biases, for the fast path's lse over all keys and over the shortlist.
// Keys can be split over blockIdx.z (each CTA writes base-2 (max, sum)
// partials that merge_row_lse combines).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kBM = 128;

// ---------------------------------------------------------------------------
// Compact log mass of each query under the fitted biases:
//   lc2_r = log2 sum_j 2^(scale*log2e * S_rj + colb2_j)   (base-2 units)
// i.e. the log-normaliser of the biased compact attention ("Latent Compaction
// ...", §3.1 Eq. (2)-(4)).  Thread = query row; key blocks of 128 streamed.
template <bool QK_BF16, int D_QK>
struct CLLayout {
  static constexpr int NQC = D_QK / 64;
  static constexpr int Q_BYTES = kBM * D_QK * 2;
  static constexpr int KC_BYTES = 128 * D_QK * 2;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_BAR = OFF_K + 2 * KC_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
};

template <bool QK_BF16, int D_QK>
__global__ void __launch_bounds__(192, 1)
    compact_lse_kernel(const __grid_constant__ CUtensorMap mQ,
                       const __grid_constant__ CUtensorMap mKc, const CompactLseParams p) {
  using L = CLLayout<QK_BF16, D_QK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sQ = base;
  uint8_t* sK = base + L::OFF_K;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* bar_q = bars;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;   // [2]
  uint64_t* s_free = bars + 7;   // [2]
  uint64_t* mma_drain = bars + 9;  // MMA completion before exit
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  __shared__ volatile int abort_flag;
  const int warp = warp_id(), lane = lane_id();
  const int q0 = blockIdx.x * kBM, h = blockIdx.y;
  // key split z covers keys [key0, key0 + t_pad) of the key_stride padded keys
  const int kstride = p.key_stride > 0 ? p.key_stride : p.t_pad;
  const int key0 = blockIdx.z * p.t_pad;
  const int nkb = max(0, min(p.t_pad, kstride - key0)) / 128;
  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(bar_q, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
    }
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, L::Q_BYTES);
      for (int c = 0; c < L::NQC; ++c) tma_load_3d(sQ + c * kBM * 128, &mQ, bar_q, 64 * c, q0, h);
      int issued = 0;
      for (int j = 0; j < nkb; ++j) {
        const int s = j & 1;
        if (j >= 2 && !wait_bar(&k_empty[s], ((j >> 1) - 1) & 1, &abort_flag, p.err)) break;
        mbar_arrive_expect_tx(&k_full[s], L::KC_BYTES);
        for (int c = 0; c < L::NQC; ++c)
          tma_load_3d(sK + s * L::KC_BYTES + c * 128 * 128, &mKc, &k_full[s], 64 * c,
                      key0 + j * 128, h);
        issued = j + 1;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      drain_wait(bar_q, 0);
      for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
        drain_wait(&k_full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(kBM, 128, QK_BF16, false, false);
      bool ok = wait_bar(bar_q, 0, &abort_flag, p.err);
      for (int j = 0; ok && j < nkb; ++j) {
        const int s = j & 1;
        if (!wait_bar(&k_full[s], (j >> 1) & 1, &abort_flag, p.err)) break;
        if (j >= 2 && !wait_bar(&s_free[s], ((j >> 1) - 1) & 1, &abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK + s * L::KC_BYTES);
#pragma unroll
        for (int k = 0; k < D_QK / 16; ++k) {
          const uint64_t da = sdesc_sw128(aQ + (k >> 2) * (kBM * 128) + (k & 3) * 32, 16, 1024);
          const uint64_t db = sdesc_sw128(aK + (k >> 2) * (128 * 128) + (k & 3) * 32, 16, 1024);
          umma_f16_ss(tbase + s * 128, da, db, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[s]);
        umma_commit(&k_empty[s]);
      }
    }
  } else {
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float* cb = p.colb2 + static_cast<size_t>(h) * kstride + key0;
    float mref = -kInf, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      if (!wait_bar(&s_full[s], (j >> 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(tbase + lane_off + s * 128 + c * 32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = v[e];
      }
      tc_fence_before();
      mbar_arrive(&s_free[s]);
      float mx = -kInf;
#pragma unroll
      for (int k = 0; k < 128; ++k) {
        x[k] = fmaf(x[k], p.scale_log2, __ldg(cb + j * 128 + k));
        mx = fmaxf(mx, x[k]);
      }
      const float nref = fmaxf(mref, mx);
      if (nref > -kInf) {
        l *= ex2(mref - nref);
#pragma unroll
        for (int k = 0; k < 128; ++k) l += ex2(x[k] - nref);
        mref = nref;
      }
    }
    if (ok) {
      const int qr = q0 + row;
      if (qr < p.n_q_pad) {
        if (p.part)
          p.part[(static_cast<size_t>(blockIdx.z) * gridDim.y + h) * p.n_q_pad + qr] =
              make_float2(mref, l);
        else
          p.lc2_pad[static_cast<size_t>(h) * p.n_q_pad + qr] =
              (qr < p.n_q) ? mref + log2f(l) : kInf;
      }
    }
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 256);
}

// Compact log mass, bf16 inputs with at most 256 selected keys: the scores of
// a 128-query tile against all keys come from one chain of MMAs with N = t_pad
// (C_k resident in shared memory for the whole CTA); S is double-buffered in
// TMEM (2 x 256 columns), alternate tiles going to two pairs of epilogue
// warpgroups.  Within a pair each warpgroup reduces half of every query row
// with an online log-sum-exp (a thread per row): the reduction is a chain of
// TMEM load, row max and exponentials per 32 columns, bound by latency, so
// four warpgroups in flight instead of two keep the exponential unit busier.
// The second half's (max, sum) reaches the first through shared memory
// (mbarriers, two buffers per pair), which combines and writes the row.
// CTAs are persistent over a contiguous range of query tiles of one head.
template <int D>
struct CL2Layout {
  static constexpr int NC = D / 64;
  static constexpr int KC_BYTES = 256 * D * 2;  // up to 256 keys
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int OFF_Q = KC_BYTES;
  static constexpr int OFF_CB = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_X = OFF_CB + 256 * 4;            // [pair][buffer][row] float2
  static constexpr int OFF_BAR = OFF_X + 2 * 2 * kBM * 8;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  static constexpr int THREADS = 64 + 4 * 128;
};

template <int D>
__global__ void __launch_bounds__(CL2Layout<D>::THREADS, 1)
    compact_lse2_kernel(const __grid_constant__ CUtensorMap mQ,
                        const __grid_constant__ CUtensorMap mKc, const CompactLseParams p,
                        int tiles_per_split) {
  using L = CL2Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sK = base;
  uint8_t* sQ = base + L::OFF_Q;
  float* sCB = reinterpret_cast<float*>(base + L::OFF_CB);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* k_full = bars + 0;
  uint64_t* q_full = bars + 1;   // [2]
  uint64_t* q_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;   // [2]
  uint64_t* s_free = bars + 7;   // [2]
  uint64_t* mma_drain = bars + 9;  // MMA completion before exit
  uint64_t* x_full = bars + 10;  // [pair][buffer]: second half's row results written
  uint64_t* x_free = bars + 14;  // [pair][buffer]: read by the first half
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 18);
  float2* xch = reinterpret_cast<float2*>(base + L::OFF_X);
  __shared__ volatile int abort_flag;
  const int warp = warp_id(), lane = lane_id();
  const int h = blockIdx.y;
  const int nkb = p.t_pad / 128;
  // key chunk z: keys [key0, key0 + t_pad) of the key_stride padded keys
  const int kstride = p.key_stride > 0 ? p.key_stride : p.t_pad;
  const int key0 = blockIdx.z * p.t_pad;
  const int ntiles_all = p.n_q_pad / kBM;
  const int t0 = blockIdx.x * tiles_per_split;
  const int nt = max(0, min(ntiles_all, t0 + tiles_per_split) - t0);
  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(k_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 256);  // both halves have read S
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&x_full[i], 128);
      mbar_init(&x_free[i], 128);
    }
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(k_full, nkb * 128 * D * 2 + p.t_pad * 4);
      for (int c = 0; c < L::NC; ++c)
        for (int j = 0; j < nkb; ++j)
          tma_load_3d(sK + c * (p.t_pad * 128) + j * (128 * 128), &mKc, k_full, 64 * c,
                      key0 + j * 128, h);
      bulk_g2s(sCB, p.colb2 + static_cast<size_t>(h) * kstride + key0, p.t_pad * 4, k_full);
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int s = i & 1;
        if (i >= 2 && !wait_bar(&q_empty[s], ((i >> 1) - 1) & 1, &abort_flag, p.err)) break;
        mbar_arrive_expect_tx(&q_full[s], L::Q_BYTES);
        for (int c = 0; c < L::NC; ++c)
          tma_load_3d(sQ + s * L::Q_BYTES + c * kBM * 128, &mQ, &q_full[s], 64 * c,
                      (t0 + i) * kBM, h);
        issued = i + 1;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      drain_wait(k_full, 0);
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i)
        drain_wait(&q_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && nt > 0) {
      const uint32_t idesc = idesc_f16(kBM, p.t_pad, true, false, false);
      bool ok = wait_bar(k_full, 0, &abort_flag, p.err);
      for (int i = 0; ok && i < nt; ++i) {
        const int s = i & 1;
        if (!wait_bar(&q_full[s], (i >> 1) & 1, &abort_flag, p.err)) break;
        if (i >= 2 && !wait_bar(&s_free[s], ((i >> 1) - 1) & 1, &abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t aQ = smem_u32(sQ + s * L::Q_BYTES), aK = smem_u32(sK);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t da = sdesc_sw128(aQ + (k >> 2) * (kBM * 128) + (k & 3) * 32, 16, 1024);
          const uint64_t db =
              sdesc_sw128(aK + (k >> 2) * (p.t_pad * 128) + (k & 3) * 32, 16, 1024);
          umma_f16_ss(tbase + s * 256, da, db, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[s]);
        umma_commit(&q_empty[s]);
      }
    }
  } else {
    const int wg = (warp - 2) >> 2;
    const int g = wg & 1, hh = wg >> 1;  // tile parity, column half
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float s2 = p.scale_log2;
    const int half = p.t_pad / 2;
    bool ok = nt > g && wait_bar(k_full, 0, &abort_flag, p.err);
    for (int i = g; ok && i < nt; i += 2) {
      const int n = i >> 1, xb = g * 2 + (n & 1);
      if (!wait_bar(&s_full[g], n & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float mref = -kInf, l = 0.f;
      for (int c = 0; c < half / 32; ++c) {
        float v[32];
        tmem_ld32(tbase + g * 256 + hh * half + c * 32 + lane_off, v);
        const float4* cb4 = reinterpret_cast<const float4*>(sCB + hh * half + c * 32);
        float mx = -kInf;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 b = cb4[q];
          v[4 * q] = fmaf(v[4 * q], s2, b.x);
          v[4 * q + 1] = fmaf(v[4 * q + 1], s2, b.y);
          v[4 * q + 2] = fmaf(v[4 * q + 2], s2, b.z);
          v[4 * q + 3] = fmaf(v[4 * q + 3], s2, b.w);
          mx = fmaxf(fmaxf(mx, fmaxf(v[4 * q], v[4 * q + 1])), fmaxf(v[4 * q + 2], v[4 * q + 3]));
        }
        const float nref = fmaxf(mref, mx);
        if (nref > -kInf) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            a0 += ex2(v[e] - nref);
            a1 += ex2(v[e + 1] - nref);
          }
          l = l * ex2(mref - nref) + (a0 + a1);
          mref = nref;
        }
      }
      tc_fence_before();
      mbar_arrive(&s_free[g]);
      if (hh == 1) {
        // hand this half's (max, sum) to the first half
        if (n >= 2 && !wait_bar(&x_free[xb], ((n >> 1) - 1) & 1, &abort_flag, p.err)) {
          ok = false;
          break;
        }
        xch[xb * kBM + row] = make_float2(mref, l);
        mbar_arrive(&x_full[xb]);
        continue;
      }
      if (!wait_bar(&x_full[xb], (n >> 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      const float2 o = xch[xb * kBM + row];
      mbar_arrive(&x_free[xb]);
      {
        const float m2 = fmaxf(mref, o.x);
        if (m2 > -kInf) {
          l = (mref > -kInf ? l * ex2(mref - m2) : 0.f) + (o.x > -kInf ? o.y * ex2(o.x - m2) : 0.f);
          mref = m2;
        }
      }
      const int qr = (t0 + i) * kBM + row;
      if (qr < p.n_q_pad) {
        if (p.part)
          p.part[(static_cast<size_t>(blockIdx.z) * gridDim.y + h) * p.n_q_pad + qr] =
              make_float2(mref, l);
        else
          p.lc2_pad[static_cast<size_t>(h) * p.n_q_pad + qr] =
              (qr < p.n_q) ? mref + log2f(l) : kInf;
      }
    }
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <bool QK_BF16, int D_QK>
cudaError_t launch_cl_t(const CUtensorMap& mQ, const CUtensorMap& mKc, const CompactLseParams& p,
                        int H, cudaStream_t st) {
  using L = CLLayout<QK_BF16, D_QK>;
  auto kern = compact_lse_kernel<QK_BF16, D_QK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  const int kstride = p.key_stride > 0 ? p.key_stride : p.t_pad;
  dim3 grid((p.n_q + kBM - 1) / kBM, H, (kstride + p.t_pad - 1) / p.t_pad);
  kern<<<grid, 192, L::SMEM, st>>>(mQ, mKc, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compact_lse_resident(OperandMode mode, const CUtensorMap& mQ,
                                        const CUtensorMap& mKc, const CompactLseParams& p, int H,
                                        int nsplit, cudaStream_t st) {
  if (p.t_pad > 256 || nsplit < 1) return cudaErrorInvalidValue;
  const int kstride = p.key_stride > 0 ? p.key_stride : p.t_pad;
  if (kstride % p.t_pad != 0 || (kstride > p.t_pad && !p.part)) return cudaErrorInvalidValue;
  const int ntiles = p.n_q_pad / kBM;
  const int tps = (ntiles + nsplit - 1) / nsplit;
  const int grid_x = (ntiles + tps - 1) / tps;
  auto go = [&](auto kern, int smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(grid_x, H, kstride / p.t_pad), 64 + 4 * 128, smem, st>>>(mQ, mKc, p, tps);
    return cudaGetLastError();
  };
  switch (mode) {
    case kBF16d128: return go(compact_lse2_kernel<128>, CL2Layout<128>::SMEM);
    case kBF16d64: return go(compact_lse2_kernel<64>, CL2Layout<64>::SMEM);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_compact_lse(OperandMode mode, const CUtensorMap& mQ, const CUtensorMap& mKc,
                               const CompactLseParams& p, int H, cudaStream_t st) {
  switch (mode) {
    case kBF16d128: return launch_cl_t<true, 128>(mQ, mKc, p, H, st);
    case kBF16d64: return launch_cl_t<true, 64>(mQ, mKc, p, H, st);
    case kSplitF16d64: return launch_cl_t<false, 192>(mQ, mKc, p, H, st);
  }
  return cudaErrorInvalidValue;
}

int compact_lse_smem(OperandMode mode) {
  switch (mode) {
    case kBF16d128: return CLLayout<true, 128>::SMEM;
    case kBF16d64: return CLLayout<true, 64>::SMEM;
    case kSplitF16d64: return CLLayout<false, 192>::SMEM;
  }
  return 0;
}

}  // namespace lc
