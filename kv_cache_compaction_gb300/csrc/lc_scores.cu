// Steps 2-3 of attention-matching compaction, plus the small data-movement
// kernels of the pipeline.
//
// Step 2 ("Latent Compaction with Test-Time Training", §3.2 Eq. (6)): each
// key's score is the largest softmax probability any reference query gives
// it.  Because exp is monotone the reduction runs in the log domain,
//   u_j = max_i (scale * q_i.k_j - lse_i),
// so the pass needs no exponential at all.  The layout is key-stationary:
// the tile S^T = K_tile Q_tile^T lands in tensor memory with one key per lane,
// so each thread reduces its own key over the query columns with one FMA and
// one max per score, and partial maxima over query splits merge with an
// atomic max on order-preserving integer codes (exact and order-free).
//
// Step 3 ("KV compaction" blog, section "Fast KV Compaction via Attention
// Matching": keep the keys with the highest attention): a per-head 4-pass
// 8-bit radix select finds the t-th largest code exactly; keys above it and
// the lowest-index keys equal to it are written in ascending index order.
#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kBK = 128;  // keys per CTA (TMEM lanes)
constexpr int kBQ = 128;  // queries per tile (TMEM columns per buffer)

template <int D_QK>
struct KSLayout {
  static constexpr int NQC = D_QK / 64;
  static constexpr int K_BYTES = kBK * D_QK * 2;
  static constexpr int QCHUNK = kBQ * 128;
  static constexpr int Q_BYTES = NQC * QCHUNK;
  static constexpr int NST = 2;
  static constexpr int OFF_Q = K_BYTES;
  static constexpr int OFF_L = OFF_Q + NST * Q_BYTES;
  static constexpr int OFF_BAR = OFF_L + NST * kBQ * 4;
  static constexpr int SMEM = 1024 + OFF_BAR + 128;
};

template <bool QK_BF16, int D_QK>
__global__ void __launch_bounds__(192, 2)
    key_scores_kernel(const __grid_constant__ CUtensorMap mK,
                      const __grid_constant__ CUtensorMap mQ, const KeyScoreParams p) {
  using L = KSLayout<D_QK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sK = base;
  uint8_t* sQ = base + L::OFF_Q;
  float* sL = reinterpret_cast<float*>(base + L::OFF_L);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* k_full = bars + 0;
  uint64_t* q_full = bars + 1;   // [2]
  uint64_t* q_empty = bars + 3;  // [2]
  uint64_t* d_full = bars + 5;   // [2]
  uint64_t* d_free = bars + 7;   // [2]
  uint64_t* mma_drain = bars + 9;  // MMA completion before exit
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  __shared__ volatile int abort_flag;

  const int warp = warp_id(), lane = lane_id();
  const int k0 = blockIdx.x * kBK, h = blockIdx.y;
  const int nqt = p.n_q_pad / kBQ;
  const int t0i = blockIdx.z * p.tiles_per_split;
  const int ntile = max(0, min(nqt, t0i + p.tiles_per_split) - t0i);

  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(k_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1 + 128);  // MMA commit + every epilogue thread
      mbar_init(&d_full[i], 1);
      mbar_init(&d_free[i], 128);
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
    if (lane == 0 && ntile > 0) {
      mbar_arrive_expect_tx(k_full, L::K_BYTES);
      for (int c = 0; c < L::NQC; ++c) tma_load_3d(sK + c * kBK * 128, &mK, k_full, 64 * c, k0, h);
      int issued = 0;
      for (int i = 0; i < ntile; ++i) {
        const int s = i & 1;
        if (i >= 2 && !wait_bar(&q_empty[s], ((i >> 1) - 1) & 1, &abort_flag, p.err)) break;
        const int q0 = (t0i + i) * kBQ;
        mbar_arrive_expect_tx(&q_full[s], L::Q_BYTES + kBQ * 4);
        for (int c = 0; c < L::NQC; ++c)
          tma_load_3d(sQ + s * L::Q_BYTES + c * L::QCHUNK, &mQ, &q_full[s], 64 * c, q0, h);
        bulk_g2s(sL + s * kBQ, p.lse_pad + static_cast<size_t>(h) * p.n_q_pad + q0, kBQ * 4,
                 &q_full[s]);
        issued = i + 1;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      drain_wait(k_full, 0);
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i)
        drain_wait(&q_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && ntile > 0) {
      constexpr uint32_t idesc = idesc_f16(kBK, kBQ, QK_BF16, false, false);
      bool ok = wait_bar(k_full, 0, &abort_flag, p.err);
      const uint32_t aK = smem_u32(sK);
      for (int i = 0; ok && i < ntile; ++i) {
        const int s = i & 1;
        if (!wait_bar(&q_full[s], (i >> 1) & 1, &abort_flag, p.err)) break;
        if (i >= 2 && !wait_bar(&d_free[s], ((i >> 1) - 1) & 1, &abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t aQ = smem_u32(sQ + s * L::Q_BYTES);
#pragma unroll
        for (int k = 0; k < D_QK / 16; ++k) {
          const uint64_t da = sdesc_sw128(aK + (k >> 2) * (kBK * 128) + (k & 3) * 32, 16, 1024);
          const uint64_t db = sdesc_sw128(aQ + (k >> 2) * L::QCHUNK + (k & 3) * 32, 16, 1024);
          umma_f16_ss(tbase + s * kBQ, da, db, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(&d_full[s]);
        umma_commit(&q_empty[s]);
      }
    }
  } else {
    const int wq = warp & 3;
    const int key = k0 + wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    float u8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) u8[e] = -kInf;
    bool ok = ntile > 0;
    for (int i = 0; ok && i < ntile; ++i) {
      const int s = i & 1;
      if (!wait_bar(&d_full[s], (i >> 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      if (!wait_bar(&q_full[s], (i >> 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      const float2* lt = reinterpret_cast<const float2*>(sL + s * kBQ);
      const float2 sc2 = make_float2(p.scale, p.scale);
      float v[kBQ];
      tmem_ld128(tbase + lane_off + s * kBQ, v);
#pragma unroll
      for (int e = 0; e < kBQ / 2; ++e) {
        const float2 l2 = lt[e];
        const float2 a = __ffma2_rn(make_float2(v[2 * e], v[2 * e + 1]), sc2,
                                    make_float2(-l2.x, -l2.y));
        u8[(2 * e) & 7] = fmaxf(u8[(2 * e) & 7], a.x);
        u8[(2 * e + 1) & 7] = fmaxf(u8[(2 * e + 1) & 7], a.y);
      }
      tc_fence_before();
      mbar_arrive(&d_free[s]);
      mbar_arrive(&q_empty[s]);
    }
    const float u = fmaxf(fmaxf(fmaxf(u8[0], u8[1]), fmaxf(u8[2], u8[3])),
                          fmaxf(fmaxf(u8[4], u8[5]), fmaxf(u8[6], u8[7])));
    if (ok && key < p.T) atomicMax(p.u_code + static_cast<size_t>(h) * p.T + key, order_code(u));
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 256);
}

// Two-tile variant for bf16 inputs: one CTA holds 256 keys as key tiles A
// and B that share every streamed query tile (halving the L2 traffic of
// re-streamed queries), with one reduction warpgroup per key tile.  Warps:
// 0 TMA, 1 MMA issue, 2..5 keys of tile A, 6..9 keys of tile B.  Tensor
// memory: D_A and D_B double-buffered, 128 columns each.
template <int D>
struct KS2Layout {
  static constexpr int NC = D / 64;
  static constexpr int K_BYTES = kBK * D * 2;    // one key tile
  static constexpr int QCHUNK = kBQ * 128;
  static constexpr int Q_BYTES = NC * QCHUNK;
  // query stages in flight: as many as fit beside the two key tiles (four
  // 32 KB stages for d = 128 keep about 28 B/clk of tile traffic per SM)
  static constexpr int NST = D == 128 ? 4 : 6;
  static constexpr int OFF_Q = 2 * K_BYTES;
  static constexpr int OFF_L = OFF_Q + NST * Q_BYTES;
  static constexpr int OFF_BAR = OFF_L + NST * kBQ * 4;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
};

// MODE 0: key scores only.  MODE 1 (mass): the same pass also reduces each
// key's column of unshifted scores to its log mass,
// L2_j = log2 sum_{i < n_rows} 2^(s log2e q_i.k_j).  MODE 2 (RMS): instead of
// the max, each key's column of squared probabilities,
// L2_j = log2 sum_i 2^(2 log2e a_ij), a_ij = s q_i.k_j - lse_i (padding rows,
// lse = +inf, drop out).  Modes 1 and 2 write one base-2 (max, sum) pair per
// query split to p.part for merge_key_lse.
template <int D, int MODE = 0>
__global__ void __launch_bounds__(320, 1)
    key_scores2_kernel(const __grid_constant__ CUtensorMap mK,
                       const __grid_constant__ CUtensorMap mQ, const KeyScoreParams p) {
  using L = KS2Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sK = base;
  uint8_t* sQ = base + L::OFF_Q;
  float* sL = reinterpret_cast<float*>(base + L::OFF_L);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* k_full = bars + 0;
  uint64_t* q_full = bars + 1;                // [NST]
  uint64_t* q_empty = bars + 1 + L::NST;      // [NST]
  uint64_t* d_full = bars + 1 + 2 * L::NST;   // [2]
  uint64_t* d_free = bars + 3 + 2 * L::NST;   // [2]
  uint64_t* mma_drain = bars + 5 + 2 * L::NST;  // MMA completion before exit
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  __shared__ volatile int abort_flag;

  const int warp = warp_id(), lane = lane_id();
  const int k0 = blockIdx.x * (2 * kBK), h = blockIdx.y;
  const int nqt = p.n_q_pad / kBQ;
  const int t0i = blockIdx.z * p.tiles_per_split;
  const int ntile = max(0, min(nqt, t0i + p.tiles_per_split) - t0i);

  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(k_full, 1);
    for (int i = 0; i < L::NST; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1 + 256);  // MMA commit + every reduction thread
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&d_full[b], 1);
      mbar_init(&d_free[b], 256);
    }
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;  // D_A(b) at 128b, D_B(b) at 256 + 128b

  if (warp == 0) {
    if (lane == 0 && ntile > 0) {
      mbar_arrive_expect_tx(k_full, 2 * L::K_BYTES);
      for (int x = 0; x < 2; ++x)
        for (int c = 0; c < L::NC; ++c)
          tma_load_3d(sK + x * L::K_BYTES + c * kBK * 128, &mK, k_full, 64 * c, k0 + x * kBK, h);
      int issued = 0;
      for (int i = 0; i < ntile; ++i) {
        const int s = i % L::NST;
        if (i >= L::NST && !wait_bar(&q_empty[s], ((i / L::NST) - 1) & 1, &abort_flag, p.err))
          break;
        const int q0 = (t0i + i) * kBQ;
        mbar_arrive_expect_tx(&q_full[s], L::Q_BYTES + kBQ * 4);
        for (int c = 0; c < L::NC; ++c)
          tma_load_3d(sQ + s * L::Q_BYTES + c * L::QCHUNK, &mQ, &q_full[s], 64 * c, q0, h);
        bulk_g2s(sL + s * kBQ, p.lse_pad + static_cast<size_t>(h) * p.n_q_pad + q0, kBQ * 4,
                 &q_full[s]);
        issued = i + 1;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      drain_wait(k_full, 0);
      for (int i = (issued > L::NST ? issued - L::NST : 0); i < issued; ++i)
        drain_wait(&q_full[i % L::NST], (i / L::NST) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && ntile > 0) {
      constexpr uint32_t idesc = idesc_f16(kBK, kBQ, true, false, false);
      bool ok = wait_bar(k_full, 0, &abort_flag, p.err);
      for (int i = 0; ok && i < ntile; ++i) {
        const int s = i % L::NST, b = i & 1;
        if (!wait_bar(&q_full[s], (i / L::NST) & 1, &abort_flag, p.err)) break;
        if (i >= 2 && !wait_bar(&d_free[b], ((i >> 1) - 1) & 1, &abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t aQ = smem_u32(sQ + s * L::Q_BYTES);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const uint32_t aK = smem_u32(sK + x * L::K_BYTES);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t da = sdesc_sw128(aK + (k >> 2) * (kBK * 128) + (k & 3) * 32, 16, 1024);
            const uint64_t db = sdesc_sw128(aQ + (k >> 2) * L::QCHUNK + (k & 3) * 32, 16, 1024);
            umma_f16_ss(tbase + x * 256 + b * kBQ, da, db, idesc, k > 0 ? 1u : 0u);
          }
        }
        umma_commit(&d_full[b]);
        umma_commit(&q_empty[s]);
      }
    }
  } else {
    const int x = (warp - 2) >> 2;
    const int wq = warp & 3;
    const int key = k0 + x * kBK + wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    float u8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) u8[e] = -kInf;
    float mass_m = -kInf, mass_s = 0.f;  // modes 1, 2: running max and sum of 2^(b - max)
    const float2 sc2 = make_float2(p.scale, p.scale);
    const float s2 = p.scale * kLog2e;
    bool ok = ntile > 0;
    for (int i = 0; ok && i < ntile; ++i) {
      const int s = i % L::NST, b = i & 1;
      if (!wait_bar(&d_full[b], (i >> 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      if (!wait_bar(&q_full[s], (i / L::NST) & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      const float2* lt = reinterpret_cast<const float2*>(sL + s * kBQ);
      float v[kBQ];
      tmem_ld128(tbase + x * 256 + b * kBQ + lane_off, v);
      tc_fence_before();
      mbar_arrive(&d_free[b]);
#pragma unroll
      for (int e = 0; e < kBQ / 2; ++e) {
        const float2 l2 = lt[e];
        const float2 a = __ffma2_rn(make_float2(v[2 * e], v[2 * e + 1]), sc2,
                                    make_float2(-l2.x, -l2.y));
        if constexpr (MODE == 2) {
          v[2 * e] = a.x * (2.f * kLog2e);
          v[2 * e + 1] = a.y * (2.f * kLog2e);
        } else {
          u8[(2 * e) & 7] = fmaxf(u8[(2 * e) & 7], a.x);
          u8[(2 * e + 1) & 7] = fmaxf(u8[(2 * e + 1) & 7], a.y);
        }
      }
      if constexpr (MODE == 2) {
        float bm0 = -kInf, bm1 = -kInf;
#pragma unroll
        for (int e = 0; e < kBQ; e += 2) {
          bm0 = fmaxf(bm0, v[e]);
          bm1 = fmaxf(bm1, v[e + 1]);
        }
        const float nm = fmaxf(mass_m, fmaxf(bm0, bm1));
        if (nm > -kInf) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int e = 0; e < kBQ; e += 2) {
            a0 += ex2(v[e] - nm);
            a1 += ex2(v[e + 1] - nm);
          }
          mass_s = mass_s * ex2(mass_m - nm) + (a0 + a1);
          mass_m = nm;
        }
      }
      if constexpr (MODE == 1) {
        // b = base-2 score; rows past n_rows (padding) carry no mass
        float bm0 = -kInf, bm1 = -kInf;
#pragma unroll
        for (int e = 0; e < kBQ; e += 2) {
          v[e] *= s2;
          v[e + 1] *= s2;
          bm0 = fmaxf(bm0, v[e]);
          bm1 = fmaxf(bm1, v[e + 1]);
        }
        const int rem = p.n_rows - (t0i + i) * kBQ;
        if (rem < kBQ) {
          bm0 = bm1 = -kInf;
#pragma unroll
          for (int e = 0; e < kBQ; ++e) {
            if (e >= rem) v[e] = -kInf;
            bm0 = fmaxf(bm0, v[e]);
          }
        }
        const float nm = fmaxf(mass_m, fmaxf(bm0, bm1));
        if (nm > -kInf) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int e = 0; e < kBQ; e += 2) {
            a0 += ex2(v[e] - nm);
            a1 += ex2(v[e + 1] - nm);
          }
          mass_s = mass_s * ex2(mass_m - nm) + (a0 + a1);
          mass_m = nm;
        }
      }
      mbar_arrive(&q_empty[s]);
    }
    const float u = fmaxf(fmaxf(fmaxf(u8[0], u8[1]), fmaxf(u8[2], u8[3])),
                          fmaxf(fmaxf(u8[4], u8[5]), fmaxf(u8[6], u8[7])));
    if (ok && key < p.T) {
      if constexpr (MODE != 2) atomicMax(p.u_code + static_cast<size_t>(h) * p.T + key, order_code(u));
      if constexpr (MODE != 0)
        p.part[(static_cast<size_t>(blockIdx.z) * gridDim.y + h) * p.T + key] =
            make_float2(mass_m, mass_s);
    }
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int D, int MODE = 0>
cudaError_t launch_ks2_t(const CUtensorMap& mK, const CUtensorMap& mQ, const KeyScoreParams& p,
                         int H, int nsplit, cudaStream_t st) {
  using L = KS2Layout<D>;
  auto kern = key_scores2_kernel<D, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((p.T + 2 * kBK - 1) / (2 * kBK), H, nsplit);
  kern<<<grid, 320, L::SMEM, st>>>(mK, mQ, p);
  return cudaGetLastError();
}

template <bool QK_BF16, int D_QK>
cudaError_t launch_ks_t(const CUtensorMap& mK, const CUtensorMap& mQ, const KeyScoreParams& p,
                        int H, int nsplit, cudaStream_t st) {
  using L = KSLayout<D_QK>;
  auto kern = key_scores_kernel<QK_BF16, D_QK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((p.T + kBK - 1) / kBK, H, nsplit);
  kern<<<grid, 192, L::SMEM, st>>>(mK, mQ, p);
  return cudaGetLastError();
}


// ------------------------------------------------------------ small kernels
__global__ void convert_bf16_f16_kernel(const __nv_bfloat16* in, __half* out, size_t n) {
  // eight elements per step when both arrays are 16-byte aligned
  const bool vec = ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15) == 0;
  const size_t n8 = vec ? n / 8 : 0;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8; i += stride) {
    const uint4 a = reinterpret_cast<const uint4*>(in)[i];
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
      r[k] = f2_to_h2(lo, hi);
    }
    reinterpret_cast<uint4*>(out)[i] = make_uint4(r[0], r[1], r[2], r[3]);
  }
  for (size_t i = n8 * 8 + blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += stride)
    out[i] = __float2half_rn(__bfloat162float(in[i]));
}

__global__ void split_f32_kernel(const float* in, __half* hi, __half* lo, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    __half a, b;
    split_f16(in[i], a, b);
    hi[i] = a;
    lo[i] = b;
  }
}

__global__ void split_rows3_kernel(const float* in, __half* out, size_t rows, int d, int order) {
  const size_t n = rows * d;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = i / d;
    const int k = static_cast<int>(i % d);
    __half a, b;
    split_f16(in[i], a, b);
    __half* o = out + r * 3 * d;
    o[k] = a;
    o[d + k] = order == 0 ? b : a;
    o[2 * d + k] = order == 0 ? a : b;
  }
}

__global__ void fill_f32_kernel(float* p, size_t n, float v) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = v;
}

__global__ void pad_rows_kernel(const float* in, float* out, int H, int n, int n_pad, float pad) {
  const size_t tot = static_cast<size_t>(H) * n_pad;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < tot;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t h = i / n_pad;
    const int r = static_cast<int>(i % n_pad);
    out[i] = r < n ? in[h * n + r] : pad;
  }
}

__global__ void decode_kernel(const uint32_t* code, float* u, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    u[i] = order_decode(code[i]);
}

__global__ void encode_kernel(const float* u, uint32_t* code, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    code[i] = order_code(u[i]);
}

// dst[h][r] = src[h][idx[h][r]] for r < t, zero rows for t <= r < t_pad.
// One warp per destination row, 16-byte moves; with `hash` set, also the
// row's hash (row_word_mix over its 32-bit words, 16-bit elements) into
// hash[h * t_pad + r].
__global__ void gather_rows_kernel(const uint8_t* src, uint8_t* dst, const int32_t* idx, int H,
                                   int T, int t, int t_pad, int row_bytes, uint32_t* hash) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = lane_id();
  if (gw >= H * t_pad) return;
  const int h = gw / t_pad, r = gw % t_pad;
  uint4* d = reinterpret_cast<uint4*>(dst + static_cast<size_t>(gw) * row_bytes);
  const int n16 = row_bytes / 16;
  const int j = r < t ? idx[static_cast<size_t>(h) * t + r] : -1;
  uint32_t acc = 0u;
  if (j >= 0 && j < T) {
    const uint4* s = reinterpret_cast<const uint4*>(src + (static_cast<size_t>(h) * T + j) * row_bytes);
    for (int k = lane; k < n16; k += 32) {
      const uint4 v = s[k];
      d[k] = v;
      acc += row_word_mix(v.x, 4 * k) + row_word_mix(v.y, 4 * k + 1) +
             row_word_mix(v.z, 4 * k + 2) + row_word_mix(v.w, 4 * k + 3);
    }
  } else {
    for (int k = lane; k < n16; k += 32) d[k] = make_uint4(0, 0, 0, 0);
  }
  if (hash) {
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) hash[gw] = acc;
  }
}

__global__ void gather_v_kernel(const void* V, int in_dtype, const int32_t* idx, float* Vc, int H,
                                int T, int t, int t_pad, int d) {
  const size_t n = static_cast<size_t>(H) * t_pad * d;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(i % d);
    const size_t hr = i / d;
    const int r = static_cast<int>(hr % t_pad), h = static_cast<int>(hr / t_pad);
    float v = 0.f;
    const int j = r < t ? idx[static_cast<size_t>(h) * t + r] : -1;
    if (j >= 0 && j < T) {
      const size_t src = (static_cast<size_t>(h) * T + j) * d + k;
      v = in_dtype == 0 ? __bfloat162float(static_cast<const __nv_bfloat16*>(V)[src])
                        : static_cast<const float*>(V)[src];
    }
    Vc[i] = v;
  }
}

// Sum over the split partials p[z * stride], z < nsplit, four loads in flight,
// in a fixed order for every element (independent of the launch).
__device__ __forceinline__ float4 sum_splits(const float4* p, size_t stride, int nsplit) {
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  int z = 0;
  for (; z + 3 < nsplit; z += 4) {
    float4 u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) u[k] = p[static_cast<size_t>(z + k) * stride];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[k].x += u[k].x; acc[k].y += u[k].y; acc[k].z += u[k].z; acc[k].w += u[k].w;
    }
  }
  for (int k = 0; z < nsplit; ++z, ++k) {
    const float4 u = p[static_cast<size_t>(z) * stride];
    acc[k].x += u.x; acc[k].y += u.y; acc[k].z += u.z; acc[k].w += u.w;
  }
  return make_float4((acc[0].x + acc[1].x) + (acc[2].x + acc[3].x),
                     (acc[0].y + acc[1].y) + (acc[2].y + acc[3].y),
                     (acc[0].z + acc[1].z) + (acc[2].z + acc[3].z),
                     (acc[0].w + acc[1].w) + (acc[2].w + acc[3].w));
}

__global__ void reduce_partials_kernel(const float4* part, float4* out, int nsplit, size_t n4) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    out[i] = sum_splits(part + i, n4, nsplit);
  }
}

// Sum of the split partials of a symmetric [H][t_pad][t_pad] system whose
// builder wrote the upper block triangle: one CTA per 32 x 32 tile (ti <= tj)
// of one head sums the tile and writes it and, through shared memory, its
// transpose.
__global__ void __launch_bounds__(256) reduce_gram_kernel(const float* part, float* out,
                                                         int nsplit, int t_pad,
                                                         const float* cpart, float* cout) {
  __shared__ float tile[32][33];
  const int h = blockIdx.y;
  int ti = 0, rem = blockIdx.x;
  const int nt = t_pad / 32;
  if (rem == nt * (nt + 1) / 2) {
    // the CTA after the tiles sums the head's right-hand-side partials
    const size_t n4 = static_cast<size_t>(gridDim.y) * t_pad / 4;
    for (int i = threadIdx.x; i < t_pad / 4; i += blockDim.x) {
      const size_t e = static_cast<size_t>(h) * t_pad / 4 + i;
      reinterpret_cast<float4*>(cout)[e] =
          sum_splits(reinterpret_cast<const float4*>(cpart) + e, n4, nsplit);
    }
    return;
  }
  while (rem >= nt - ti) {
    rem -= nt - ti;
    ++ti;
  }
  const int tj = ti + rem;
  const int ty = threadIdx.x >> 3, tx = threadIdx.x & 7;
  const size_t tt = static_cast<size_t>(t_pad) * t_pad;
  const size_t off = static_cast<size_t>(h) * tt + static_cast<size_t>(ti * 32 + ty) * t_pad +
                     tj * 32 + tx * 4;
  const size_t stride4 = static_cast<size_t>(gridDim.y) * tt / 4;
  const float4 r = sum_splits(reinterpret_cast<const float4*>(part + off), stride4, nsplit);
  *reinterpret_cast<float4*>(out + off) = r;
  if (ti == tj) return;  // diagonal tiles hold both triangles already
  tile[ty][tx * 4 + 0] = r.x;
  tile[ty][tx * 4 + 1] = r.y;
  tile[ty][tx * 4 + 2] = r.z;
  tile[ty][tx * 4 + 3] = r.w;
  __syncthreads();
  const size_t toff = static_cast<size_t>(h) * tt + static_cast<size_t>(tj * 32 + ty) * t_pad +
                      ti * 32 + tx * 4;
  *reinterpret_cast<float4*>(out + toff) =
      make_float4(tile[tx * 4 + 0][ty], tile[tx * 4 + 1][ty], tile[tx * 4 + 2][ty],
                  tile[tx * 4 + 3][ty]);
}

// Copy the upper triangle to the lower one (the Gram builder writes the
// upper block triangle only).
__global__ void symmetrize_kernel(float* G, int H, int t_pad) {
  const size_t n = static_cast<size_t>(H) * t_pad * t_pad;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % t_pad);
    const size_t hr = i / t_pad;
    const int r = static_cast<int>(hr % t_pad);
    if (r > c) {
      const size_t h = hr / t_pad;
      G[i] = G[(h * t_pad + c) * t_pad + r];
    }
  }
}

// Per-query shift and right-hand side of the mass fit, base 2:
// rowsh2 = m * log2(e) (+inf in padded rows), row_b = exp(lse - m) (0 there).
// Per-query shift and mass of the mass system and, when colb2 is given, its
// per-key base-2 biases (0 for the t kept keys, -inf for the padding): one
// launch for both.
__global__ void mass_rows_kernel(const float* m_pad, const float* lse_pad, float* rowsh2,
                                 float* row_b, int H, int n_q, int n_q_pad, float* colb2, int t,
                                 int t_pad) {
  const size_t n = static_cast<size_t>(H) * n_q_pad;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n; i += stride) {
    const int r = static_cast<int>(i % n_q_pad);
    if (r < n_q) {
      rowsh2[i] = m_pad[i] * kLog2e;
      row_b[i] = ex2((lse_pad[i] - m_pad[i]) * kLog2e);
    } else {
      rowsh2[i] = kInf;
      row_b[i] = 0.f;
    }
  }
  if (colb2) {
    const size_t nc = static_cast<size_t>(H) * t_pad;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < nc; i += stride)
      colb2[i] = static_cast<int>(i % t_pad) < t ? 0.f : -kInf;
  }
}

__global__ void fill_colb2_kernel(float* colb2, int H, int t, int t_pad) {
  const size_t n = static_cast<size_t>(H) * t_pad;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    colb2[i] = static_cast<int>(i % t_pad) < t ? 0.f : -kInf;
}

__global__ void merge_key_lse_kernel(const float2* part, float* L2, int nsplit, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float m = -kInf;
    for (int z = 0; z < nsplit; ++z) m = fmaxf(m, part[z * n + i].x);
    float sum = 0.f;
    if (m > -kInf)
      for (int z = 0; z < nsplit; ++z) {
        const float2 q = part[z * n + i];
        if (q.x > -kInf) sum += q.y * ex2(q.x - m);
      }
    L2[i] = m > -kInf ? m + log2f(sum) : -kInf;
  }
}

__global__ void merge_row_lse_kernel(const float2* part, float* out, int nsplit, int n, int n_pad,
                                     size_t total) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    if (static_cast<int>(i % n_pad) >= n) {
      out[i] = kInf;
      continue;
    }
    float m = -kInf;
    for (int z = 0; z < nsplit; ++z) m = fmaxf(m, part[z * total + i].x);
    float sum = 0.f;
    if (m > -kInf)
      for (int z = 0; z < nsplit; ++z) {
        const float2 q = part[z * total + i];
        if (q.x > -kInf) sum += q.y * ex2(q.x - m);
      }
    out[i] = m > -kInf ? m + log2f(sum) : -kInf;
  }
}

// u_j = log of the RMS probability = (L2_j ln 2 - ln n) / 2, as an order
// code for the selection and optionally as a float.
__global__ void rms_finish_kernel(const float* L2, float half_log_n, uint32_t* code, float* u,
                                  size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float v = 0.5f * L2[i] * kLn2 - half_log_n;
    if (code) code[i] = order_code(v);
    if (u) u[i] = v;
  }
}

__global__ void scale_f32_kernel(const float* in, float* out, size_t n, float mul) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    out[i] = in[i] * mul;
}

__global__ void compose_idx_kernel(const int32_t* short_idx, const int32_t* pos, int32_t* idx,
                                   uint8_t* chosen, int H, int kt, int t) {
  const size_t n = static_cast<size_t>(H) * t;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t h = i / t;
    const int r = pos[i];
    const bool ok = r >= 0 && r < kt;
    idx[i] = ok ? short_idx[h * kt + r] : -1;
    if (ok) chosen[h * kt + r] = 1;
  }
}

// Base-2 log-sum-exp of get(i) over i < n, whole block (256 threads).
template <class F>
__device__ float block_lse2_256(F get, int n, float* red) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  float m = -kInf;
  for (int i = tid; i < n; i += 256) m = fmaxf(m, get(i));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[w] = m;
  __syncthreads();
  float M = -kInf;
  for (int k = 0; k < 8; ++k) M = fmaxf(M, red[k]);
  __syncthreads();
  float sum = 0.f;
  if (M > -kInf)
    for (int i = tid; i < n; i += 256) sum += ex2(get(i) - M);
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[w] = sum;
  __syncthreads();
  float S = 0.f;
  for (int k = 0; k < 8; ++k) S += red[k];
  __syncthreads();
  return M > -kInf ? M + log2f(S) : -kInf;
}

// One CTA per head.  D2 = log2 of the missing mass (the column masses of the
// shortlist keys that were not chosen), then for each chosen key
//   beta_j = ln(1 + 2^x),  x = D2 - log2 t - L2_j,
// evaluated as x ln2 + ln(1 + 2^-x) for x > 0 (no overflow); no missing
// mass gives beta = 0.
__global__ void __launch_bounds__(256) redistribute_beta_kernel(const float* L2,
                                                                const uint8_t* chosen,
                                                                const int32_t* pos, float* beta,
                                                                int kt, int t) {
  __shared__ float red[8];
  const int h = blockIdx.x, tid = threadIdx.x;
  const float* Lh = L2 + static_cast<size_t>(h) * kt;
  const uint8_t* ch = chosen + static_cast<size_t>(h) * kt;
  const float D2 = block_lse2_256([&](int j) { return ch[j] ? -kInf : Lh[j]; }, kt, red);
  const float log2t = log2f(static_cast<float>(t));
  for (int r = tid; r < t; r += 256) {
    const int j = pos[static_cast<size_t>(h) * t + r];
    float b = 0.f;
    if (D2 > -kInf && j >= 0 && j < kt) {
      const float x = D2 - log2t - Lh[j];
      b = x > 0.f ? x * kLn2 + log1pf(ex2(-x)) : log1pf(ex2(x));
    }
    beta[static_cast<size_t>(h) * t + r] = b;
  }
}

inline int grid_for(size_t n, int block = 256) {
  size_t g = (n + block - 1) / block;
  if (g > 152 * 16) g = 152 * 16;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_key_scores_mass(OperandMode mode, const CUtensorMap& mK,
                                   const CUtensorMap& mQ, const KeyScoreParams& p, int H,
                                   int nsplit, cudaStream_t st) {
  if (!p.part || !p.u_code) return cudaErrorInvalidValue;
  switch (mode) {
    case kBF16d128: return launch_ks2_t<128, 1>(mK, mQ, p, H, nsplit, st);
    case kBF16d64: return launch_ks2_t<64, 1>(mK, mQ, p, H, nsplit, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_key_scores_rms(OperandMode mode, const CUtensorMap& mK,
                                  const CUtensorMap& mQ, const KeyScoreParams& p, int H,
                                  int nsplit, cudaStream_t st) {
  if (!p.part) return cudaErrorInvalidValue;
  switch (mode) {
    case kBF16d128: return launch_ks2_t<128, 2>(mK, mQ, p, H, nsplit, st);
    case kBF16d64: return launch_ks2_t<64, 2>(mK, mQ, p, H, nsplit, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rms_finish(const float* L2, int n_rows, uint32_t* code, float* u, size_t n,
                              cudaStream_t st) {
  rms_finish_kernel<<<grid_for(n), 256, 0, st>>>(L2, 0.5f * logf(static_cast<float>(n_rows)),
                                                 code, u, n);
  return cudaGetLastError();
}

cudaError_t launch_merge_key_lse(const float2* part, float* L, int nsplit, int H, int T,
                                 cudaStream_t st) {
  const size_t n = static_cast<size_t>(H) * T;
  merge_key_lse_kernel<<<grid_for(n), 256, 0, st>>>(part, L, nsplit, n);
  return cudaGetLastError();
}

cudaError_t launch_merge_row_lse(const float2* part, float* lc2_pad, int nsplit, int H, int n,
                                 int n_pad, cudaStream_t st) {
  const size_t total = static_cast<size_t>(H) * n_pad;
  merge_row_lse_kernel<<<grid_for(total), 256, 0, st>>>(part, lc2_pad, nsplit, n, n_pad, total);
  return cudaGetLastError();
}

cudaError_t launch_scale_f32(const float* in, float* out, size_t n, float mul, cudaStream_t st) {
  scale_f32_kernel<<<grid_for(n), 256, 0, st>>>(in, out, n, mul);
  return cudaGetLastError();
}

cudaError_t launch_compose_idx(const int32_t* short_idx, const int32_t* pos, int32_t* idx,
                               uint8_t* chosen, int H, int kt, int t, cudaStream_t st) {
  compose_idx_kernel<<<grid_for(static_cast<size_t>(H) * t), 256, 0, st>>>(short_idx, pos, idx,
                                                                            chosen, H, kt, t);
  return cudaGetLastError();
}

cudaError_t launch_redistribute_beta(const float* L2, const uint8_t* chosen, const int32_t* pos,
                                     float* beta, int H, int kt, int t, cudaStream_t st) {
  redistribute_beta_kernel<<<H, 256, 0, st>>>(L2, chosen, pos, beta, kt, t);
  return cudaGetLastError();
}

cudaError_t launch_key_scores(OperandMode mode, const CUtensorMap& mK, const CUtensorMap& mQ,
                              const KeyScoreParams& p, int H, int nsplit, cudaStream_t st) {
  switch (mode) {
    case kBF16d128: return launch_ks2_t<128>(mK, mQ, p, H, nsplit, st);
    case kBF16d64: return launch_ks2_t<64>(mK, mQ, p, H, nsplit, st);
    case kSplitF16d64: return launch_ks_t<false, 192>(mK, mQ, p, H, nsplit, st);
  }
  return cudaErrorInvalidValue;
}

int key_scores_smem(OperandMode mode) {
  switch (mode) {
    case kBF16d128: return KS2Layout<128>::SMEM;
    case kBF16d64: return KS2Layout<64>::SMEM;
    case kSplitF16d64: return KSLayout<192>::SMEM;
  }
  return 0;
}

cudaError_t launch_convert_bf16_to_f16(const __nv_bfloat16* in, __half* out, size_t n,
                                       cudaStream_t st) {
  convert_bf16_f16_kernel<<<grid_for(n / 8 + 1), 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

cudaError_t launch_split_f32(const float* in, __half* hi, __half* lo, size_t n, cudaStream_t st) {
  split_f32_kernel<<<grid_for(n), 256, 0, st>>>(in, hi, lo, n);
  return cudaGetLastError();
}

cudaError_t launch_split_rows3(const float* in, __half* out, size_t rows, int d, int qk_order,
                               cudaStream_t st) {
  split_rows3_kernel<<<grid_for(rows * d), 256, 0, st>>>(in, out, rows, d, qk_order);
  return cudaGetLastError();
}

cudaError_t launch_fill_f32(float* p, size_t n, float v, cudaStream_t st) {
  fill_f32_kernel<<<grid_for(n), 256, 0, st>>>(p, n, v);
  return cudaGetLastError();
}

cudaError_t launch_pad_rows(const float* in, float* out, int H, int n, int n_pad, float pad,
                            cudaStream_t st) {
  pad_rows_kernel<<<grid_for(static_cast<size_t>(H) * n_pad), 256, 0, st>>>(in, out, H, n, n_pad,
                                                                          pad);
  return cudaGetLastError();
}

cudaError_t launch_decode_scores(const uint32_t* code, float* u, size_t n, cudaStream_t st) {
  decode_kernel<<<grid_for(n), 256, 0, st>>>(code, u, n);
  return cudaGetLastError();
}

cudaError_t launch_encode_scores(const float* u, uint32_t* code, size_t n, cudaStream_t st) {
  encode_kernel<<<grid_for(n), 256, 0, st>>>(u, code, n);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* src, void* dst, const int32_t* idx, int H, int T,
                               int t, int t_pad, int row_bytes, cudaStream_t st, uint32_t* hash) {
  const int warps = H * t_pad;
  gather_rows_kernel<<<(warps * 32 + 255) / 256, 256, 0, st>>>(
      static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), idx, H, T, t, t_pad,
      row_bytes, hash);
  return cudaGetLastError();
}

cudaError_t launch_gather_v(const void* V, int in_dtype, const int32_t* idx, float* Vc, int H,
                            int T, int t, int t_pad, int d, cudaStream_t st) {
  gather_v_kernel<<<grid_for(static_cast<size_t>(H) * t_pad * d), 256, 0, st>>>(
      V, in_dtype, idx, Vc, H, T, t, t_pad, d);
  return cudaGetLastError();
}

cudaError_t launch_reduce_partials(const float* part, float* out, int nsplit, size_t n,
                                   cudaStream_t st) {
  if (n % 4) return cudaErrorInvalidValue;
  reduce_partials_kernel<<<grid_for(n / 4), 256, 0, st>>>(reinterpret_cast<const float4*>(part),
                                                          reinterpret_cast<float4*>(out), nsplit,
                                                          n / 4);
  return cudaGetLastError();
}

cudaError_t launch_reduce_gram(const float* part, float* out, int nsplit, int H, int t_pad,
                               cudaStream_t st, const float* cpart, float* cout) {
  if (t_pad % 32) return cudaErrorInvalidValue;
  const int nt = t_pad / 32;
  const int ntile = nt * (nt + 1) / 2;
  reduce_gram_kernel<<<dim3(ntile + (cpart ? 1 : 0), H), 256, 0, st>>>(part, out, nsplit, t_pad,
                                                                       cpart, cout);
  return cudaGetLastError();
}

cudaError_t launch_symmetrize(float* G, int H, int t_pad, cudaStream_t st) {
  symmetrize_kernel<<<grid_for(static_cast<size_t>(H) * t_pad * t_pad), 256, 0, st>>>(G, H, t_pad);
  return cudaGetLastError();
}

cudaError_t launch_mass_rows(const float* rowmax_pad, const float* lse_pad, float* rowsh2,
                             float* row_b, int H, int n_q, int n_q_pad, cudaStream_t st,
                             float* colb2, int t, int t_pad) {
  mass_rows_kernel<<<grid_for(static_cast<size_t>(H) * n_q_pad), 256, 0, st>>>(
      rowmax_pad, lse_pad, rowsh2, row_b, H, n_q, n_q_pad, colb2, t, t_pad);
  return cudaGetLastError();
}

cudaError_t launch_fill_colb2(float* colb2, int H, int t, int t_pad, cudaStream_t st) {
  fill_colb2_kernel<<<grid_for(static_cast<size_t>(H) * t_pad), 256, 0, st>>>(colb2, H, t, t_pad);
  return cudaGetLastError();
}

}  // namespace lc
