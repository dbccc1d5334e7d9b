// Step 1 of attention-matching compaction: full-cache statistics of every
// reference query ("Latent Compaction with Test-Time Training", §3
// Preliminaries, Eq. (1)): row max m, log mass lse and output O.
//
// One CTA owns 128 query rows of one KV head and streams the head's keys in
// tiles of BN.  Warp roles:
//   warp 0      TMA producer: the Q tile once, then K/V tiles into a 2-stage ring;
//   warp 1      tensor-core issuer: S_j = Q K_j^T into a double-buffered TMEM
//               accumulator, then O += P_j V_j with P in fp16 (for fp32
//               inputs P and V are split into fp16 hi + lo pairs);
//   warps 2..5  softmax: thread = query row; reads S_j from TMEM, keeps a
//               running row max and sum, writes P_j to shared memory.
// The exponent reference of a row moves only when the row max grows by more
// than 8 (base 2), so the O accumulator in TMEM is rescaled rarely; the final
// division by the row sum makes the result independent of the reference.
#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kBM = 128;

template <int D_QK, int D_V, int V_TERMS, int BN, int P_TERMS>
struct AttnLayout {
  static constexpr int NQC = D_QK / 64;
  static constexpr int NVC = D_V / 64;
  static constexpr int Q_BYTES = kBM * D_QK * 2;
  static constexpr int KCHUNK = BN * 128;
  static constexpr int K_BYTES = NQC * KCHUNK;
  static constexpr int V_BYTES = NVC * KCHUNK;
  static constexpr int STAGE = K_BYTES + V_TERMS * V_BYTES;
  static constexpr int NST = 2;
  static constexpr int PCHUNK = kBM * 128;
  static constexpr int P_BYTES = (BN / 64) * PCHUNK;
  static constexpr int OFF_STAGE = Q_BYTES;
  static constexpr int OFF_PHI = OFF_STAGE + NST * STAGE;
  static constexpr int OFF_PLO = OFF_PHI + P_BYTES;
  static constexpr int OFF_BAR = OFF_PLO + (P_TERMS == 2 ? P_BYTES : 0);
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
};

template <bool QK_BF16, int D_QK, int D_V, int V_TERMS, int BN, int P_TERMS>
__global__ void __launch_bounds__(192, 1)
    attn_stats_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                      const __grid_constant__ CUtensorMap mV,
                      const __grid_constant__ CUtensorMap mVlo, const AttnStatsParams p) {
  using L = AttnLayout<D_QK, D_V, V_TERMS, BN, P_TERMS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sQ = base;
  uint8_t* sStage = base + L::OFF_STAGE;
  uint8_t* sPhi = base + L::OFF_PHI;
  uint8_t* sPlo = base + L::OFF_PLO;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* bar_q = bars + 0;
  uint64_t* kv_full = bars + 1;             // [NST]
  uint64_t* kv_empty = bars + 1 + L::NST;   // [NST]
  uint64_t* s_full = bars + 1 + 2 * L::NST; // [2]
  uint64_t* s_free = s_full + 2;            // [2]
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* mma_drain = pv_done + 1;  // MMA completion before exit
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  __shared__ volatile int abort_flag;

  const int warp = warp_id(), lane = lane_id();
  const int q0 = blockIdx.x * kBM;
  const int h = blockIdx.y;
  const int nkt = (p.T + BN - 1) / BN;

  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::NST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tO = tbase + 2 * BN;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      mbar_arrive_expect_tx(bar_q, L::Q_BYTES);
      for (int c = 0; c < L::NQC; ++c) tma_load_3d(sQ + c * kBM * 128, &mQ, bar_q, 64 * c, q0, h);
      int issued = 0;
      for (int j = 0; j < nkt; ++j) {
        const int s = j % L::NST;
        if (j >= L::NST && !wait_bar(&kv_empty[s], ((j / L::NST) - 1) & 1, &abort_flag, p.err))
          break;
        uint8_t* st = sStage + s * L::STAGE;
        mbar_arrive_expect_tx(&kv_full[s], L::STAGE);
        for (int c = 0; c < L::NQC; ++c)
          tma_load_3d(st + c * L::KCHUNK, &mK, &kv_full[s], 64 * c, j * BN, h);
        for (int c = 0; c < L::NVC; ++c)
          tma_load_3d(st + L::K_BYTES + c * L::KCHUNK, &mV, &kv_full[s], 64 * c, j * BN, h);
        if (V_TERMS == 2)
          for (int c = 0; c < L::NVC; ++c)
            tma_load_3d(st + L::K_BYTES + L::V_BYTES + c * L::KCHUNK, &mVlo, &kv_full[s], 64 * c,
                        j * BN, h);
        issued = j + 1;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      drain_wait(bar_q, 0);
      for (int j = (issued > L::NST ? issued - L::NST : 0); j < issued; ++j)
        drain_wait(&kv_full[j % L::NST], (j / L::NST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBM, BN, QK_BF16, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kBM, D_V, false, false, true);
      const uint32_t aQ = smem_u32(sQ);
      bool ok = wait_bar(bar_q, 0, &abort_flag, p.err);
      auto issue_s = [&](int j) -> bool {
        const int s = j % L::NST, b = j & 1;
        if (!wait_bar(&kv_full[s], (j / L::NST) & 1, &abort_flag, p.err)) return false;
        if (j >= 2 && !wait_bar(&s_free[b], ((j >> 1) - 1) & 1, &abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t aK = smem_u32(sStage + s * L::STAGE);
#pragma unroll
        for (int k = 0; k < D_QK / 16; ++k) {
          const uint64_t da = sdesc_sw128(aQ + (k >> 2) * (kBM * 128) + (k & 3) * 32, 16, 1024);
          const uint64_t db = sdesc_sw128(aK + (k >> 2) * L::KCHUNK + (k & 3) * 32, 16, 1024);
          umma_f16_ss(tbase + b * BN, da, db, idesc_s, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nkt; ++j) {
        if (j + 1 < nkt && !issue_s(j + 1)) break;
        if (!wait_bar(p_full, j & 1, &abort_flag, p.err)) break;
        tc_fence_after();
        const int s = j % L::NST;
        const uint32_t aV = smem_u32(sStage + s * L::STAGE + L::K_BYTES);
        const uint32_t aPh = smem_u32(sPhi), aPl = smem_u32(sPlo);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint32_t poff = (k >> 2) * L::PCHUNK + (k & 3) * 32;
          const uint64_t dph = sdesc_sw128(aPh + poff, 16, 1024);
          const uint64_t dpl = sdesc_sw128(aPl + poff, 16, 1024);
          const uint64_t dv = sdesc_sw128(aV + k * 2048, L::KCHUNK, 1024);
          umma_f16_ss(tO, dph, dv, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
          if (P_TERMS == 2) umma_f16_ss(tO, dpl, dv, idesc_pv, 1u);
          if (V_TERMS == 2) {
            const uint64_t dvl = sdesc_sw128(aV + L::V_BYTES + k * 2048, L::KCHUNK, 1024);
            umma_f16_ss(tO, dph, dvl, idesc_pv, 1u);
          }
        }
        umma_commit(&kv_empty[s]);
        umma_commit(pv_done);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_ref = -kInf;   // exponent reference (base 2)
    float m_true = -kInf;  // exact running row max (base 2)
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int b = j & 1;
      if (!wait_bar(&s_full[b], (j >> 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float x[BN];
      if constexpr (BN == 128) {
        tmem_ld128(tbase + lane_off + b * BN, x);
      } else {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(tbase + lane_off + b * BN + c * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c * 32 + e] = v[e];
        }
      }
      tc_fence_before();
      mbar_arrive(&s_free[b]);
      const int valid = p.T - j * BN;
      if (valid < BN) {  // ragged last tile: keys past T do not exist
#pragma unroll
        for (int k = 0; k < BN; ++k)
          if (k >= valid) x[k] = -kInf;
      }
      // row max of the raw scores (scale > 0), eight independent chains
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = x[e];
#pragma unroll
      for (int k = 8; k < BN; k += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(m8[e], x[k + e]);
      const float mx =
          fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
      m_true = fmaxf(m_true, mx);
      const bool resc = mx > m_ref + 8.f;
      const float new_ref = resc ? mx : m_ref;
      const float alpha = resc ? ex2(m_ref - new_ref) : 1.f;
      // P buffer free and O up to date once the previous P.V has completed.
      if (j > 0) {
        if (!wait_bar(pv_done, (j - 1) & 1, &abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int c = 0; c < D_V / 32; ++c) {
            float o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tO + lane_off + c * 32, o);
          }
        }
      }
      m_ref = new_ref;
      // p = 2^(S * scale*log2e - m_ref): packed FMA, hardware exp2, eight
      // partial sums
      const float2 s2 = make_float2(sl2, sl2);
      const float2 nm2 = make_float2(-m_ref, -m_ref);
      float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
#pragma unroll
      for (int c8 = 0; c8 < BN / 8; ++c8) {
        float pv[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a = __ffma2_rn(make_float2(x[c8 * 8 + 2 * e], x[c8 * 8 + 2 * e + 1]), s2, nm2);
          pv[2 * e] = ex2(a.x);
          pv[2 * e + 1] = ex2(a.y);
          l4[e] = __fadd2_rn(l4[e], make_float2(pv[2 * e], pv[2 * e + 1]));
        }
        const uint32_t off = (c8 >> 3) * L::PCHUNK + sw128_offset(row, (c8 & 7) * 8);
        if (P_TERMS == 2) {
          uint4 hi, lo;
          split8(pv, hi, lo);
          *reinterpret_cast<uint4*>(sPhi + off) = hi;
          *reinterpret_cast<uint4*>(sPlo + off) = lo;
        } else {
          *reinterpret_cast<uint4*>(sPhi + off) = pack8_f16(pv);
        }
      }
      l = fmaf(l, alpha, ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) +
                             ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y)));
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && wait_bar(pv_done, (nkt - 1) & 1, &abort_flag, p.err)) {
      tc_fence_after();
      const int qr = q0 + row;
      const size_t hq = static_cast<size_t>(h) * p.n_q;
      const float inv_l = 1.f / l;
      if (qr < p.n_q) {
        const float m_nat = m_true * kLn2;
        const float lse_nat = (m_ref + log2f(l)) * kLn2;
        if (p.rowmax) p.rowmax[hq + qr] = m_nat;
        if (p.lse) p.lse[hq + qr] = lse_nat;
        if (p.rowmax_pad) p.rowmax_pad[static_cast<size_t>(h) * p.n_q_pad + qr] = m_nat;
        if (p.lse_pad) p.lse_pad[static_cast<size_t>(h) * p.n_q_pad + qr] = lse_nat;
      } else if (qr < p.n_q_pad) {
        if (p.rowmax_pad) p.rowmax_pad[static_cast<size_t>(h) * p.n_q_pad + qr] = kInf;
        if (p.lse_pad) p.lse_pad[static_cast<size_t>(h) * p.n_q_pad + qr] = kInf;
      }
#pragma unroll
      for (int c = 0; c < D_V / 32; ++c) {
        float o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        if (qr < p.n_q) {
          const size_t off = (hq + qr) * D_V + c * 32;
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= inv_l;
          if (p.O) {
            float4* dst = reinterpret_cast<float4*>(p.O + off);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          }
          if (p.O_hi) {
            uint4* dh = reinterpret_cast<uint4*>(p.O_hi + off);
            uint4* dl = reinterpret_cast<uint4*>(p.O_lo + off);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 hi, lo;
              split8(o + 8 * e, hi, lo);
              dh[e] = hi;
              dl[e] = lo;
            }
          }
        }
      }
    }
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// Two-tile pass with P kept in tensor memory (bf16 inputs, P.V in one fp16
// product).  One CTA owns 256 query rows as two tiles, each with its own
// softmax warpgroup.  The softmax writes P_x (fp16 pairs) over the first 64
// columns of its score buffer S_x, and P_x V_j reads it from tensor memory
// (A operand in TMEM), so P never touches shared memory; the next scores
// S_x(j+1) are issued after P_x V_j (same thread, in order).  Completion of
// S_x(j+1) therefore also means P_x V_j is done: the softmax rescales O_x and
// overwrites the buffer with no further wait.  K and V tiles stream through
// a 5-slot ring (load n: K_{n/2} if n is even, V_{n/2} if odd).  Tensor
// memory: S_A, S_B, O_A, O_B, 128 columns each.  Warps: 0 TMA, 1 MMA issue,
// 2..5 softmax of tile A, 6..9 softmax of tile B.
template <int D>
struct Attn3Layout {
  static constexpr int NC = D / 64;
  static constexpr int BN = 128;
  static constexpr int NSLOT = 5;
  static constexpr int Q_BYTES = kBM * D * 2;  // one tile
  static constexpr int SLOT = BN * D * 2;      // one K or V tile
  static constexpr int OFF_RING = 2 * Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * SLOT;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
};

__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    attn_stats3_kernel(const __grid_constant__ CUtensorMap mQ,
                       const __grid_constant__ CUtensorMap mK,
                       const __grid_constant__ CUtensorMap mV, const AttnStatsParams p) {
  using L = Attn3Layout<D>;
  constexpr int BN = L::BN;
  constexpr int NS = L::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sQ = base;
  uint8_t* sRing = base + L::OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* r_full = bars + 1;            // [NS]
  uint64_t* r_empty = bars + 1 + NS;      // [NS]
  uint64_t* s_full = bars + 1 + 2 * NS;   // [2] tile A, B
  uint64_t* p_full = bars + 3 + 2 * NS;   // [2]
  uint64_t* pv_done = bars + 5 + 2 * NS;  // [2]
  uint64_t* mma_drain = bars + 7 + 2 * NS;  // MMA completion before exit
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  __shared__ volatile int abort_flag;

  const int warp = warp_id(), lane = lane_id();
  const int q0 = blockIdx.x * (2 * kBM);
  const int h = blockIdx.y;
  const int nkt = (p.T + BN - 1) / BN;

  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(q_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);
      mbar_init(&pv_done[x], 1);
    }
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;  // S_A 0, S_B 128, O_A 256, O_B 384

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mV);
      mbar_arrive_expect_tx(q_full, 2 * L::Q_BYTES);
      for (int x = 0; x < 2; ++x)
        for (int c = 0; c < L::NC; ++c)
          tma_load_3d(sQ + x * L::Q_BYTES + c * kBM * 128, &mQ, q_full, 64 * c, q0 + x * kBM, h);
      int issued = 0;
      for (int n = 0; n < 2 * nkt; ++n) {
        const int sl = n % NS;
        if (n >= NS && !wait_bar(&r_empty[sl], ((n / NS) - 1) & 1, &abort_flag, p.err)) break;
        uint8_t* dst = sRing + sl * L::SLOT;
        mbar_arrive_expect_tx(&r_full[sl], L::SLOT);
        const CUtensorMap* m = (n & 1) ? &mV : &mK;
        for (int c = 0; c < L::NC; ++c)
          tma_load_3d(dst + c * BN * 128, m, &r_full[sl], 64 * c, (n >> 1) * BN, h);
        issued = n + 1;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      drain_wait(q_full, 0);
      for (int n = (issued > NS ? issued - NS : 0); n < issued; ++n)
        drain_wait(&r_full[n % NS], (n / NS) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBM, BN, true, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kBM, D, false, false, true);
      bool ok = wait_bar(q_full, 0, &abort_flag, p.err);
      auto ring_ready = [&](int n) { return mbar_test_wait(&r_full[n % NS], (n / NS) & 1); };
      // S_x(j) = Q_x K_j^T
      auto issue_s = [&](int x, int j) {
        const uint32_t aQ = smem_u32(sQ + x * L::Q_BYTES);
        const uint32_t aK = smem_u32(sRing + ((2 * j) % NS) * L::SLOT);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t da = sdesc_sw128(aQ + (k >> 2) * (kBM * 128) + (k & 3) * 32, 16, 1024);
          const uint64_t db = sdesc_sw128(aK + (k >> 2) * (BN * 128) + (k & 3) * 32, 16, 1024);
          umma_f16_ss(tbase + x * 128, da, db, idesc_s, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[x]);
      };
      // O_x += P_x V_j, P_x in tensor memory (16 keys = 8 columns per step)
      auto issue_pv = [&](int x, int j) {
        const uint32_t aV = smem_u32(sRing + ((2 * j + 1) % NS) * L::SLOT);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t dv = sdesc_sw128(aV + k * 2048, BN * 128, 1024);
          umma_f16_ts(tbase + 256 + x * 128, tbase + x * 128 + k * 8, dv, idesc_pv,
                      (j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&pv_done[x]);
      };
      // Event loop over both tiles: S_x(0); then per j: P_x V_j once P_x(j)
      // is written, followed by S_x(j+1) once K_{j+1} has landed.  A ring
      // slot is released once both tiles have issued the product reading it.
      int ns[2] = {0, 0}, np[2] = {0, 0};
      int kr = 0, vr = 0;  // K and V loads released so far
      uint64_t t_last = globaltimer_ns();
      uint32_t spins = 0;
      while (ok && (np[0] < nkt || np[1] < nkt)) {
        bool did = false;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (np[x] < ns[x]) {  // scores issued, P.V pending
            const int j = np[x];
            if (mbar_test_wait(&p_full[x], j & 1) && ring_ready(2 * j + 1)) {
              tc_fence_after();
              issue_pv(x, j);
              ++np[x];
              did = true;
            }
          }
          if (ns[x] == np[x] && ns[x] < nkt && ring_ready(2 * ns[x])) {
            tc_fence_after();
            issue_s(x, ns[x]);
            ++ns[x];
            did = true;
          }
        }
        if (did) {
          for (; kr < min(ns[0], ns[1]); ++kr) umma_commit(&r_empty[(2 * kr) % NS]);
          for (; vr < min(np[0], np[1]); ++vr) umma_commit(&r_empty[(2 * vr + 1) % NS]);
          t_last = globaltimer_ns();
        } else if ((++spins & 63u) == 0) {
          if (abort_flag) break;
          if (*reinterpret_cast<volatile uint32_t*>(p.err) & kErrWaitTimeout) {
            abort_flag = 1;
            break;
          }
          if (globaltimer_ns() - t_last > kWaitLimitNs) {
            atomicOr(p.err, kErrWaitTimeout);
            abort_flag = 1;
            break;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = (warp - 2) >> 2;  // tile
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + x * 128, tO = tbase + 256 + x * 128;
    const float sl2 = p.scale_log2;
    float m_ref = -kInf, m_true = -kInf, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      if (!wait_bar(&s_full[x], j & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float xs[BN];
      tmem_ld128(tS + lane_off, xs);
      const int valid = p.T - j * BN;
      if (valid < BN) {
#pragma unroll
        for (int k = 0; k < BN; ++k)
          if (k >= valid) xs[k] = -kInf;
      }
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = xs[e];
#pragma unroll
      for (int k = 8; k < BN; k += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(m8[e], xs[k + e]);
      const float mx =
          fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
      m_true = fmaxf(m_true, mx);
      const bool resc = mx > m_ref + 8.f;
      const float new_ref = resc ? mx : m_ref;
      const float alpha = resc ? ex2(m_ref - new_ref) : 1.f;
      m_ref = new_ref;
      const float2 s2 = make_float2(sl2, sl2);
      const float2 nm2 = make_float2(-m_ref, -m_ref);
      float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      float pw[BN / 2];  // P as fp16 pairs (bit patterns), key 2c in the low half
#pragma unroll
      for (int c8 = 0; c8 < BN / 8; ++c8) {
        float pv[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a =
              __ffma2_rn(make_float2(xs[c8 * 8 + 2 * e], xs[c8 * 8 + 2 * e + 1]), s2, nm2);
          pv[2 * e] = ex2(a.x);
          pv[2 * e + 1] = ex2(a.y);
          l4[e] = __fadd2_rn(l4[e], make_float2(pv[2 * e], pv[2 * e + 1]));
        }
        const uint4 q = pack8_f16(pv);
        pw[c8 * 4 + 0] = __uint_as_float(q.x);
        pw[c8 * 4 + 1] = __uint_as_float(q.y);
        pw[c8 * 4 + 2] = __uint_as_float(q.z);
        pw[c8 * 4 + 3] = __uint_as_float(q.w);
      }
      l = fmaf(l, alpha, ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) +
                             ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y)));
      // S_x(j) complete implies P_x V_{j-1} complete: O may be rescaled and
      // the score buffer overwritten by P_x(j) right away
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(tO + lane_off + c * 32, o);
        }
      }
      {
        float w0[32], w1[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          w0[e] = pw[e];
          w1[e] = pw[32 + e];
        }
        tmem_st32(tS + lane_off, w0);
        tmem_st32(tS + lane_off + 32, w1);
      }
      tc_fence_before();
      mbar_arrive(&p_full[x]);
    }
    if (ok && wait_bar(&pv_done[x], (nkt - 1) & 1, &abort_flag, p.err)) {
      tc_fence_after();
      const int qr = q0 + x * kBM + row;
      const size_t hq = static_cast<size_t>(h) * p.n_q;
      const float inv_l = 1.f / l;
      if (qr < p.n_q) {
        const float m_nat = m_true * kLn2;
        const float lse_nat = (m_ref + log2f(l)) * kLn2;
        if (p.rowmax) p.rowmax[hq + qr] = m_nat;
        if (p.lse) p.lse[hq + qr] = lse_nat;
        if (p.rowmax_pad) p.rowmax_pad[static_cast<size_t>(h) * p.n_q_pad + qr] = m_nat;
        if (p.lse_pad) p.lse_pad[static_cast<size_t>(h) * p.n_q_pad + qr] = lse_nat;
      } else if (qr < p.n_q_pad) {
        if (p.rowmax_pad) p.rowmax_pad[static_cast<size_t>(h) * p.n_q_pad + qr] = kInf;
        if (p.lse_pad) p.lse_pad[static_cast<size_t>(h) * p.n_q_pad + qr] = kInf;
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        if (qr < p.n_q) {
          const size_t off = (hq + qr) * D + c * 32;
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= inv_l;
          if (p.O) {
            float4* dst = reinterpret_cast<float4*>(p.O + off);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          }
          if (p.O_hi) {
            uint4* dh = reinterpret_cast<uint4*>(p.O_hi + off);
            uint4* dl = reinterpret_cast<uint4*>(p.O_lo + off);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 hi, lo;
              split8(o + 8 * e, hi, lo);
              dh[e] = hi;
              dl[e] = lo;
            }
          }
        }
      }
    }
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <bool QK_BF16, int D_QK, int D_V, int V_TERMS, int BN, int P_TERMS>
cudaError_t launch_attn_t(const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                          const CUtensorMap& mVlo, const AttnStatsParams& p, int H,
                          cudaStream_t st) {
  using L = AttnLayout<D_QK, D_V, V_TERMS, BN, P_TERMS>;
  auto kern = attn_stats_kernel<QK_BF16, D_QK, D_V, V_TERMS, BN, P_TERMS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((p.n_q + kBM - 1) / kBM, H);
  kern<<<grid, 192, L::SMEM, st>>>(mQ, mK, mV, mVlo, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_attn3_t(const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                           const AttnStatsParams& p, int H, cudaStream_t st) {
  using L = Attn3Layout<D>;
  auto kern = attn_stats3_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((p.n_q + 2 * kBM - 1) / (2 * kBM), H);
  kern<<<grid, 320, L::SMEM, st>>>(mQ, mK, mV, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_stats(OperandMode mode, bool split_p, const CUtensorMap& mQ,
                              const CUtensorMap& mK, const CUtensorMap& mV,
                              const CUtensorMap& mVlo, const AttnStatsParams& p, int H,
                              cudaStream_t st) {
  switch (mode) {
    case kBF16d128:
      return split_p ? launch_attn_t<true, 128, 128, 1, 128, 2>(mQ, mK, mV, mVlo, p, H, st)
                     : launch_attn3_t<128>(mQ, mK, mV, p, H, st);
    case kBF16d64:
      return split_p ? launch_attn_t<true, 64, 64, 1, 128, 2>(mQ, mK, mV, mVlo, p, H, st)
                     : launch_attn3_t<64>(mQ, mK, mV, p, H, st);
    case kSplitF16d64: return launch_attn_t<false, 192, 64, 2, 64, 2>(mQ, mK, mV, mVlo, p, H, st);
  }
  return cudaErrorInvalidValue;
}

int attn_stats_smem(OperandMode mode) {
  switch (mode) {
    case kBF16d128: return AttnLayout<128, 128, 1, 128, 2>::SMEM;
    case kBF16d64: return Attn3Layout<64>::SMEM;
    case kSplitF16d64: return AttnLayout<192, 64, 2, 64, 2>::SMEM;
  }
  return 0;
}

}  // namespace lc
