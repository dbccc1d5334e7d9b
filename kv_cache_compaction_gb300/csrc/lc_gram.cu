// Normal equations of the two fits of attention-matching compaction ("KV
// compaction" blog, section "Fast KV Compaction via Attention Matching"):
//   mass fit   (step 4):  G = A^T A, c = A^T b with
//                         A_ri = exp(s q_r.C_ki - m_r), b_r = exp(lse_r - m_r);
//   output fit (step 5):  H = X^T X, R = X^T O with
//                         X_ri = softmax_i(s q_r.C_ki + beta_i).
// Both are the same computation, E_ir = 2^(s2 S_ir + colb2_i - rowsh2_r), with
// a different per-key bias and per-query shift; A and X are never stored.
//
// Layout is key-stationary: the score tile S^T = C_k q^T lands in tensor
// memory with one selected key per lane, so each thread owns one key and
// writes its row of E in the K-major layout the Gram products read, and
// c_i = sum_r E_ir b_r is a per-thread dot product.  E is split into fp16
// hi + lo and each Gram block is the sum of three tensor-core products
// (hi.hi + hi.lo + lo.hi), which keeps fp32-level accuracy.  With two key
// blocks per CTA the blocks G00 and G01 are formed together as 128 x 256
// products (the second block's E rows follow the first's in shared memory),
// six products per step instead of nine: issuing tensor-core instructions,
// not executing them, limits these kernels.
//
// CTA kinds (blockIdx.x):
//   [0, npairs)           key-block pair (bi <= bj): G[bi][bj], and c[bi]
//                         for diagonal pairs when row_b is given;
//   [npairs, npairs+nblk) R[bi] = E_bi O (output fit only).
// blockIdx.z splits the query slabs; partial sums are reduced afterwards in
// a fixed order.
#include <algorithm>

#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kSL = 64;  // query rows per slab

template <int D_QK, int D_V, int NST_>
struct GramLayout {
  static constexpr int NQC = D_QK / 64;
  static constexpr int NVC = D_V / 64;
  static constexpr int KC_BYTES = 128 * D_QK * 2;
  static constexpr int QCHUNK = kSL * 128;
  static constexpr int Q_BYTES = NQC * QCHUNK;
  static constexpr int O_BYTES = 2 * NVC * QCHUNK;  // hi + lo
  static constexpr int STAGE = Q_BYTES + O_BYTES;    // multiple of 1024
  static constexpr int NST = NST_;
  static constexpr int ROW_STAGE = 2 * kSL * 4;      // row shift + row b
  static constexpr int E_BYTES = 128 * 128;          // 128 keys x 64 queries x 2 B
  static constexpr int OFF_STAGE = 2 * KC_BYTES;
  static constexpr int OFF_E = OFF_STAGE + NST * STAGE;
  static constexpr int OFF_ROWS = OFF_E + 4 * E_BYTES;
  static constexpr int OFF_BAR = OFF_ROWS + NST * ROW_STAGE;
  static constexpr int SMEM = 1024 + OFF_BAR + 128;
};

// Adds the finished chunk's accumulator into the CTA's running sum, NCOL
// columns of this thread's tensor-memory lane, 16 at a time.
template <int NCOL>
__device__ __forceinline__ void fold_acc(uint32_t tsum, uint32_t tchunk) {
#pragma unroll 1
  for (int c = 0; c < NCOL / 16; ++c) {
    float a[16], b[16];
    tmem_ld16(tsum + c * 16, a);
    tmem_ld16(tchunk + c * 16, b);
#pragma unroll
    for (int e = 0; e < 16; ++e) a[e] += b[e];
    tmem_st16(tsum + c * 16, a);
  }
}

// Writes this thread's row of the CTA's partial: the running sum, plus the
// last chunk's accumulator when there was more than one chunk.
template <int NCOL>
__device__ __forceinline__ void store_acc_row(uint32_t tsum, uint32_t tchunk, bool add_chunk,
                                              float* dst) {
#pragma unroll
  for (int c = 0; c < NCOL / 32; ++c) {
    float v[32];
    tmem_ld32(tsum + c * 32, v);
    if (add_chunk) {
      float w[32];
      tmem_ld32(tchunk + c * 32, w);
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] += w[e];
    }
    float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
    for (int e = 0; e < 8; ++e) d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
  }
}

template <bool QK_BF16, int D_QK, int D_V, int NST>
__global__ void __launch_bounds__(192, 1)
    gram_kernel(const __grid_constant__ CUtensorMap mKc, const __grid_constant__ CUtensorMap mQ,
                const __grid_constant__ CUtensorMap mOhi, const __grid_constant__ CUtensorMap mOlo,
                const GramParams p) {
  using L = GramLayout<D_QK, D_V, NST>;
  // With a single stage the next slab's scores cannot be issued before the
  // current slab's products have released that stage.
  constexpr bool kPrefetchS = NST > 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sRows = base + L::OFF_ROWS;
  uint8_t* sKi = base;
  uint8_t* sKj = base + L::KC_BYTES;
  uint8_t* sStage = base + L::OFF_STAGE;
  uint8_t* sEih = base + L::OFF_E;
  uint8_t* sEil = sEih + L::E_BYTES;
  uint8_t* sEjh = sEil + L::E_BYTES;
  uint8_t* sEjl = sEjh + L::E_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* k_full = bars + 0;
  uint64_t* st_full = bars + 1;   // [2]
  uint64_t* st_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* s_free = bars + 7;    // [2]
  uint64_t* e_full = bars + 9;
  uint64_t* e_free = bars + 10;
  uint64_t* mma_drain = bars + 11;  // MMA completion before exit
  uint64_t* acc_free = bars + 12;   // a chunk's accumulator folded into the sum
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 13);
  __shared__ volatile int abort_flag;

  const int warp = warp_id(), lane = lane_id();
  const int h = blockIdx.y, z = blockIdx.z;
  const int npairs = p.nblk * (p.nblk + 1) / 2;
  const bool is_r = static_cast<int>(blockIdx.x) >= npairs;
  int bi = 0, bj = 0;
  if (!is_r) {
    int rem = blockIdx.x;
    while (rem >= p.nblk - bi) {
      rem -= p.nblk - bi;
      ++bi;
    }
    bj = bi + rem;
  } else {
    bi = bj = blockIdx.x - npairs;
  }
  const bool two = !is_r && bi != bj;
  const bool with_c = !is_r && bi == bj && p.row_b != nullptr;
  const int total_slabs = p.n_q_pad / kSL;
  const int s0 = z * p.slabs_per_split;
  const int s1 = min(total_slabs, s0 + p.slabs_per_split);
  const int nsl = max(0, s1 - s0);

  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(k_full, 1);
    for (int s = 0; s < L::NST; ++s) {
      mbar_init(&st_full[s], 1);
      mbar_init(&st_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
    }
    mbar_init(e_full, 128);
    mbar_init(e_free, 1);
    mbar_init(mma_drain, 1);
    mbar_init(acc_free, 128);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  // G block or R block: chunk 0 (of kGramChain slabs) accumulates at column
  // 256 and stays there as the running sum; later chunks at column 384
  const uint32_t tAcc = tbase + 256;
  const uint32_t tChunk = tbase + 384;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0 && nsl > 0) {
      mbar_arrive_expect_tx(k_full, (two ? 2 : 1) * L::KC_BYTES);
      for (int c = 0; c < L::NQC; ++c) {
        tma_load_3d(sKi + c * 128 * 128, &mKc, k_full, 64 * c, bi * 128, h);
        if (two) tma_load_3d(sKj + c * 128 * 128, &mKc, k_full, 64 * c, bj * 128, h);
      }
      const uint32_t bytes = L::Q_BYTES + (is_r ? L::O_BYTES : 0) + kSL * 4 + (with_c ? kSL * 4 : 0);
      int issued = 0;
      for (int i = 0; i < nsl; ++i) {
        const int s = i % L::NST;
        if (i >= L::NST && !wait_bar(&st_empty[s], ((i / L::NST) - 1) & 1, &abort_flag, p.err))
          break;
        uint8_t* st = sStage + s * L::STAGE;
        const int r0 = (s0 + i) * kSL;
        mbar_arrive_expect_tx(&st_full[s], bytes);
        for (int c = 0; c < L::NQC; ++c)
          tma_load_3d(st + c * L::QCHUNK, &mQ, &st_full[s], 64 * c, r0, h);
        if (is_r) {
          for (int c = 0; c < L::NVC; ++c) {
            tma_load_3d(st + L::Q_BYTES + c * L::QCHUNK, &mOhi, &st_full[s], 64 * c, r0, h);
            tma_load_3d(st + L::Q_BYTES + (L::NVC + c) * L::QCHUNK, &mOlo, &st_full[s], 64 * c,
                        r0, h);
          }
        }
        const size_t roff = static_cast<size_t>(h) * p.n_q_pad + r0;
        uint8_t* rw = sRows + s * L::ROW_STAGE;
        bulk_g2s(rw, p.rowsh2 + roff, kSL * 4, &st_full[s]);
        if (with_c) bulk_g2s(rw + kSL * 4, p.row_b + roff, kSL * 4, &st_full[s]);
        issued = i + 1;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      drain_wait(k_full, 0);
      for (int i = (issued > L::NST ? issued - L::NST : 0); i < issued; ++i)
        drain_wait(&st_full[i % L::NST], (i / L::NST) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nsl > 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, kSL, QK_BF16, false, false);
      constexpr uint32_t idesc_g = idesc_f16(128, 128, false, false, false);
      constexpr uint32_t idesc_r = idesc_f16(128, D_V, false, false, true);
      bool ok = wait_bar(k_full, 0, &abort_flag, p.err);
      auto issue_s = [&](int i) -> bool {
        const int s = i % L::NST, b = i & 1;
        if (!wait_bar(&st_full[s], (i / L::NST) & 1, &abort_flag, p.err)) return false;
        if (i >= 2 && !wait_bar(&s_free[b], ((i >> 1) - 1) & 1, &abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t aQ = smem_u32(sStage + s * L::STAGE);
#pragma unroll
        for (int k = 0; k < D_QK / 16; ++k) {
          const uint64_t dq = sdesc_sw128(aQ + (k >> 2) * L::QCHUNK + (k & 3) * 32, 16, 1024);
          const uint32_t koff = (k >> 2) * (128 * 128) + (k & 3) * 32;
          umma_f16_ss(tbase + b * 128, sdesc_sw128(smem_u32(sKi) + koff, 16, 1024), dq, idesc_s,
                      k > 0 ? 1u : 0u);
          if (two)
            umma_f16_ss(tbase + b * 128 + 64, sdesc_sw128(smem_u32(sKj) + koff, 16, 1024), dq,
                        idesc_s, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int i = 0; ok && i < nsl; ++i) {
        if (kPrefetchS && i + 1 < nsl && !issue_s(i + 1)) break;
        if (!wait_bar(e_full, i & 1, &abort_flag, p.err)) break;
        const int ch = i / kGramChain;
        // chunk ch - 1 has been folded into the sum before chunk ch reuses
        // its accumulator
        if (i % kGramChain == 0 && ch >= 2 &&
            !wait_bar(acc_free, (ch - 2) & 1, &abort_flag, p.err))
          break;
        tc_fence_after();
        const int s = i % L::NST;
        const uint32_t tA = ch == 0 ? tAcc : tChunk;
        const bool cont = i % kGramChain > 0;
        const uint32_t eih = smem_u32(sEih), eil = smem_u32(sEil);
        if (!is_r) {
          const uint32_t ejh = two ? smem_u32(sEjh) : eih;
          const uint32_t ejl = two ? smem_u32(sEjl) : eil;
#pragma unroll
          for (int k = 0; k < kSL / 16; ++k) {
            const uint32_t o = k * 32;
            const uint32_t acc0 = (cont || k > 0) ? 1u : 0u;
            umma_f16_ss(tA, sdesc_sw128(eih + o, 16, 1024), sdesc_sw128(ejh + o, 16, 1024),
                        idesc_g, acc0);
            umma_f16_ss(tA, sdesc_sw128(eih + o, 16, 1024), sdesc_sw128(ejl + o, 16, 1024),
                        idesc_g, 1u);
            umma_f16_ss(tA, sdesc_sw128(eil + o, 16, 1024), sdesc_sw128(ejh + o, 16, 1024),
                        idesc_g, 1u);
          }
        } else {
          const uint32_t aO = smem_u32(sStage + s * L::STAGE + L::Q_BYTES);
          const uint32_t aOl = aO + L::NVC * L::QCHUNK;
#pragma unroll
          for (int k = 0; k < kSL / 16; ++k) {
            const uint32_t o = k * 32;
            const uint32_t acc0 = (cont || k > 0) ? 1u : 0u;
            const uint64_t doh = sdesc_sw128(aO + k * 2048, L::QCHUNK, 1024);
            const uint64_t dol = sdesc_sw128(aOl + k * 2048, L::QCHUNK, 1024);
            umma_f16_ss(tA, sdesc_sw128(eih + o, 16, 1024), doh, idesc_r, acc0);
            umma_f16_ss(tA, sdesc_sw128(eih + o, 16, 1024), dol, idesc_r, 1u);
            umma_f16_ss(tA, sdesc_sw128(eil + o, 16, 1024), doh, idesc_r, 1u);
          }
        }
        umma_commit(&st_empty[s]);
        umma_commit(e_free);
        if (!kPrefetchS && i + 1 < nsl && !issue_s(i + 1)) break;
      }
    }
  } else {
    // ---------------------------------------------------------- E rows
    const int wq = warp & 3;
    const int j = wq * 32 + lane;  // key row within the block
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const size_t cb_off = static_cast<size_t>(h) * p.t_pad;
    const float cbi = p.colb2[cb_off + bi * 128 + j];
    const float cbj = two ? p.colb2[cb_off + bj * 128 + j] : 0.f;
    const float s2 = p.scale_log2;
    float cacc = 0.f;
    bool ok = nsl > 0;
    for (int i = 0; ok && i < nsl; ++i) {
      const int b = i & 1, s = i % L::NST;
      // slab i - 1 closed chunk ch >= 1: once its products are complete,
      // fold it into the sum so that chunk ch + 1 can reuse its accumulator
      if (i >= 2 * kGramChain && (i - 1) % kGramChain == kGramChain - 1) {
        if (!wait_bar(e_free, (i - 1) & 1, &abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        if (!is_r) fold_acc<128>(tAcc + lane_off, tChunk + lane_off);
        else fold_acc<D_V>(tAcc + lane_off, tChunk + lane_off);
        tc_fence_before();
        mbar_arrive(acc_free);
      }
      float cs = 0.f;  // the slab's share of c
      if (!wait_bar(&s_full[b], (i >> 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      float xi[kSL], xj[kSL];
#pragma unroll
      for (int c = 0; c < kSL / 32; ++c) {
        float v[32];
        tmem_ld32(tbase + lane_off + b * 128 + c * 32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) xi[c * 32 + e] = v[e];
        if (two) {
          tmem_ld32(tbase + lane_off + b * 128 + 64 + c * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) xj[c * 32 + e] = v[e];
        }
      }
      tc_fence_before();
      mbar_arrive(&s_free[b]);
      if (i > 0 && !wait_bar(e_free, (i - 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      // the row data arrived with the stage's copies
      if (!wait_bar(&st_full[s], (i / L::NST) & 1, &abort_flag, p.err)) { ok = false; break; }
      const float* rs = reinterpret_cast<const float*>(sRows + s * L::ROW_STAGE);
      const float* rb = rs + kSL;
#pragma unroll
      for (int c8 = 0; c8 < kSL / 8; ++c8) {
        float e8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float sh = rs[c8 * 8 + e];
          e8[e] = ex2(fmaf(xi[c8 * 8 + e], s2, cbi) - sh);
          if (with_c) cs = fmaf(e8[e], rb[c8 * 8 + e], cs);
        }
        uint4 hi, lo;
        split8(e8, hi, lo);
        const uint32_t off = sw128_offset(j, c8 * 8);
        *reinterpret_cast<uint4*>(sEih + off) = hi;
        *reinterpret_cast<uint4*>(sEil + off) = lo;
        if (two) {
#pragma unroll
          for (int e = 0; e < 8; ++e) e8[e] = ex2(fmaf(xj[c8 * 8 + e], s2, cbj) - rs[c8 * 8 + e]);
          split8(e8, hi, lo);
          *reinterpret_cast<uint4*>(sEjh + off) = hi;
          *reinterpret_cast<uint4*>(sEjl + off) = lo;
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(e_full);
      cacc += cs;
    }
    if (ok && nsl > 0 && wait_bar(e_free, (nsl - 1) & 1, &abort_flag, p.err)) {
      tc_fence_after();
      const int H = gridDim.y;
      const size_t zh = static_cast<size_t>(z) * H + h;
      const int key = bi * 128 + j;
      const bool chunks = nsl > kGramChain;  // the last chunk is still apart
      if (!is_r) {
        store_acc_row<128>(tAcc + lane_off, tChunk + lane_off, chunks,
                           p.Gpart + (zh * p.t_pad + key) * p.t_pad + bj * 128);
        if (with_c) p.cpart[zh * p.t_pad + key] = cacc;
      } else {
        store_acc_row<D_V>(tAcc + lane_off, tChunk + lane_off, chunks,
                           p.Rpart + (zh * p.t_pad + key) * p.d_v);
      }
    }
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// Two-group variant for bf16 inputs (d = 64 or 128): query slabs alternate
// between two epilogue warpgroups with their own E buffer and score buffer,
// so the Gram products of one slab run on the tensor core while the other
// group forms the next slab's E.  Warps: 0 TMA, 1 MMA issue, 2..5 group 0
// (even slabs), 6..9 group 1 (odd slabs).  A ring stage is refilled as soon
// as its scores are formed (pair CTAs) or its O slab's product is done (R
// CTAs); the per-query row data are read through L1.  Tensor memory: S[2] (two blocks of
// 64 columns each) at 0 and 128, accumulator at 256.  Shared memory (pair /
// R CTAs): C_k blocks, a 2-stage ring of query (and O) slabs, E[2].
template <int D>
struct Gram2Layout {
  static constexpr int NC = D / 64;
  static constexpr int KC_BYTES = 128 * D * 2;
  static constexpr int QCHUNK = kSL * 128;
  static constexpr int Q_BYTES = NC * QCHUNK;
  static constexpr int O_BYTES = 2 * NC * QCHUNK;   // hi + lo (R CTAs only)
  static constexpr int E_BLK = 128 * 128;           // one block's E (hi or lo)
  // pair CTAs: Kc_i, Kc_j | ring 2 x Q | E[2] = 4 blocks each
  static constexpr int P_OFF_RING = 2 * KC_BYTES;
  static constexpr int P_STAGE = Q_BYTES;
  static constexpr int P_OFF_E = P_OFF_RING + 2 * P_STAGE;
  static constexpr int P_END = P_OFF_E + 2 * 4 * E_BLK;
  // R CTAs: Kc_i | ring 2 x (Q + O) | E[2] = 2 blocks each
  static constexpr int R_OFF_RING = KC_BYTES;
  static constexpr int R_STAGE = Q_BYTES + O_BYTES;
  static constexpr int R_OFF_E = R_OFF_RING + 2 * R_STAGE;
  static constexpr int R_END = R_OFF_E + 2 * 2 * E_BLK;
  static constexpr int OFF_BAR = (P_END > R_END ? P_END : R_END);
  static constexpr int OFF_CX = OFF_BAR + 256;      // group-1 partial c
  static constexpr int SMEM = 1024 + OFF_CX + 128 * 4;
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    gram2_kernel(const __grid_constant__ CUtensorMap mKc, const __grid_constant__ CUtensorMap mQ,
                 const __grid_constant__ CUtensorMap mOhi, const __grid_constant__ CUtensorMap mOlo,
                 const GramParams p) {
  using L = Gram2Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* k_full = bars + 0;
  uint64_t* st_full = bars + 1;   // [2]
  uint64_t* st_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2] per group
  uint64_t* s_free = bars + 7;    // [2]
  uint64_t* e_full = bars + 9;    // [2]
  uint64_t* e_free = bars + 11;   // [2]
  uint64_t* done = bars + 13;
  uint64_t* mma_drain = bars + 14;  // MMA completion before exit
  uint64_t* acc_free = bars + 15;   // a chunk's accumulator folded into the sum
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 16);
  float* cx = reinterpret_cast<float*>(base + L::OFF_CX);
  __shared__ volatile int abort_flag;

  const int warp = warp_id(), lane = lane_id();
  const int h = blockIdx.y, z = blockIdx.z;
  const int npairs = p.nblk * (p.nblk + 1) / 2;
  const bool is_r = p.r_only || static_cast<int>(blockIdx.x) >= npairs;
  int bi = 0, bj = 0;
  if (!is_r) {
    int rem = blockIdx.x;
    while (rem >= p.nblk - bi) {
      rem -= p.nblk - bi;
      ++bi;
    }
    bj = bi + rem;
  } else {
    bi = bj = p.r_only ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) - npairs;
  }
  const bool two = !is_r && bi != bj;
  const bool with_c = !is_r && bi == bj && p.row_b != nullptr;
  const int total_slabs = p.n_q_pad / kSL;
  const int s0 = z * p.slabs_per_split;
  const int nsl = max(0, min(total_slabs, s0 + p.slabs_per_split) - s0);

  uint8_t* sKi = base;
  uint8_t* sKj = base + L::KC_BYTES;
  uint8_t* sRing = base + (is_r ? L::R_OFF_RING : L::P_OFF_RING);
  const int stage_bytes = is_r ? L::R_STAGE : L::P_STAGE;
  uint8_t* sE = base + (is_r ? L::R_OFF_E : L::P_OFF_E);
  const int e_buf = (is_r ? 2 : 4) * L::E_BLK;  // one group's E buffer

  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(k_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&st_full[i], 1);
      mbar_init(&st_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
      mbar_init(&e_full[i], 128);
      mbar_init(&e_free[i], 1);
    }
    mbar_init(done, 1);
    mbar_init(mma_drain, 1);
    mbar_init(acc_free, 128);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  // chunk 0 (of kGramChain slabs) accumulates at column 256 and stays there
  // as the running sum; later chunks at column 384
  const uint32_t tAcc = tbase + 256;
  const uint32_t tChunk = tbase + 384;

  if (warp == 0) {
    if (lane == 0 && nsl > 0) {
      mbar_arrive_expect_tx(k_full, (two ? 2 : 1) * L::KC_BYTES);
      for (int c = 0; c < L::NC; ++c) {
        tma_load_3d(sKi + c * 128 * 128, &mKc, k_full, 64 * c, bi * 128, h);
        if (two) tma_load_3d(sKj + c * 128 * 128, &mKc, k_full, 64 * c, bj * 128, h);
      }
      const uint32_t bytes = L::Q_BYTES + (is_r ? L::O_BYTES : 0);
      int issued = 0;
      for (int i = 0; i < nsl; ++i) {
        const int s = i & 1;
        if (i >= 2 && !wait_bar(&st_empty[s], ((i >> 1) - 1) & 1, &abort_flag, p.err)) break;
        uint8_t* st = sRing + s * stage_bytes;
        const int r0 = (s0 + i) * kSL;
        mbar_arrive_expect_tx(&st_full[s], bytes);
        for (int c = 0; c < L::NC; ++c)
          tma_load_3d(st + c * L::QCHUNK, &mQ, &st_full[s], 64 * c, r0, h);
        if (is_r) {
          for (int c = 0; c < L::NC; ++c) {
            tma_load_3d(st + L::Q_BYTES + c * L::QCHUNK, &mOhi, &st_full[s], 64 * c, r0, h);
            tma_load_3d(st + L::Q_BYTES + (L::NC + c) * L::QCHUNK, &mOlo, &st_full[s], 64 * c,
                        r0, h);
          }
        }
        issued = i + 1;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      drain_wait(k_full, 0);
      for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i)
        drain_wait(&st_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && nsl > 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, kSL, true, false, false);
      constexpr uint32_t idesc_g = idesc_f16(128, 128, false, false, false);
      constexpr uint32_t idesc_r = idesc_f16(128, D, false, false, true);
      bool ok = wait_bar(k_full, 0, &abort_flag, p.err);
      auto issue_s = [&](int i) {  // scores of slab i into S[i & 1]
        const int s = i & 1;
        tc_fence_after();
        const uint32_t aQ = smem_u32(sRing + s * stage_bytes);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t dq = sdesc_sw128(aQ + (k >> 2) * L::QCHUNK + (k & 3) * 32, 16, 1024);
          const uint32_t koff = (k >> 2) * (128 * 128) + (k & 3) * 32;
          umma_f16_ss(tbase + s * 128, sdesc_sw128(smem_u32(sKi) + koff, 16, 1024), dq, idesc_s,
                      k > 0 ? 1u : 0u);
          if (two)
            umma_f16_ss(tbase + s * 128 + 64, sdesc_sw128(smem_u32(sKj) + koff, 16, 1024), dq,
                        idesc_s, k > 0 ? 1u : 0u);
        }
        // a pair CTA is done with the query slab once its scores are formed
        if (!is_r) umma_commit(&st_empty[s]);
        umma_commit(&s_full[s]);
      };
      auto issue_g = [&](int i) {  // Gram (or R) products of slab i
        const int g = i & 1;
        tc_fence_after();
        const uint32_t eb = smem_u32(sE + g * e_buf);
        const uint32_t eih = eb, eil = eb + L::E_BLK;
        const uint32_t tA = i < kGramChain ? tAcc : tChunk;
        const bool cont = i % kGramChain > 0;
        if (!is_r) {
          const uint32_t ejh = two ? eb + 2 * L::E_BLK : eih;
          const uint32_t ejl = two ? eb + 3 * L::E_BLK : eil;
#pragma unroll
          for (int k = 0; k < kSL / 16; ++k) {
            const uint32_t o = k * 32;
            const uint32_t acc0 = (cont || k > 0) ? 1u : 0u;
            umma_f16_ss(tA, sdesc_sw128(eih + o, 16, 1024), sdesc_sw128(ejh + o, 16, 1024),
                        idesc_g, acc0);
            umma_f16_ss(tA, sdesc_sw128(eih + o, 16, 1024), sdesc_sw128(ejl + o, 16, 1024),
                        idesc_g, 1u);
            umma_f16_ss(tA, sdesc_sw128(eil + o, 16, 1024), sdesc_sw128(ejh + o, 16, 1024),
                        idesc_g, 1u);
          }
        } else {
          const uint32_t aO = smem_u32(sRing + g * stage_bytes + L::Q_BYTES);
          const uint32_t aOl = aO + L::NC * L::QCHUNK;
#pragma unroll
          for (int k = 0; k < kSL / 16; ++k) {
            const uint32_t o = k * 32;
            const uint32_t acc0 = (cont || k > 0) ? 1u : 0u;
            const uint64_t doh = sdesc_sw128(aO + k * 2048, L::QCHUNK, 1024);
            const uint64_t dol = sdesc_sw128(aOl + k * 2048, L::QCHUNK, 1024);
            umma_f16_ss(tA, sdesc_sw128(eih + o, 16, 1024), doh, idesc_r, acc0);
            umma_f16_ss(tA, sdesc_sw128(eih + o, 16, 1024), dol, idesc_r, 1u);
            umma_f16_ss(tA, sdesc_sw128(eil + o, 16, 1024), doh, idesc_r, 1u);
          }
          umma_commit(&st_empty[g]);  // the O slab feeds the products above
        }
        umma_commit(&e_free[g]);
      };
      // a chunk's first products wait until the previous chunk has been
      // folded into the sum (its accumulator is reused)
      auto acc_ready = [&](int i) {
        const int ch = i / kGramChain;
        return i % kGramChain != 0 || ch < 2 || mbar_test_wait(acc_free, (ch - 2) & 1);
      };
      // Event loop: the scores of a slab are issued as soon as its query slab
      // is loaded and its S buffer has been read (up to two slabs ahead of
      // the Gram products), the Gram products as soon as its E is formed.
      int ns = 0, ng = 0;
      uint64_t t_last = globaltimer_ns();
      uint32_t spins = 0;
      while (ok && ng < nsl) {
        if (ns < nsl && mbar_test_wait(&st_full[ns & 1], (ns >> 1) & 1) &&
            (ns < 2 || mbar_test_wait(&s_free[ns & 1], ((ns >> 1) - 1) & 1))) {
          issue_s(ns++);
          t_last = globaltimer_ns();
        } else if (ng < ns && mbar_test_wait(&e_full[ng & 1], (ng >> 1) & 1) && acc_ready(ng)) {
          issue_g(ng++);
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
      umma_commit(done);
    }
  } else {
    // ---------------------------------------------------------- E rows
    const int g = (warp - 2) >> 2;
    const int wq = warp & 3;
    const int j = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const size_t cb_off = static_cast<size_t>(h) * p.t_pad;
    const float cbi = p.colb2[cb_off + bi * 128 + j];
    const float cbj = two ? p.colb2[cb_off + bj * 128 + j] : 0.f;
    const float s2 = p.scale_log2;
    uint8_t* eb = sE + g * e_buf;
    uint8_t* sEih = eb;
    uint8_t* sEil = eb + L::E_BLK;
    uint8_t* sEjh = eb + 2 * L::E_BLK;
    uint8_t* sEjl = eb + 3 * L::E_BLK;
    // slab e closed chunk ch >= 1 (not the last): once its products are
    // complete, fold it into the sum so that chunk ch + 1 can reuse its
    // accumulator.  The group that formed slab e does this, before its next
    // slab or after its last one.
    auto closes_chunk = [&](int e) {
      return e >= 2 * kGramChain - 1 && e % kGramChain == kGramChain - 1 && e < nsl - 1;
    };
    auto fold = [&](int e) -> bool {
      if (!wait_bar(&e_free[g], (e >> 1) & 1, &abort_flag, p.err)) return false;
      tc_fence_after();
      if (!is_r) fold_acc<128>(tAcc + lane_off, tChunk + lane_off);
      else fold_acc<D>(tAcc + lane_off, tChunk + lane_off);
      tc_fence_before();
      mbar_arrive(acc_free);
      return true;
    };
    float cacc = 0.f;
    bool ok = nsl > 0;
    for (int i = g; ok && i < nsl; i += 2) {
      const int n = i >> 1;  // this group's n-th slab
      if (i >= 2 && closes_chunk(i - 2) && !fold(i - 2)) { ok = false; break; }
      float cs = 0.f;  // the slab's share of c
      // per-query shifts (and mass) of this slab, read through L1: every
      // thread of the group reads the same 64 values
      const size_t roff = static_cast<size_t>(h) * p.n_q_pad + static_cast<size_t>(s0 + i) * kSL;
      const float* rs = p.rowsh2 + roff;
      const float* rb = with_c ? p.row_b + roff : rs;
      asm volatile("prefetch.global.L1 [%0];" ::"l"(rs));
      asm volatile("prefetch.global.L1 [%0];" ::"l"(rs + 32));
      if (with_c) {
        asm volatile("prefetch.global.L1 [%0];" ::"l"(rb));
        asm volatile("prefetch.global.L1 [%0];" ::"l"(rb + 32));
      }
      if (!wait_bar(&s_full[g], n & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {  // 32 query columns at a time
        // row data of these columns first: their latency overlaps the TMEM load
        float4 sh4[8], b4[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) sh4[q] = __ldg(reinterpret_cast<const float4*>(rs + hf * 32) + q);
        if (with_c) {
#pragma unroll
          for (int q = 0; q < 8; ++q) b4[q] = __ldg(reinterpret_cast<const float4*>(rb + hf * 32) + q);
        }
        float xi[32], xj[32];
        const uint32_t ts = tbase + g * 128 + hf * 32 + lane_off;
        if (two) tmem_ld32x2(ts, ts + 64, xi, xj);
        else tmem_ld32(ts, xi);
        if (hf == 1) {
          tc_fence_before();
          mbar_arrive(&s_free[g]);
        } else {
          if (n > 0 && !wait_bar(&e_free[g], (n - 1) & 1, &abort_flag, p.err)) { ok = false; break; }
        }
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          const int c8 = hf * 4 + q8;
          const float sh8[8] = {sh4[2 * q8].x, sh4[2 * q8].y, sh4[2 * q8].z, sh4[2 * q8].w,
                                sh4[2 * q8 + 1].x, sh4[2 * q8 + 1].y, sh4[2 * q8 + 1].z,
                                sh4[2 * q8 + 1].w};
          float e8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) e8[e] = ex2(fmaf(xi[q8 * 8 + e], s2, cbi) - sh8[e]);
          if (with_c) {
            const float b8[8] = {b4[2 * q8].x, b4[2 * q8].y, b4[2 * q8].z, b4[2 * q8].w,
                                 b4[2 * q8 + 1].x, b4[2 * q8 + 1].y, b4[2 * q8 + 1].z,
                                 b4[2 * q8 + 1].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) cs = fmaf(e8[e], b8[e], cs);
          }
          uint4 hi, lo;
          split8(e8, hi, lo);
          const uint32_t off = sw128_offset(j, c8 * 8);
          *reinterpret_cast<uint4*>(sEih + off) = hi;
          *reinterpret_cast<uint4*>(sEil + off) = lo;
          if (two) {
#pragma unroll
            for (int e = 0; e < 8; ++e) e8[e] = ex2(fmaf(xj[q8 * 8 + e], s2, cbj) - sh8[e]);
            split8(e8, hi, lo);
            *reinterpret_cast<uint4*>(sEjh + off) = hi;
            *reinterpret_cast<uint4*>(sEjl + off) = lo;
          }
        }
      }
      if (!ok) break;
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&e_full[g]);
      cacc += cs;
    }
    // a chunk closed by this group's last slab (the next chunk has one slab)
    if (ok && nsl >= 2 && ((nsl - 2) & 1) == g && closes_chunk(nsl - 2) && !fold(nsl - 2))
      ok = false;
    // combine the groups' partial c and publish the block accumulator
    if (with_c && g == 1) cx[j] = cacc;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (ok && g == 0 && nsl > 0 && wait_bar(done, 0, &abort_flag, p.err)) {
      tc_fence_after();
      const int H = gridDim.y;
      const size_t zh = static_cast<size_t>(z) * H + h;
      const int key = bi * 128 + j;
      const bool chunks = nsl > kGramChain;  // the last chunk is still apart
      if (!is_r) {
        store_acc_row<128>(tAcc + lane_off, tChunk + lane_off, chunks,
                           p.Gpart + (zh * p.t_pad + key) * p.t_pad + bj * 128);
        if (with_c) p.cpart[zh * p.t_pad + key] = cacc + (nsl > 1 ? cx[j] : 0.f);
      } else {
        store_acc_row<D>(tAcc + lane_off, tChunk + lane_off, chunks,
                         p.Rpart + (zh * p.t_pad + key) * p.d_v);
      }
    }
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// Both key blocks of a 256-key system in one CTA per (head, query range): the
// scores of a query slab are formed once for both blocks (S at TMEM columns 0
// and 64) and E once per block by eight epilogue warps (warp w holds key rows
// 32 (w % 4) .. +31 of block (w - 2) / 4, the TMEM lanes it may access).
// Gram mode accumulates G00, G01 and G11 at TMEM columns 128, 256 and 384
// (and c for the mass system); R mode accumulates R_b = E_b O at columns
// 128 + 128 b.  Compared with one CTA per block pair each slab's scores and E
// are formed once instead of twice.  Warps: 0 TMA, 1 MMA issue, 2..9 E rows.
// Shared memory: C_k of both blocks, 2-stage rings of query slabs, of O slabs
// (R mode) and of per-query row data, and E (two buffers in Gram mode, one in
// R mode).
template <int D, bool RM>
struct Gram3Layout {
  static constexpr int NC = D / 64;
  static constexpr int KC_BYTES = 128 * D * 2;
  static constexpr int QCHUNK = kSL * 128;
  static constexpr int Q_BYTES = NC * QCHUNK;
  static constexpr int O_BYTES = RM ? 2 * NC * QCHUNK : 0;  // hi + lo
  static constexpr int E_BLK = 128 * 128;  // 128 keys x 64 queries, fp16
  static constexpr int NE = RM ? 1 : 2;    // E buffers
  static constexpr int OFF_RING = 2 * KC_BYTES;
  static constexpr int OFF_O = OFF_RING + 2 * Q_BYTES;
  static constexpr int OFF_E = OFF_O + 2 * O_BYTES;
  static constexpr int OFF_ROWS = OFF_E + NE * 4 * E_BLK;
  static constexpr int ROW_STAGE = 2 * kSL * 4;  // row shift + row mass
  static constexpr int OFF_BAR = OFF_ROWS + 2 * ROW_STAGE;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
};

template <int D, bool RM>
__global__ void __launch_bounds__(320, 1)
    gram3_kernel(const __grid_constant__ CUtensorMap mKc, const __grid_constant__ CUtensorMap mQ,
                 const __grid_constant__ CUtensorMap mOhi,
                 const __grid_constant__ CUtensorMap mOlo, const GramParams p) {
  using L = Gram3Layout<D, RM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::OFF_BAR);
  uint64_t* k_full = bars + 0;
  uint64_t* st_full = bars + 1;   // [2] query slab
  uint64_t* st_empty = bars + 3;  // [2]
  uint64_t* o_full = bars + 5;    // [2] O slab (R mode)
  uint64_t* o_empty = bars + 7;   // [2]
  uint64_t* r_full = bars + 9;    // [2] row data
  uint64_t* r_empty = bars + 11;  // [2]
  uint64_t* s_full = bars + 13;
  uint64_t* s_free = bars + 14;
  uint64_t* e_full = bars + 15;   // [2]
  uint64_t* e_free = bars + 17;   // [2]
  uint64_t* done = bars + 19;
  uint64_t* mma_drain = bars + 20;  // MMA completion before exit
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  __shared__ volatile int abort_flag;

  const int warp = warp_id(), lane = lane_id();
  const int h = blockIdx.y, z = blockIdx.z;
  const bool with_c = !RM && p.row_b != nullptr;
  const int total_slabs = p.n_q_pad / kSL;
  const int s0 = z * p.slabs_per_split;
  const int nsl = max(0, min(total_slabs, s0 + p.slabs_per_split) - s0);
  uint8_t* sK0 = base;
  uint8_t* sK1 = base + L::KC_BYTES;
  uint8_t* sRing = base + L::OFF_RING;
  uint8_t* sO = base + L::OFF_O;
  uint8_t* sE = base + L::OFF_E;
  float* sRows = reinterpret_cast<float*>(base + L::OFF_ROWS);
  // E buffer of slab i and the phase of its barriers
  auto ebuf = [](int i) { return RM ? 0 : (i & 1); };
  auto ephase = [](int i) { return static_cast<uint32_t>(RM ? (i & 1) : ((i >> 1) & 1)); };

  if (threadIdx.x == 0) {
    abort_flag = launch_aborted(p.err) ? 1 : 0;
    mbar_init(k_full, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&st_full[i], 1);
      mbar_init(&st_empty[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 1);
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], 256);
      mbar_init(&e_full[i], 256);
      mbar_init(&e_free[i], 1);
    }
    mbar_init(done, 1);
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    if (lane == 0 && nsl > 0) {
      mbar_arrive_expect_tx(k_full, 2 * L::KC_BYTES);
      for (int c = 0; c < L::NC; ++c) {
        tma_load_3d(sK0 + c * 128 * 128, &mKc, k_full, 64 * c, 0, h);
        tma_load_3d(sK1 + c * 128 * 128, &mKc, k_full, 64 * c, 128, h);
      }
      // per slab: query slab, row data, O slab -- each stage refilled once
      // its consumers (scores / E / R products of slab i - 2) are done
      int nq = 0, nr = 0, no = 0;  // slabs whose copies are issued, per kind
      for (int i = 0; i < nsl; ++i) {
        const int s = i & 1;
        const uint32_t ph = ((i >> 1) - 1) & 1;
        const int r0 = (s0 + i) * kSL;
        if (i >= 2 && !wait_bar(&st_empty[s], ph, &abort_flag, p.err)) break;
        uint8_t* st = sRing + s * L::Q_BYTES;
        mbar_arrive_expect_tx(&st_full[s], L::Q_BYTES);
        for (int c = 0; c < L::NC; ++c)
          tma_load_3d(st + c * L::QCHUNK, &mQ, &st_full[s], 64 * c, r0, h);
        nq = i + 1;
        if (i >= 2 && !wait_bar(&r_empty[s], ph, &abort_flag, p.err)) break;
        const size_t roff = static_cast<size_t>(h) * p.n_q_pad + r0;
        float* rw = sRows + s * (L::ROW_STAGE / 4);
        mbar_arrive_expect_tx(&r_full[s], (with_c ? 2 : 1) * kSL * 4);
        bulk_g2s(rw, p.rowsh2 + roff, kSL * 4, &r_full[s]);
        if (with_c) bulk_g2s(rw + kSL, p.row_b + roff, kSL * 4, &r_full[s]);
        nr = i + 1;
        if (RM) {
          if (i >= 2 && !wait_bar(&o_empty[s], ph, &abort_flag, p.err)) break;
          uint8_t* so = sO + s * L::O_BYTES;
          mbar_arrive_expect_tx(&o_full[s], L::O_BYTES);
          for (int c = 0; c < L::NC; ++c) {
            tma_load_3d(so + c * L::QCHUNK, &mOhi, &o_full[s], 64 * c, r0, h);
            tma_load_3d(so + (L::NC + c) * L::QCHUNK, &mOlo, &o_full[s], 64 * c, r0, h);
          }
        }
        no = RM ? i + 1 : 0;
      }
      // the copies in flight land before the CTA exits, also when the pipeline
      // was abandoned after a wait gave up elsewhere in the CTA
      auto drain = [&](uint64_t* full, int n) {
        for (int i = (n > 2 ? n - 2 : 0); i < n; ++i) drain_wait(&full[i & 1], (i >> 1) & 1);
      };
      drain_wait(k_full, 0);
      drain(st_full, nq);
      drain(r_full, nr);
      drain(o_full, no);
    }
  } else if (warp == 1) {
    if (lane == 0 && nsl > 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, kSL, true, false, false);
      constexpr uint32_t idesc_g = idesc_f16(128, 128, false, false, false);
      constexpr uint32_t idesc_g2 = idesc_f16(128, 256, false, false, false);
      constexpr uint32_t idesc_r = idesc_f16(128, D, false, false, true);
      bool ok = wait_bar(k_full, 0, &abort_flag, p.err);
      auto issue_s = [&](int i) {  // scores of slab i for both key blocks
        const int s = i & 1;
        tc_fence_after();
        const uint32_t aQ = smem_u32(sRing + s * L::Q_BYTES);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t dq = sdesc_sw128(aQ + (k >> 2) * L::QCHUNK + (k & 3) * 32, 16, 1024);
          const uint32_t koff = (k >> 2) * (128 * 128) + (k & 3) * 32;
          umma_f16_ss(tbase, sdesc_sw128(smem_u32(sK0) + koff, 16, 1024), dq, idesc_s,
                      k > 0 ? 1u : 0u);
          umma_f16_ss(tbase + 64, sdesc_sw128(smem_u32(sK1) + koff, 16, 1024), dq, idesc_s,
                      k > 0 ? 1u : 0u);
        }
        umma_commit(&st_empty[s]);
        umma_commit(s_full);
      };
      auto issue_g = [&](int i) {  // Gram blocks (or R) of slab i
        tc_fence_after();
        // E tiles [E0 hi, E1 hi, E0 lo, E1 lo]: E1 follows E0, so one
        // 256-row operand covers both key blocks
        const uint32_t eb = smem_u32(sE + ebuf(i) * 4 * L::E_BLK);
        const uint32_t e0h = eb, e1h = eb + L::E_BLK;
        const uint32_t e0l = eb + 2 * L::E_BLK, e1l = eb + 3 * L::E_BLK;
        if constexpr (!RM) {
#pragma unroll
          for (int k = 0; k < kSL / 16; ++k) {
            const uint32_t o = k * 32;
            const uint32_t acc0 = (i > 0 || k > 0) ? 1u : 0u;
            const uint64_t a0h = sdesc_sw128(e0h + o, 16, 1024);
            const uint64_t a0l = sdesc_sw128(e0l + o, 16, 1024);
            const uint64_t a1h = sdesc_sw128(e1h + o, 16, 1024);
            const uint64_t a1l = sdesc_sw128(e1l + o, 16, 1024);
            // G00 | G01 (TMEM columns 128..383) as 128 x 256 products
            umma_f16_ss(tbase + 128, a0h, a0h, idesc_g2, acc0);
            umma_f16_ss(tbase + 128, a0h, a0l, idesc_g2, 1u);
            umma_f16_ss(tbase + 128, a0l, a0h, idesc_g2, 1u);
            umma_f16_ss(tbase + 384, a1h, a1h, idesc_g, acc0);
            umma_f16_ss(tbase + 384, a1h, a1l, idesc_g, 1u);
            umma_f16_ss(tbase + 384, a1l, a1h, idesc_g, 1u);
          }
        } else {
          const uint32_t aO = smem_u32(sO + (i & 1) * L::O_BYTES);
          const uint32_t aOl = aO + L::NC * L::QCHUNK;
#pragma unroll
          for (int k = 0; k < kSL / 16; ++k) {
            const uint32_t o = k * 32;
            const uint32_t acc0 = (i > 0 || k > 0) ? 1u : 0u;
            const uint64_t doh = sdesc_sw128(aO + k * 2048, L::QCHUNK, 1024);
            const uint64_t dol = sdesc_sw128(aOl + k * 2048, L::QCHUNK, 1024);
            const uint64_t a0h = sdesc_sw128(e0h + o, 16, 1024);
            const uint64_t a0l = sdesc_sw128(e0l + o, 16, 1024);
            const uint64_t a1h = sdesc_sw128(e1h + o, 16, 1024);
            const uint64_t a1l = sdesc_sw128(e1l + o, 16, 1024);
            umma_f16_ss(tbase + 128, a0h, doh, idesc_r, acc0);
            umma_f16_ss(tbase + 128, a0h, dol, idesc_r, 1u);
            umma_f16_ss(tbase + 128, a0l, doh, idesc_r, 1u);
            umma_f16_ss(tbase + 256, a1h, doh, idesc_r, acc0);
            umma_f16_ss(tbase + 256, a1h, dol, idesc_r, 1u);
            umma_f16_ss(tbase + 256, a1l, doh, idesc_r, 1u);
          }
          umma_commit(&o_empty[i & 1]);
        }
        umma_commit(&e_free[ebuf(i)]);
      };
      // Event loop: a slab's scores are issued once its query slab is loaded
      // and the previous scores have been read; its products once its E (and
      // in R mode its O slab) is ready.
      int ns = 0, ng = 0;
      uint64_t t_last = globaltimer_ns();
      uint32_t spins = 0;
      while (ok && ng < nsl) {
        if (ns < nsl && mbar_test_wait(&st_full[ns & 1], (ns >> 1) & 1) &&
            (ns == 0 || mbar_test_wait(s_free, (ns - 1) & 1))) {
          issue_s(ns++);
          t_last = globaltimer_ns();
        } else if (ng < ns && mbar_test_wait(&e_full[ebuf(ng)], ephase(ng)) &&
                   (!RM || mbar_test_wait(&o_full[ng & 1], (ng >> 1) & 1))) {
          issue_g(ng++);
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
      umma_commit(done);
    }
  } else {
    // ---------------------------------------------------------- E rows
    const int b = (warp - 2) >> 2;
    const int q = warp & 3;
    const int j = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const float cb = p.colb2[static_cast<size_t>(h) * p.t_pad + b * 128 + j];
    const float s2 = p.scale_log2;
    float cacc = 0.f;
    bool ok = nsl > 0;
    for (int i = 0; ok && i < nsl; ++i) {
      if (!wait_bar(&r_full[i & 1], (i >> 1) & 1, &abort_flag, p.err)) { ok = false; break; }
      if (!wait_bar(s_full, i & 1, &abort_flag, p.err)) { ok = false; break; }
      tc_fence_after();
      const float* rs = sRows + (i & 1) * (L::ROW_STAGE / 4);
      const float* rb = rs + kSL;
      uint8_t* sEh = sE + ebuf(i) * 4 * L::E_BLK + b * L::E_BLK;
      uint8_t* sEl = sEh + 2 * L::E_BLK;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {  // 32 query columns at a time
        float x[32];
        tmem_ld32(tbase + b * 64 + hf * 32 + lane_off, x);
        if (hf == 1) {
          tc_fence_before();
          mbar_arrive(s_free);
        } else if (i >= (RM ? 1 : 2) &&
                   !wait_bar(&e_free[ebuf(i)], ephase(i) ^ 1u, &abort_flag, p.err)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          const int c8 = hf * 4 + q8;
          const float4 sa = *reinterpret_cast<const float4*>(rs + c8 * 8);
          const float4 sb = *reinterpret_cast<const float4*>(rs + c8 * 8 + 4);
          const float sh8[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
          float e8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) e8[e] = ex2(fmaf(x[q8 * 8 + e], s2, cb) - sh8[e]);
          if (with_c) {
            const float4 ba = *reinterpret_cast<const float4*>(rb + c8 * 8);
            const float4 bb = *reinterpret_cast<const float4*>(rb + c8 * 8 + 4);
            const float b8[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) cacc = fmaf(e8[e], b8[e], cacc);
          }
          uint4 hi, lo;
          split8(e8, hi, lo);
          const uint32_t off = sw128_offset(j, c8 * 8);
          *reinterpret_cast<uint4*>(sEh + off) = hi;
          *reinterpret_cast<uint4*>(sEl + off) = lo;
        }
      }
      if (!ok) break;
      mbar_arrive(&r_empty[i & 1]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&e_full[ebuf(i)]);
    }
    // publish: Gram mode G00 / G11 (own block), half of G01 (block-0 rows)
    // and c; R mode the block's R rows
    if (ok && nsl > 0 && wait_bar(done, 0, &abort_flag, p.err)) {
      tc_fence_after();
      const int H = gridDim.y;
      const size_t zh = static_cast<size_t>(z) * H + h;
      const int key = b * 128 + j;
      auto put32 = [&](uint32_t tcol, float* dst) {
        float v[32];
        tmem_ld32(tbase + tcol + lane_off, v);
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int e = 0; e < 8; ++e) d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
      };
      if constexpr (!RM) {
        float* dst = p.Gpart + (zh * p.t_pad + key) * p.t_pad + b * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) put32(128 + b * 256 + c * 32, dst + c * 32);
        float* dst01 = p.Gpart + (zh * p.t_pad + j) * p.t_pad + 128 + b * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) put32(256 + b * 64 + c * 32, dst01 + c * 32);
        if (with_c) p.cpart[zh * p.t_pad + key] = cacc;
      } else {
        float* dst = p.Rpart + (zh * p.t_pad + key) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) put32(128 + b * 128 + c * 32, dst + c * 32);
      }
    }
  }
  if (warp == 1 && lane_id() == 0) drain_mma(mma_drain);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int D>
cudaError_t launch_gram2_t(bool with_r, const CUtensorMap& mKc, const CUtensorMap& mQ,
                           const CUtensorMap& mOhi, const CUtensorMap& mOlo, const GramParams& p,
                           int H, int nsplit, cudaStream_t st) {
  using L = Gram2Layout<D>;
  auto kern = gram2_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  const int npairs = p.nblk * (p.nblk + 1) / 2;
  dim3 grid(npairs + (with_r ? p.nblk : 0), H, nsplit);
  kern<<<grid, 320, L::SMEM, st>>>(mKc, mQ, mOhi, mOlo, p);
  return cudaGetLastError();
}

template <bool QK_BF16, int D_QK, int D_V, int NST>
cudaError_t launch_gram_t(bool with_r, const CUtensorMap& mKc, const CUtensorMap& mQ,
                          const CUtensorMap& mOhi, const CUtensorMap& mOlo, const GramParams& p,
                          int H, int nsplit, cudaStream_t st) {
  using L = GramLayout<D_QK, D_V, NST>;
  auto kern = gram_kernel<QK_BF16, D_QK, D_V, NST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  const int npairs = p.nblk * (p.nblk + 1) / 2;
  dim3 grid(npairs + (with_r ? p.nblk : 0), H, nsplit);
  kern<<<grid, 192, L::SMEM, st>>>(mKc, mQ, mOhi, mOlo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gram(OperandMode mode, bool with_r, const CUtensorMap& mKc,
                        const CUtensorMap& mQ, const CUtensorMap& mOhi, const CUtensorMap& mOlo,
                        const GramParams& p, int H, int nsplit, cudaStream_t st) {
  switch (mode) {
    case kBF16d128: return launch_gram2_t<128>(with_r, mKc, mQ, mOhi, mOlo, p, H, nsplit, st);
    case kBF16d64: return launch_gram2_t<64>(with_r, mKc, mQ, mOhi, mOlo, p, H, nsplit, st);
    case kSplitF16d64:
      return launch_gram_t<false, 192, 64, 1>(with_r, mKc, mQ, mOhi, mOlo, p, H, nsplit, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gram_all_pairs(OperandMode mode, const CUtensorMap& mKc, const CUtensorMap& mQ,
                                  const CUtensorMap& mOhi, const CUtensorMap& mOlo,
                                  const GramParams& p, int H, int nsplit, cudaStream_t st) {
  if (p.nblk != 2) return cudaErrorInvalidValue;
  auto go = [&](auto kern, int smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(1, H, nsplit), 320, smem, st>>>(mKc, mQ, mOhi, mOlo, p);
    return cudaGetLastError();
  };
  switch (mode) {
    case kBF16d128: return go(gram3_kernel<128, false>, Gram3Layout<128, false>::SMEM);
    case kBF16d64: return go(gram3_kernel<64, false>, Gram3Layout<64, false>::SMEM);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gram_r(OperandMode mode, const CUtensorMap& mKc, const CUtensorMap& mQ,
                          const CUtensorMap& mOhi, const CUtensorMap& mOlo, const GramParams& p,
                          int H, int nsplit, cudaStream_t st) {
  if (p.nblk != 2 || !p.Rpart) return cudaErrorInvalidValue;
  auto go = [&](auto kern, int smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(1, H, nsplit), 320, smem, st>>>(mKc, mQ, mOhi, mOlo, p);
    return cudaGetLastError();
  };
  switch (mode) {
    case kBF16d128: return go(gram3_kernel<128, true>, Gram3Layout<128, true>::SMEM);
    case kBF16d64: return go(gram3_kernel<64, true>, Gram3Layout<64, true>::SMEM);
    default: return cudaErrorInvalidValue;
  }
}

int gram_smem(OperandMode mode) {
  switch (mode) {
    case kBF16d128:
      return std::max({Gram2Layout<128>::SMEM, Gram3Layout<128, false>::SMEM,
                       Gram3Layout<128, true>::SMEM});
    case kBF16d64:
      return std::max({Gram2Layout<64>::SMEM, Gram3Layout<64, false>::SMEM,
                       Gram3Layout<64, true>::SMEM});
    case kSplitF16d64: return GramLayout<192, 64, 1>::SMEM;
  }
  return 0;
}

}  // namespace lc
