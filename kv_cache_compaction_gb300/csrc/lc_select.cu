// Step 3 of attention-matching compaction: the t keys with the highest score
// ("KV compaction" blog, section "Fast KV Compaction via Attention Matching":
// C_k is the set of keys with the highest attention), ties to the lower
// index, returned in ascending order.
//
// Scores are compared through an order-preserving map of fp32 to uint32
// (order_code; -0 and +0 share a code).  Two algorithms:
//
// * select_topt_kernel: one CTA per head, four 8-bit radix passes over the
//   head's codes find the t-th largest code exactly; a block scan writes the
//   keys above it and the lowest-index keys equal to it.  Latency-bound; used
//   for short heads (the benchmark layer has T = 8192 per head).
//
// * the wide path, for long heads (T >= kWideMinT): (1) one CTA per head
//   samples the scores and takes as threshold theta the sample value
//   expected to have about 4t scores of the head at or above it; (2) a
//   streaming filter over every SM reads each score once (bulk copies into a
//   shared-memory ring) and writes the (code, index) pairs at or above theta
//   in index order, each CTA to its own region of the head's candidate list;
//   (3) one CTA per head reads the regions in order and writes the exact top
//   t, which come out in ascending index order without a sort.  If the
//   sample misjudged (fewer than t candidates, or more than a region or the
//   list holds), step (3) runs the exact single-CTA selection over the whole
//   head instead, so the result never depends on the sample: the top t of a
//   head are always among the scores >= theta when at least t scores are.
#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kWideSample = 16384;  // sampled scores per head
constexpr int kWideCap = 16384;     // candidate list length per head
constexpr int kWideTarget = 4;      // expected candidates: kWideTarget * t
constexpr int kSampleBlocks = 64;   // runs of consecutive keys in the sample
constexpr int kWideRegions = 256;   // filter warps per head, at most (one region each)
constexpr int kFilterWarps = 8;     // consumer warps per filter CTA (plus one producer)
constexpr int kFilterThreads = 32 * (kFilterWarps + 1);
constexpr int kSlice = 512;         // 16-byte words per warp and stage (8 KB)
constexpr int kFilterStages = 3;    // stages in flight per CTA (64 KB each)

// Source of the codes of one head: the codes themselves, or fp32 scores
// mapped on the fly.
struct CodeSrc {
  const uint32_t* c;
  static constexpr bool kCodes = true;
  __device__ __forceinline__ uint32_t operator()(int j) const { return c[j]; }
};
struct ScoreSrc {
  const float* u;
  static constexpr bool kCodes = false;
  __device__ __forceinline__ uint32_t operator()(int j) const { return order_code(u[j]); }
};

__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int& total) {
  // tmp: 32 ints of shared memory
  const int lane = lane_id(), w = warp_id();
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < static_cast<int>(blockDim.x >> 5) ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    tmp[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before_warp = w > 0 ? tmp[w - 1] : 0;
  total = tmp[31];
  __syncthreads();
  return before_warp + x - v;
}

// Locate, from a 256-bin histogram of one radix digit (counts of keys in the
// current bucket), the bin that holds rank `need` counted from the top, and
// the rank inside that bin.  Run by warp 0; lane l owns bins 255-8l..248-8l.
__device__ __forceinline__ void radix_pick_bin(const int* hist, int need, int shift,
                                               uint32_t prefix, uint32_t* s_prefix,
                                               int* s_need) {
  const int lane = lane_id();
  int cnt[8], own = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    cnt[k] = hist[255 - 8 * lane - k];
    own += cnt[k];
  }
  int incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int excl = incl - own;
  const uint32_t hit = __ballot_sync(0xffffffffu, incl >= need);
  const int src = hit ? __ffs(hit) - 1 : 31;
  if (lane == src) {
    int acc = excl, b = 255 - 8 * lane - 7;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (acc + cnt[k] >= need) {
        b = 255 - 8 * lane - k;
        break;
      }
      acc += cnt[k];
    }
    *s_prefix = prefix | (static_cast<uint32_t>(b) << shift);
    *s_need = need - acc;
  }
}

// Shared scratch of the selection routines.
struct SelShared {
  int hist[256];
  int tmp[32];
  uint32_t prefix;
  int need;
  int count;
};

// The t largest codes of one head (src(j), j < T), lowest index first on
// ties, written in ascending index order to dst[0..t).  NT threads.
// CPT > 0: thread i holds codes [CPT i, CPT i + CPT) in registers (T <= 1024
// CPT); CPT == 0: codes are re-read from the source in each pass.  Four 8-bit
// radix passes find the code of the t-th largest; equal bins within a
// thread's run are counted before the shared atomic.
template <int CPT, int NT, class Src>
__device__ void select_head(Src src, int T, int t, int32_t* dst, SelShared& sh) {
  const int tid = threadIdx.x;
  constexpr int R = CPT > 0 ? CPT : 1;
  uint32_t v[R];
  const int chunk = CPT > 0 ? CPT : (T + NT - 1) / NT;
  const int j0 = min(T, tid * chunk), j1 = min(T, j0 + chunk);
  if constexpr (CPT > 0) {
    bool vec = false;
    if constexpr (Src::kCodes)
      vec = j0 + CPT <= T && CPT % 4 == 0 && (reinterpret_cast<uintptr_t>(src.c + j0) & 15) == 0;
    if (vec) {
#pragma unroll
      for (int q = 0; q < CPT / 4; ++q) {
        const uint4 u = reinterpret_cast<const uint4*>(src.c + j0)[q];
        v[4 * q] = u.x;
        v[4 * q + 1] = u.y;
        v[4 * q + 2] = u.z;
        v[4 * q + 3] = u.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < CPT; ++k) v[k] = j0 + k < j1 ? src(j0 + k) : 0u;
    }
  }
  auto get = [&](int k) -> uint32_t {
    if constexpr (CPT > 0) return v[k];
    else return src(j0 + k);
  };
  uint32_t prefix = 0, mask = 0;
  int need = t;  // rank (from the top) still to locate inside the current bucket
  const int n = j1 - j0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += NT) sh.hist[b] = 0;
    __syncthreads();
    int run_bin = -1, run_cnt = 0;
    auto count = [&](uint32_t x) {
      if ((x & mask) == prefix) {
        const int bin = static_cast<int>((x >> shift) & 255u);
        if (bin == run_bin) {
          ++run_cnt;
        } else {
          if (run_cnt) atomicAdd(&sh.hist[run_bin], run_cnt);
          run_bin = bin;
          run_cnt = 1;
        }
      }
    };
    if constexpr (CPT > 0) {
#pragma unroll
      for (int k = 0; k < CPT; ++k)
        if (k < n) count(get(k));
    } else {
      for (int k = 0; k < n; ++k) count(get(k));
    }
    if (run_cnt) atomicAdd(&sh.hist[run_bin], run_cnt);
    __syncthreads();
    if (tid < 32) radix_pick_bin(sh.hist, need, shift, prefix, &sh.prefix, &sh.need);
    __syncthreads();
    prefix = sh.prefix;
    need = sh.need;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix = code of the t-th largest; take all larger codes and the first
  // `need` (lowest-index) codes equal to it.
  const uint32_t tau = prefix;
  int gt = 0, eq = 0;
  if constexpr (CPT > 0) {
#pragma unroll
    for (int k = 0; k < CPT; ++k)
      if (k < n) {
        gt += v[k] > tau;
        eq += v[k] == tau;
      }
  } else {
    for (int k = 0; k < n; ++k) {
      const uint32_t x = get(k);
      gt += x > tau;
      eq += x == tau;
    }
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, sh.tmp, tot);
  const int take_eq = max(0, min(eq, need - eq_before));
  const int out0 = block_exclusive_scan(gt + take_eq, sh.tmp, tot);
  int o = out0, te = 0;
  if constexpr (CPT > 0) {
#pragma unroll
    for (int k = 0; k < CPT; ++k)
      if (k < n && (v[k] > tau || (v[k] == tau && te++ < take_eq)) && o < t) dst[o++] = j0 + k;
  } else {
    for (int k = 0; k < n; ++k) {
      const uint32_t x = get(k);
      if ((x > tau || (x == tau && te++ < take_eq)) && o < t) dst[o++] = j0 + k;
    }
  }
}

template <int CPT>
__global__ void __launch_bounds__(kSelThreads)
    select_topt_kernel(const uint32_t* __restrict__ code, int T, int t, int32_t* __restrict__ idx) {
  __shared__ SelShared sh;
  const int h = blockIdx.x;
  select_head<CPT, kSelThreads>(CodeSrc{code + static_cast<size_t>(h) * T}, T, t,
                                idx + static_cast<size_t>(h) * t, sh);
}

// ------------------------------------------------------------- wide path

constexpr int kSmallThreads = 512;  // CTAs of the sample and final stages
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSampleRegs = kWideSample / kSmallThreads;  // sampled codes per thread
constexpr int kFinalRegs = kWideCap / kSmallThreads;      // candidates per thread

// Sum of v over the CTA (kSmallThreads threads), returned to every thread.
// red: 2 * kSmallWarps ints, used in turn by `phase` so that consecutive
// calls need one barrier each.
__device__ __forceinline__ int small_sum(int v, int* red, int phase) {
  v = __reduce_add_sync(0xffffffffu, v);
  int* r = red + (phase & 1) * kSmallWarps;
  if (lane_id() == 0) r[warp_id()] = v;
  __syncthreads();
  int s = 0;
#pragma unroll
  for (int w = 0; w < kSmallWarps; ++w) s += r[w];
  return s;
}

// Largest code c with at least k of the CTA's codes >= c, found one bit at a
// time from the top (bits 31 .. 32 - nbits; the lower bits of the result are
// zero).  With nbits = 32 and at least k codes, c is exactly the k-th
// largest code.  Each thread holds R codes in registers (nv valid).
template <int R>
__device__ uint32_t small_bisect_kth(const uint32_t (&v)[R], int nv, int k, int nbits, int* red) {
  uint32_t prefix = 0;
  for (int b = 0; b < nbits; ++b) {
    const uint32_t cand = prefix | (0x80000000u >> b);
    int c = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) c += (r < nv && v[r] >= cand) ? 1 : 0;
    if (small_sum(c, red, b) >= k) prefix = cand;
  }
  return prefix;
}

// (1) One CTA per head: a sample of kWideSample scores in kSampleBlocks
// runs of consecutive keys spread evenly over the head (whole sectors, few
// requests); theta = the sample's ceil(kWideTarget * t * S / T)-th largest
// code to 24 bits, so that about kWideTarget * t scores of the head lie at or
// above it (the threshold only steers how many candidates pass; the result
// does not depend on it).
template <class Src>
__global__ void __launch_bounds__(kSmallThreads)
    select_sample_kernel(Src src, int T, int t, WideScratch ws) {
  __shared__ int red[2 * kSmallWarps];
  const int h = blockIdx.x;
  Src s = src;
  if constexpr (Src::kCodes) s.c += static_cast<size_t>(h) * T;
  else s.u += static_cast<size_t>(h) * T;
  // piece p = 16 consecutive keys of run p / (keys per run / 16), 16-byte
  // loads (T % 4 == 0 and run starts rounded down to a multiple of 4)
  constexpr int kRun = kWideSample / kSampleBlocks;
  constexpr int kPieces = kSampleRegs / 16;  // pieces per thread
  uint4 raw[kPieces][4];
#pragma unroll
  for (int r = 0; r < kPieces; ++r) {
    const int piece = r * kSmallThreads + threadIdx.x;
    const int run = piece / (kRun / 16);
    const int start = static_cast<int>((static_cast<long long>(T - kRun) * run /
                                        (kSampleBlocks - 1)) & ~3ll);
    const int j = start + (piece % (kRun / 16)) * 16;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if constexpr (Src::kCodes) raw[r][q] = __ldg(reinterpret_cast<const uint4*>(s.c + j) + q);
      else raw[r][q] = __ldg(reinterpret_cast<const uint4*>(s.u + j) + q);
    }
  }
  uint32_t v[kSampleRegs];
#pragma unroll
  for (int r = 0; r < kPieces; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w4[4] = {raw[r][q].x, raw[r][q].y, raw[r][q].z, raw[r][q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        v[16 * r + 4 * q + e] = Src::kCodes ? w4[e] : order_code(__uint_as_float(w4[e]));
    }
  const double want = static_cast<double>(kWideTarget) * t * kWideSample / T;
  const int k = max(1, min(kWideSample, static_cast<int>(ceil(want))));
  const uint32_t theta = small_bisect_kth(v, kSampleRegs, k, 24, red);
  if (threadIdx.x == 0) ws.theta[h] = theta;
}

// (2) Streaming filter: every score of every head read once.  Each CTA owns
// a contiguous range of its head, split into kFilterWarps contiguous
// sub-ranges, one per consumer warp; each consumer warp writes its
// candidates, in index order, to its own region of the head's list (region
// c * kFilterWarps + w, `region` slots; the count goes to count[h][...],
// past `region` only counted).  A producer warp copies the next kSlice words
// of every sub-range into a kFilterStages-deep shared-memory ring by bulk
// asynchronous copies (stage i complete: full[i]; released by all consumer
// warps: empty[i]), so the copies run ahead of the scan and no CTA-wide
// barrier sits in the loop.  A consumer lane scans words r * 32 + lane of its
// slice; a warp scan of the lanes' hit counts per word row keeps the appends
// in index order.  Waits are bounded: on a timeout the error bit is set, the
// warps stop, and their regions are marked overflowed.
template <class Src>
__global__ void __launch_bounds__(kFilterThreads)
    select_filter_kernel(Src src, int T, int region, WideScratch ws) {
  extern __shared__ __align__(128) uint4 ring[];  // kFilterStages x kFilterWarps x kSlice
  __shared__ __align__(8) uint64_t full[kFilterStages];
  __shared__ __align__(8) uint64_t empty[kFilterStages];
  __shared__ volatile int abort_flag;
  const int h = blockIdx.y, warp = warp_id(), lane = lane_id();
  const size_t base = static_cast<size_t>(h) * T;
  const uint4* row;
  if constexpr (Src::kCodes) row = reinterpret_cast<const uint4*>(src.c + base);
  else row = reinterpret_cast<const uint4*>(src.u + base);
  const int nv = T / 4;
  const int per = (nv + gridDim.x - 1) / gridDim.x;
  const int c0 = min(nv, blockIdx.x * per), c1 = min(nv, c0 + per);
  const int sub = (c1 - c0 + kFilterWarps - 1) / kFilterWarps;  // words per sub-range
  const int nstage = (sub + kSlice - 1) / kSlice;
  auto range = [&](int w, int& a, int& b) {
    a = min(c1, c0 + w * sub);
    b = min(c1, a + sub);
  };
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kFilterStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kFilterWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == kFilterWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nstage; ++i) {
        const int s = i % kFilterStages;
        if (i >= kFilterStages &&
            !wait_bar(&empty[s], ((i / kFilterStages) - 1) & 1, &abort_flag, ws.err))
          break;
        uint32_t bytes = 0;
        for (int w = 0; w < kFilterWarps; ++w) {
          int a, b;
          range(w, a, b);
          const int q = a + i * kSlice;
          bytes += static_cast<uint32_t>(max(0, min(kSlice, b - q))) * 16u;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        for (int w = 0; w < kFilterWarps; ++w) {
          int a, b;
          range(w, a, b);
          const int q = a + i * kSlice;
          const int nq = min(kSlice, b - q);
          if (nq > 0)
            bulk_g2s(ring + (s * kFilterWarps + w) * kSlice, row + q,
                     static_cast<uint32_t>(nq) * 16u, &full[s]);
        }
        issued = i + 1;
      }
      // copies in flight land before the CTA exits (after an abort too)
      for (int i = max(0, issued - kFilterStages); i < issued; ++i)
        drain_wait(&full[i % kFilterStages], (i / kFilterStages) & 1);
    }
    return;
  }
  // -------------------------------------------------------------- consumers
  const uint32_t theta = ws.theta[h];
  // scores compare as floats against the threshold mapped back (the order
  // map is monotone and -0 == +0 in both); codes compare as codes
  const float theta_f = order_decode(theta);
  auto hit_of = [&](uint32_t w) -> bool {
    if constexpr (Src::kCodes) return w >= theta;
    else return __uint_as_float(w) >= theta_f;
  };
  auto code_of = [](uint32_t w) -> uint32_t {
    if constexpr (Src::kCodes) return w;
    else return order_code(__uint_as_float(w));
  };
  const int reg = blockIdx.x * kFilterWarps + warp;
  const size_t reg0 = static_cast<size_t>(h) * kWideCap + static_cast<size_t>(reg) * region;
  uint32_t* cc = ws.cand_code + reg0;
  int32_t* ci = ws.cand_idx + reg0;
  int a, b;
  range(warp, a, b);
  int count = 0;
  bool ok = true;
  constexpr int kRows = kSlice / 32;  // words per lane and stage
  for (int i = 0; i < nstage; ++i) {
    const int s = i % kFilterStages;
    if (!wait_bar(&full[s], (i / kFilterStages) & 1, &abort_flag, ws.err)) {
      ok = false;
      break;
    }
    const int q = a + i * kSlice;
    const int nq = max(0, min(kSlice, b - q));
    const uint4* sl = ring + (s * kFilterWarps + warp) * kSlice;
    uint4 v[kRows];
    uint64_t hitmask = 0u;  // bit 4r + e: element e of word r * 32 + lane
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int j = r * 32 + lane;
      v[r] = j < nq ? sl[j] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int j = r * 32 + lane;
      const uint64_t m4 = (hit_of(v[r].x) ? 1u : 0u) | (hit_of(v[r].y) ? 2u : 0u) |
                          (hit_of(v[r].z) ? 4u : 0u) | (hit_of(v[r].w) ? 8u : 0u);
      hitmask |= j < nq ? m4 << (4 * r) : 0ull;
    }
    // every lane has used every loaded word (the hit mask depends on all of
    // them), so the loads have completed: the slice may be refilled
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (__any_sync(0xffffffffu, hitmask != 0u)) {
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const unsigned m4 = static_cast<unsigned>((hitmask >> (4 * r)) & 15u);
        const unsigned rows_hit = __ballot_sync(0xffffffffu, m4 != 0u);
        if (rows_hit == 0u) continue;
        // lanes in order, a lane's elements in order: index order
        const int c = __popc(m4);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int pos = count + incl - c;
        const uint32_t w4[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((m4 >> e) & 1u) {
            if (pos < region) {
              cc[pos] = code_of(w4[e]);
              ci[pos] = 4 * (q + r * 32 + lane) + e;
            }
            ++pos;
          }
        }
        count += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
  }
  if (lane == 0) ws.count[h * kWideRegions + reg] = ok ? count : region + 1;
}

// (3) One CTA per head: the exact top t of the candidates.  The regions are
// read in order, so the list is sorted by key index.  tau = the t-th largest
// code (32-step bisection), then every code above tau and the first
// (lowest-index) codes equal to it are written, in list order, i.e. in
// ascending index order.  When the candidates cannot hold the top t (fewer
// than t, a region that overflowed, or more than a thread's share of the
// list), the exact selection over the whole head runs instead (with this
// CTA's kSmallThreads threads).
template <class Src>
__global__ void __launch_bounds__(kSmallThreads)
    select_final_kernel(Src src, int T, int t, int nreg, int region, WideScratch ws,
                        int32_t* __restrict__ idx) {
  __shared__ SelShared sh;
  __shared__ int red[2 * kSmallWarps];
  __shared__ int roff[kWideRegions + 1];
  const int h = blockIdx.x, tid = threadIdx.x;
  int32_t* dst = idx + static_cast<size_t>(h) * t;
  if (tid < 32) {
    // region offsets in the concatenated list (warp scan over <= 5 x 32)
    int carry = 0;
    bool overflow = false;
    for (int r0 = 0; r0 < nreg; r0 += 32) {
      const int r = r0 + tid;
      const int c = r < nreg ? ws.count[h * kWideRegions + r] : 0;
      overflow |= c > region;
      int incl = min(c, region);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      if (r < nreg) roff[r] = carry + incl - min(c, region);
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    overflow = __any_sync(0xffffffffu, overflow);
    if (tid == 0) roff[nreg] = overflow ? -1 : carry;
  }
  __syncthreads();
  const int n = roff[nreg];
  if (n < t || n > kWideCap) {
    Src s = src;
    if constexpr (Src::kCodes) s.c += static_cast<size_t>(h) * T;
    else s.u += static_cast<size_t>(h) * T;
    select_head<0, kSmallThreads>(s, T, t, dst, sh);
    return;
  }
  // thread i: entries [kFinalRegs i, kFinalRegs i + kFinalRegs) of the list
  // the regions form in order; the region of the first one by binary search
  // over the region offsets, every load issued before any is used
  uint32_t code[kFinalRegs];
  int32_t cid[kFinalRegs];
  const int e0 = min(n, tid * kFinalRegs);
  const int nv = min(n, e0 + kFinalRegs) - e0;
  {
    int lo = 0, hi = nreg - 1;  // last region whose offset is <= e0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (roff[mid] <= e0) lo = mid;
      else hi = mid - 1;
    }
    int r = lo;
    int g[kFinalRegs];
#pragma unroll
    for (int k = 0; k < kFinalRegs; ++k) {
      const int e = e0 + k;
      while (r + 1 < nreg && roff[r + 1] <= e) ++r;
      g[k] = k < nv ? r * region + (e - roff[r]) : 0;
    }
    const uint32_t* gc = ws.cand_code + static_cast<size_t>(h) * kWideCap;
    const int32_t* gi = ws.cand_idx + static_cast<size_t>(h) * kWideCap;
#pragma unroll
    for (int k = 0; k < kFinalRegs; ++k) {
      code[k] = k < nv ? gc[g[k]] : 0u;
      cid[k] = k < nv ? gi[g[k]] : 0;
    }
  }
  const uint32_t tau = small_bisect_kth(code, nv, t, 32, red);
  int above = 0, eq = 0;
#pragma unroll
  for (int k = 0; k < kFinalRegs; ++k) {
    above += (k < nv && code[k] > tau) ? 1 : 0;
    eq += (k < nv && code[k] == tau) ? 1 : 0;
  }
  const int take_eq = t - small_sum(above, red, 0);
  int tot;
  const int eq_before = block_exclusive_scan(eq, sh.tmp, tot);
  const int my_eq = max(0, min(eq, take_eq - eq_before));
  int o = block_exclusive_scan(above + my_eq, sh.tmp, tot);
  int te = 0;
#pragma unroll
  for (int k = 0; k < kFinalRegs; ++k)
    if (k < nv && (code[k] > tau || (code[k] == tau && te++ < my_eq)) && o < t) dst[o++] = cid[k];
}

constexpr size_t kRingBytes = static_cast<size_t>(kFilterStages) * kFilterWarps * kSlice * 16;

template <class Src>
cudaError_t wide_attributes() {
  constexpr int kDevices = 64;
  static volatile bool done[kDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kDevices && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(select_filter_kernel<Src>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kRingBytes));
  if (e == cudaSuccess && dev >= 0 && dev < kDevices) done[dev] = true;
  return e;
}

// CTAs per head of the filter: one wave over all heads, at most
// kWideRegions / kFilterWarps per head.
template <class Src>
cudaError_t filter_ctas(int H, int T, int sm_count, int* per_head) {
  int occ = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &occ, select_filter_kernel<Src>, kFilterThreads, kRingBytes);
  if (e != cudaSuccess) return e;
  const int per_head_max = max(1, (T / 4) / (kFilterWarps * kSlice));
  *per_head = max(1, min(min(per_head_max, kWideRegions / kFilterWarps),
                         max(1, occ) * sm_count / H));
  return cudaSuccess;
}

template <class Src>
cudaError_t launch_wide(Src src, int H, int T, int t, int32_t* idx, const WideScratch& ws,
                        int sm_count, int stage, cudaStream_t st) {
  const cudaError_t ea = wide_attributes<Src>();
  if (ea != cudaSuccess) return ea;
  int per_head = 1;
  const cudaError_t ef = filter_ctas<Src>(H, T, sm_count, &per_head);
  if (ef != cudaSuccess) return ef;
  const int nreg = per_head * kFilterWarps;
  const int region = kWideCap / nreg;
  if (stage == 0) {
    select_sample_kernel<Src><<<H, kSmallThreads, 0, st>>>(src, T, t, ws);
  } else if (stage == 1) {
    select_filter_kernel<Src><<<dim3(per_head, H), kFilterThreads, kRingBytes, st>>>(src, T,
                                                                                      region, ws);
  } else {
    select_final_kernel<Src><<<H, kSmallThreads, 0, st>>>(src, T, t, nreg, region, ws, idx);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select_topt(const uint32_t* code, int H, int T, int t, int32_t* idx,
                               cudaStream_t st) {
  if (T <= 4 * kSelThreads)
    select_topt_kernel<4><<<H, kSelThreads, 0, st>>>(code, T, t, idx);
  else if (T <= 8 * kSelThreads)
    select_topt_kernel<8><<<H, kSelThreads, 0, st>>>(code, T, t, idx);
  else if (T <= 32 * kSelThreads)
    select_topt_kernel<32><<<H, kSelThreads, 0, st>>>(code, T, t, idx);
  else
    select_topt_kernel<0><<<H, kSelThreads, 0, st>>>(code, T, t, idx);
  return cudaGetLastError();
}

bool select_wide_applies(int T, int t) { return T >= kWideMinT && t <= 1024 && T % 4 == 0; }

size_t select_wide_bytes(int H) {
  const size_t a = 256;
  const size_t theta = (static_cast<size_t>(H) * 4 + a - 1) / a * a;
  const size_t count = (static_cast<size_t>(H) * kWideRegions * 4 + a - 1) / a * a;
  return theta + count + static_cast<size_t>(H) * kWideCap * 8;
}

WideScratch wide_scratch(void* base, int H, uint32_t* err) {
  uint8_t* p = static_cast<uint8_t*>(base);
  const size_t a = 256;
  const size_t theta = (static_cast<size_t>(H) * 4 + a - 1) / a * a;
  const size_t count = (static_cast<size_t>(H) * kWideRegions * 4 + a - 1) / a * a;
  WideScratch w;
  w.theta = reinterpret_cast<uint32_t*>(p);
  w.count = reinterpret_cast<int*>(p + theta);
  w.cand_code = reinterpret_cast<uint32_t*>(p + theta + count);
  w.cand_idx = reinterpret_cast<int32_t*>(p + theta + count + static_cast<size_t>(H) * kWideCap * 4);
  w.err = err;
  return w;
}

cudaError_t launch_select_wide_codes(const uint32_t* code, int H, int T, int t, int32_t* idx,
                                     void* scratch, int sm_count, uint32_t* err, int stage,
                                     cudaStream_t st) {
  return launch_wide(CodeSrc{code}, H, T, t, idx, wide_scratch(scratch, H, err), sm_count, stage,
                     st);
}

cudaError_t launch_select_wide_scores(const float* u, int H, int T, int t, int32_t* idx,
                                      void* scratch, int sm_count, uint32_t* err, int stage,
                                      cudaStream_t st) {
  return launch_wide(ScoreSrc{u}, H, T, t, idx, wide_scratch(scratch, H, err), sm_count, stage,
                     st);
}

}  // namespace lc
