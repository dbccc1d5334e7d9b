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
//   draws a strided sample of the scores and takes as threshold theta the
//   sample value expected to have about 4t scores of the head at or above
//   it; (2) a streaming filter over every SM reads each score once (16-byte
//   loads) and appends the (code, index) pairs at or above theta to a
//   per-head candidate list; (3) one CTA per head selects the exact top t
//   among the candidates and sorts their indices.  If the sample misjudged
//   (fewer than t candidates, or more than the list holds), step (3) runs
//   the exact single-CTA selection over the whole head instead, so the
//   result never depends on the sample: the top t of a head are always
//   among the scores >= theta when at least t scores are.
#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kWideSample = 16384;  // sampled scores per head
constexpr int kWideCap = 16384;     // candidate list length per head
constexpr int kWideTarget = 4;      // expected candidates: kWideTarget * t
constexpr int kFilterThreads = 256;
constexpr int kFilterUnroll = 4;    // 16-byte loads in flight per thread

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
// ties, written in ascending index order to dst[0..t).  kSelThreads threads.
// CPT > 0: thread i holds codes [CPT i, CPT i + CPT) in registers (T <= 1024
// CPT); CPT == 0: codes are re-read from the source in each pass.  Four 8-bit
// radix passes find the code of the t-th largest; equal bins within a
// thread's run are counted before the shared atomic.
template <int CPT, class Src>
__device__ void select_head(Src src, int T, int t, int32_t* dst, SelShared& sh) {
  const int tid = threadIdx.x;
  constexpr int R = CPT > 0 ? CPT : 1;
  uint32_t v[R];
  const int chunk = CPT > 0 ? CPT : (T + kSelThreads - 1) / kSelThreads;
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
    for (int b = tid; b < 256; b += kSelThreads) sh.hist[b] = 0;
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
  select_head<CPT>(CodeSrc{code + static_cast<size_t>(h) * T}, T, t,
                   idx + static_cast<size_t>(h) * t, sh);
}

// ------------------------------------------------------------- wide path

// Rank-k largest of keys key(i) over the i < n with pred(i), by four 8-bit
// radix passes over shared memory: returns the key value (all four digits)
// and, in *rank, how many keys equal to it belong to the top k.  Histogram
// updates are aggregated over the lanes of a warp that share a bin.
template <class Key, class Pred>
__device__ uint32_t block_kth_largest(Key key, Pred pred, int n, int k, SelShared& sh, int* rank) {
  const int tid = threadIdx.x, lane = lane_id();
  uint32_t prefix = 0, mask = 0;
  int need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += blockDim.x) sh.hist[b] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += blockDim.x) {
      const int i = i0 + tid;
      int bin = -1;
      if (i < n && pred(i)) {
        const uint32_t x = key(i);
        if ((x & mask) == prefix) bin = static_cast<int>((x >> shift) & 255u);
      }
      const unsigned active = __activemask();
      const unsigned peers = __match_any_sync(active, bin);
      if (bin >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[bin], __popc(peers));
    }
    __syncthreads();
    if (tid < 32) radix_pick_bin(sh.hist, need, shift, prefix, &sh.prefix, &sh.need);
    __syncthreads();
    prefix = sh.prefix;
    need = sh.need;
    mask |= 255u << shift;
    __syncthreads();
  }
  *rank = need;
  return prefix;
}

// (1) One CTA per head: a strided sample of kWideSample scores; theta = the
// sample's ceil(kWideTarget * t * S / T)-th largest code, so that about
// kWideTarget * t scores of the head lie at or above it.  Also clears the
// head's candidate count.
template <class Src>
__global__ void __launch_bounds__(kSelThreads)
    select_sample_kernel(Src src, int T, int t, WideScratch ws) {
  extern __shared__ uint32_t smp[];  // kWideSample codes
  __shared__ SelShared sh;
  const int h = blockIdx.x;
  Src s = src;
  if constexpr (Src::kCodes) s.c += static_cast<size_t>(h) * T;
  else s.u += static_cast<size_t>(h) * T;
  const int stride = T / kWideSample;
  constexpr int kPer = kWideSample / kSelThreads;
  uint32_t v[kPer];
#pragma unroll
  for (int r = 0; r < kPer; ++r) v[r] = s((threadIdx.x + r * kSelThreads) * stride);
#pragma unroll
  for (int r = 0; r < kPer; ++r) smp[threadIdx.x + r * kSelThreads] = v[r];
  __syncthreads();
  const double want = static_cast<double>(kWideTarget) * t * kWideSample / T;
  const int k = max(1, min(kWideSample, static_cast<int>(ceil(want))));
  int rank;
  const uint32_t theta = block_kth_largest([&](int i) { return smp[i]; }, [](int) { return true; },
                                           kWideSample, k, sh, &rank);
  if (threadIdx.x == 0) {
    ws.theta[h] = theta;
    ws.count[h] = 0;
  }
}

// (2) Streaming filter: every score of every head read once with 16-byte
// loads (T % 4 == 0, 16-byte aligned rows), the next batch of loads issued
// before the current one is examined; the (code, index) pairs with code >=
// theta of their head are appended to the head's candidate list, one atomic
// per warp and batch (a warp scan of the lanes' hit counts places them).
// Pairs past the list's end are counted but not stored.
template <class Src>
__global__ void __launch_bounds__(kFilterThreads)
    select_filter_kernel(Src src, int T, WideScratch ws) {
  const int h = blockIdx.y, lane = lane_id();
  const uint32_t theta = ws.theta[h];
  const size_t base = static_cast<size_t>(h) * T;
  const uint4* row;
  if constexpr (Src::kCodes) row = reinterpret_cast<const uint4*>(src.c + base);
  else row = reinterpret_cast<const uint4*>(src.u + base);
  int* cnt = ws.count + h;
  uint32_t* cc = ws.cand_code + static_cast<size_t>(h) * kWideCap;
  int32_t* ci = ws.cand_idx + static_cast<size_t>(h) * kWideCap;
  const int nv = T / 4;
  constexpr int kBatch = kFilterThreads * kFilterUnroll;
  const int step = gridDim.x * kBatch;
  auto code_of = [](uint32_t w) -> uint32_t {
    if constexpr (Src::kCodes) return w;
    else return order_code(__uint_as_float(w));
  };
  uint4 cur[kFilterUnroll], nxt[kFilterUnroll];
  auto load = [&](uint4 (&v)[kFilterUnroll], int q0) {
#pragma unroll
    for (int k = 0; k < kFilterUnroll; ++k) {
      const int q = q0 + k * kFilterThreads + threadIdx.x;
      v[k] = q < nv ? __ldcs(row + q) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  int q0 = blockIdx.x * kBatch;
  if (q0 < nv) load(cur, q0);
  for (; q0 < nv; q0 += step) {
    const int qn = q0 + step;
    if (qn < nv) load(nxt, qn);
    uint32_t code[kFilterUnroll * 4];
    int hits = 0;
#pragma unroll
    for (int k = 0; k < kFilterUnroll; ++k) {
      const int q = q0 + k * kFilterThreads + threadIdx.x;
      const uint32_t w[4] = {cur[k].x, cur[k].y, cur[k].z, cur[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t c = code_of(w[e]);
        code[4 * k + e] = c;
        hits += (q < nv && c >= theta) ? 1 : 0;
      }
    }
    if (__any_sync(0xffffffffu, hits > 0)) {
      int incl = hits;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int pos = 0;
      if (lane == 31) pos = atomicAdd(cnt, incl);
      pos = __shfl_sync(0xffffffffu, pos, 31) + incl - hits;
#pragma unroll
      for (int k = 0; k < kFilterUnroll; ++k) {
        const int q = q0 + k * kFilterThreads + threadIdx.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t c = code[4 * k + e];
          if (q < nv && c >= theta) {
            if (pos < kWideCap) {
              cc[pos] = c;
              ci[pos] = 4 * q + e;
            }
            ++pos;
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kFilterUnroll; ++k) cur[k] = nxt[k];
  }
}

// (3) One CTA per head: the exact top t of the candidates (the t-th largest
// code tau, all codes above it, and of the codes equal to it those with the
// lowest indices), indices sorted ascending by a bitonic network.  When the
// candidates cannot hold the top t (fewer than t, or the list overflowed),
// the exact single-CTA selection over the whole head runs instead.
template <class Src>
__global__ void __launch_bounds__(kSelThreads)
    select_final_kernel(Src src, int T, int t, WideScratch ws, int32_t* __restrict__ idx) {
  extern __shared__ uint32_t dyn[];
  __shared__ SelShared sh;
  __shared__ int sorted[1024];
  const int h = blockIdx.x, tid = threadIdx.x, lane = lane_id();
  int32_t* dst = idx + static_cast<size_t>(h) * t;
  const int n = ws.count[h];
  if (n < t || n > kWideCap) {
    Src s = src;
    if constexpr (Src::kCodes) s.c += static_cast<size_t>(h) * T;
    else s.u += static_cast<size_t>(h) * T;
    select_head<0>(s, T, t, dst, sh);
    return;
  }
  uint32_t* code = dyn;
  int32_t* cid = reinterpret_cast<int32_t*>(dyn + kWideCap);
  {
    constexpr int kPer = kWideCap / kSelThreads;
    const uint32_t* gc = ws.cand_code + static_cast<size_t>(h) * kWideCap;
    const int32_t* gi = ws.cand_idx + static_cast<size_t>(h) * kWideCap;
    uint32_t vc[kPer];
    int32_t vi[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = tid + r * kSelThreads;
      vc[r] = i < n ? gc[i] : 0u;
      vi[r] = i < n ? gi[i] : 0;
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = tid + r * kSelThreads;
      if (i < n) {
        code[i] = vc[r];
        cid[i] = vi[r];
      }
    }
  }
  __syncthreads();
  int take_eq;
  const uint32_t tau = block_kth_largest([&](int i) { return code[i]; }, [](int) { return true; },
                                         n, t, sh, &take_eq);
  // among the codes equal to tau, the take_eq lowest indices: the
  // take_eq-th largest of ~index
  int ties = 0;
  for (int i = tid; i < n; i += blockDim.x) ties += code[i] == tau;
  for (int o = 16; o > 0; o >>= 1) ties += __shfl_xor_sync(0xffffffffu, ties, o);
  if (tid == 0) sh.count = 0;
  __syncthreads();
  if (lane == 0) atomicAdd(&sh.count, ties);
  __syncthreads();
  ties = sh.count;
  __syncthreads();
  uint32_t cut = 0xffffffffu;  // keep ties with index <= cut
  if (take_eq < ties) {
    int r;
    const uint32_t ncut = block_kth_largest([&](int i) { return ~static_cast<uint32_t>(cid[i]); },
                                            [&](int i) { return code[i] == tau; }, n, take_eq, sh,
                                            &r);
    cut = ~ncut;
  }
  // compact the t kept indices (any order), then sort them
  if (tid == 0) sh.count = 0;
  for (int i = tid; i < 1024; i += blockDim.x) sorted[i] = 0x7fffffff;
  __syncthreads();
  for (int i0 = 0; i0 < n; i0 += blockDim.x) {
    const int i = i0 + tid;
    const bool keep = i < n && (code[i] > tau || (code[i] == tau &&
                                                  static_cast<uint32_t>(cid[i]) <= cut));
    const unsigned active = __activemask();
    const unsigned m = __ballot_sync(active, keep);
    int pos = 0;
    if (m) {
      const int leader = __ffs(m) - 1;
      if (lane == leader) pos = atomicAdd(&sh.count, __popc(m));
      pos = __shfl_sync(active, pos, leader) + __popc(m & ((1u << lane) - 1u));
    }
    if (keep && pos < 1024) sorted[pos] = cid[i];
  }
  __syncthreads();
  // bitonic sort of the 1024 slots (padding sorts last)
  for (int k = 2; k <= 1024; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < 1024; i += blockDim.x) {
        const int p = i ^ j;
        if (p > i) {
          const int a = sorted[i], b = sorted[p];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            sorted[i] = b;
            sorted[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < t; i += blockDim.x) dst[i] = sorted[i];
}

// Opt the two shared-memory-heavy kernels of one source type into their
// dynamic shared memory, once per device (setting it twice is harmless, so
// concurrent first calls need no lock).
template <class Src>
cudaError_t wide_attributes() {
  constexpr int kDevices = 64;
  static volatile bool done[kDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kDevices && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(select_sample_kernel<Src>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kWideSample * 4));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(select_final_kernel<Src>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(static_cast<size_t>(kWideCap) * 8));
  if (e == cudaSuccess && dev >= 0 && dev < kDevices) done[dev] = true;
  return e;
}

template <class Src>
cudaError_t launch_wide(Src src, int H, int T, int t, int32_t* idx, const WideScratch& ws,
                        int sm_count, int stage, cudaStream_t st) {
  const cudaError_t ea = wide_attributes<Src>();
  if (ea != cudaSuccess) return ea;
  if (stage == 0) {
    select_sample_kernel<Src><<<H, kSelThreads, kWideSample * 4, st>>>(src, T, t, ws);
  } else if (stage == 1) {
    // eight 256-thread CTAs per SM over all heads
    const int per_head_max =
        (T / 4 + kFilterThreads * kFilterUnroll - 1) / (kFilterThreads * kFilterUnroll);
    const int per_head = max(1, min(per_head_max, (8 * sm_count + H - 1) / H));
    select_filter_kernel<Src><<<dim3(per_head, H), kFilterThreads, 0, st>>>(src, T, ws);
  } else {
    select_final_kernel<Src><<<H, kSelThreads, static_cast<size_t>(kWideCap) * 8, st>>>(
        src, T, t, ws, idx);
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
  const size_t head = 256;  // theta and count, padded
  return 2 * head * ((static_cast<size_t>(H) * 4 + head - 1) / head) +
         static_cast<size_t>(H) * kWideCap * 8;
}

WideScratch wide_scratch(void* base, int H) {
  uint8_t* p = static_cast<uint8_t*>(base);
  const size_t hb = ((static_cast<size_t>(H) * 4 + 255) / 256) * 256;
  WideScratch w;
  w.theta = reinterpret_cast<uint32_t*>(p);
  w.count = reinterpret_cast<int*>(p + hb);
  w.cand_code = reinterpret_cast<uint32_t*>(p + 2 * hb);
  w.cand_idx = reinterpret_cast<int32_t*>(p + 2 * hb + static_cast<size_t>(H) * kWideCap * 4);
  return w;
}

cudaError_t launch_select_wide_codes(const uint32_t* code, int H, int T, int t, int32_t* idx,
                                     void* scratch, int sm_count, int stage, cudaStream_t st) {
  return launch_wide(CodeSrc{code}, H, T, t, idx, wide_scratch(scratch, H), sm_count, stage, st);
}

cudaError_t launch_select_wide_scores(const float* u, int H, int T, int t, int32_t* idx,
                                      void* scratch, int sm_count, int stage, cudaStream_t st) {
  return launch_wide(ScoreSrc{u}, H, T, t, idx, wide_scratch(scratch, H), sm_count, stage, st);
}

}  // namespace lc
