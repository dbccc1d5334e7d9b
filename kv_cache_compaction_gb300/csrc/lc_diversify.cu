// Farthest-first traversal of a head's keys ("Latent Compaction with
// Test-Time Training", §3.2 Eq. (7), after Gonzalez 1985): starting from the
// seed set S, repeatedly add i* = argmax_{i not in S} min_{j in S} ||k_i - k_j||^2.
//
// One thread-block cluster per KV head.  CTA r of the cluster owns the key
// slice [r P, (r + 1) P) and keeps, per key, the squared distance to its
// nearest selected key (-inf once the key is selected, so it never wins
// again).  When the slice fits, its keys stay in shared memory for the whole
// traversal; otherwise they are re-read from global memory at every step.
// Per step: every CTA finds its slice's farthest key (block reduction, ties
// to the lower index), publishes it in shared memory, and after one cluster
// barrier every CTA reads all published candidates through distributed
// shared memory and takes the same winner; then every CTA folds the winner's
// distance into its slice.  The candidate slots alternate between two
// buffers by step parity, so one barrier per step orders each write after
// the previous step's reads.  Distances are fp32 sums of squared
// differences of the bf16 keys, one warp per key (lanes over d, coalesced
// row reads, a shuffle reduction).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace lc {
namespace {

constexpr int kFFThreads = 256;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ float2 ld_dsmem_f2(const float2* local, uint32_t rank) {
  uint32_t a = smem_u32(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(ra)
               : "memory");
  return v;
}

// (value, index) with ties to the lower index; index -1 = none.
__device__ __forceinline__ bool ff_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i >= 0 && (bi < 0 || i < bi));
}

// Squared distance of key row `kr` (D bf16 values, read by the whole warp)
// to the center `c` (D floats in shared memory); every lane gets the sum.
template <int D>
__device__ __forceinline__ float warp_dist2(const __nv_bfloat16* kr, const float* c, int lane) {
  constexpr int PER = D / 32;
  float s = 0.f;
  if constexpr (PER == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(kr + lane * 4);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    const float e0 = a.x - c[lane * 4], e1 = a.y - c[lane * 4 + 1];
    const float e2 = b.x - c[lane * 4 + 2], e3 = b.y - c[lane * 4 + 3];
    s = fmaf(e0, e0, fmaf(e1, e1, fmaf(e2, e2, e3 * e3)));
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(kr + lane * 2);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
    const float e0 = a.x - c[lane * 2], e1 = a.y - c[lane * 2 + 1];
    s = fmaf(e0, e0, e1 * e1);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

template <int D, bool RESIDENT>
__global__ void __launch_bounds__(kFFThreads, 1)
    farthest_first_kernel(const __nv_bfloat16* __restrict__ K, int T, const int32_t* seeds,
                          int n_seed, int n_add, int P, int32_t* out) {
  extern __shared__ uint8_t ff_smem[];
  __shared__ float2 slot[2];     // this CTA's candidate, by step parity
  __shared__ float2 wred[kFFThreads / 32];
  __shared__ float center[D];
  __shared__ int s_winner;
  const uint32_t rank = cluster_ctarank(), ncl = cluster_nctarank();
  const int h = blockIdx.x / ncl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int base = static_cast<int>(rank) * P;
  const int cnt = max(0, min(P, T - base));
  const __nv_bfloat16* Kh = K + static_cast<size_t>(h) * T * D;
  float* mind = reinterpret_cast<float*>(ff_smem);
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(ff_smem + ((P * 4 + 15) & ~15));

  for (int i = tid; i < P; i += kFFThreads) mind[i] = i < cnt ? kInf : -kInf;
  if constexpr (RESIDENT) {
    const uint4* src = reinterpret_cast<const uint4*>(Kh + static_cast<size_t>(base) * D);
    uint4* dst = reinterpret_cast<uint4*>(sK);
    for (int i = tid; i < cnt * D / 8; i += kFFThreads) dst[i] = src[i];
  }
  if (rank == 0)
    for (int i = tid; i < n_add; i += kFFThreads) out[static_cast<size_t>(h) * n_add + i] = -1;
  __syncthreads();

  // fold the distance to key `c` into the slice and mark c selected
  auto fold = [&](int c) {
    for (int k = tid; k < D; k += kFFThreads) center[k] = __bfloat162float(Kh[static_cast<size_t>(c) * D + k]);
    __syncthreads();
    for (int i = warp; i < cnt; i += kFFThreads / 32) {
      const __nv_bfloat16* kr = RESIDENT ? sK + static_cast<size_t>(i) * D
                                         : Kh + static_cast<size_t>(base + i) * D;
      const float d2 = warp_dist2<D>(kr, center, lane);
      if (lane == 0) mind[i] = fminf(mind[i], d2);
    }
    __syncthreads();
    if (tid == 0 && c >= base && c < base + cnt) mind[c - base] = -kInf;
    __syncthreads();
  };

  for (int s = 0; s < n_seed; ++s) {
    const int c = seeds[static_cast<size_t>(h) * n_seed + s];
    if (c >= 0 && c < T) fold(c);
  }
  cluster_sync_all();  // every CTA of the cluster is running before DSMEM reads

  for (int it = 0; it < n_add; ++it) {
    // local farthest key
    float bv = -kInf;
    int bi = -1;
    for (int i = tid; i < cnt; i += kFFThreads) {
      const float v = mind[i];
      if (ff_better(v, base + i, bv, bi) && v > -kInf) {
        bv = v;
        bi = base + i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ff_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) wred[warp] = make_float2(bv, __int_as_float(bi));
    __syncthreads();
    if (tid == 0) {
      float v = -kInf;
      int ix = -1;
      for (int w = 0; w < kFFThreads / 32; ++w) {
        const float2 c = wred[w];
        if (ff_better(c.x, __float_as_int(c.y), v, ix)) {
          v = c.x;
          ix = __float_as_int(c.y);
        }
      }
      slot[it & 1] = make_float2(v, __int_as_float(ix));
    }
    cluster_sync_all();
    if (tid == 0) {
      float v = -kInf;
      int ix = -1;
      for (uint32_t r = 0; r < ncl; ++r) {
        const float2 c = ld_dsmem_f2(&slot[it & 1], r);
        if (ff_better(c.x, __float_as_int(c.y), v, ix)) {
          v = c.x;
          ix = __float_as_int(c.y);
        }
      }
      s_winner = (v > -kInf) ? ix : -1;
      if (rank == 0 && s_winner >= 0) out[static_cast<size_t>(h) * n_add + it] = s_winner;
    }
    __syncthreads();
    const int c = s_winner;
    if (c < 0) break;  // no key left (uniform across the cluster)
    fold(c);
  }
  cluster_sync_all();  // no CTA leaves while another may still read its slots
}

template <int D, bool RESIDENT>
cudaError_t launch_ff_t(const __nv_bfloat16* K, int H, int T, const int32_t* seeds, int n_seed,
                        int n_add, int cl, int P, size_t smem, int32_t* out, cudaStream_t st) {
  auto kern = farthest_first_kernel<D, RESIDENT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (cl > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(H * cl);
  cfg.blockDim = dim3(kFFThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nclusters = 0;
  e = cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (nclusters < 1) return cudaErrorInvalidConfiguration;
  e = cudaLaunchKernelEx(&cfg, kern, K, T, seeds, n_seed, n_add, P, out);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_ff_d(const __nv_bfloat16* K, int H, int T, const int32_t* seeds, int n_seed,
                        int n_add, int32_t* out, cudaStream_t st) {
  constexpr size_t kBudget = 200 * 1024;  // dynamic shared memory per CTA
  // smallest cluster whose slices (keys and distances) fit in shared memory
  for (int cl = 1; cl <= 16; cl *= 2) {
    const int P = (T + cl - 1) / cl;
    const size_t smem = ((static_cast<size_t>(P) * 4 + 15) & ~size_t(15)) +
                        static_cast<size_t>(P) * D * 2;
    if (smem <= kBudget) {
      cudaError_t e = launch_ff_t<D, true>(K, H, T, seeds, n_seed, n_add, cl, P, smem, out, st);
      if (e != cudaErrorInvalidConfiguration || cl <= 8) return e;
      (void)cudaGetLastError();  // cluster of 16 not schedulable here: stream instead
      break;
    }
  }
  // keys re-read from global memory at every step; distances stay resident
  for (int cl = 8; cl <= 16; cl *= 2) {
    const int P = (T + cl - 1) / cl;
    const size_t smem = (static_cast<size_t>(P) * 4 + 15) & ~size_t(15);
    if (smem <= kBudget || cl == 16) {
      if (smem > kBudget) return cudaErrorInvalidValue;
      return launch_ff_t<D, false>(K, H, T, seeds, n_seed, n_add, cl, P, smem, out, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_farthest_first(int d, const __nv_bfloat16* K, int H, int T,
                                  const int32_t* seeds, int n_seed, int n_add, int32_t* out,
                                  cudaStream_t st) {
  switch (d) {
    case 64: return launch_ff_d<64>(K, H, T, seeds, n_seed, n_add, out, st);
    case 128: return launch_ff_d<128>(K, H, T, seeds, n_seed, n_add, out, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lc
