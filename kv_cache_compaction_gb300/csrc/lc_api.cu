// Host orchestrator behind include/lc.h: argument checks, workspace carving,
// TMA tensor maps, and the launch sequence of the five compaction steps.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/lc.h"
#include "lc_common.cuh"
#include "lc_kernels.cuh"

using namespace lc;

namespace {

constexpr int kMaxHeads = 4096;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// [H][rows][inner] 16-bit tensor, 64-element x box_rows boxes, 128B swizzle,
// zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* ptr, bool bf16, int inner, int rows, int H,
              int box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(H)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2,
                           static_cast<cuuint64_t>(inner) * 2 * rows};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct Plan {
  OperandMode mode;
  bool bf16_in;
  int H, n_q, T, d, t, d_qk, n_q_pad, t_pad, nblk;
  float scale;
  int max_iter;
  bool all_pairs;              // one CTA forms all three Gram blocks (bf16, nblk == 2)
  int ks_max, g5_max, g7_max, r_max;  // largest query splits the workspace holds
  // workspace offsets (bytes)
  size_t qop, kop, vhi, vlo;            // operand copies (16-bit)
  size_t m_pad, lse_pad, ohi, olo;      // step-1 results
  size_t ucode, idx, selw;              // steps 2-3 (selw: wide-select scratch)
  bool selw_on;                         // step 3 through the wide path
  size_t kc, khash;                     // kept-key rows and their hashes
  size_t rowsh2, rowb, colb2, lc2;      // fit inputs
  size_t gpart, cpart, G, c;            // mass system
  size_t hpart, rpart, Hm, R, vc;       // output system
  size_t mat, vec, wbuf;                // solver scratch
  size_t w_tmp, beta_tmp;               // steps 4 results when the caller gives none
  size_t total;
};

// Query-range split for a launch of `units` independent CTAs (times the
// split) on `sms` SMs with `occ` CTAs resident per SM: the split in
// [1, max_split] whose last wave is fullest (ties to the smaller split).
int best_split(int units, int sms, int occ, int max_split) {
  const int slots = sms * occ;
  int best = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= max_split; ++s) {
    const long long ctas = static_cast<long long>(units) * s;
    const long long waves = (ctas + slots - 1) / slots;
    const double eff = static_cast<double>(ctas) / static_cast<double>(waves * slots);
    if (eff > best_eff + 1e-3) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

// Upper bound on the split used for `units` CTAs: about four full waves of
// a 160-SM device, never more than the number of query tiles.
int max_split(int units, int occ, int tiles) {
  int s = (4 * 160 * occ + units - 1) / units;
  if (s < 1) s = 1;
  if (s > tiles) s = tiles;
  if (s > 64) s = 64;
  return s;
}

lc_status validate(const lc_shape* s) {
  if (!s) return LC_ERR_INVALID_ARG;
  if (s->n_kv_heads < 1 || s->n_kv_heads > kMaxHeads || s->n_q < 1 || s->T < 1 || s->t < 1)
    return LC_ERR_INVALID_ARG;
  if (s->t > s->T) return LC_ERR_INVALID_ARG;
  if (s->t > 1024) return LC_ERR_UNSUPPORTED;
  if (s->d != 64 && s->d != 128) return LC_ERR_UNSUPPORTED;
  if (s->in_dtype != LC_BF16 && s->in_dtype != LC_FP32) return LC_ERR_INVALID_ARG;
  if (s->in_dtype == LC_FP32 && s->d != 64) return LC_ERR_UNSUPPORTED;
  if (!(s->scale >= 0.f) || !std::isfinite(s->scale)) return LC_ERR_INVALID_ARG;
  if (s->nnls_max_iter < 0) return LC_ERR_INVALID_ARG;
  // tensor-map extents are 32-bit
  if (static_cast<long long>(s->n_q) + 256 > (1ll << 31) || static_cast<long long>(s->T) + 256 > (1ll << 31))
    return LC_ERR_UNSUPPORTED;
  return LC_OK;
}

Plan make_plan(const lc_shape* s) {
  Plan p{};
  p.H = s->n_kv_heads;
  p.n_q = s->n_q;
  p.T = s->T;
  p.d = s->d;
  p.t = s->t;
  p.bf16_in = s->in_dtype == LC_BF16;
  p.mode = p.bf16_in ? (s->d == 128 ? kBF16d128 : kBF16d64) : kSplitF16d64;
  p.d_qk = p.bf16_in ? s->d : 3 * s->d;
  p.n_q_pad = static_cast<int>(round_up(s->n_q, 128));
  p.t_pad = static_cast<int>(round_up(s->t, 128));
  p.nblk = p.t_pad / 128;
  p.scale = s->scale > 0.f ? s->scale : 1.f / std::sqrt(static_cast<float>(s->d));
  p.max_iter = s->nnls_max_iter > 0 ? s->nnls_max_iter : 3 * s->t;

  const int nqt = p.n_q_pad / 128;
  const int slabs = p.n_q_pad / 64;
  const int npairs = p.nblk * (p.nblk + 1) / 2;
  p.ks_max = max_split(((p.T + 255) / 256) * p.H, 2, nqt);
  p.all_pairs = p.bf16_in && p.nblk == 2;
  if (p.all_pairs) {
    // long CTAs: at most two waves of a 160-SM device, but no CTA sums more
    // than kGramChain slabs in one accumulator
    const int cap = std::max(gram_min_split(slabs),
                             std::max(1, std::min(max_split(p.H, 1, slabs), 320 / p.H)));
    p.g5_max = p.g7_max = cap;
    p.r_max = cap;
  } else {
    p.g5_max = max_split(npairs * p.H, 1, slabs);
    p.g7_max = p.r_max = max_split((npairs + p.nblk) * p.H, 1, slabs);
  }

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  };
  const size_t H = p.H;
  if (p.bf16_in) {
    p.qop = p.kop = 0;  // caller's Q and K are used directly
    p.vhi = take(H * p.T * p.d * 2);
    p.vlo = 0;
  } else {
    p.qop = take(H * p.n_q * p.d_qk * 2);
    p.kop = take(H * p.T * p.d_qk * 2);
    p.vhi = take(H * p.T * p.d * 2);
    p.vlo = take(H * p.T * p.d * 2);
  }
  p.m_pad = take(H * p.n_q_pad * 4);
  p.lse_pad = take(H * p.n_q_pad * 4);
  p.ohi = take(H * p.n_q * p.d * 2);
  p.olo = take(H * p.n_q * p.d * 2);
  p.ucode = take(H * p.T * 4);
  p.selw_on = select_wide_applies(p.T, p.t);
  p.selw = take(p.selw_on ? select_wide_bytes(p.H) : 0);
  p.idx = take(H * p.t * 4);
  p.kc = take(H * p.t_pad * p.d_qk * 2);
  p.khash = take(H * p.t_pad * 4);
  p.rowsh2 = take(H * p.n_q_pad * 4);
  p.rowb = take(H * p.n_q_pad * 4);
  p.colb2 = take(H * p.t_pad * 4);
  p.lc2 = take(H * p.n_q_pad * 4);
  const size_t tt = static_cast<size_t>(p.t_pad) * p.t_pad;
  p.gpart = take(static_cast<size_t>(p.g5_max) * H * tt * 4);
  p.cpart = take(static_cast<size_t>(p.g5_max) * H * p.t_pad * 4);
  p.G = take(H * tt * 4);
  p.c = take(H * p.t_pad * 4);
  p.hpart = take(static_cast<size_t>(p.g7_max) * H * tt * 4);
  p.rpart = take(static_cast<size_t>(p.r_max) * H * p.t_pad * p.d * 4);
  p.Hm = take(H * tt * 4);
  p.R = take(H * p.t_pad * p.d * 4);
  p.vc = take(H * p.t_pad * p.d * 4);
  p.mat = take(H * tt * 4);
  p.vec = take(H * 8 * p.t_pad * 4);
  p.wbuf = take(H * p.t_pad * 64 * 4);
  p.w_tmp = take(H * p.t * 4);
  p.beta_tmp = take(H * p.t * 4);
  p.total = off;
  return p;
}

#define LC_CUDA(call)                                   \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) {                            \
      std::fprintf(stderr, "lc: %s failed: %s\n", #call, cudaGetErrorString(e_)); \
      return LC_ERR_CUDA;                               \
    }                                                   \
  } while (0)

}  // namespace

// Optional per-kernel timing: CUDA events recorded on the call's stream
// around each of the library's launches, resolved when read.
struct Profiler {
  bool on = false;
  struct Pending {
    std::string name;
    int launches;
    cudaEvent_t a, b;
  };
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> pool;
  std::map<std::string, std::pair<double, int>> acc;

  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  void resolve() {
    for (auto& p : pending) {
      float ms = 0.f;
      cudaEventSynchronize(p.b);
      cudaEventElapsedTime(&ms, p.a, p.b);
      auto& a = acc[p.name];
      a.first += ms;
      a.second += p.launches;
      pool.push_back(p.a);
      pool.push_back(p.b);
    }
    pending.clear();
  }
  ~Profiler() {
    for (auto& p : pending) {
      cudaEventDestroy(p.a);
      cudaEventDestroy(p.b);
    }
    for (auto e : pool) cudaEventDestroy(e);
  }
};

struct lc_context {
  int device = 0;
  int sm_count = 148;
  int32_t* d_status = nullptr;  // [kMaxHeads]
  int32_t* d_iters = nullptr;   // [kMaxHeads]
  uint32_t* d_err = nullptr;
  Profiler prof;
  // host entry point: copy stream, per-group step-1 streams and events of
  // the pipelined upload
  static constexpr int kGroups = 8;
  cudaStream_t copy_st = nullptr;
  cudaStream_t grp_st[kGroups] = {};
  cudaEvent_t ev_start = nullptr;
  cudaEvent_t ev_copy[kGroups] = {};
  cudaEvent_t ev_p1[kGroups] = {};
  // multi-layer entry point: the solve stream and its hand-off events
  cudaStream_t fit_st = nullptr;
  cudaEvent_t ev_mass[2] = {}, ev_fit[2] = {}, ev_begin = nullptr;
  // step 5: the auxiliary stream of the output-system factorisation
  cudaStream_t aux_st = nullptr;
  cudaEvent_t ev_h = nullptr, ev_f = nullptr;
};

namespace {

struct Ctx {
  lc_context* h;
  Plan p;
  uint8_t* ws;
  cudaStream_t st;
  template <class T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(ws + off);
  }
};

// Brackets one kernel launch with profiler events when profiling is on.
struct ProfScope {
  lc_context* h;
  cudaStream_t st;
  cudaEvent_t b = nullptr;
  ProfScope(lc_context* h_, cudaStream_t st_, const char* name, int launches)
      : h(h_), st(st_) {
    if (!h->prof.on) return;
    if (h->prof.pending.size() > 8192) h->prof.resolve();
    cudaEvent_t a = h->prof.get();
    b = h->prof.get();
    cudaEventRecord(a, st);
    h->prof.pending.push_back({name, launches, a, b});
  }
  ~ProfScope() {
    if (b) cudaEventRecord(b, st);
  }
};
// `n`: kernel launches inside the scope (0 for a memset).
#define LC_PROF(c, name, n) ProfScope prof_scope_##__LINE__((c).h, (c).st, name, n)

lc_status check_ws(const Plan& p, void* ws, size_t bytes) {
  if (!ws) return LC_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % 256) return LC_ERR_WORKSPACE;
  if (bytes < p.total) return LC_ERR_WORKSPACE;
  return LC_OK;
}

lc_status enter(lc_context* h) {
  if (!h) return LC_ERR_INVALID_ARG;
  if (!get_encode()) return LC_ERR_CUDA;
  LC_CUDA(cudaSetDevice(h->device));
  return LC_OK;
}

// Operand copies: fp16 V for bf16 inputs; split fp16 Q/K/V for fp32 inputs.
lc_status prepare_operands(const Ctx& c, const void* Q, const void* K, const void* V, bool need_v,
                           const void** qop, const void** kop) {
  const Plan& p = c.p;
  const size_t nv = static_cast<size_t>(p.H) * p.T * p.d;
  if (p.bf16_in) {
    *qop = Q;
    *kop = K;
    if (need_v) {
      LC_PROF(c, "convert_v", 1);
      LC_CUDA(launch_convert_bf16_to_f16(static_cast<const __nv_bfloat16*>(V), c.at<__half>(p.vhi),
                                         nv, c.st));
    }
  } else {
    LC_CUDA(launch_split_rows3(static_cast<const float*>(Q), c.at<__half>(p.qop),
                               static_cast<size_t>(p.H) * p.n_q, p.d, 0, c.st));
    LC_CUDA(launch_split_rows3(static_cast<const float*>(K), c.at<__half>(p.kop),
                               static_cast<size_t>(p.H) * p.T, p.d, 1, c.st));
    if (need_v)
      LC_CUDA(launch_split_f32(static_cast<const float*>(V), c.at<__half>(p.vhi), c.at<__half>(p.vlo),
                               nv, c.st));
    *qop = c.ws + p.qop;
    *kop = c.ws + p.kop;
  }
  return LC_OK;
}

// Step 1 for heads [h0, h0 + nh) (all heads by default).
lc_status run_pass1(const Ctx& c, const void* qop, const void* kop, float* rowmax, float* lse,
                    float* O, bool to_ws, int h0 = 0, int nh = -1) {
  const Plan& p = c.p;
  if (nh < 0) nh = p.H;
  const bool qk_bf16 = p.bf16_in;
  // below 2x compression the output fit amplifies P's rounding: split P.V
  const bool split_p = 2 * p.t > p.T;
  const int bn = (p.mode == kSplitF16d64) ? 64 : 128;
  // operands are 16-bit (bf16 inputs, or the split fp16 copies of fp32 ones)
  const size_t q_off = static_cast<size_t>(h0) * p.n_q * p.d_qk * 2;
  const size_t k_off = static_cast<size_t>(h0) * p.T * p.d_qk * 2;
  const size_t v_off = static_cast<size_t>(h0) * p.T * p.d * 2;
  CUtensorMap mQ, mK, mV, mVlo;
  if (!make_map(&mQ, static_cast<const uint8_t*>(qop) + q_off, qk_bf16, p.d_qk, p.n_q, nh, 128))
    return LC_ERR_CUDA;
  if (!make_map(&mK, static_cast<const uint8_t*>(kop) + k_off, qk_bf16, p.d_qk, p.T, nh, bn))
    return LC_ERR_CUDA;
  if (!make_map(&mV, c.ws + p.vhi + v_off, false, p.d, p.T, nh, bn)) return LC_ERR_CUDA;
  if (!make_map(&mVlo, (p.bf16_in ? c.ws + p.vhi : c.ws + p.vlo) + v_off, false, p.d, p.T, nh, bn))
    return LC_ERR_CUDA;
  const size_t rq = static_cast<size_t>(h0) * p.n_q, rqp = static_cast<size_t>(h0) * p.n_q_pad;
  AttnStatsParams a{};
  a.n_q = p.n_q;
  a.T = p.T;
  a.n_q_pad = p.n_q_pad;
  a.scale_log2 = p.scale * kLog2e;
  a.rowmax = rowmax ? rowmax + rq : nullptr;
  a.lse = lse ? lse + rq : nullptr;
  a.O = O ? O + rq * p.d : nullptr;
  if (to_ws) {
    a.rowmax_pad = c.at<float>(p.m_pad) + rqp;
    a.lse_pad = c.at<float>(p.lse_pad) + rqp;
    a.O_hi = c.at<__half>(p.ohi) + rq * p.d;
    a.O_lo = c.at<__half>(p.olo) + rq * p.d;
  }
  a.err = c.h->d_err;
  {
    LC_PROF(c, "attn_stats", 1);
    LC_CUDA(launch_attn_stats(p.mode, split_p, mQ, mK, mV, mVlo, a, nh, c.st));
  }
  return LC_OK;
}

lc_status run_pass2(const Ctx& c, const void* qop, const void* kop) {
  const Plan& p = c.p;
  CUtensorMap mQ, mK;
  if (!make_map(&mQ, qop, p.bf16_in, p.d_qk, p.n_q, p.H, 128)) return LC_ERR_CUDA;
  if (!make_map(&mK, kop, p.bf16_in, p.d_qk, p.T, p.H, 128)) return LC_ERR_CUDA;
  {
    LC_PROF(c, "clear_scores", 0);
    LC_CUDA(cudaMemsetAsync(c.ws + p.ucode, 0, static_cast<size_t>(p.H) * p.T * 4, c.st));
  }
  const int nqt = p.n_q_pad / 128;
  // bf16 inputs: 256 keys and one CTA per SM; fp32 inputs: 128 keys, two per SM
  const int kpc = p.bf16_in ? 256 : 128, occ = p.bf16_in ? 1 : 2;
  int split = best_split(((p.T + kpc - 1) / kpc) * p.H, c.h->sm_count, occ, p.ks_max);
  const int tiles = (nqt + split - 1) / split;
  split = (nqt + tiles - 1) / tiles;
  KeyScoreParams k{};
  k.n_q_pad = p.n_q_pad;
  k.T = p.T;
  k.tiles_per_split = tiles;
  k.scale = p.scale;
  k.lse_pad = c.at<float>(p.lse_pad);
  k.u_code = c.at<uint32_t>(p.ucode);
  k.err = c.h->d_err;
  {
    LC_PROF(c, "key_scores", 1);
    LC_CUDA(launch_key_scores(p.mode, mK, mQ, k, p.H, split, c.st));
  }
  return LC_OK;
}

// Step 2 as RMS attention (bf16 operands): merged base-2 column masses of
// the squared probabilities into L2, then order codes of u = log RMS in the
// workspace's ucode (and u as floats when given).
lc_status run_pass2_rms(const Ctx& c, const void* qop, const void* kop, float2* part, float* L2,
                        float* u) {
  const Plan& p = c.p;
  CUtensorMap mQ, mK;
  if (!make_map(&mQ, qop, true, p.d_qk, p.n_q, p.H, 128)) return LC_ERR_CUDA;
  if (!make_map(&mK, kop, true, p.d_qk, p.T, p.H, 128)) return LC_ERR_CUDA;
  const int nqt = p.n_q_pad / 128;
  int split = best_split(((p.T + 255) / 256) * p.H, c.h->sm_count, 1, p.ks_max);
  const int tiles = (nqt + split - 1) / split;
  split = (nqt + tiles - 1) / tiles;
  KeyScoreParams k{};
  k.n_q_pad = p.n_q_pad;
  k.T = p.T;
  k.tiles_per_split = tiles;
  k.scale = p.scale;
  k.lse_pad = c.at<float>(p.lse_pad);
  k.part = part;
  k.err = c.h->d_err;
  {
    LC_PROF(c, "key_scores_rms", 3);
    LC_CUDA(launch_key_scores_rms(p.mode, mK, mQ, k, p.H, split, c.st));
    LC_CUDA(launch_merge_key_lse(part, L2, split, p.H, p.T, c.st));
    LC_CUDA(launch_rms_finish(L2, p.n_q, c.at<uint32_t>(p.ucode), u,
                              static_cast<size_t>(p.H) * p.T, c.st));
  }
  return LC_OK;
}

// Steps 4-5 from the workspace's m_pad, lse_pad, O hi/lo and the given idx.
lc_status run_fit_solve(const Ctx& c, const void* qop, const void* V, const int32_t* idx,
                        float* w, float* beta, float* Cv, int bounded_iters, int status_off,
                        const CUtensorMap& mKc, const CUtensorMap& mQ64, const CUtensorMap& mOhi,
                        const CUtensorMap& mOlo, GramParams g, int g7_split, int g7_slabs,
                        int r_split, int r_slabs);

// bounded_iters > 0: step 4 as the bounded variant (w in [e^-3, e^3], that
// many iterations) instead of the NNLS.  The mass system is built on c's
// stream; from the solve on, the work goes to `cs` (the same context, or one
// on another stream that waits for `handoff`).  Per-head outcomes go to the
// report at head offset status_off.
lc_status run_fit(const Ctx& ca, const void* qop, const void* kop, const void* V,
                  const int32_t* idx, float* w, float* beta, float* Cv, int bounded_iters = 0,
                  const Ctx* cs = nullptr, cudaEvent_t handoff = nullptr, int status_off = 0) {
  const Ctx* cp = &ca;
  const Plan& p = ca.p;
  const size_t H = p.H;
  const int row_bytes = p.d_qk * 2;
  const Ctx& c = ca;
  {
    LC_PROF(c, "gather_keys", 1);
    LC_CUDA(launch_gather_rows(kop, c.ws + p.kc, idx, p.H, p.T, p.t, p.t_pad, row_bytes, c.st,
                               c.at<uint32_t>(p.khash)));
  }
  CUtensorMap mQ64, mKc, mOhi, mOlo;
  if (!make_map(&mQ64, qop, p.bf16_in, p.d_qk, p.n_q, p.H, 64)) return LC_ERR_CUDA;
  if (!make_map(&mKc, c.ws + p.kc, p.bf16_in, p.d_qk, p.t_pad, p.H, 128)) return LC_ERR_CUDA;
  if (!make_map(&mOhi, c.ws + p.ohi, false, p.d, p.n_q, p.H, 64)) return LC_ERR_CUDA;
  if (!make_map(&mOlo, c.ws + p.olo, false, p.d, p.n_q, p.H, 64)) return LC_ERR_CUDA;

  // ---- step 4: mass system and NNLS
  {
    LC_PROF(c, "mass_rows", 1);
    LC_CUDA(launch_mass_rows(c.at<float>(p.m_pad), c.at<float>(p.lse_pad), c.at<float>(p.rowsh2),
                             c.at<float>(p.rowb), p.H, p.n_q, p.n_q_pad, c.st,
                             c.at<float>(p.colb2), p.t, p.t_pad));
  }
  const int slabs = p.n_q_pad / 64;
  const int npairs = p.nblk * (p.nblk + 1) / 2;
  // the all-pairs kernels hold one accumulator per block: their chains are
  // bounded by the split alone
  const int min_split = p.all_pairs ? gram_min_split(slabs) : 1;
  auto split_of = [&](int units, int cap, int* per) {
    int sp = std::max(min_split, best_split(units, c.h->sm_count, 1, cap));
    *per = (slabs + sp - 1) / sp;
    return (slabs + *per - 1) / *per;
  };
  int g5_slabs = 0, g7_slabs = 0, r_slabs = 0;
  const int g5_split = split_of((p.all_pairs ? 1 : npairs) * p.H, p.g5_max, &g5_slabs);
  const int g7_split =
      split_of((p.all_pairs ? 1 : npairs + p.nblk) * p.H, p.g7_max, &g7_slabs);
  const int r_split = p.all_pairs ? split_of(p.H, p.r_max, &r_slabs) : g7_split;
  GramParams g{};
  g.n_q_pad = p.n_q_pad;
  g.n_q = p.n_q;
  g.t_pad = p.t_pad;
  g.nblk = p.nblk;
  g.slabs_per_split = g5_slabs;
  g.scale_log2 = p.scale * kLog2e;
  g.rowsh2 = c.at<float>(p.rowsh2);
  g.row_b = c.at<float>(p.rowb);
  g.colb2 = c.at<float>(p.colb2);
  g.Gpart = c.at<float>(p.gpart);
  g.cpart = c.at<float>(p.cpart);
  g.Rpart = nullptr;
  g.d_v = p.d;
  g.err = c.h->d_err;
  {
    LC_PROF(c, "gram_mass", 1);
    if (p.all_pairs)
      LC_CUDA(launch_gram_all_pairs(p.mode, mKc, mQ64, mOhi, mOlo, g, p.H, g5_split, c.st));
    else
      LC_CUDA(launch_gram(p.mode, false, mKc, mQ64, mOhi, mOlo, g, p.H, g5_split, c.st));
  }
  {
    LC_PROF(c, "reduce_mass", 1);
    LC_CUDA(launch_reduce_gram(c.at<float>(p.gpart), c.at<float>(p.G), g5_split, p.H, p.t_pad, c.st,
                               c.at<float>(p.cpart), c.at<float>(p.c)));
  }
  if (cs && cs->st != ca.st) {
    LC_CUDA(cudaEventRecord(handoff, ca.st));
    LC_CUDA(cudaStreamWaitEvent(cs->st, handoff, 0));
    cp = cs;
  }
  return run_fit_solve(*cp, qop, V, idx, w, beta, Cv, bounded_iters, status_off, mKc, mQ64, mOhi,
                       mOlo, g, g7_split, g7_slabs, r_split, r_slabs);
}

// Steps 4 (solve) and 5 of run_fit.
lc_status run_fit_solve(const Ctx& c, const void* qop, const void* V, const int32_t* idx,
                        float* w, float* beta, float* Cv, int bounded_iters, int status_off,
                        const CUtensorMap& mKc, const CUtensorMap& mQ64, const CUtensorMap& mOhi,
                        const CUtensorMap& mOlo, GramParams g, int g7_split, int g7_slabs,
                        int r_split, int r_slabs) {
  const Plan& p = c.p;
  const size_t H = p.H;
  SolveParams sp{};
  sp.H = p.H;
  sp.t = p.t;
  sp.t_pad = p.t_pad;
  sp.d_v = p.d;
  sp.max_iter = p.max_iter;
  sp.G = c.at<float>(p.G);
  sp.c = c.at<float>(p.c);
  sp.w = w;
  sp.beta = beta;
  sp.colb2 = c.at<float>(p.colb2);
  sp.mat = c.at<float>(p.mat);
  sp.vec = c.at<float>(p.vec);
  sp.wbuf = c.at<float>(p.wbuf);
  sp.head_status = c.h->d_status + status_off;
  sp.head_iters = c.h->d_iters + status_off;
  sp.err = c.h->d_err;
  sp.krows = c.ws + p.kc;
  sp.khash = c.at<uint32_t>(p.khash);
  sp.k_row_bytes = p.d_qk * 2;
  if (bounded_iters > 0) {
    LC_PROF(c, "bounded_ls", 1);
    sp.max_iter = bounded_iters;
    LC_CUDA(launch_bounded_ls(sp, std::exp(-3.f), std::exp(3.f), c.st));
  } else {
    LC_PROF(c, "nnls", 1);
    LC_CUDA(launch_nnls(sp, c.st));
  }

  // ---- step 5: compact log mass, output system, OLS
  CUtensorMap mQ128;
  if (!make_map(&mQ128, qop, p.bf16_in, p.d_qk, p.n_q, p.H, 128)) return LC_ERR_CUDA;
  CompactLseParams cl{};
  cl.n_q = p.n_q;
  cl.n_q_pad = p.n_q_pad;
  cl.t_pad = p.t_pad;
  cl.scale_log2 = p.scale * kLog2e;
  cl.colb2 = c.at<float>(p.colb2);
  cl.lc2_pad = c.at<float>(p.lc2);
  cl.err = c.h->d_err;
  {
    LC_PROF(c, "compact_lse", 1);
    if (p.bf16_in && p.nblk <= 2) {
      const int ntiles = p.n_q_pad / 128;
      const int sp = best_split(p.H, c.h->sm_count, 1, ntiles);
      LC_CUDA(launch_compact_lse_resident(p.mode, mQ128, mKc, cl, p.H, sp, c.st));
    } else {
      LC_CUDA(launch_compact_lse(p.mode, mQ128, mKc, cl, p.H, c.st));
    }
  }
  g.slabs_per_split = g7_slabs;
  g.rowsh2 = c.at<float>(p.lc2);
  g.row_b = nullptr;
  g.Gpart = c.at<float>(p.hpart);
  g.cpart = nullptr;
  g.Rpart = c.at<float>(p.rpart);
  OlsParams op{};
  op.H = p.H;
  op.t = p.t;
  op.t_pad = p.t_pad;
  op.d_v = p.d;
  op.Hm = c.at<float>(p.Hm);
  op.R = c.at<float>(p.R);
  op.Vc = c.at<float>(p.vc);
  op.w = w;
  op.mat = c.at<float>(p.mat);
  op.dinv = c.at<float>(p.vec);
  op.Cv = Cv;
  op.head_status = c.h->d_status + status_off;
  op.err = c.h->d_err;
  if (p.all_pairs) {
    // H first; its factorisation (a CTA per head) runs on the auxiliary
    // stream while R is formed on the SMs left free
    {
      LC_PROF(c, "gram_out", 1);
      LC_CUDA(launch_gram_all_pairs(p.mode, mKc, mQ64, mOhi, mOlo, g, p.H, g7_split, c.st));
    }
    {
      LC_PROF(c, "reduce_out", 1);
      LC_CUDA(launch_reduce_gram(c.at<float>(p.hpart), c.at<float>(p.Hm), g7_split, p.H, p.t_pad,
                                 c.st));
    }
    lc_context* hc = c.h;
    if (!hc->aux_st) LC_CUDA(cudaStreamCreateWithFlags(&hc->aux_st, cudaStreamNonBlocking));
    if (!hc->ev_h) LC_CUDA(cudaEventCreateWithFlags(&hc->ev_h, cudaEventDisableTiming));
    if (!hc->ev_f) LC_CUDA(cudaEventCreateWithFlags(&hc->ev_f, cudaEventDisableTiming));
    LC_CUDA(cudaEventRecord(hc->ev_h, c.st));
    LC_CUDA(cudaStreamWaitEvent(hc->aux_st, hc->ev_h, 0));
    {
      Ctx ca{c.h, c.p, c.ws, hc->aux_st};
      LC_PROF(ca, "ols_factor", 1);
      LC_CUDA(launch_ols_factor(op, hc->aux_st));
    }
    LC_CUDA(cudaEventRecord(hc->ev_f, hc->aux_st));
    const int free_sms = std::max(1, c.h->sm_count - p.H);
    int rs = std::max(gram_min_split(p.n_q_pad / 64), best_split(p.H, free_sms, 1, p.r_max));
    const int r_per = (p.n_q_pad / 64 + rs - 1) / rs;
    rs = (p.n_q_pad / 64 + r_per - 1) / r_per;
    GramParams gr = g;
    gr.r_only = 1;
    gr.slabs_per_split = r_per;
    {
      LC_PROF(c, "gram_r", 1);
      LC_CUDA(launch_gram_r(p.mode, mKc, mQ64, mOhi, mOlo, gr, p.H, rs, c.st));
    }
    {
      LC_PROF(c, "reduce_out", 2);
      LC_CUDA(launch_reduce_partials(c.at<float>(p.rpart), c.at<float>(p.R), rs,
                                     H * p.t_pad * p.d, c.st));
      LC_CUDA(launch_gather_v(V, p.bf16_in ? 0 : 1, idx, c.at<float>(p.vc), p.H, p.T, p.t,
                              p.t_pad, p.d, c.st));
    }
    LC_CUDA(cudaStreamWaitEvent(c.st, hc->ev_f, 0));
    {
      LC_PROF(c, "ols", 1);
      LC_CUDA(launch_ols_solve(op, c.st));
    }
    return LC_OK;
  }
  {
    LC_PROF(c, "gram_out", 1);
    LC_CUDA(launch_gram(p.mode, true, mKc, mQ64, mOhi, mOlo, g, p.H, g7_split, c.st));
  }
  {
    LC_PROF(c, "reduce_out", 3);
    LC_CUDA(launch_reduce_gram(c.at<float>(p.hpart), c.at<float>(p.Hm), g7_split, p.H, p.t_pad, c.st));
    LC_CUDA(launch_reduce_partials(c.at<float>(p.rpart), c.at<float>(p.R), r_split,
                                   H * p.t_pad * p.d, c.st));
    LC_CUDA(launch_gather_v(V, p.bf16_in ? 0 : 1, idx, c.at<float>(p.vc), p.H, p.T, p.t, p.t_pad,
                            p.d, c.st));
  }
  {
    LC_PROF(c, "ols", 2);
    LC_CUDA(launch_ols(op, c.st));
  }
  return LC_OK;
}

// Step 3 in the pipeline, from the order codes of the key scores: the wide
// path for long heads, else one CTA per head.
cudaError_t select_step(const Ctx& c, int32_t* idx, cudaStream_t st) {
  const Plan& p = c.p;
  if (!p.selw_on) return launch_select_topt(c.at<uint32_t>(p.ucode), p.H, p.T, p.t, idx, st);
  for (int stage = 0; stage < 3; ++stage) {
    const cudaError_t e = launch_select_wide_codes(c.at<uint32_t>(p.ucode), p.H, p.T, p.t, idx,
                                                   c.ws + p.selw, c.h->sm_count, c.h->d_err,
                                                   stage, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

lc_status reset_report(const Ctx& c) {
  LC_CUDA(cudaMemsetAsync(c.h->d_status, 0, sizeof(int32_t) * c.p.H, c.st));
  LC_CUDA(cudaMemsetAsync(c.h->d_iters, 0, sizeof(int32_t) * c.p.H, c.st));
  LC_CUDA(cudaMemsetAsync(c.h->d_err, 0, sizeof(uint32_t), c.st));
  return LC_OK;
}

#define LC_TRY(x)                \
  do {                           \
    lc_status s_ = (x);          \
    if (s_ != LC_OK) return s_;  \
  } while (0)

// ---------------------------------------------------------------- fast path
// Two-pass selection, uniform redistribution of the missing mass, direct
// values ("KV compaction" blog, "Attempt #3: Two-Pass", "Choosing beta",
// "Choosing C_v").  bf16 operands only.
struct FastPlan {
  OperandMode mode;
  int H, n_q, T, d, t, n_sub, kt;
  int n_sub_pad, T_pad, kt_pad, n_q_pad, t_pad;
  float scale;
  int mass_units, mass_max;  // pass 2 scores: CTAs per query split, largest split
  int sub_kb, sub_splits;    // pass 1 lse: key blocks per split, splits
  int sl_chunk, sl_chunks;   // pass 2 lse: keys per resident chunk, chunks
  // workspace offsets (bytes)
  size_t qs, colb_all, lc2_sub, lse_sub;  // pass 1 over the query subset
  size_t ucode, shrt, kp, colb_short;     // scores, shortlist, its keys
  size_t lc2_q, lse_q, pos;               // pass 2 over all queries
  size_t part, L2, chosen;                // column masses of the shortlist keys
  size_t part1, part3;                    // split partials of the two lse passes
  size_t total;
};

lc_status fast_plan(const lc_shape* s, int n_sub, int k, FastPlan* out) {
  LC_TRY(validate(s));
  if (s->in_dtype != LC_BF16) return LC_ERR_UNSUPPORTED;
  if (n_sub < 1 || n_sub > s->n_q || k < 1) return LC_ERR_INVALID_ARG;
  FastPlan p{};
  p.mode = s->d == 128 ? kBF16d128 : kBF16d64;
  p.H = s->n_kv_heads;
  p.n_q = s->n_q;
  p.T = s->T;
  p.d = s->d;
  p.t = s->t;
  p.n_sub = n_sub;
  p.kt = static_cast<int>(std::min<long long>(static_cast<long long>(k) * s->t, s->T));
  p.n_sub_pad = static_cast<int>(round_up(n_sub, 128));
  p.T_pad = static_cast<int>(round_up(s->T, 128));
  p.kt_pad = static_cast<int>(round_up(p.kt, 128));
  p.n_q_pad = static_cast<int>(round_up(s->n_q, 128));
  p.t_pad = static_cast<int>(round_up(s->t, 128));
  p.scale = s->scale > 0.f ? s->scale : 1.f / std::sqrt(static_cast<float>(s->d));
  p.mass_units = ((p.kt + 255) / 256) * p.H;
  p.mass_max = max_split(p.mass_units, 2, p.n_q_pad / 128);
  {
    // the subset's lse over all T keys: split the keys so that about two
    // waves of CTAs run (the subset alone gives only n_sub/128 per head)
    const int nkb = p.T_pad / 128, units = (p.n_sub_pad / 128) * p.H;
    int ns = std::max(1, std::min(std::min(nkb, 64), (2 * 152 + units - 1) / units));
    p.sub_kb = (nkb + ns - 1) / ns;
    p.sub_splits = (nkb + p.sub_kb - 1) / p.sub_kb;
    p.sl_chunk = p.kt_pad <= 256 ? p.kt_pad : (p.kt_pad % 256 == 0 ? 256 : 128);
    p.sl_chunks = p.kt_pad / p.sl_chunk;
  }

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  };
  const size_t H = p.H;
  p.qs = take(H * p.n_sub_pad * p.d * 2);
  p.colb_all = take(H * p.T_pad * 4);
  p.lc2_sub = take(H * p.n_sub_pad * 4);
  p.lse_sub = take(H * p.n_sub_pad * 4);
  p.ucode = take(H * p.T * 4);
  p.shrt = take(H * p.kt * 4);
  p.kp = take(H * p.kt_pad * p.d * 2);
  p.colb_short = take(H * p.kt_pad * 4);
  p.part1 = take(static_cast<size_t>(p.sub_splits) * H * p.n_sub_pad * 8);
  p.part3 = p.sl_chunks > 1 ? take(static_cast<size_t>(p.sl_chunks) * H * p.n_q_pad * 8) : 0;
  p.lc2_q = take(H * p.n_q_pad * 4);
  p.lse_q = take(H * p.n_q_pad * 4);
  p.pos = take(H * p.t * 4);
  p.part = take(static_cast<size_t>(p.mass_max) * H * p.kt * 8);
  p.L2 = take(H * p.kt * 4);
  p.chosen = take(H * p.kt);
  p.total = off;
  *out = p;
  return LC_OK;
}

// Query split of a key-column pass over `units` CTAs and `tiles` query tiles.
int column_split(const lc_context* h, int units, int occ, int tiles, int cap, int* per) {
  int split = best_split(units, h->sm_count, occ, std::min(cap, tiles));
  *per = (tiles + split - 1) / split;
  return (tiles + *per - 1) / *per;
}

struct FastCtx {
  lc_context* h;
  cudaStream_t st;
};

lc_status run_fast(const FastCtx& c, const FastPlan& p, uint8_t* ws, const void* Q, const void* K,
                   const void* V, const int32_t* qsel, int32_t* idx, float* beta, float* Cv,
                   int32_t* short_out) {
  auto F = [&](size_t o) { return reinterpret_cast<float*>(ws + o); };
  auto I = [&](size_t o) { return reinterpret_cast<int32_t*>(ws + o); };
  auto U = [&](size_t o) { return reinterpret_cast<uint32_t*>(ws + o); };
  const size_t H = p.H;
  const int row_bytes = p.d * 2;
  const float s2 = p.scale * kLog2e;
  LC_CUDA(cudaMemsetAsync(c.h->d_status, 0, sizeof(int32_t) * p.H, c.st));
  LC_CUDA(cudaMemsetAsync(c.h->d_iters, 0, sizeof(int32_t) * p.H, c.st));
  LC_CUDA(cudaMemsetAsync(c.h->d_err, 0, sizeof(uint32_t), c.st));

  CUtensorMap mQ, mK, mQs, mKp;
  if (!make_map(&mQ, Q, true, p.d, p.n_q, p.H, 128)) return LC_ERR_CUDA;
  if (!make_map(&mK, K, true, p.d, p.T, p.H, 128)) return LC_ERR_CUDA;
  if (!make_map(&mQs, ws + p.qs, true, p.d, p.n_sub_pad, p.H, 128)) return LC_ERR_CUDA;
  if (!make_map(&mKp, ws + p.kp, true, p.d, p.kt_pad, p.H, 128)) return LC_ERR_CUDA;

  // ---- pass 1: the query subset Q' scores every key under full attention
  {
    LC_PROF(c, "fast_prepare", 3);
    LC_CUDA(launch_gather_rows(Q, ws + p.qs, qsel, p.H, p.n_q, p.n_sub, p.n_sub_pad, row_bytes,
                               c.st));
    LC_CUDA(launch_fill_colb2(F(p.colb_all), p.H, p.T, p.T_pad, c.st));
    LC_CUDA(launch_fill_colb2(F(p.colb_short), p.H, p.kt, p.kt_pad, c.st));
  }
  CompactLseParams cl{};
  cl.n_q = p.n_sub;
  cl.n_q_pad = p.n_sub_pad;
  cl.t_pad = p.sub_kb * 128;
  cl.key_stride = p.T_pad;
  cl.part = reinterpret_cast<float2*>(ws + p.part1);
  cl.scale_log2 = s2;
  cl.colb2 = F(p.colb_all);
  cl.lc2_pad = nullptr;
  cl.err = c.h->d_err;
  {
    LC_PROF(c, "subset_lse", 3);
    LC_CUDA(launch_compact_lse(p.mode, mQs, mK, cl, p.H, c.st));
    LC_CUDA(launch_merge_row_lse(cl.part, F(p.lc2_sub), p.sub_splits, p.H, p.n_sub, p.n_sub_pad,
                                 c.st));
    LC_CUDA(launch_scale_f32(F(p.lc2_sub), F(p.lse_sub), H * p.n_sub_pad, kLn2, c.st));
  }
  KeyScoreParams ks{};
  ks.scale = p.scale;
  ks.err = c.h->d_err;
  {
    LC_PROF(c, "subset_scores", 1);
    LC_CUDA(cudaMemsetAsync(ws + p.ucode, 0, H * p.T * 4, c.st));
    const int units = ((p.T + 255) / 256) * p.H, tiles = p.n_sub_pad / 128;
    ks.n_q_pad = p.n_sub_pad;
    ks.T = p.T;
    const int split = column_split(c.h, units, 1, tiles, max_split(units, 2, tiles),
                                   &ks.tiles_per_split);
    ks.lse_pad = F(p.lse_sub);
    ks.u_code = U(p.ucode);
    LC_CUDA(launch_key_scores(p.mode, mK, mQs, ks, p.H, split, c.st));
  }
  {
    LC_PROF(c, "shortlist", 2);
    LC_CUDA(launch_select_topt(U(p.ucode), p.H, p.T, p.kt, I(p.shrt), c.st));
    LC_CUDA(launch_gather_rows(K, ws + p.kp, I(p.shrt), p.H, p.T, p.kt, p.kt_pad, row_bytes,
                               c.st));
  }

  // ---- pass 2: every query scores the shortlist, normalised over it
  // every query's lse over the shortlist: resident key chunks of at most
  // 256, one partial per chunk when there are several
  cl.n_q = p.n_q;
  cl.n_q_pad = p.n_q_pad;
  cl.t_pad = p.sl_chunk;
  cl.key_stride = p.kt_pad;
  cl.part = p.sl_chunks > 1 ? reinterpret_cast<float2*>(ws + p.part3) : nullptr;
  cl.colb2 = F(p.colb_short);
  cl.lc2_pad = F(p.lc2_q);
  {
    LC_PROF(c, "shortlist_lse", 3);
    const int sp = best_split(p.H * p.sl_chunks, c.h->sm_count, 1, p.n_q_pad / 128);
    LC_CUDA(launch_compact_lse_resident(p.mode, mQ, mKp, cl, p.H, sp, c.st));
    if (cl.part)
      LC_CUDA(launch_merge_row_lse(cl.part, F(p.lc2_q), p.sl_chunks, p.H, p.n_q, p.n_q_pad,
                                   c.st));
    LC_CUDA(launch_scale_f32(F(p.lc2_q), F(p.lse_q), H * p.n_q_pad, kLn2, c.st));
  }
  {
    // scores and column masses of the shortlist in one pass
    LC_PROF(c, "shortlist_scores", 2);
    LC_CUDA(cudaMemsetAsync(ws + p.ucode, 0, H * p.kt * 4, c.st));
    const int tiles = p.n_q_pad / 128;
    ks.n_q_pad = p.n_q_pad;
    ks.T = p.kt;
    ks.n_rows = p.n_q;
    const int split = column_split(c.h, p.mass_units, 1, tiles, p.mass_max, &ks.tiles_per_split);
    ks.lse_pad = F(p.lse_q);
    ks.part = reinterpret_cast<float2*>(ws + p.part);
    LC_CUDA(launch_key_scores_mass(p.mode, mKp, mQ, ks, p.H, split, c.st));
    LC_CUDA(launch_merge_key_lse(ks.part, F(p.L2), split, p.H, p.kt, c.st));
  }
  {
    LC_PROF(c, "select_compose", 3);
    LC_CUDA(cudaMemsetAsync(ws + p.chosen, 0, H * p.kt, c.st));
    LC_CUDA(launch_select_topt(U(p.ucode), p.H, p.kt, p.t, I(p.pos), c.st));
    LC_CUDA(launch_compose_idx(I(p.shrt), I(p.pos), idx, ws + p.chosen, p.H, p.kt, p.t, c.st));
  }
  {
    // beta from the column masses: missing mass = the shortlist keys not chosen
    LC_PROF(c, "redistribute_values", 2);
    LC_CUDA(launch_redistribute_beta(F(p.L2), ws + p.chosen, I(p.pos), beta, p.H, p.kt, p.t,
                                     c.st));
    LC_CUDA(launch_gather_v(V, 0, idx, Cv, p.H, p.T, p.t, p.t, p.d, c.st));
  }
  if (short_out)
    LC_CUDA(cudaMemcpyAsync(short_out, ws + p.shrt, H * p.kt * 4, cudaMemcpyDeviceToDevice,
                            c.st));
  return LC_OK;
}

}  // namespace

extern "C" {

lc_status lc_create(lc_handle* out, int device) {
  if (!out) return LC_ERR_INVALID_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) return LC_ERR_INVALID_ARG;
  if (!get_encode()) return LC_ERR_CUDA;
  lc_context* h = new lc_context();
  h->device = device;
  cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device);
  if (h->sm_count < 1) h->sm_count = 148;
  if (cudaSetDevice(device) != cudaSuccess ||
      cudaMalloc(&h->d_status, sizeof(int32_t) * kMaxHeads) != cudaSuccess ||
      cudaMalloc(&h->d_iters, sizeof(int32_t) * kMaxHeads) != cudaSuccess ||
      cudaMalloc(&h->d_err, sizeof(uint32_t)) != cudaSuccess) {
    cudaFree(h->d_status);
    cudaFree(h->d_iters);
    cudaFree(h->d_err);
    delete h;
    return LC_ERR_CUDA;
  }
  cudaMemset(h->d_status, 0, sizeof(int32_t) * kMaxHeads);
  cudaMemset(h->d_iters, 0, sizeof(int32_t) * kMaxHeads);
  cudaMemset(h->d_err, 0, sizeof(uint32_t));
  *out = h;
  return LC_OK;
}

lc_status lc_destroy(lc_handle h) {
  if (!h) return LC_ERR_INVALID_ARG;
  cudaSetDevice(h->device);
  cudaFree(h->d_status);
  cudaFree(h->d_iters);
  cudaFree(h->d_err);
  for (int g = 0; g < lc_context::kGroups; ++g) {
    if (h->ev_copy[g]) cudaEventDestroy(h->ev_copy[g]);
    if (h->ev_p1[g]) cudaEventDestroy(h->ev_p1[g]);
    if (h->grp_st[g]) cudaStreamDestroy(h->grp_st[g]);
  }
  if (h->ev_start) cudaEventDestroy(h->ev_start);
  if (h->copy_st) cudaStreamDestroy(h->copy_st);
  for (int b = 0; b < 2; ++b) {
    if (h->ev_mass[b]) cudaEventDestroy(h->ev_mass[b]);
    if (h->ev_fit[b]) cudaEventDestroy(h->ev_fit[b]);
  }
  if (h->ev_begin) cudaEventDestroy(h->ev_begin);
  if (h->fit_st) cudaStreamDestroy(h->fit_st);
  if (h->ev_h) cudaEventDestroy(h->ev_h);
  if (h->ev_f) cudaEventDestroy(h->ev_f);
  if (h->aux_st) cudaStreamDestroy(h->aux_st);
  delete h;
  return LC_OK;
}

lc_status lc_workspace_bytes(const lc_shape* shape, size_t* bytes) {
  LC_TRY(validate(shape));
  if (!bytes) return LC_ERR_INVALID_ARG;
  *bytes = make_plan(shape).total;
  return LC_OK;
}

lc_status lc_full_attn_stats(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                             const void* V, float* rowmax, float* lse, float* O, void* workspace,
                             size_t workspace_bytes, void* stream) {
  LC_TRY(validate(shape));
  if (!Q || !K || !V) return LC_ERR_INVALID_ARG;
  const Plan p = make_plan(shape);
  LC_TRY(check_ws(p, workspace, workspace_bytes));
  LC_TRY(enter(h));
  Ctx c{h, p, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream)};
  const void *qop, *kop;
  LC_TRY(prepare_operands(c, Q, K, V, true, &qop, &kop));
  return run_pass1(c, qop, kop, rowmax, lse, O, false);
}

lc_status lc_key_scores(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                        const float* lse, float* u, void* workspace, size_t workspace_bytes,
                        void* stream) {
  LC_TRY(validate(shape));
  if (!Q || !K || !lse || !u) return LC_ERR_INVALID_ARG;
  const Plan p = make_plan(shape);
  LC_TRY(check_ws(p, workspace, workspace_bytes));
  LC_TRY(enter(h));
  Ctx c{h, p, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream)};
  const void *qop, *kop;
  LC_TRY(prepare_operands(c, Q, K, nullptr, false, &qop, &kop));
  LC_CUDA(launch_pad_rows(lse, c.at<float>(p.lse_pad), p.H, p.n_q, p.n_q_pad, kInf, c.st));
  LC_TRY(run_pass2(c, qop, kop));
  LC_CUDA(launch_decode_scores(c.at<uint32_t>(p.ucode), u, static_cast<size_t>(p.H) * p.T, c.st));
  return LC_OK;
}

lc_status lc_select_topt(lc_handle h, int n_heads, int T, int t, const float* u, int32_t* idx,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (n_heads < 1 || T < 1 || t < 1 || t > T || !u || !idx) return LC_ERR_INVALID_ARG;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256) return LC_ERR_WORKSPACE;
  const size_t need = static_cast<size_t>(n_heads) * T * 4;
  if (workspace_bytes < need) return LC_ERR_WORKSPACE;
  LC_TRY(enter(h));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* code = static_cast<uint32_t*>(workspace);
  if (select_wide_applies(T, t) && (reinterpret_cast<uintptr_t>(u) & 15) == 0 &&
      workspace_bytes >= select_wide_bytes(n_heads)) {
    static const char* const kStage[3] = {"select_sample", "select_filter", "select_final"};
    for (int stage = 0; stage < 3; ++stage) {
      ProfScope prof(h, st, kStage[stage], 1);
      LC_CUDA(launch_select_wide_scores(u, n_heads, T, t, idx, workspace, h->sm_count, h->d_err,
                                        stage, st));
    }
    return LC_OK;
  }
  LC_CUDA(launch_encode_scores(u, code, static_cast<size_t>(n_heads) * T, st));
  LC_CUDA(launch_select_topt(code, n_heads, T, t, idx, st));
  return LC_OK;
}

lc_status lc_fit_only(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                      const void* V, const int32_t* idx, const float* rowmax, const float* lse,
                      const float* O, float* w, float* beta, float* Cv, void* workspace,
                      size_t workspace_bytes, void* stream) {
  LC_TRY(validate(shape));
  if (!Q || !K || !V || !idx || !rowmax || !lse || !O || !w || !beta || !Cv)
    return LC_ERR_INVALID_ARG;
  const Plan p = make_plan(shape);
  LC_TRY(check_ws(p, workspace, workspace_bytes));
  LC_TRY(enter(h));
  Ctx c{h, p, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream)};
  LC_TRY(reset_report(c));
  const void *qop, *kop;
  LC_TRY(prepare_operands(c, Q, K, V, false, &qop, &kop));
  LC_CUDA(launch_pad_rows(rowmax, c.at<float>(p.m_pad), p.H, p.n_q, p.n_q_pad, kInf, c.st));
  LC_CUDA(launch_pad_rows(lse, c.at<float>(p.lse_pad), p.H, p.n_q, p.n_q_pad, kInf, c.st));
  LC_CUDA(launch_split_f32(O, c.at<__half>(p.ohi), c.at<__half>(p.olo),
                           static_cast<size_t>(p.H) * p.n_q * p.d, c.st));
  return run_fit(c, qop, kop, V, idx, w, beta, Cv);
}

lc_status lc_compact_layer(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                           const void* V, int32_t* idx, float* w, float* beta, float* Cv,
                           void* workspace, size_t workspace_bytes, void* stream) {
  LC_TRY(validate(shape));
  if (!Q || !K || !V || !idx || !w || !beta || !Cv) return LC_ERR_INVALID_ARG;
  const Plan p = make_plan(shape);
  LC_TRY(check_ws(p, workspace, workspace_bytes));
  LC_TRY(enter(h));
  Ctx c{h, p, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream)};
  LC_TRY(reset_report(c));
  const void *qop, *kop;
  LC_TRY(prepare_operands(c, Q, K, V, true, &qop, &kop));
  LC_TRY(run_pass1(c, qop, kop, nullptr, nullptr, nullptr, true));
  LC_TRY(run_pass2(c, qop, kop));
  {
    LC_PROF(c, "select_topt", c.p.selw_on ? 3 : 1);
    LC_CUDA(select_step(c, idx, c.st));
  }
  return run_fit(c, qop, kop, V, idx, w, beta, Cv);
}

lc_status lc_host_workspace_bytes(const lc_shape* shape, size_t* bytes) {
  LC_TRY(validate(shape));
  if (!bytes) return LC_ERR_INVALID_ARG;
  const Plan p = make_plan(shape);
  const size_t el = shape->in_dtype == LC_BF16 ? 2 : 4;
  const size_t H = p.H;
  size_t extra = round_up(H * p.n_q * p.d * el, 256) + 2 * round_up(H * p.T * p.d * el, 256) +
                 3 * round_up(H * p.t * 4, 256) + round_up(H * p.t * p.d * 4, 256);
  *bytes = p.total + extra;
  return LC_OK;
}

lc_status lc_compact_layer_host(lc_handle h, const lc_shape* shape, const void* Q_host,
                                const void* K_host, const void* V_host, int32_t* idx_host,
                                float* w_host, float* beta_host, float* Cv_host, void* workspace,
                                size_t workspace_bytes, void* stream) {
  LC_TRY(validate(shape));
  if (!Q_host || !K_host || !V_host || !idx_host || !w_host || !beta_host || !Cv_host)
    return LC_ERR_INVALID_ARG;
  size_t need = 0;
  LC_TRY(lc_host_workspace_bytes(shape, &need));
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 || workspace_bytes < need)
    return LC_ERR_WORKSPACE;
  LC_TRY(enter(h));
  const Plan p = make_plan(shape);
  const size_t el = shape->in_dtype == LC_BF16 ? 2 : 4;
  const size_t H = p.H;
  uint8_t* base = static_cast<uint8_t*>(workspace) + p.total;
  const size_t qb = H * p.n_q * p.d * el, kb = H * p.T * p.d * el;
  uint8_t* dQ = base;
  uint8_t* dK = dQ + round_up(qb, 256);
  uint8_t* dV = dK + round_up(kb, 256);
  uint8_t* dIdx = dV + round_up(kb, 256);
  uint8_t* dW = dIdx + round_up(H * p.t * 4, 256);
  uint8_t* dB = dW + round_up(H * p.t * 4, 256);
  uint8_t* dC = dB + round_up(H * p.t * 4, 256);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!p.bf16_in || H < 2) {
    LC_CUDA(cudaMemcpyAsync(dQ, Q_host, qb, cudaMemcpyHostToDevice, st));
    LC_CUDA(cudaMemcpyAsync(dK, K_host, kb, cudaMemcpyHostToDevice, st));
    LC_CUDA(cudaMemcpyAsync(dV, V_host, kb, cudaMemcpyHostToDevice, st));
    LC_TRY(lc_compact_layer(h, shape, dQ, dK, dV, reinterpret_cast<int32_t*>(dIdx),
                            reinterpret_cast<float*>(dW), reinterpret_cast<float*>(dB),
                            reinterpret_cast<float*>(dC), workspace, p.total, stream));
  } else {
    // Pipelined upload: the heads go up in groups (one head per group for up
    // to eight heads) on a copy stream; each group's step 1 runs on its own
    // stream as soon as its copy lands, so all but the first group's upload
    // hides under step-1 work, and the groups' CTAs fill the GPU together.
    constexpr int kG = lc_context::kGroups;
    if (!h->copy_st) LC_CUDA(cudaStreamCreateWithFlags(&h->copy_st, cudaStreamNonBlocking));
    if (!h->ev_start) LC_CUDA(cudaEventCreateWithFlags(&h->ev_start, cudaEventDisableTiming));
    for (int g = 0; g < kG; ++g) {
      if (!h->grp_st[g]) LC_CUDA(cudaStreamCreateWithFlags(&h->grp_st[g], cudaStreamNonBlocking));
      if (!h->ev_copy[g]) LC_CUDA(cudaEventCreateWithFlags(&h->ev_copy[g], cudaEventDisableTiming));
      if (!h->ev_p1[g]) LC_CUDA(cudaEventCreateWithFlags(&h->ev_p1[g], cudaEventDisableTiming));
    }
    const int ng = static_cast<int>(std::min<size_t>(H, kG));
    const int per = static_cast<int>((H + ng - 1) / ng);
    Ctx c{h, p, static_cast<uint8_t*>(workspace), st};
    LC_TRY(reset_report(c));
    // everything below is ordered after earlier work on the caller's stream
    // (which may still read the staging buffers) and after the report reset
    LC_CUDA(cudaEventRecord(h->ev_start, st));
    LC_CUDA(cudaStreamWaitEvent(h->copy_st, h->ev_start, 0));
    const size_t qh = static_cast<size_t>(p.n_q) * p.d * el, kh = static_cast<size_t>(p.T) * p.d * el;
    for (int g = 0; g < ng; ++g) {
      const int h0 = g * per, nh = std::min(per, static_cast<int>(H) - h0);
      if (nh <= 0) break;
      const size_t o = static_cast<size_t>(h0), n = static_cast<size_t>(nh);
      LC_CUDA(cudaMemcpyAsync(dK + o * kh, static_cast<const uint8_t*>(K_host) + o * kh, n * kh,
                              cudaMemcpyHostToDevice, h->copy_st));
      LC_CUDA(cudaMemcpyAsync(dV + o * kh, static_cast<const uint8_t*>(V_host) + o * kh, n * kh,
                              cudaMemcpyHostToDevice, h->copy_st));
      LC_CUDA(cudaMemcpyAsync(dQ + o * qh, static_cast<const uint8_t*>(Q_host) + o * qh, n * qh,
                              cudaMemcpyHostToDevice, h->copy_st));
      LC_CUDA(cudaEventRecord(h->ev_copy[g], h->copy_st));
      Ctx cg{h, p, static_cast<uint8_t*>(workspace), h->grp_st[g]};
      LC_CUDA(cudaStreamWaitEvent(cg.st, h->ev_copy[g], 0));
      const size_t nv = n * p.T * p.d, ov = o * p.T * p.d;
      {
        LC_PROF(cg, "convert_v", 1);
        LC_CUDA(launch_convert_bf16_to_f16(reinterpret_cast<const __nv_bfloat16*>(dV) + ov,
                                           cg.at<__half>(p.vhi) + ov, nv, cg.st));
      }
      LC_TRY(run_pass1(cg, dQ, dK, nullptr, nullptr, nullptr, true, h0, nh));
      LC_CUDA(cudaEventRecord(h->ev_p1[g], cg.st));
      LC_CUDA(cudaStreamWaitEvent(st, h->ev_p1[g], 0));
    }
    int32_t* idx = reinterpret_cast<int32_t*>(dIdx);
    LC_TRY(run_pass2(c, dQ, dK));
    {
      LC_PROF(c, "select_topt", c.p.selw_on ? 3 : 1);
      LC_CUDA(select_step(c, idx, st));
    }
    LC_TRY(run_fit(c, dQ, dK, dV, idx, reinterpret_cast<float*>(dW), reinterpret_cast<float*>(dB),
                   reinterpret_cast<float*>(dC)));
  }
  LC_CUDA(cudaMemcpyAsync(idx_host, dIdx, H * p.t * 4, cudaMemcpyDeviceToHost, st));
  LC_CUDA(cudaMemcpyAsync(w_host, dW, H * p.t * 4, cudaMemcpyDeviceToHost, st));
  LC_CUDA(cudaMemcpyAsync(beta_host, dB, H * p.t * 4, cudaMemcpyDeviceToHost, st));
  LC_CUDA(cudaMemcpyAsync(Cv_host, dC, H * p.t * p.d * 4, cudaMemcpyDeviceToHost, st));
  LC_CUDA(cudaStreamSynchronize(st));
  return LC_OK;
}

lc_status lc_fast_workspace_bytes(const lc_shape* shape, int n_sub, int k, size_t* bytes) {
  FastPlan p;
  LC_TRY(fast_plan(shape, n_sub, k, &p));
  if (!bytes) return LC_ERR_INVALID_ARG;
  *bytes = p.total;
  return LC_OK;
}

lc_status lc_compact_layer_fast(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                                const void* V, const int32_t* qsel, int n_sub, int k,
                                int32_t* idx, float* beta, float* Cv, int32_t* short_out,
                                void* workspace, size_t workspace_bytes, void* stream) {
  FastPlan p;
  LC_TRY(fast_plan(shape, n_sub, k, &p));
  if (!Q || !K || !V || !qsel || !idx || !beta || !Cv) return LC_ERR_INVALID_ARG;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 || workspace_bytes < p.total)
    return LC_ERR_WORKSPACE;
  LC_TRY(enter(h));
  FastCtx c{h, static_cast<cudaStream_t>(stream)};
  return run_fast(c, p, static_cast<uint8_t*>(workspace), Q, K, V, qsel, idx, beta, Cv,
                  short_out);
}

lc_status lc_compact_attention(lc_handle h, int n_heads, int n, int t, int n_new, int d,
                               float scale, const void* q, const void* Ck, const float* beta,
                               const float* Cv, const void* Knew, const void* Vnew,
                               const int32_t* n_vis, float* A, float* log_z, void* stream) {
  if (n_heads < 1 || n_heads > kMaxHeads || n < 1 || t < 0 || n_new < 0) return LC_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return LC_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return LC_ERR_INVALID_ARG;
  if (!q || !A || (t > 0 && (!Ck || !beta || !Cv)) || (n_new > 0 && (!Knew || !Vnew)))
    return LC_ERR_INVALID_ARG;
  LC_TRY(enter(h));
  CompactAttnParams p{};
  p.n = n;
  p.t = t;
  p.n_new = n_new;
  p.scale = scale > 0.f ? scale : 1.f / std::sqrt(static_cast<float>(d));
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.Ck = static_cast<const __nv_bfloat16*>(Ck);
  p.beta = beta;
  p.Cv = Cv;
  p.Knew = static_cast<const __nv_bfloat16*>(Knew);
  p.Vnew = static_cast<const __nv_bfloat16*>(Vnew);
  p.n_vis = n_vis;
  p.A = A;
  p.log_z = log_z;
  FastCtx c{h, static_cast<cudaStream_t>(stream)};
  LC_PROF(c, "compact_attention", 1);
  LC_CUDA(launch_compact_attention(d, p, n_heads, c.st));
  return LC_OK;
}

namespace {
// Held-out evaluation: step-1 statistics and the compacted attention of the
// held-out rows, placed after the compaction plan's own workspace.
struct HeldoutPlan {
  Plan p;
  size_t lse, O, ck, A, lz, total;
};

lc_status heldout_plan(const lc_shape* s, HeldoutPlan* out) {
  LC_TRY(validate(s));
  if (s->in_dtype != LC_BF16) return LC_ERR_UNSUPPORTED;
  HeldoutPlan hp{};
  hp.p = make_plan(s);
  size_t off = hp.p.total;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  };
  const size_t H = s->n_kv_heads, n = s->n_q, d = s->d, t = s->t;
  hp.lse = take(H * n * 4);
  hp.O = take(H * n * d * 4);
  hp.ck = take(H * t * d * 2);
  hp.A = take(H * n * d * 4);
  hp.lz = take(H * n * 4);
  hp.total = off;
  *out = hp;
  return LC_OK;
}
}  // namespace

lc_status lc_heldout_workspace_bytes(const lc_shape* shape, size_t* bytes) {
  HeldoutPlan hp;
  LC_TRY(heldout_plan(shape, &hp));
  if (!bytes) return LC_ERR_INVALID_ARG;
  *bytes = hp.total;
  return LC_OK;
}

lc_status lc_heldout_errors(lc_handle h, const lc_shape* shape, const void* Qh, const void* K,
                            const void* V, const int32_t* idx, const float* beta,
                            const float* Cv, float* mass_err, float* out_err, void* workspace,
                            size_t workspace_bytes, void* stream) {
  HeldoutPlan hp;
  LC_TRY(heldout_plan(shape, &hp));
  if (!Qh || !K || !V || !idx || !beta || !Cv || !mass_err || !out_err) return LC_ERR_INVALID_ARG;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 || workspace_bytes < hp.total)
    return LC_ERR_WORKSPACE;
  LC_TRY(enter(h));
  const Plan& p = hp.p;
  Ctx c{h, p, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream)};
  LC_CUDA(cudaMemsetAsync(h->d_err, 0, sizeof(uint32_t), c.st));
  const void *qop, *kop;
  LC_TRY(prepare_operands(c, Qh, K, V, true, &qop, &kop));
  LC_TRY(run_pass1(c, qop, kop, nullptr, c.at<float>(hp.lse), c.at<float>(hp.O), false));
  {
    LC_PROF(c, "gather_keys", 1);
    LC_CUDA(launch_gather_rows(K, c.ws + hp.ck, idx, p.H, p.T, p.t, p.t, p.d * 2, c.st));
  }
  CompactAttnParams a{};
  a.n = p.n_q;
  a.t = p.t;
  a.n_new = 0;
  a.scale = p.scale;
  a.q = static_cast<const __nv_bfloat16*>(Qh);
  a.Ck = c.at<__nv_bfloat16>(hp.ck);
  a.beta = beta;
  a.Cv = Cv;
  a.A = c.at<float>(hp.A);
  a.log_z = c.at<float>(hp.lz);
  {
    LC_PROF(c, "compact_attention", 1);
    LC_CUDA(launch_compact_attention(p.d, a, p.H, c.st));
  }
  {
    LC_PROF(c, "heldout_reduce", 1);
    LC_CUDA(launch_heldout_reduce(p.d, c.at<float>(hp.A), c.at<float>(hp.lz), c.at<float>(hp.O),
                                  c.at<float>(hp.lse), p.H, p.n_q, mass_err, out_err, c.st));
  }
  return LC_OK;
}

lc_status lc_farthest_first(lc_handle h, int n_heads, int T, int d, const void* K,
                            const int32_t* seeds, int n_seed, int M, int32_t* out, void* stream) {
  if (n_heads < 1 || n_heads > kMaxHeads || T < 1 || n_seed < 1 || M < n_seed || M > T)
    return LC_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return LC_ERR_UNSUPPORTED;
  if (!K || !seeds || (M > n_seed && !out)) return LC_ERR_INVALID_ARG;
  if (M == n_seed) return LC_OK;
  LC_TRY(enter(h));
  FastCtx c{h, static_cast<cudaStream_t>(stream)};
  LC_PROF(c, "farthest_first", 1);
  LC_CUDA(launch_farthest_first(d, static_cast<const __nv_bfloat16*>(K), n_heads, T, seeds, n_seed,
                                M - n_seed, out, c.st));
  return LC_OK;
}

namespace {
// The baseline variant's extra workspace: per-split column partials and the
// merged column masses of the RMS pass, after the compaction plan's own.
struct BaselinePlan {
  Plan p;
  size_t part, L2, total;
};

lc_status baseline_plan(const lc_shape* s, BaselinePlan* out) {
  LC_TRY(validate(s));
  if (s->in_dtype != LC_BF16) return LC_ERR_UNSUPPORTED;
  BaselinePlan bp{};
  bp.p = make_plan(s);
  size_t off = bp.p.total;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  };
  const size_t H = s->n_kv_heads, T = s->T;
  bp.part = take(static_cast<size_t>(bp.p.ks_max) * H * T * 8);
  bp.L2 = take(H * T * 4);
  bp.total = off;
  *out = bp;
  return LC_OK;
}
}  // namespace

lc_status lc_baseline_workspace_bytes(const lc_shape* shape, size_t* bytes) {
  BaselinePlan bp;
  LC_TRY(baseline_plan(shape, &bp));
  if (!bytes) return LC_ERR_INVALID_ARG;
  *bytes = bp.total;
  return LC_OK;
}

lc_status lc_key_scores_rms(lc_handle h, const lc_shape* shape, const void* Q, const void* K,
                            const float* lse, float* u, void* workspace, size_t workspace_bytes,
                            void* stream) {
  BaselinePlan bp;
  LC_TRY(baseline_plan(shape, &bp));
  if (!Q || !K || !lse || !u) return LC_ERR_INVALID_ARG;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 || workspace_bytes < bp.total)
    return LC_ERR_WORKSPACE;
  LC_TRY(enter(h));
  const Plan& p = bp.p;
  Ctx c{h, p, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream)};
  LC_CUDA(launch_pad_rows(lse, c.at<float>(p.lse_pad), p.H, p.n_q, p.n_q_pad, kInf, c.st));
  return run_pass2_rms(c, Q, K, c.at<float2>(bp.part), c.at<float>(bp.L2), u);
}

lc_status lc_compact_layer_baseline(lc_handle h, const lc_shape* shape, const void* Q,
                                    const void* K, const void* V, int32_t* idx, float* w,
                                    float* beta, float* Cv, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  BaselinePlan bp;
  LC_TRY(baseline_plan(shape, &bp));
  if (!Q || !K || !V || !idx || !w || !beta || !Cv) return LC_ERR_INVALID_ARG;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 || workspace_bytes < bp.total)
    return LC_ERR_WORKSPACE;
  LC_TRY(enter(h));
  const Plan& p = bp.p;
  Ctx c{h, p, static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream)};
  LC_TRY(reset_report(c));
  const void *qop, *kop;
  LC_TRY(prepare_operands(c, Q, K, V, true, &qop, &kop));
  LC_TRY(run_pass1(c, qop, kop, nullptr, nullptr, nullptr, true));
  LC_TRY(run_pass2_rms(c, qop, kop, c.at<float2>(bp.part), c.at<float>(bp.L2), nullptr));
  {
    LC_PROF(c, "select_topt", c.p.selw_on ? 3 : 1);
    LC_CUDA(select_step(c, idx, c.st));
  }
  const int iters = shape->nnls_max_iter > 0 ? shape->nnls_max_iter : 2;
  return run_fit(c, qop, kop, V, idx, w, beta, Cv, iters);
}

lc_status lc_layers_workspace_bytes(const lc_shape* shape, int n_layers, size_t* bytes) {
  LC_TRY(validate(shape));
  if (!bytes || n_layers < 1) return LC_ERR_INVALID_ARG;
  *bytes = (n_layers > 1 ? 2 : 1) * make_plan(shape).total;
  return LC_OK;
}

lc_status lc_compact_layers(lc_handle h, const lc_shape* shape, int n_layers, const void* Q,
                            const void* K, const void* V, int32_t* idx, float* w, float* beta,
                            float* Cv, void* workspace, size_t workspace_bytes, void* stream) {
  LC_TRY(validate(shape));
  if (n_layers < 1 || static_cast<long long>(n_layers) * shape->n_kv_heads > kMaxHeads)
    return LC_ERR_INVALID_ARG;
  if (!Q || !K || !V || !idx || !w || !beta || !Cv) return LC_ERR_INVALID_ARG;
  const Plan p = make_plan(shape);
  const int nb = n_layers > 1 ? 2 : 1;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 ||
      workspace_bytes < nb * p.total)
    return LC_ERR_WORKSPACE;
  LC_TRY(enter(h));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!h->fit_st) LC_CUDA(cudaStreamCreateWithFlags(&h->fit_st, cudaStreamNonBlocking));
  if (!h->ev_begin) LC_CUDA(cudaEventCreateWithFlags(&h->ev_begin, cudaEventDisableTiming));
  for (int b = 0; b < 2; ++b) {
    if (!h->ev_mass[b]) LC_CUDA(cudaEventCreateWithFlags(&h->ev_mass[b], cudaEventDisableTiming));
    if (!h->ev_fit[b]) LC_CUDA(cudaEventCreateWithFlags(&h->ev_fit[b], cudaEventDisableTiming));
  }
  const size_t H = p.H, LH = static_cast<size_t>(n_layers) * H;
  LC_CUDA(cudaMemsetAsync(h->d_status, 0, sizeof(int32_t) * LH, st));
  LC_CUDA(cudaMemsetAsync(h->d_iters, 0, sizeof(int32_t) * LH, st));
  LC_CUDA(cudaMemsetAsync(h->d_err, 0, sizeof(uint32_t), st));
  // the solve stream starts after the caller's earlier work and the resets
  LC_CUDA(cudaEventRecord(h->ev_begin, st));
  LC_CUDA(cudaStreamWaitEvent(h->fit_st, h->ev_begin, 0));
  const size_t el = p.bf16_in ? 2 : 4;
  const size_t qs = H * p.n_q * p.d * el, ks = H * p.T * p.d * el;
  for (int l = 0; l < n_layers; ++l) {
    const int b = l & 1;
    uint8_t* wsb = static_cast<uint8_t*>(workspace) + b * p.total;
    Ctx ca{h, p, wsb, st};
    Ctx cs{h, p, wsb, h->fit_st};
    // workspace b is free once layer l - 2 has finished its solve
    if (l >= 2) LC_CUDA(cudaStreamWaitEvent(st, h->ev_fit[b], 0));
    const void* Ql = static_cast<const uint8_t*>(Q) + l * qs;
    const void* Kl = static_cast<const uint8_t*>(K) + l * ks;
    const void* Vl = static_cast<const uint8_t*>(V) + l * ks;
    int32_t* idxl = idx + l * H * p.t;
    const void *qop, *kop;
    LC_TRY(prepare_operands(ca, Ql, Kl, Vl, true, &qop, &kop));
    LC_TRY(run_pass1(ca, qop, kop, nullptr, nullptr, nullptr, true));
    LC_TRY(run_pass2(ca, qop, kop));
    {
      LC_PROF(ca, "select_topt", ca.p.selw_on ? 3 : 1);
      LC_CUDA(select_step(ca, idxl, st));
    }
    LC_TRY(run_fit(ca, qop, kop, Vl, idxl, w + l * H * p.t, beta + l * H * p.t,
                   Cv + l * H * p.t * p.d, 0, &cs, h->ev_mass[b], l * p.H));
    LC_CUDA(cudaEventRecord(h->ev_fit[b], h->fit_st));
  }
  // the caller's stream resumes when the last solve is done (the solve
  // stream is in order, so that covers every layer)
  LC_CUDA(cudaStreamWaitEvent(st, h->ev_fit[(n_layers - 1) & 1], 0));
  return LC_OK;
}

lc_status lc_get_report(lc_handle h, int n_heads, int32_t* head_status, int32_t* nnls_iters,
                        uint32_t* device_error_bits, void* stream) {
  if (!h || n_heads < 1 || n_heads > kMaxHeads) return LC_ERR_INVALID_ARG;
  LC_TRY(enter(h));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LC_CUDA(cudaStreamSynchronize(st));
  if (head_status)
    LC_CUDA(cudaMemcpy(head_status, h->d_status, sizeof(int32_t) * n_heads, cudaMemcpyDeviceToHost));
  if (nnls_iters)
    LC_CUDA(cudaMemcpy(nnls_iters, h->d_iters, sizeof(int32_t) * n_heads, cudaMemcpyDeviceToHost));
  if (device_error_bits)
    LC_CUDA(cudaMemcpy(device_error_bits, h->d_err, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  return LC_OK;
}

lc_status lc_profile_enable(lc_handle h, int on) {
  if (!h) return LC_ERR_INVALID_ARG;
  h->prof.on = on != 0;
  return LC_OK;
}

lc_status lc_profile_read(lc_handle h, int max_kernels, char* names, double* total_ms,
                          int32_t* launches, int* n_kernels) {
  if (!h || max_kernels < 0 || !n_kernels) return LC_ERR_INVALID_ARG;
  LC_TRY(enter(h));
  h->prof.resolve();
  int i = 0;
  for (auto& kv : h->prof.acc) {
    if (i < max_kernels) {
      if (names) {
        std::strncpy(names + 32 * i, kv.first.c_str(), 31);
        names[32 * i + 31] = 0;
      }
      if (total_ms) total_ms[i] = kv.second.first;
      if (launches) launches[i] = kv.second.second;
    }
    ++i;
  }
  *n_kernels = i;
  h->prof.acc.clear();
  return LC_OK;
}

const char* lc_status_string(lc_status s) {
  switch (s) {
    case LC_OK: return "ok";
    case LC_ERR_INVALID_ARG: return "invalid argument";
    case LC_ERR_UNSUPPORTED: return "unsupported shape or type";
    case LC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case LC_ERR_CUDA: return "CUDA call failed";
    case LC_ERR_NOT_CONVERGED: return "NNLS iteration cap reached";
    case LC_ERR_SINGULAR: return "singular system (ridge added)";
    case LC_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
