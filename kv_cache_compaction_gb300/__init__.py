"""GB300-native attention-matching compaction of a layer's KV cache.

Thin ctypes binding over ``liblc.so`` (C ABI declared in ``include/lc.h``).
Every step runs in the library's CUDA kernels; this module only checks and
marshals arguments (device pointers of torch tensors, the current CUDA
stream) and owns a cached device workspace.  There is no CPU fallback: if the
library is missing, importing the binding's entry points raises.

Typical use::

    import torch, kv_cache_compaction_gb300 as lc
    comp = lc.Compactor(device=0)
    idx, w, beta, Cv = comp.compact_layer(Q, K, V, t=256)   # bf16 CUDA tensors

Q is [H, n_q, d] (the reference queries of every query head of each KV
head's group), K and V are [H, T, d].
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

__all__ = ["Compactor", "LCError", "load_library", "LIB_PATH", "STATUS", "EXPORTS"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblc.so")

STATUS = {
    0: "LC_OK", 1: "LC_ERR_INVALID_ARG", 2: "LC_ERR_UNSUPPORTED", 3: "LC_ERR_WORKSPACE",
    4: "LC_ERR_CUDA", 5: "LC_ERR_NOT_CONVERGED", 6: "LC_ERR_SINGULAR", 7: "LC_ERR_TIMEOUT",
}

# Every symbol include/lc.h declares.
EXPORTS = [
    "lc_create", "lc_destroy", "lc_workspace_bytes", "lc_full_attn_stats", "lc_key_scores",
    "lc_select_topt", "lc_fit_only", "lc_compact_layer", "lc_host_workspace_bytes",
    "lc_compact_layer_host", "lc_get_report", "lc_profile_enable", "lc_profile_read",
    "lc_select_topt_noalloc", "lc_status_string", "lc_fast_workspace_bytes",
    "lc_compact_layer_fast", "lc_compact_attention", "lc_heldout_workspace_bytes",
    "lc_heldout_errors", "lc_farthest_first", "lc_baseline_workspace_bytes",
    "lc_compact_layer_baseline", "lc_key_scores_rms", "lc_layers_workspace_bytes",
    "lc_compact_layers",
]

LC_BF16, LC_FP32 = 0, 1


class LCError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("n_kv_heads", ctypes.c_int), ("n_q", ctypes.c_int), ("T", ctypes.c_int),
                ("d", ctypes.c_int), ("t", ctypes.c_int), ("in_dtype", ctypes.c_int),
                ("scale", ctypes.c_float), ("nnls_max_iter", ctypes.c_int)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load liblc.so and declare its signatures (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not found: build it with kv_cache_compaction_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, sz, i32, f32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
    sp = ctypes.POINTER(Shape)
    sig = {
        "lc_create": ([ctypes.POINTER(vp), i32], i32),
        "lc_destroy": ([vp], i32),
        "lc_workspace_bytes": ([sp, ctypes.POINTER(sz)], i32),
        "lc_host_workspace_bytes": ([sp, ctypes.POINTER(sz)], i32),
        "lc_full_attn_stats": ([vp, sp, vp, vp, vp, f32p, f32p, f32p, vp, sz, vp], i32),
        "lc_key_scores": ([vp, sp, vp, vp, vp, vp, vp, sz, vp], i32),
        "lc_select_topt": ([vp, i32, i32, i32, vp, vp, vp, sz, vp], i32),
        "lc_select_topt_noalloc": ([i32, i32, i32, vp, vp, vp], i32),
        "lc_fit_only": ([vp, sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
        "lc_compact_layer": ([vp, sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
        "lc_compact_layer_host": ([vp, sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
        "lc_fast_workspace_bytes": ([sp, i32, i32, ctypes.POINTER(sz)], i32),
        "lc_compact_layer_fast": ([vp, sp, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp, sz, vp],
                                  i32),
        "lc_compact_attention": ([vp, i32, i32, i32, i32, i32, ctypes.c_float, vp, vp, vp, vp,
                                  vp, vp, vp, vp, vp, vp], i32),
        "lc_heldout_workspace_bytes": ([sp, ctypes.POINTER(sz)], i32),
        "lc_heldout_errors": ([vp, sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
        "lc_farthest_first": ([vp, i32, i32, i32, vp, vp, i32, i32, vp, vp], i32),
        "lc_baseline_workspace_bytes": ([sp, ctypes.POINTER(sz)], i32),
        "lc_compact_layer_baseline": ([vp, sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
        "lc_key_scores_rms": ([vp, sp, vp, vp, vp, vp, vp, sz, vp], i32),
        "lc_layers_workspace_bytes": ([sp, i32, ctypes.POINTER(sz)], i32),
        "lc_compact_layers": ([vp, sp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
        "lc_get_report": ([vp, i32, vp, vp, vp, vp], i32),
        "lc_profile_enable": ([vp, i32], i32),
        "lc_profile_read": ([vp, i32, vp, vp, vp, vp], i32),
        "lc_status_string": ([i32], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(code: int, where: str):
    if code != 0:
        raise LCError(code, where)


def _ptr(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


@dataclass
class Report:
    head_status: list
    nnls_iters: list
    device_error_bits: int


class Compactor:
    """One library handle on one CUDA device, plus a cached workspace."""

    def __init__(self, device: int = 0):
        import torch
        self._torch = torch
        self.lib = load_library()
        self.device = torch.device("cuda", device)
        h = ctypes.c_void_p()
        _check(self.lib.lc_create(ctypes.byref(h), device), "lc_create")
        self.handle = h
        self._ws = None

    def close(self):
        if getattr(self, "handle", None):
            self.lib.lc_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ helpers
    def shape(self, Q, K, t: int = 1, scale: float = 0.0, nnls_max_iter: int = 0) -> Shape:
        torch = self._torch
        if Q.dim() != 3 or K.dim() != 3 or Q.shape[0] != K.shape[0] or Q.shape[2] != K.shape[2]:
            raise ValueError("Q must be [H, n_q, d] and K [H, T, d]")
        if Q.dtype == torch.bfloat16:
            dt = LC_BF16
        elif Q.dtype == torch.float32:
            dt = LC_FP32
        else:
            raise ValueError("Q, K, V must be bfloat16 or float32")
        return Shape(int(Q.shape[0]), int(Q.shape[1]), int(K.shape[1]), int(Q.shape[2]), int(t),
                     dt, float(scale), int(nnls_max_iter))

    def _check_inputs(self, *xs):
        for x in xs:
            if x is None:
                continue
            if not x.is_cuda or x.device != self.device:
                raise ValueError("tensors must live on " + str(self.device))
            if not x.is_contiguous():
                raise ValueError("tensors must be contiguous")

    def workspace_bytes(self, shape: Shape, host: bool = False) -> int:
        n = ctypes.c_size_t()
        fn = self.lib.lc_host_workspace_bytes if host else self.lib.lc_workspace_bytes
        _check(fn(ctypes.byref(shape), ctypes.byref(n)), "workspace_bytes")
        return n.value

    def workspace(self, nbytes: int):
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = self._torch.empty(max(nbytes, 256), dtype=self._torch.uint8, device=self.device)
        return self._ws

    def _stream(self):
        return ctypes.c_void_p(self._torch.cuda.current_stream(self.device).cuda_stream)

    def _empty(self, shape, dtype):
        return self._torch.empty(shape, dtype=dtype, device=self.device)

    # ------------------------------------------------------------ entry points
    def full_attn_stats(self, Q, K, V, scale: float = 0.0):
        """Step 1: (rowmax, lse, O) for every reference query."""
        torch = self._torch
        self._check_inputs(Q, K, V)
        s = self.shape(Q, K, 1, scale)
        ws = self.workspace(self.workspace_bytes(s))
        H, n_q, d = Q.shape
        m = self._empty((H, n_q), torch.float32)
        lse = self._empty((H, n_q), torch.float32)
        O = self._empty((H, n_q, d), torch.float32)
        _check(self.lib.lc_full_attn_stats(self.handle, ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V),
                                           _ptr(m), _ptr(lse), _ptr(O), _ptr(ws), ws.numel(),
                                           self._stream()), "lc_full_attn_stats")
        return m, lse, O

    def key_scores(self, Q, K, lse, scale: float = 0.0):
        """Step 2: u[h, j] = max_i (scale q_i.k_j - lse_i)."""
        torch = self._torch
        self._check_inputs(Q, K, lse)
        s = self.shape(Q, K, 1, scale)
        ws = self.workspace(self.workspace_bytes(s))
        u = self._empty((K.shape[0], K.shape[1]), torch.float32)
        _check(self.lib.lc_key_scores(self.handle, ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(lse),
                                      _ptr(u), _ptr(ws), ws.numel(), self._stream()),
               "lc_key_scores")
        return u

    def select_topt(self, u, t: int):
        """Step 3: ascending indices of the t largest scores per row of u."""
        torch = self._torch
        self._check_inputs(u)
        if u.dtype != torch.float32 or u.dim() != 2:
            raise ValueError("u must be a [H, T] float32 tensor")
        H, T = u.shape
        ws = self.workspace(max(256, H * T * 4))
        idx = self._empty((H, t), torch.int32)
        _check(self.lib.lc_select_topt(self.handle, H, T, t, _ptr(u), _ptr(idx), _ptr(ws),
                                       ws.numel(), self._stream()), "lc_select_topt")
        return idx

    def fit_only(self, Q, K, V, idx, rowmax, lse, O, scale: float = 0.0, nnls_max_iter: int = 0):
        """Steps 4-5 for given keys and statistics: (w, beta, Cv)."""
        torch = self._torch
        self._check_inputs(Q, K, V, idx, rowmax, lse, O)
        t = int(idx.shape[1])
        s = self.shape(Q, K, t, scale, nnls_max_iter)
        ws = self.workspace(self.workspace_bytes(s))
        H, _, d = Q.shape
        w = self._empty((H, t), torch.float32)
        beta = self._empty((H, t), torch.float32)
        Cv = self._empty((H, t, d), torch.float32)
        _check(self.lib.lc_fit_only(self.handle, ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V),
                                    _ptr(idx), _ptr(rowmax), _ptr(lse), _ptr(O), _ptr(w),
                                    _ptr(beta), _ptr(Cv), _ptr(ws), ws.numel(), self._stream()),
               "lc_fit_only")
        return w, beta, Cv

    def compact_layer(self, Q, K, V, t: int, scale: float = 0.0, nnls_max_iter: int = 0, out=None):
        """Steps 1-5: (idx, w, beta, Cv).  ``out`` may supply preallocated outputs."""
        torch = self._torch
        self._check_inputs(Q, K, V)
        s = self.shape(Q, K, t, scale, nnls_max_iter)
        ws = self.workspace(self.workspace_bytes(s))
        H, _, d = Q.shape
        if out is None:
            out = (self._empty((H, t), torch.int32), self._empty((H, t), torch.float32),
                   self._empty((H, t), torch.float32), self._empty((H, t, d), torch.float32))
        idx, w, beta, Cv = out
        _check(self.lib.lc_compact_layer(self.handle, ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V),
                                         _ptr(idx), _ptr(w), _ptr(beta), _ptr(Cv), _ptr(ws),
                                         ws.numel(), self._stream()), "lc_compact_layer")
        return idx, w, beta, Cv

    def compact_layers(self, Q, K, V, t: int, scale: float = 0.0, nnls_max_iter: int = 0,
                       out=None):
        """compact_layer for L layers in one pipelined call: Q [L, H, n_q, d],
        K, V [L, H, T, d] -> (idx [L, H, t], w, beta [L, H, t], Cv [L, H, t, d])."""
        torch = self._torch
        self._check_inputs(Q, K, V)
        L, H, _, d = Q.shape
        s = self.shape(Q[0], K[0], t, scale, nnls_max_iter)
        n = ctypes.c_size_t()
        _check(self.lib.lc_layers_workspace_bytes(ctypes.byref(s), L, ctypes.byref(n)),
               "lc_layers_workspace_bytes")
        ws = self.workspace(n.value)
        if out is None:
            out = (self._empty((L, H, t), torch.int32), self._empty((L, H, t), torch.float32),
                   self._empty((L, H, t), torch.float32), self._empty((L, H, t, d), torch.float32))
        idx, w, beta, Cv = out
        _check(self.lib.lc_compact_layers(self.handle, ctypes.byref(s), L, _ptr(Q), _ptr(K),
                                          _ptr(V), _ptr(idx), _ptr(w), _ptr(beta), _ptr(Cv),
                                          _ptr(ws), ws.numel(), self._stream()),
               "lc_compact_layers")
        return idx, w, beta, Cv

    def compact_layer_host(self, Q, K, V, t: int, out, scale: float = 0.0, nnls_max_iter: int = 0):
        """Steps 1-5 on host (preferably pinned) CPU tensors, results written to
        the CPU tensors in ``out`` = (idx, w, beta, Cv); synchronises."""
        s = self.shape(Q, K, t, scale, nnls_max_iter)
        ws = self.workspace(self.workspace_bytes(s, host=True))
        idx, w, beta, Cv = out
        for x in (Q, K, V, idx, w, beta, Cv):
            if x.is_cuda or not x.is_contiguous():
                raise ValueError("host entry point takes contiguous CPU tensors")
        _check(self.lib.lc_compact_layer_host(self.handle, ctypes.byref(s), _ptr(Q), _ptr(K),
                                              _ptr(V), _ptr(idx), _ptr(w), _ptr(beta), _ptr(Cv),
                                              _ptr(ws), ws.numel(), self._stream()),
               "lc_compact_layer_host")
        return idx, w, beta, Cv

    def compact_layer_fast(self, Q, K, V, qsel, t: int, k: int = 4, scale: float = 0.0,
                           out=None, with_shortlist: bool = False):
        """Two-pass selection, redistributed beta and direct values:
        (idx, beta, Cv[, shortlist]).  ``qsel`` [H, n_sub] int32 holds the rows
        of Q that form the query subset of the first pass (the random draw is
        the caller's); the shortlist keeps min(k t, T) keys."""
        torch = self._torch
        self._check_inputs(Q, K, V, qsel)
        if qsel.dtype != torch.int32 or qsel.dim() != 2 or qsel.shape[0] != Q.shape[0]:
            raise ValueError("qsel must be an [H, n_sub] int32 tensor")
        s = self.shape(Q, K, t, scale)
        n_sub = int(qsel.shape[1])
        n = ctypes.c_size_t()
        _check(self.lib.lc_fast_workspace_bytes(ctypes.byref(s), n_sub, k, ctypes.byref(n)),
               "lc_fast_workspace_bytes")
        ws = self.workspace(n.value)
        H, _, d = Q.shape
        if out is None:
            out = (self._empty((H, t), torch.int32), self._empty((H, t), torch.float32),
                   self._empty((H, t, d), torch.float32))
        idx, beta, Cv = out
        short = self._empty((H, min(k * t, K.shape[1])), torch.int32) if with_shortlist else None
        _check(self.lib.lc_compact_layer_fast(self.handle, ctypes.byref(s), _ptr(Q), _ptr(K),
                                              _ptr(V), _ptr(qsel), n_sub, k, _ptr(idx),
                                              _ptr(beta), _ptr(Cv), _ptr(short), _ptr(ws),
                                              ws.numel(), self._stream()),
               "lc_compact_layer_fast")
        return (idx, beta, Cv, short) if with_shortlist else (idx, beta, Cv)

    def compact_attention(self, q, Ck, beta, Cv, Knew=None, Vnew=None, n_vis=None,
                          scale: float = 0.0):
        """Attention of q [H, n, d] over a compacted cache (Ck bf16 [H, t, d],
        beta, Cv fp32) plus appended tokens (Knew, Vnew bf16 [H, n_new, d];
        row r sees the first n_vis[h, r] of them, all if n_vis is None):
        (A [H, n, d] fp32, log_z [H, n] fp32)."""
        torch = self._torch
        self._check_inputs(q, Ck, beta, Cv, Knew, Vnew, n_vis)
        H, n, d = q.shape
        t = int(Ck.shape[1])
        n_new = 0 if Knew is None else int(Knew.shape[1])
        A = self._empty((H, n, d), torch.float32)
        lz = self._empty((H, n), torch.float32)
        _check(self.lib.lc_compact_attention(self.handle, H, n, t, n_new, d, scale, _ptr(q),
                                             _ptr(Ck), _ptr(beta), _ptr(Cv), _ptr(Knew),
                                             _ptr(Vnew), _ptr(n_vis), _ptr(A), _ptr(lz),
                                             self._stream()), "lc_compact_attention")
        return A, lz

    def heldout_errors(self, Qh, K, V, idx, beta, Cv, scale: float = 0.0):
        """Mean |log Z_cmp - log Z_full| and mean ||A_cmp - A_full|| per head
        on held-out queries Qh for the compaction (idx, beta, Cv)."""
        torch = self._torch
        self._check_inputs(Qh, K, V, idx, beta, Cv)
        s = self.shape(Qh, K, int(idx.shape[1]), scale)
        n = ctypes.c_size_t()
        _check(self.lib.lc_heldout_workspace_bytes(ctypes.byref(s), ctypes.byref(n)),
               "lc_heldout_workspace_bytes")
        ws = self.workspace(n.value)
        H = Qh.shape[0]
        me = self._empty((H,), torch.float32)
        oe = self._empty((H,), torch.float32)
        _check(self.lib.lc_heldout_errors(self.handle, ctypes.byref(s), _ptr(Qh), _ptr(K), _ptr(V),
                                          _ptr(idx), _ptr(beta), _ptr(Cv), _ptr(me), _ptr(oe),
                                          _ptr(ws), ws.numel(), self._stream()),
               "lc_heldout_errors")
        return me, oe

    def farthest_first(self, K, seeds, M: int):
        """Farthest-first traversal per head from the seeds [H, n_seed] int32
        until M keys are selected: the added indices [H, M - n_seed] int32."""
        torch = self._torch
        self._check_inputs(K, seeds)
        H, T, d = K.shape
        n_seed = int(seeds.shape[1])
        out = self._empty((H, max(M - n_seed, 0)), torch.int32)
        _check(self.lib.lc_farthest_first(self.handle, H, T, d, _ptr(K), _ptr(seeds), n_seed, M,
                                          _ptr(out), self._stream()), "lc_farthest_first")
        return out

    def _baseline_ws(self, s):
        n = ctypes.c_size_t()
        _check(self.lib.lc_baseline_workspace_bytes(ctypes.byref(s), ctypes.byref(n)),
               "lc_baseline_workspace_bytes")
        return self.workspace(n.value)

    def key_scores_rms(self, Q, K, lse, scale: float = 0.0):
        """RMS key scores u[h, j] = log sqrt(mean_i p_ij^2) (bf16 Q, K)."""
        torch = self._torch
        self._check_inputs(Q, K, lse)
        s = self.shape(Q, K, 1, scale)
        ws = self._baseline_ws(s)
        u = self._empty((K.shape[0], K.shape[1]), torch.float32)
        _check(self.lib.lc_key_scores_rms(self.handle, ctypes.byref(s), _ptr(Q), _ptr(K),
                                          _ptr(lse), _ptr(u), _ptr(ws), ws.numel(),
                                          self._stream()), "lc_key_scores_rms")
        return u

    def compact_layer_baseline(self, Q, K, V, t: int, scale: float = 0.0, iters: int = 0):
        """The baseline variant (RMS key scores, bounded biases in
        [e^-3, e^3] with `iters` iterations, 0 = two): (idx, w, beta, Cv)."""
        torch = self._torch
        self._check_inputs(Q, K, V)
        s = self.shape(Q, K, t, scale, iters)
        ws = self._baseline_ws(s)
        H, _, d = Q.shape
        idx = self._empty((H, t), torch.int32)
        w = self._empty((H, t), torch.float32)
        beta = self._empty((H, t), torch.float32)
        Cv = self._empty((H, t, d), torch.float32)
        _check(self.lib.lc_compact_layer_baseline(self.handle, ctypes.byref(s), _ptr(Q), _ptr(K),
                                                  _ptr(V), _ptr(idx), _ptr(w), _ptr(beta),
                                                  _ptr(Cv), _ptr(ws), ws.numel(),
                                                  self._stream()), "lc_compact_layer_baseline")
        return idx, w, beta, Cv

    def profile(self, on: bool):
        """Turn per-kernel CUDA-event timing of the library's launches on/off."""
        _check(self.lib.lc_profile_enable(self.handle, int(on)), "lc_profile_enable")

    def profile_read(self) -> dict:
        """{kernel name: (total ms, launches)} since the last read; synchronises
        with the recorded events and clears the totals."""
        cap = 64
        names = ctypes.create_string_buffer(32 * cap)
        ms = (ctypes.c_double * cap)()
        cnt = (ctypes.c_int32 * cap)()
        n = ctypes.c_int()
        _check(self.lib.lc_profile_read(self.handle, cap, names, ms, cnt, ctypes.byref(n)),
               "lc_profile_read")
        out = {}
        for i in range(min(n.value, cap)):
            nm = names.raw[32 * i:32 * i + 32].split(b"\0", 1)[0].decode()
            out[nm] = (ms[i], cnt[i])
        return out

    def report(self, n_heads: int) -> Report:
        st = (ctypes.c_int32 * n_heads)()
        it = (ctypes.c_int32 * n_heads)()
        err = ctypes.c_uint32()
        _check(self.lib.lc_get_report(self.handle, n_heads, st, it, ctypes.byref(err),
                                      self._stream()), "lc_get_report")
        return Report(list(st), list(it), err.value)
