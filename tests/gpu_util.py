"""Helpers for the GPU parity tests: upload seeded inputs, compare with the
oracle.  Tolerances are the gates of the method's accuracy contract:
  - log mass lse: 1e-3 absolute;
  - key scores a_j = exp(u_j): 2e-3 relative, i.e. 2e-3 absolute on u_j;
  - selection: bit-exact on identical score arrays;
  - beta and C_v: 1e-3 relative Frobenius (beta on the common support, with
    the denominator floored at 1).
The attention output O has no gate of its own; it is checked at 2e-3 relative
Frobenius because it feeds C_v.
"""
from __future__ import annotations

import numpy as np

import synth

LSE_ABS = 1e-3
SCORE_ABS = 2e-3
FIT_REL = 1e-3
O_REL = 2e-3


def torch():
    import torch as _t
    return _t


def compactor():
    from kv_cache_compaction_gb300 import build as b
    b.build()
    import kv_cache_compaction_gb300 as lc
    return lc.Compactor(0)


def dev(a: np.ndarray, dtype: str):
    """Upload a float32 array holding bf16-exact (dtype 'bf16') or fp32 values."""
    t = torch()
    if dtype == "bf16":
        bits = synth.bf16_bits(a).view(np.int16)
        return t.from_numpy(np.ascontiguousarray(bits)).view(t.bfloat16).cuda()
    return t.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_f32(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_i32(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host(x) -> np.ndarray:
    return x.detach().cpu().numpy()


def relf(a, b) -> float:
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def beta_err(b_gpu, b_ref) -> float:
    """||beta_gpu - beta_ref|| / max(||beta_ref||, 1) over keys where both are
    finite (w > 0 on both sides)."""
    b_gpu, b_ref = np.asarray(b_gpu, np.float64), np.asarray(b_ref, np.float64)
    m = np.isfinite(b_gpu) & np.isfinite(b_ref)
    return float(np.linalg.norm(b_gpu[m] - b_ref[m]) / max(np.linalg.norm(b_ref[m]), 1.0))


def inputs(w: synth.Workload, heads=None):
    d = synth.make(w, heads)
    return d, dev(d["Q"], w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype)
