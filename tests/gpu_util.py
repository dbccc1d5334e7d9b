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


def near_tie_swap(got, ref, u, n_keep, where=""):
    """Check that the selections ``got`` and ``ref`` (ascending key indices)
    agree except for keys whose reference score ties the n_keep-th largest
    within the score tolerance (rounding may order such keys either way).
    Returns the overlap |got & ref| / n_keep."""
    got, ref = np.asarray(got), np.asarray(ref)
    if not np.array_equal(got, ref):
        tau = np.sort(np.asarray(u))[::-1][n_keep - 1]
        diff = np.setxor1d(got, ref)
        assert np.all(np.abs(np.asarray(u)[diff] - tau) <= SCORE_ABS), \
            f"{where}: selection differs beyond near-ties"
    return np.intersect1d(got, ref).size / n_keep


def gate_fit(wg, bg, cg, ref, where=""):
    """w, beta and C_v of one head against the oracle's fit ``ref``."""
    assert relf(wg, ref["w"]) <= FIT_REL, f"{where} w relF {relf(wg, ref['w']):.2e}"
    assert beta_err(bg, ref["beta"]) <= FIT_REL, f"{where} beta {beta_err(bg, ref['beta']):.2e}"
    assert relf(cg, ref["Cv"]) <= FIT_REL, f"{where} Cv relF {relf(cg, ref['Cv']):.2e}"


def check_layer_fits(comp, w, Q, K, V, refs, idx, wg, bg, cg):
    """Steps 3-5 of a GPU compaction, head by head, against the oracle's
    compaction of each head (``refs``: head -> oracle.compact_head result).

    Heads whose selection equals the oracle's compare w, beta and C_v
    directly.  Where a near-tie made the selections differ, the GPU's fit
    is compared on the oracle's own selection and statistics instead,
    through lc_fit_only: every head gets its fit compared, and every oracle
    input still comes from the generator or the oracle.  Returns the
    selection overlaps."""
    overlaps, refit = {}, []
    for h, r in refs.items():
        overlaps[h] = near_tie_swap(idx[h], r["idx"], r["u"], w.t, f"head {h}")
        if overlaps[h] == 1.0:
            gate_fit(wg[h], bg[h], cg[h], r, f"head {h}")
        else:
            refit.append(h)
    if refit:
        sel = [refs[h] for h in refit]
        wf, bf, cf = comp.fit_only(Q[refit], K[refit], V[refit],
                                   dev_i32(np.stack([r["idx"] for r in sel])),
                                   dev_f32(np.stack([r["m"] for r in sel])),
                                   dev_f32(np.stack([r["lse"] for r in sel])),
                                   dev_f32(np.stack([r["O"] for r in sel])), scale=w.scale)
        rep = comp.report(len(refit))
        assert rep.device_error_bits == 0
        wf, bf, cf = host(wf), host(bf), host(cf)
        for i, h in enumerate(refit):
            assert rep.head_status[i] == 0, f"head {h} refit status {rep.head_status[i]}"
            gate_fit(wf[i], bf[i], cf[i], refs[h], f"head {h} (on the oracle's selection)")
    return overlaps
