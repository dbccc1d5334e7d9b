"""Degenerate systems and host-side errors, through the C ABI.

* Two kept keys with equal vectors: the mass system has two equal columns, so
  its minimiser is not unique.  Library and oracle both give the copy at the
  later position w = 0 (the minimiser Lawson-Hanson reaches with its argmax
  ties going to the lower index), so the whole compaction still matches the
  oracle's at the usual tolerances.
* All reference queries at q = 0 ("KV compaction" blog, "Fast KV Compaction
  via Attention Matching": the case that shows why beta is needed): every key
  gets the same attention, the mass system is rank one and the output system
  too.  The library's factorisations break down, it adds its ridge and
  reports LC_ERR_SINGULAR; the solutions are not unique, so the test compares
  what is: the compact mass sum(w) = T (oracle: the same), and the compact
  output at q = 0, which must equal the full one, mean(V).
* A workspace that is too small or misaligned returns LC_ERR_WORKSPACE and
  enqueues nothing: preset output buffers keep their contents.
"""
import ctypes
import math

import numpy as np
import pytest

import oracle
import synth
from gpu_util import (FIT_REL, check_layer_fits, compactor, dev, dev_f32, dev_i32, gate_fit,
                      host, relf, torch)

pytestmark = pytest.mark.gpu

LC_ERR_WORKSPACE, LC_ERR_SINGULAR = 3, 6


@pytest.fixture(scope="module")
def comp():
    return compactor()


def _with_duplicates(seed):
    """A small peaked layer in which each head's highest-scoring key has an
    exact copy at a later position.  With peaked queries many keys reach a
    probability near 1, and the copy halves that of the duplicated key, so
    half the keys are kept to keep both copies."""
    w = synth.workload("cfg2", H=2, T=384, G=2, t=192, seed=seed)
    d = synth.make(w)
    pairs = []
    for h in range(w.H):
        r = oracle.compact_head(d["Q"][h], d["K"][h], d["V"][h], w.t, w.softmax_scale)
        a = int(np.argmax(r["u"]))
        b = (a + w.T // 2) % w.T
        a, b = min(a, b), max(a, b)
        d["K"][h][b] = d["K"][h][a]
        pairs.append((a, b))
    return w, d, pairs


def test_duplicate_kept_keys(comp):
    w, d, pairs = _with_duplicates(31)
    refs = {h: oracle.compact_head(d["Q"][h], d["K"][h], d["V"][h], w.t, w.softmax_scale)
            for h in range(w.H)}
    for h, (a, b) in enumerate(pairs):
        r = refs[h]
        assert a in r["idx"] and b in r["idx"], "both copies must be kept (test is not testing)"
        pb = int(np.flatnonzero(r["idx"] == b)[0])
        assert r["w"][pb] == 0.0 and r["w"][r["idx"] == a][0] > 0.0
    Q, K, V = dev(d["Q"], w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype)
    idx, wg, bg, cg = (host(x) for x in comp.compact_layer(Q, K, V, w.t))
    rep = comp.report(w.H)
    assert rep.device_error_bits == 0 and rep.head_status == [0] * w.H, rep
    check_layer_fits(comp, w, Q, K, V, refs, idx, wg, bg, cg)
    for h, (a, b) in enumerate(pairs):
        pb = int(np.flatnonzero(idx[h] == b)[0])
        assert wg[h][pb] == 0.0 and np.isneginf(bg[h][pb]), "later copy has a weight"
        assert np.array_equal(cg[h][pb], d["V"][h][b]), "later copy's value row changed"
    # the same fit through lc_fit_only on the oracle's selection and statistics
    sel = [refs[h] for h in range(w.H)]
    wf, bf, cf = comp.fit_only(Q, K, V, dev_i32(np.stack([r["idx"] for r in sel])),
                               dev_f32(np.stack([r["m"] for r in sel])),
                               dev_f32(np.stack([r["lse"] for r in sel])),
                               dev_f32(np.stack([r["O"] for r in sel])))
    rep = comp.report(w.H)
    assert rep.head_status == [0] * w.H, rep
    for h in range(w.H):
        gate_fit(host(wf)[h], host(bf)[h], host(cf)[h], refs[h], f"head {h} fit_only")


@pytest.mark.parametrize("T,t", [(256, 32), (500, 100), (2048, 256)])
def test_zero_queries_singular(comp, T, t):
    w = synth.workload("cfg2", H=2, T=T, G=1, t=t, seed=32)
    d = synth.make(w)
    d["Q"][:] = 0.0
    Q, K, V = dev(d["Q"], w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype)
    idx, wg, bg, cg = (host(x) for x in comp.compact_layer(Q, K, V, t))
    rep = comp.report(w.H)
    assert rep.device_error_bits == 0
    assert rep.head_status == [LC_ERR_SINGULAR] * w.H, rep.head_status
    r = oracle.compact_head(d["Q"][0], d["K"][0], d["V"][0], t, w.softmax_scale)
    assert abs(r["w"].sum() - T) <= 1e-9 * T, "oracle: compact mass at q = 0 is not T"
    for h in range(w.H):
        # every key scores 1/T: the selection is the t lowest indices
        assert np.array_equal(idx[h], np.arange(t))
        assert np.all(np.isfinite(wg[h])) and np.all(wg[h] >= 0) and np.all(np.isfinite(cg[h]))
        assert abs(wg[h].sum() - T) <= FIT_REL * T, f"head {h}: sum w = {wg[h].sum()}"
        # compact output at q = 0: softmax of beta over the kept keys times C_v
        b = bg[h].astype(np.float64)
        p = np.exp(b - b.max())
        p /= p.sum()
        out = p @ cg[h].astype(np.float64)
        ref = d["V"][h].astype(np.float64).mean(axis=0)
        assert relf(out, ref) <= FIT_REL, f"head {h}: compact output {relf(out, ref):.2e}"
        assert abs(math.log(wg[h].sum()) - math.log(T)) <= 1e-3


def test_workspace_errors_enqueue_nothing(comp):
    w = synth.workload("cfg2", H=2, T=300, t=20, seed=7)
    d = synth.make(w)
    Q, K, V = dev(d["Q"], w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype)
    t_ = torch()
    s = comp.shape(Q, K, w.t)
    need = comp.workspace_bytes(s)
    ws = t_.empty(need + 512, dtype=t_.uint8, device="cuda")
    base = ws.data_ptr()
    assert base % 256 == 0
    outs = [t_.full((w.H, w.t), 7, dtype=t_.int32, device="cuda"),
            t_.full((w.H, w.t), 7.0, device="cuda"), t_.full((w.H, w.t), 7.0, device="cuda"),
            t_.full((w.H, w.t, w.d), 7.0, device="cuda")]
    ptr = [ctypes.c_void_p(x.data_ptr()) for x in (Q, K, V, *outs)]
    t_.cuda.synchronize()
    for wsp, nbytes in [(base, need - 1), (base + 16, need), (0, need)]:
        code = comp.lib.lc_compact_layer(comp.handle, ctypes.byref(s), *ptr[:3], *ptr[3:],
                                         ctypes.c_void_p(wsp), nbytes, comp._stream())
        assert code == LC_ERR_WORKSPACE, code
    t_.cuda.synchronize()
    for x in outs:
        assert bool((x == 7).all()), "an output changed although the call was rejected"
    # the same call with a valid workspace runs
    code = comp.lib.lc_compact_layer(comp.handle, ctypes.byref(s), *ptr[:3], *ptr[3:],
                                     ctypes.c_void_p(base), need, comp._stream())
    assert code == 0
    t_.cuda.synchronize()
    assert not bool((outs[0] == 7).all())
