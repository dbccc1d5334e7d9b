"""Parity of the baseline attention-matching variant (RMS key scores, bounded
biases in [e^-3, e^3] with two iterations, least-squares values) with the
float64 oracle's compact_head_variant on the same seeded inputs.  Gates as
for the main path: scores 2e-3 absolute in the log domain, selection exact
up to near-ties, w, beta and C_v 1e-3 relative Frobenius."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (FIT_REL, LSE_ABS, O_REL, SCORE_ABS, beta_err, compactor, dev_f32, host,
                      inputs, relf)

pytestmark = pytest.mark.gpu

CASES = {
    "d128_ragged": synth.workload("cfg2", H=2, T=300, t=20, seed=7),
    "d64_ragged": synth.workload("cfg2", H=2, T=257, d=64, t=33, seed=8),
    "t_over_128": synth.workload("cfg2", H=2, T=700, G=2, t=160, seed=10),
    "iid": synth.workload("cfg2", H=1, T=640, G=2, t=64, kind="iid", seed=11),
    "t256": synth.workload("cfg2", H=2, T=1024, G=4, t=256, seed=12),
    # edge cases: one kept key (its bias meets the upper bound e^3); one
    # cached key
    "t1": synth.workload("cfg2", H=2, T=200, G=1, t=1, kind="iid", seed=18),
    "T1": synth.workload("cfg2", H=1, T=1, G=2, t=1, seed=17),
}


@pytest.fixture(scope="module")
def comp():
    return compactor()


@pytest.mark.parametrize("name", list(CASES))
def test_rms_scores(comp, name):
    w = CASES[name]
    d, Q, K, _ = inputs(w)
    lse = np.stack([oracle.full_stats(d["Q"][h], d["K"][h], d["V"][h], w.softmax_scale)[1]
                    for h in range(w.H)])
    u = host(comp.key_scores_rms(Q, K, dev_f32(lse)))
    for h in range(w.H):
        ref = oracle.rms_key_scores(d["Q"][h], d["K"][h], lse[h], w.softmax_scale)
        err = np.max(np.abs(u[h] - ref))
        assert err <= SCORE_ABS, f"head {h}: max |u - u_ref| = {err:.2e}"


def _check(w, d, h, idx, wg, bg, cg, rep_iters):
    r = oracle.compact_head_variant(d["Q"][h], d["K"][h], d["V"][h], w.t, w.softmax_scale)
    if not np.array_equal(idx, r["idx"]):
        tau = np.sort(r["u"])[::-1][w.t - 1]
        diff = np.setxor1d(idx, r["idx"])
        assert np.all(np.abs(r["u"][diff] - tau) <= SCORE_ABS), f"head {h}: selection differs"
        return False
    lo, hi = np.exp(-3.0), np.exp(3.0)
    assert np.all(wg >= lo * (1 - 1e-6)) and np.all(wg <= hi * (1 + 1e-6))
    assert relf(wg, r["w"]) <= FIT_REL, f"head {h} w relF {relf(wg, r['w']):.2e}"
    assert beta_err(bg, r["beta"]) <= FIT_REL, f"head {h} beta"
    assert relf(cg, r["Cv"]) <= FIT_REL, f"head {h} Cv relF {relf(cg, r['Cv']):.2e}"
    assert rep_iters == r["iters"], f"head {h}: {rep_iters} iterations vs {r['iters']}"
    return True


def _run(comp, w, heads=None):
    d, Q, K, V = inputs(w)
    idx, wg, bg, cg = (host(x) for x in comp.compact_layer_baseline(Q, K, V, w.t))
    rep = comp.report(w.H)
    assert rep.device_error_bits == 0
    full = 0
    for h in (range(w.H) if heads is None else heads):
        assert rep.head_status[h] == 0, rep.head_status
        full += _check(w, d, h, idx[h], wg[h], bg[h], cg[h], rep.nnls_iters[h])
    return full


@pytest.mark.parametrize("name", list(CASES))
def test_baseline_small(comp, name):
    assert _run(comp, CASES[name]) >= 1


def test_baseline_full_size_layer(comp):
    """The 8-head T = 4096, n_q = 16384 layer, heads 0 and 3."""
    assert _run(comp, synth.workload("cfg2"), heads=(0, 3)) >= 1


def test_baseline_keeps_every_key(comp):
    """t = T: every key is kept and the compacted cache reproduces the full
    one: for every query the compact log mass matches lse and the compact
    output matches O (w itself is only determined up to the conditioning of
    the T x T mass system in fp32)."""
    w = synth.workload("cfg2", H=1, T=200, G=2, t=200, seed=21)
    d, Q, K, V = inputs(w)
    idx, wg, bg, cg = (host(x) for x in comp.compact_layer_baseline(Q, K, V, w.t))
    assert np.array_equal(idx[0], np.arange(w.T))
    s = w.softmax_scale
    _, lse, O = oracle.full_stats(d["Q"][0], d["K"][0], d["V"][0], s)
    logits = s * (d["Q"][0].astype(np.float64) @ d["K"][0].astype(np.float64).T) + bg[0][None, :]
    mx = logits.max(axis=1)
    mass = mx + np.log(np.exp(logits - mx[:, None]).sum(axis=1))
    assert np.max(np.abs(mass - lse)) <= LSE_ABS
    X = oracle.compact_weights(d["Q"][0], d["K"][0], bg[0], s)
    assert relf(X @ cg[0], O) <= O_REL
