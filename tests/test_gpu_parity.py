"""Parity of the CUDA path (through the C ABI) with the float64 oracle on the
same seeded inputs.  Every oracle input comes from the generator or from the
oracle itself, never from the GPU."""
import math

import numpy as np
import pytest

import oracle
import synth
from gpu_util import (FIT_REL, LSE_ABS, O_REL, SCORE_ABS, beta_err, check_layer_fits,
                      compactor, dev, dev_f32, dev_i32, host, inputs, relf, torch)

pytestmark = pytest.mark.gpu

# Small cases the oracle finishes in seconds; they span several tiles and end
# in ragged tails (T, n_q and t not multiples of the tile sizes).
CASES = {
    "cfg1_fp32_d64": synth.workload("cfg1"),
    "bf16_d128_ragged": synth.workload("cfg2", H=2, T=300, t=20, seed=7),
    "bf16_d64_ragged": synth.workload("cfg2", H=2, T=257, d=64, t=33, seed=8),
    "bf16_tiny": synth.workload("cfg2", H=1, G=1, T=5, t=3, seed=9),
    "bf16_t_over_128": synth.workload("cfg2", H=2, T=700, G=2, t=160, seed=10),
    "bf16_iid_d128": synth.workload("cfg2", H=1, T=640, G=2, t=64, kind="iid", seed=11),
    "bf16_t256": synth.workload("cfg2", H=2, T=1024, G=4, t=256, seed=12),
    "bf16_t300_ragged": synth.workload("cfg2", H=1, T=1100, G=3, t=300, seed=13),
    # edge cases: a single kept key, a single cached key (t = T = 1), the
    # fp32 path at ragged sizes, more than half the keys kept over several tiles
    "bf16_t1": synth.workload("cfg2", H=2, T=200, G=1, t=1, seed=14),
    "bf16_T1": synth.workload("cfg2", H=1, T=1, G=2, t=1, seed=15),
    "fp32_ragged": synth.workload("cfg1", T=300, t=17, G=1, seed=16),
    "bf16_split_p_ragged": synth.workload("cfg2", H=1, T=130, G=2, t=100, seed=17),
}


@pytest.fixture(scope="module")
def comp():
    return compactor()


_oracle_cache = {}


def oracle_run(name):
    if name not in _oracle_cache:
        w = CASES[name]
        d = synth.make(w)
        res = oracle.compact_layer(d["Q"], d["K"], d["V"], w.t, w.softmax_scale)
        _oracle_cache[name] = (d, res)
    return _oracle_cache[name]


@pytest.mark.parametrize("name", list(CASES))
def test_full_attn_stats(comp, name):
    w = CASES[name]
    d, res = oracle_run(name)
    Q, K, V = dev(d["Q"], w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype)
    m, lse, O = comp.full_attn_stats(Q, K, V)
    m, lse, O = host(m), host(lse), host(O)
    for h, r in enumerate(res):
        assert np.max(np.abs(lse[h] - r["lse"])) <= LSE_ABS, f"head {h} lse"
        assert np.max(np.abs(m[h] - r["m"])) <= LSE_ABS, f"head {h} rowmax"
        assert relf(O[h], r["O"]) <= O_REL, f"head {h} O relF {relf(O[h], r['O']):.2e}"


@pytest.mark.parametrize("name", list(CASES))
def test_key_scores(comp, name):
    w = CASES[name]
    d, res = oracle_run(name)
    Q, K = dev(d["Q"], w.dtype), dev(d["K"], w.dtype)
    lse = dev_f32(np.stack([r["lse"] for r in res]))
    u = host(comp.key_scores(Q, K, lse))
    for h, r in enumerate(res):
        err = np.max(np.abs(u[h] - r["u"]))
        assert err <= SCORE_ABS, f"head {h}: max |u_gpu - u| = {err:.2e}"


SELECT_CASES = [
    ("continuous", lambda: synth.continuous_scores(4, 8192, 1), [1, 7, 256, 8192]),
    ("ties", lambda: synth.tie_heavy_scores(3, 1000, 2), [1, 100, 333, 999, 1000]),
    ("signed_zero", lambda: synth.tie_heavy_scores(2, 300, 3, levels=(0.0, -0.0, -1.0)), [5, 150]),
    ("long", lambda: synth.continuous_scores(2, 131072, 4), [1024]),
    ("single", lambda: synth.continuous_scores(1, 1, 5), [1]),
    # long heads take the sampled-threshold path; these cases drive its
    # branches: candidates found (several t, 2^20 keys), too many
    # candidates (ties everywhere), too few (the high scores sit exactly at
    # the sampled positions, so the sample overestimates the threshold)
    ("wide_continuous", lambda: synth.continuous_scores(3, 1 << 20, 6), [1, 100, 1024]),
    ("wide_ties", lambda: synth.tie_heavy_scores(2, 131072, 7), [1, 1024]),
    ("wide_sample_misjudged", lambda: _sampled_positions_high(2, 131072), [1024]),
]


def _sampled_positions_high(n_heads, T, stride=8):
    """Scores 0 except at every stride-th key, where they rise with the key:
    a strided sample sees only the high values."""
    u = np.zeros((n_heads, T), np.float32)
    u[:, ::stride] = 1.0 + 1e-3 * np.arange(T // stride, dtype=np.float32)
    return u


@pytest.mark.parametrize("case", SELECT_CASES, ids=lambda c: c[0])
def test_select_bit_exact(comp, case):
    _, make, ts = case
    u = make().astype(np.float32)
    ud = dev_f32(u)
    for t in ts:
        idx = host(comp.select_topt(ud, t))
        for h in range(u.shape[0]):
            ref = oracle.select(u[h], t)
            assert np.array_equal(idx[h], ref), f"t={t} head {h}"


def _fit_ref(d, res, w):
    """Oracle fit on the oracle's own selection."""
    return [oracle.fit_head(d["Q"][h], d["K"][h], d["V"][h], r["idx"], r["m"], r["lse"], r["O"],
                            w.softmax_scale) for h, r in enumerate(res)]


@pytest.mark.parametrize("name", list(CASES))
def test_fit_only(comp, name):
    w = CASES[name]
    d, res = oracle_run(name)
    Q, K, V = dev(d["Q"], w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype)
    idx = dev_i32(np.stack([r["idx"] for r in res]))
    m = dev_f32(np.stack([r["m"] for r in res]))
    lse = dev_f32(np.stack([r["lse"] for r in res]))
    O = dev_f32(np.stack([r["O"] for r in res]))
    wg, bg, cg = comp.fit_only(Q, K, V, idx, m, lse, O)
    rep = comp.report(w.H)
    wg, bg, cg = host(wg), host(bg), host(cg)
    for h, r in enumerate(res):
        assert rep.head_status[h] == 0, f"head {h} status {rep.head_status[h]}"
        assert relf(wg[h], r["w"]) <= FIT_REL, f"head {h} w relF {relf(wg[h], r['w']):.2e}"
        assert beta_err(bg[h], r["beta"]) <= FIT_REL, f"head {h} beta {beta_err(bg[h], r['beta']):.2e}"
        assert relf(cg[h], r["Cv"]) <= FIT_REL, f"head {h} Cv relF {relf(cg[h], r['Cv']):.2e}"
    assert rep.device_error_bits == 0


@pytest.mark.parametrize("name", list(CASES))
def test_compact_layer(comp, name):
    w = CASES[name]
    d, res = oracle_run(name)
    Q, K, V = dev(d["Q"], w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype)
    idx, wg, bg, cg = comp.compact_layer(Q, K, V, w.t)
    rep = comp.report(w.H)
    idx, wg, bg, cg = host(idx), host(wg), host(bg), host(cg)
    assert rep.device_error_bits == 0
    check_layer_fits(comp, w, Q, K, V, dict(enumerate(res)), idx, wg, bg, cg)


def test_keep_every_key(comp):
    """t = T: the compact cache is the full cache, w = 1 and C_v = V."""
    w = synth.workload("cfg2", H=2, T=96, G=3, t=96, seed=21)
    d, Q, K, V = inputs(w)
    idx, wg, bg, cg = comp.compact_layer(Q, K, V, w.t)
    idx, wg, cg = host(idx), host(wg), host(cg)
    for h in range(w.H):
        assert np.array_equal(idx[h], np.arange(w.T))
        assert relf(wg[h], np.ones(w.T)) <= FIT_REL
        assert relf(cg[h], d["V"][h]) <= FIT_REL


def test_zero_queries(comp):
    """Queries at q = 0 see every key with probability 1/T (the pages'
    argument for the bias); their lse is log T and their output mean(V)."""
    w = synth.workload("cfg2", H=1, T=200, G=2, t=16, seed=22)
    d = synth.make(w)
    d["Q"][0, ::7] = 0.0
    Q, K, V = dev(d["Q"], w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype)
    m, lse, O = comp.full_attn_stats(Q, K, V)
    lse, O = host(lse), host(O)
    z = np.arange(0, w.n_q, 7)
    assert np.max(np.abs(lse[0, z] - math.log(w.T))) <= LSE_ABS
    assert np.max(np.abs(O[0, z] - d["V"][0].mean(0))) <= 1e-3
    r = oracle.compact_head(d["Q"][0], d["K"][0], d["V"][0], w.t, w.softmax_scale)
    idx, wg, bg, cg = comp.compact_layer(Q, K, V, w.t)
    idx, wg, bg, cg = host(idx)[0], host(wg)[0], host(bg)[0], host(cg)[0]
    if np.array_equal(idx, r["idx"]):
        assert relf(wg, r["w"]) <= FIT_REL
        assert relf(cg, r["Cv"]) <= FIT_REL


def test_nnls_iteration_cap_reported(comp):
    """With the cap at one iteration the NNLS reports LC_ERR_NOT_CONVERGED on a
    head whose unconstrained least-squares solution is infeasible, and every
    output stays finite (beta may be -inf).  The fit runs on the oracle's
    selection so that both sides solve the same problem."""
    w = synth.workload("cfg2", H=2, T=2048, G=4, t=256, seed=23)
    d, Q, K, V = inputs(w)
    r = [oracle.compact_head(d["Q"][h], d["K"][h], d["V"][h], w.t, w.softmax_scale) for h in range(w.H)]
    infeasible = []
    for x in r:
        z = np.linalg.solve(x["G"], x["c"])
        infeasible.append(bool(np.any(z < -1e-3 * np.abs(z).max())))
    assert any(infeasible), "test case has no infeasible head"
    args = (dev_i32(np.stack([x["idx"] for x in r])), dev_f32(np.stack([x["m"] for x in r])),
            dev_f32(np.stack([x["lse"] for x in r])), dev_f32(np.stack([x["O"] for x in r])))
    wg, bg, cg = comp.fit_only(Q, K, V, *args, nnls_max_iter=1)
    rep = comp.report(w.H)
    for h in range(w.H):
        if infeasible[h]:
            assert rep.head_status[h] == 5
        assert np.all(np.isfinite(host(cg)[h])) and np.all(np.isfinite(host(wg)[h]))
    wg, bg, cg = comp.fit_only(Q, K, V, *args)
    rep = comp.report(w.H)
    for h in range(w.H):
        assert rep.head_status[h] == 0
        assert relf(host(wg)[h], r[h]["w"]) <= FIT_REL
        assert relf(host(cg)[h], r[h]["Cv"]) <= FIT_REL


def test_host_entry_matches_device(comp):
    t_ = torch()
    w = CASES["bf16_d128_ragged"]
    d, Q, K, V = inputs(w)
    ref = [host(x) for x in comp.compact_layer(Q, K, V, w.t)]
    out = (t_.empty((w.H, w.t), dtype=t_.int32), t_.empty((w.H, w.t)), t_.empty((w.H, w.t)),
           t_.empty((w.H, w.t, w.d)))
    comp.compact_layer_host(Q.cpu(), K.cpu(), V.cpu(), w.t, out)
    for a, b in zip(out, ref):
        assert np.array_equal(a.numpy(), b)


def test_reruns_are_bitwise_identical(comp):
    """Repeated compactions of the same layer give the same bits: every sum
    on the path runs in a fixed order (no floating-point atomics), including
    the active-set solves of the NNLS, which this two-head slice of the
    benchmark layer reaches (at least one step with active indices)."""
    w = synth.workload("cfg3", H=2)
    _, Q, K, V = inputs(w)
    runs = [[host(x) for x in comp.compact_layer(Q, K, V, w.t)] for _ in range(3)]
    iters = comp.report(w.H).nnls_iters
    assert min(iters) >= 2, iters  # the capacitance-form steps ran
    for other in runs[1:]:
        for x, y in zip(runs[0], other):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
