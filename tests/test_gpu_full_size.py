"""Parity at the full sizes of the benchmark configurations, in the launch
configuration the benchmark uses (one compact_layer call over all heads of a
layer).  The oracle recomputes sampled outputs: whole heads where it finishes
in seconds (cfg2 every head, cfg3 and cfg4 sampled heads and layers), single
query rows and properties of the GPU's own outputs where the layer is too
large for a float64 CPU pass (cfg5, 131072 keys).  Every expected value comes
from the generator or the oracle."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (FIT_REL, LSE_ABS, O_REL, SCORE_ABS, beta_err, compactor, dev, dev_f32,
                      dev_i32, host, inputs, relf)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def comp():
    return compactor()


def _check_head(w, d, h, idx, wg, bg, cg, m=None, lse=None):
    """One head of a GPU compaction against the oracle's compaction of it."""
    r = oracle.compact_head(d["Q"][h], d["K"][h], d["V"][h], w.t, w.softmax_scale)
    if lse is not None:
        assert np.max(np.abs(lse - r["lse"])) <= LSE_ABS, f"head {h} lse"
        assert np.max(np.abs(m - r["m"])) <= LSE_ABS, f"head {h} rowmax"
    if not np.array_equal(idx, r["idx"]):
        # only keys whose oracle scores tie within the score tolerance may swap
        tau = np.sort(r["u"])[::-1][w.t - 1]
        diff = np.setxor1d(idx, r["idx"])
        assert np.all(np.abs(r["u"][diff] - tau) <= SCORE_ABS), f"head {h}: selection differs"
        return
    assert relf(wg, r["w"]) <= FIT_REL, f"head {h} w relF {relf(wg, r['w']):.2e}"
    assert beta_err(bg, r["beta"]) <= FIT_REL, f"head {h} beta {beta_err(bg, r['beta']):.2e}"
    assert relf(cg, r["Cv"]) <= FIT_REL, f"head {h} Cv relF {relf(cg, r['Cv']):.2e}"


def _layer(comp, w, heads_checked, with_stats=True):
    d, Q, K, V = inputs(w)
    stats = None
    if with_stats:
        m, lse, _ = comp.full_attn_stats(Q, K, V)
        stats = (host(m), host(lse))
    idx, wg, bg, cg = (host(x) for x in comp.compact_layer(Q, K, V, w.t))
    rep = comp.report(w.H)
    assert rep.device_error_bits == 0
    assert all(s == 0 for s in rep.head_status), rep.head_status
    for h in heads_checked:
        kw = {} if stats is None else {"m": stats[0][h], "lse": stats[1][h]}
        _check_head(w, d, h, idx[h], wg[h], bg[h], cg[h], **kw)


def test_cfg2_full_layer_every_head(comp):
    """Qwen3-8B-like layer: 8 KV heads, T = 4096, n_q = 16384, t = 128."""
    w = synth.workload("cfg2")
    _layer(comp, w, range(w.H))


def test_cfg3_layer_sampled_heads(comp):
    """The benchmark layer (T = 8192, n_q = 32768, t = 256), heads 0 and 5."""
    _layer(comp, synth.workload("cfg3"), (0, 5))


@pytest.mark.parametrize("layer", [0, 35])
def test_cfg4_sampled_layers(comp, layer):
    """Layers of the 36-layer sweep (per-layer seeds), one sampled head each."""
    w = synth.workload("cfg4").layer(layer)
    _layer(comp, w, (3,), with_stats=False)


CFG5_HEADS = 2  # heads 0 and 1 of the layer (a prefix of the full draw)


@pytest.fixture(scope="module")
def cfg5(comp):
    w = synth.workload("cfg5", H=CFG5_HEADS)
    d, Q, K, V = inputs(w)
    m, lse, O = comp.full_attn_stats(Q, K, V)
    out = comp.compact_layer(Q, K, V, w.t)
    rep = comp.report(w.H)
    u = comp.key_scores(Q, K, lse)
    idx_u = comp.select_topt(u, w.t)
    return {"w": w, "d": d, "m": host(m), "lse": host(lse), "O": host(O),
            "out": [host(x) for x in out], "rep": rep, "idx_u": host(idx_u), "u": host(u)}


def test_cfg5_sampled_rows(cfg5):
    """Long context (T = 131072, n_q = 524288): m, lse and O of sampled query
    rows -- every needle row and a seeded sample of the rest -- recomputed by
    the oracle over all 131072 keys."""
    w, d = cfg5["w"], cfg5["d"]
    rng = np.random.default_rng(5)
    for h in range(w.H):
        rows = np.unique(np.concatenate([np.asarray(d["needle_rows"][h]),
                                         rng.choice(w.n_q, 32, replace=False)]))
        m, lse, O = oracle.full_stats(d["Q"][h][rows], d["K"][h], d["V"][h], w.softmax_scale)
        assert np.max(np.abs(cfg5["lse"][h][rows] - lse)) <= LSE_ABS, f"head {h} lse"
        assert np.max(np.abs(cfg5["m"][h][rows] - m)) <= LSE_ABS, f"head {h} rowmax"
        assert relf(cfg5["O"][h][rows], O) <= O_REL, f"head {h} O"


def test_cfg5_layer_properties(cfg5):
    """Properties of the full-size compaction that hold at any size: the
    selection is the exact top-t of the layer's own score array (ties to the
    lower index), every key score is a log-probability (<= 0 up to rounding)
    and at least the best needle pairing's value, the NNLS converged with
    w >= 0 and beta = log w, and every output is finite."""
    w, d = cfg5["w"], cfg5["d"]
    idx, wg, bg, cg = cfg5["out"]
    rep = cfg5["rep"]
    assert rep.device_error_bits == 0
    assert all(s == 0 for s in rep.head_status), rep.head_status
    assert np.array_equal(idx, cfg5["idx_u"])
    for h in range(w.H):
        u = cfg5["u"][h]
        assert np.all(u <= SCORE_ABS)
        # lower bound at each needle key: its paired row's log-probability,
        # from the oracle's own statistics of that row
        pos = np.asarray(d["needle_pos"][h])
        rows = np.asarray(d["needle_rows"][h])
        _, lse_r, _ = oracle.full_stats(d["Q"][h][rows], d["K"][h], d["V"][h], w.softmax_scale)
        s = w.softmax_scale * np.einsum("nd,nd->n", d["Q"][h][rows].astype(np.float64),
                                        d["K"][h][pos].astype(np.float64))
        assert np.all(u[pos] >= s - lse_r - SCORE_ABS)
        assert np.all(np.diff(idx[h]) > 0)
        assert np.all(wg[h] >= 0) and np.all(np.isfinite(wg[h]))
        pos_w = wg[h] > 0
        assert np.allclose(bg[h][pos_w], np.log(wg[h][pos_w]), rtol=0, atol=1e-5)
        assert np.all(np.isneginf(bg[h][~pos_w]))
        assert np.all(np.isfinite(cg[h]))


def test_cfg5_fit_t1024(comp):
    """The 1024 x 1024 NNLS and OLS of the long-context configuration against
    the oracle: head 0 of cfg5 at full T, a seeded sample of 2048 query rows
    (every needle row included), the oracle's own top-1024 keys for those rows;
    m, lse and O of the rows from the oracle over all 131072 keys."""
    w = synth.workload("cfg5", H=1)
    d = synth.make(w)
    rng = np.random.default_rng(6)
    needle_rows = np.asarray(d["needle_rows"][0])
    rest = np.setdiff1d(np.arange(w.n_q), needle_rows)
    rows = np.sort(np.concatenate([needle_rows,
                                   rng.choice(rest, 2048 - needle_rows.size, replace=False)]))
    Qs, K, V = d["Q"][0][rows], d["K"][0], d["V"][0]
    m, lse, O = oracle.full_stats(Qs, K, V, w.softmax_scale)
    idx = oracle.select(oracle.key_scores(Qs, K, lse, w.softmax_scale), w.t)
    r = oracle.fit_head(Qs, K, V, idx, m, lse, O, w.softmax_scale)
    wg, bg, cg = comp.fit_only(dev(Qs[None], w.dtype), dev(K[None], w.dtype), dev(V[None], w.dtype),
                               dev_i32(idx[None]), dev_f32(m[None]), dev_f32(lse[None]),
                               dev_f32(O[None]))
    rep = comp.report(1)
    assert rep.device_error_bits == 0 and rep.head_status[0] == 0, rep
    wg, bg, cg = host(wg)[0], host(bg)[0], host(cg)[0]
    assert relf(wg, r["w"]) <= FIT_REL, f"w relF {relf(wg, r['w']):.2e}"
    assert beta_err(bg, r["beta"]) <= FIT_REL, f"beta {beta_err(bg, r['beta']):.2e}"
    assert relf(cg, r["Cv"]) <= FIT_REL, f"Cv relF {relf(cg, r['Cv']):.2e}"
