"""Parity of the decode-time consumer (attention over a compacted cache plus
appended tokens) and of the held-out error metrics with the float64 oracle.

Every input comes from the seeded generator or from the oracle: the compacted
caches fed to the held-out metrics are the oracle's own compactions.  The
consumer computes in fp32, so its outputs are held to 2e-5 relative Frobenius
(A) and 2e-5 absolute (log Z); the held-out errors to the step-1 gates (log
mass 1e-3 absolute, output 2e-3 relative)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import LSE_ABS, O_REL, compactor, dev, dev_f32, dev_i32, host, relf

pytestmark = pytest.mark.gpu

A_REL = 2e-5
LZ_ABS = 2e-5


@pytest.fixture(scope="module")
def comp():
    return compactor()


def _consumer_case(seed, H, n, t, n_new, d, drop=0.2, causal=True):
    rng = np.random.default_rng(seed)
    w = synth.workload("cfg2", H=H, T=max(t, 1), d=d, t=max(t, 1), seed=seed)
    q = synth.bf16_round(rng.standard_normal((H, n, d)).astype(np.float32))
    Ck = synth.bf16_round(rng.standard_normal((H, t, d)).astype(np.float32))
    Cv = rng.standard_normal((H, t, d)).astype(np.float32)
    beta = rng.normal(0.0, 1.5, size=(H, t)).astype(np.float32)
    beta[rng.random((H, t)) < drop] = -np.inf
    Kn, Vn = synth.appended_tokens(synth.workload("cfg2", H=H, d=d, seed=seed), n_new, seed + 1)
    if causal:
        n_vis = (np.arange(n)[None, :] + rng.integers(0, 3, size=(H, 1))) % (n_new + 1)
    else:
        n_vis = np.full((H, n), n_new)
    return dict(q=q, Ck=Ck, Cv=Cv, beta=beta, Kn=Kn, Vn=Vn, n_vis=n_vis.astype(np.int32),
                scale=w.softmax_scale)


def _check_consumer(comp, c, pass_vis=True):
    H = c["q"].shape[0]
    A, lz = comp.compact_attention(
        dev(c["q"], "bf16"), dev(c["Ck"], "bf16"), dev_f32(c["beta"]), dev_f32(c["Cv"]),
        dev(c["Kn"], "bf16") if c["Kn"].shape[1] else None,
        dev(c["Vn"], "bf16") if c["Kn"].shape[1] else None,
        dev_i32(c["n_vis"]) if pass_vis else None)
    A, lz = host(A), host(lz)
    for h in range(H):
        Ar, lr = oracle.combine_attention(c["q"][h], c["Ck"][h], c["beta"][h], c["Cv"][h],
                                          c["Kn"][h], c["Vn"][h], c["n_vis"][h], c["scale"])
        fin = np.isfinite(lr)
        assert np.array_equal(np.isfinite(lz[h]), fin), f"head {h}: empty rows differ"
        assert np.all(A[h][~fin] == 0)
        if fin.any():
            assert np.max(np.abs(lz[h][fin] - lr[fin])) <= LZ_ABS, f"head {h} log Z"
            assert relf(A[h][fin], Ar[fin]) <= A_REL, f"head {h} A {relf(A[h][fin], Ar[fin]):.2e}"


@pytest.mark.parametrize("d", [64, 128])
def test_consumer_causal_ragged(comp, d):
    """Ragged rows, compacted size and appended count (none a tile multiple),
    dropped entries, a causal count per row (some rows see no appended
    token)."""
    _check_consumer(comp, _consumer_case(61 + d, 2, 45, 37, 50, d))


def test_consumer_no_appended_tokens(comp):
    c = _consumer_case(62, 3, 70, 256, 0, 128, causal=False)
    _check_consumer(comp, c, pass_vis=False)


def test_consumer_all_appended_visible(comp):
    c = _consumer_case(63, 1, 33, 64, 96, 128, causal=False)
    _check_consumer(comp, c, pass_vis=False)


def test_consumer_empty_rows(comp):
    """Every compacted entry dropped and row 0 sees no appended token."""
    c = _consumer_case(64, 1, 8, 5, 4, 64, drop=1.0)
    c["n_vis"][0, 0] = 0
    _check_consumer(comp, c)


def test_consumer_identity_compaction_is_full_attention(comp):
    """C_k = K, beta = 0, C_v = V and no appended token: the consumer's output
    and log Z are the full cache's (step 1 of the library on the same keys)."""
    w = synth.workload("cfg2", H=2, T=300, t=300, seed=65)
    d = synth.make(w)
    Q, K, V = (dev(d[k], "bf16") for k in ("Q", "K", "V"))
    m, lse, O = comp.full_attn_stats(Q, K, V)
    A, lz = comp.compact_attention(Q, K, dev_f32(np.zeros((w.H, w.T))), dev_f32(d["V"]))
    assert np.max(np.abs(host(lz) - host(lse))) <= LSE_ABS
    assert relf(host(A), host(O)) <= O_REL


def _heldout_check(comp, w, res, n_h, seed):
    d = synth.make(w)
    Qh = synth.heldout_queries(w, d["K"], n_h, seed)
    idx = np.stack([r["idx"] for r in res]).astype(np.int32)
    beta = np.stack([r["beta"] for r in res]).astype(np.float32)
    Cv = np.stack([r["Cv"] for r in res]).astype(np.float32)
    me, oe = comp.heldout_errors(dev(Qh, w.dtype), dev(d["K"], w.dtype), dev(d["V"], w.dtype),
                                 dev_i32(idx), dev_f32(beta), dev_f32(Cv))
    me, oe = host(me), host(oe)
    rep = comp.report(w.H)
    assert rep.device_error_bits == 0
    for h in range(w.H):
        mr, orr = oracle.heldout_errors(Qh[h], d["K"][h], d["V"][h], d["K"][h][idx[h]],
                                        beta[h], Cv[h].astype(np.float64), w.softmax_scale)
        assert abs(me[h] - mr) <= LSE_ABS, f"head {h}: mass error {me[h]} vs {mr}"
        assert abs(oe[h] - orr) <= O_REL * max(orr, 1e-3) + 1e-5, f"head {h}: output error"
    return me, oe


def test_heldout_errors_am_compaction(comp):
    """Held-out errors of the oracle's attention-matching compaction of a
    small layer (2 heads, T = 1024, t = 128), 700 held-out queries."""
    w = synth.workload("cfg2", H=2, T=1024, t=128, seed=66)
    d = synth.make(w)
    res = oracle.compact_layer(d["Q"], d["K"], d["V"], w.t, w.softmax_scale)
    _heldout_check(comp, w, res, 700, 1066)


def test_heldout_errors_fast_compaction_full_size(comp):
    """The benchmark layer (8 heads, T = 8192, t = 256) compacted by the
    oracle's fast path (256-query subsets, k = 4); 4096 held-out queries per
    head."""
    w = synth.workload("cfg3")
    d = synth.make(w)
    rng = np.random.default_rng(67)
    res = [oracle.compact_head_fast(d["Q"][h], d["K"][h], d["V"][h],
                                    rng.choice(w.n_q, 256, replace=False), w.t, 4,
                                    w.softmax_scale) for h in range(w.H)]
    _heldout_check(comp, w, res, 4096, 1067)
