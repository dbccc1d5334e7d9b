"""The stored oracle compactions of two long-context heads (cfg5: 131072 keys,
524288 queries, t = 1024), checked on the CPU before any GPU run uses them:
the generator still draws the layer they were computed on (input digest);
the stored selection is the oracle's top-t of the stored scores; the stored
weights satisfy beta = log w, w >= 0; and the stored m and lse of sampled
rows equal the oracle's, recomputed over all keys."""
import hashlib
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def layer():
    w = synth.workload("cfg5", H=2)
    return w, synth.make(w)


@pytest.mark.parametrize("h", [0, 1])
def test_stored_cfg5_head(layer, h):
    w, d = layer
    g = np.load(os.path.join(GOLDEN, f"cfg5_head{h}.npz"))
    dig = hashlib.sha256()
    for k in ("Q", "K", "V"):
        dig.update(synth.bf16_bits(d[k][h]).tobytes())
    assert dig.hexdigest() == str(g["inputs_sha256"]), "the generator draws another layer"
    assert int(g["nnls_status"]) == oracle.OK and int(g["ols_status"]) == oracle.OK
    assert g["u"].shape == (w.T,) and g["idx"].shape == (w.t,)
    assert np.array_equal(g["idx"], oracle.select(g["u"], w.t))
    wv, beta = g["w"], g["beta"]
    assert np.all(wv >= 0)
    pos = wv > 0
    assert np.array_equal(beta[pos], np.log(wv[pos])) and np.all(np.isneginf(beta[~pos]))
    assert g["Cv"].shape == (w.t, w.d) and np.all(np.isfinite(g["Cv"]))
    rows = g["rows"][:: max(1, g["rows"].size // 16)]
    sel = np.searchsorted(g["rows"], rows)
    m, lse, _ = oracle.full_stats(d["Q"][h][rows], d["K"][h], d["V"][h], w.softmax_scale)
    assert np.allclose(m, g["m"][sel], rtol=1e-12, atol=0)
    assert np.allclose(lse, g["lse"][sel], rtol=1e-12, atol=0)
