"""The hand-derived worked example in tests/golden/am_worked_4key.txt.

Four keys k_j = j and two queries q_1 = ln 2, q_2 = -2 ln 2 (scale 1) make
every step of attention-matching compaction come out in closed form: log
masses ln 15 and ln(85/64), outputs with denominators 15 and 85, the kept
keys {0, 3}, weights 95/73 and 125/73 and values with denominators 95 and
125.  The two weights differ and the output system is not symmetric, so a
dropped term, a mean in place of the max over queries or a bias on the
wrong key moves some value far beyond float64 rounding (the mass system is
symmetric here, so its transposition is left to the other oracle pins).
The oracle must reproduce them to that rounding; the CUDA path, run in fp32
with the vectors zero-padded to d = 64, must meet the method's tolerances."""
import math
import os

import numpy as np
import pytest

import oracle

FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                       "am_worked_4key.txt")


def load_fixture():
    vals = {}
    for line in open(FIXTURE):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        parts = line.split()
        name = parts[0]
        nidx = {"m": 1, "lse": 1, "u": 1, "idx": 1, "w": 1, "beta": 1, "O": 2, "Cv": 2}[name]
        key = tuple(int(x) for x in parts[1:1 + nidx])
        vals.setdefault(name, {})[key] = float(parts[1 + nidx])
    out = {}
    for name, d in vals.items():
        shape = tuple(max(k[i] for k in d) + 1 for i in range(len(next(iter(d)))))
        a = np.zeros(shape)
        for k, v in d.items():
            a[k] = v
        out[name] = a
    out["idx"] = out["idx"].astype(np.int64)
    return out


def worked_inputs(d=1):
    """Q [2, d], K [4, d], V [4, max(d, 4)] of the worked example (zero-padded)."""
    ln2 = math.log(2.0)
    Q = np.zeros((2, d))
    Q[:, 0] = [ln2, -2.0 * ln2]
    K = np.zeros((4, d))
    K[:, 0] = np.arange(4)
    V = np.zeros((4, max(d, 4)))
    V[:, :4] = np.eye(4)
    return Q, K, V


def test_fixture_is_consistent():
    g = load_fixture()
    # the values are the exact expressions the header derives
    assert np.allclose(g["lse"], [math.log(15), math.log(85 / 64)], rtol=0, atol=1e-15)
    assert np.allclose(g["w"], [95 / 73, 125 / 73], rtol=0, atol=1e-15)
    assert np.allclose(g["beta"], np.log(g["w"]), rtol=0, atol=1e-15)
    assert np.allclose(g["Cv"].sum(axis=1), 1.0, rtol=0, atol=1e-15)
    assert np.allclose(g["O"].sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_oracle_reproduces_the_worked_example():
    g = load_fixture()
    Q, K, V = worked_inputs()
    r = oracle.compact_head(Q, K, V, 2, 1.0)
    assert np.allclose(r["m"], g["m"], rtol=0, atol=1e-14)
    assert np.allclose(r["lse"], g["lse"], rtol=0, atol=1e-14)
    assert np.allclose(r["O"], g["O"], rtol=0, atol=1e-14)
    assert np.allclose(r["u"], g["u"], rtol=0, atol=1e-14)
    assert np.array_equal(np.asarray(r["idx"]), g["idx"])
    assert np.allclose(r["w"], g["w"], rtol=1e-12, atol=0)
    assert np.allclose(r["beta"], g["beta"], rtol=0, atol=1e-12)
    assert np.allclose(r["Cv"], g["Cv"], rtol=0, atol=1e-12)


@pytest.mark.gpu
def test_cuda_path_reproduces_the_worked_example():
    import torch
    from gpu_util import FIT_REL, LSE_ABS, O_REL, SCORE_ABS, beta_err, compactor, relf

    g = load_fixture()
    comp = compactor()
    d = 64  # fp32 inputs run at d = 64
    Q, K, V = (torch.from_numpy(np.ascontiguousarray(a[None], dtype=np.float32)).cuda()
               for a in worked_inputs(d))
    V = V[..., :d].contiguous()
    m, lse, O = comp.full_attn_stats(Q, K, V, scale=1.0)
    u = comp.key_scores(Q, K, lse, scale=1.0)
    idx, w, beta, Cv = comp.compact_layer(Q, K, V, 2, scale=1.0)
    torch.cuda.synchronize()
    assert comp.report(1).device_error_bits == 0
    h = lambda x: x.detach().cpu().numpy()[0].astype(np.float64)
    assert np.max(np.abs(h(m) - g["m"])) <= LSE_ABS
    assert np.max(np.abs(h(lse) - g["lse"])) <= LSE_ABS
    assert relf(h(O)[:, :4], g["O"]) <= O_REL
    assert np.max(np.abs(h(u) - g["u"])) <= SCORE_ABS
    assert np.array_equal(h(idx).astype(np.int64), g["idx"])
    assert relf(h(w), g["w"]) <= FIT_REL
    assert beta_err(h(beta), g["beta"]) <= FIT_REL
    assert relf(h(Cv)[:, :4], g["Cv"]) <= FIT_REL
    assert np.max(np.abs(h(Cv)[:, 4:])) <= 1e-6
