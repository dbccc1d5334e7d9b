"""The pipelined multi-layer entry point against one compact_layer call per
layer on the same inputs: the same kernels run with the same parameters, so
the selections are identical and the fitted values agree to fp32 rounding
(the solver's order of accumulation may differ); every layer's report is
kept.  The single-layer results themselves are checked against the oracle
by the other parity tests."""
import numpy as np
import pytest

import synth
from gpu_util import compactor, dev, host, relf

pytestmark = pytest.mark.gpu

TIGHT = 1e-5


@pytest.fixture(scope="module")
def comp():
    return compactor()


def _stack(ws):
    ds = [synth.make(w) for w in ws]
    return tuple(dev(np.stack([d[k] for d in ds]), ws[0].dtype) for k in ("Q", "K", "V"))


def _compare(comp, ws):
    Q, K, V = _stack(ws)
    L, H = Q.shape[0], Q.shape[1]
    t = ws[0].t
    idx, w, beta, Cv = (host(x) for x in comp.compact_layers(Q, K, V, t))
    rep = comp.report(L * H)
    assert rep.device_error_bits == 0
    for l in range(L):
        i1, w1, b1, c1 = (host(x) for x in comp.compact_layer(Q[l].contiguous(), K[l].contiguous(),
                                                               V[l].contiguous(), t))
        r1 = comp.report(H)
        assert np.array_equal(idx[l], i1), f"layer {l}: selection differs"
        assert relf(w[l], w1) <= TIGHT and relf(c1, Cv[l]) <= TIGHT, f"layer {l}"
        fin = np.isfinite(b1)
        assert np.array_equal(np.isfinite(beta[l]), fin)
        assert np.max(np.abs(beta[l][fin] - b1[fin]), initial=0.0) <= 1e-4
        assert list(rep.head_status[l * H:(l + 1) * H]) == list(r1.head_status)


def test_three_small_layers(comp):
    _compare(comp, [synth.workload("cfg2", H=2, T=700, G=2, t=160, seed=90 + l) for l in range(3)])


def test_single_layer(comp):
    _compare(comp, [synth.workload("cfg2", H=2, T=300, t=20, seed=7)])


def test_benchmark_layers(comp):
    """Four layers of the 36-layer sweep at full size (cfg4, layers 0-3)."""
    w = synth.workload("cfg4")
    _compare(comp, [w.layer(l) for l in range(4)])


def test_fp32_layers(comp):
    _compare(comp, [synth.workload("cfg1", seed=101 + l) for l in range(2)])
