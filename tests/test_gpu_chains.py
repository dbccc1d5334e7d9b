"""Gram accumulation chains at their edge lengths, through lc_fit_only.

The tensor core's fp32 accumulation truncates, so no Gram accumulator sums
more than 64 query slabs of 64 rows: the per-block kernels keep a running sum
in tensor memory and fold each later chunk into it, and the all-pairs kernel
takes at least ceil(slabs / 64) query splits.  These cases put exactly P
slabs on every CTA of the mass and output Grams (one head, one block of
kept keys: the query range is split 64 ways, so n_q = 64 * 64 * P) and
compare the fit with the oracle's on the same selection (every T/t-th key)
and statistics:

* P = 64: one chunk, nothing folded;
* P = 65: a second chunk of one slab, added at the end;
* P = 129: chunk 1 closed by the last slab but one (bf16 kernel: folded by
  its group after its loop; fp32 kernel: in the loop);
* P = 130, 193: folds in the loop, and for 193 also after the loop;
* a ragged query count whose last CTA has a shorter chain than the others.

The all-pairs kernel (t = 256, bf16) is run where the minimum split decides
the launch (8320 slabs for one head).  Every expected value comes from the
oracle and the generator.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import compactor, dev, dev_f32, dev_i32, gate_fit, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def comp():
    return compactor()


def _fit_case(comp, w):
    d = synth.make(w)
    Q, K, V = d["Q"][0], d["K"][0], d["V"][0]
    s = w.softmax_scale
    m, lse, O = oracle.full_stats(Q, K, V, s)
    idx = np.arange(0, w.T, w.T // w.t)[: w.t].astype(np.int64)  # every other key
    ref = oracle.fit_head(Q, K, V, idx, m, lse, O, s)
    wg, bg, cg = comp.fit_only(dev(Q[None], w.dtype), dev(K[None], w.dtype), dev(V[None], w.dtype),
                               dev_i32(idx[None]), dev_f32(m[None]), dev_f32(lse[None]),
                               dev_f32(O[None]))
    rep = comp.report(1)
    assert rep.device_error_bits == 0 and rep.head_status[0] == 0, rep
    gate_fit(host(wg)[0], host(bg)[0], host(cg)[0], ref, f"{w.name} n_q={w.n_q}")


@pytest.mark.parametrize("P", [64, 65, 129, 130, 193])
def test_bf16_block_kernel_chains(comp, P):
    w = synth.workload("cfg2", H=1, T=256, t=128, n_q_override=64 * 64 * P, seed=700 + P)
    _fit_case(comp, w)


@pytest.mark.parametrize("P", [129, 130])
def test_bf16_block_kernel_chains_d64(comp, P):
    # d = 64: the output system's R blocks fold 64-column accumulators
    w = synth.workload("cfg2", H=1, T=256, d=64, t=128, n_q_override=64 * 64 * P, seed=750 + P)
    _fit_case(comp, w)


@pytest.mark.parametrize("P", [64, 65, 129, 130])
def test_fp32_block_kernel_chains(comp, P):
    # cfg1's own shape and compression (T = 512, t = 32): with iid scores and
    # half of the keys kept the output system is too ill-conditioned for an
    # fp32 fit to meet the tolerance whatever the chain length
    w = synth.workload("cfg1", n_q_override=64 * 64 * P, seed=800 + P)
    _fit_case(comp, w)


@pytest.mark.parametrize("name", ["cfg2", "cfg1"])
def test_ragged_chains(comp, name):
    # n_q = 64 * 64 * 129 + 77: 8258 slabs of 64 rows (the last one partial)
    # split 130 per CTA, so the last CTA sums 68 slabs (one chunk and four
    # slabs) while the others fold two chunks
    kw = {"H": 1, "T": 256, "t": 128} if name == "cfg2" else {}
    w = synth.workload(name, n_q_override=64 * 64 * 129 + 77, seed=950, **kw)
    _fit_case(comp, w)


def test_all_pairs_minimum_split(comp):
    w = synth.workload("cfg3", H=1, T=512, t=256, n_q_override=64 * 8320, seed=901)
    _fit_case(comp, w)
