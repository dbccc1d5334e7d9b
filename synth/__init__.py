"""Seeded synthetic inputs for attention-matching layer compaction.

This module only draws random numbers and rounds them to the storage type.
It contains none of the compaction arithmetic: both the CUDA path (through
the tests and the benchmark) and the float64 oracle read their inputs from
here, and neither imports the other.

Workload shapes follow the settings on the pages: grouped-query attention with
``G`` query heads sharing each of ``H`` KV heads, head dimension ``d``, ``T``
cached positions and context-prefill reference queries, ``n_q = G*T`` per KV
head ("KV compaction", section "The Problem with Attention Matching": the
reference queries come from re-running the context through the model).  No
model or dataset is available, so the values are synthetic:

* ``iid``     -- Q, K, V iid N(0, 1).
* ``peaked``  -- keys N(0, 1) with 4 outlier channels per head scaled by 8;
  each query row is 0.5 * (a uniformly drawn key of the same head) plus
  N(0, 1) noise, so attention is peaked; values N(0, 1).
* ``needles`` -- ``peaked`` plus planted needle keys: for each of ``n`` distinct
  (key position, query row) pairs the key is moved along its query so that the
  query's logit on it exceeds its best other logit by a fixed margin.

Query layout per KV head is ``[G*T, d]`` with row ``g*T + p`` holding query
head ``g`` at position ``p`` (queries are iid, so this only fixes naming).
bf16 workloads are rounded to bfloat16 with round-to-nearest-even before
either side sees them; arrays are returned as float32 holding those exact
values (``bf16_bits`` gives the 16-bit patterns for device upload).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "make", "bf16_round", "bf16_bits",
    "tie_heavy_scores", "continuous_scores", "workload",
]


@dataclass(frozen=True)
class Workload:
    name: str
    H: int          # KV heads
    G: int          # query heads per KV head (GQA group)
    T: int          # cached positions per head
    d: int          # head dimension
    t: int          # keys kept per head
    dtype: str      # "bf16" or "fp32": storage type of Q, K, V
    seed: int
    kind: str       # "iid" | "peaked"
    needles: int = 0
    needle_margin: float = 6.0
    n_q_override: int = 0      # 0 -> G*T
    layers: int = 1            # >1: a model of identically shaped layers
    scale: float = 0.0         # 0 -> 1/sqrt(d)

    @property
    def n_q(self) -> int:
        return self.n_q_override if self.n_q_override > 0 else self.G * self.T

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0 else 1.0 / math.sqrt(self.d)

    def layer(self, l: int) -> "Workload":
        """The ``l``-th layer of a multi-layer workload: same shape, own seed."""
        return replace(self, name=f"{self.name}.L{l}", seed=self.seed + l, layers=1)


# The five settings: single-head fp32 sanity case; Qwen3-8B-like GQA layer at
# T=4096; the headline layer at T=8192; a 36-layer model of headline layers;
# long context with needles.
WORKLOADS = {
    "cfg1": Workload("cfg1", H=1, G=1, T=512, d=64, t=32, dtype="fp32", seed=101, kind="iid"),
    "cfg2": Workload("cfg2", H=8, G=4, T=4096, d=128, t=128, dtype="bf16", seed=201, kind="peaked"),
    "cfg3": Workload("cfg3", H=8, G=4, T=8192, d=128, t=256, dtype="bf16", seed=301, kind="peaked"),
    "cfg4": Workload("cfg4", H=8, G=4, T=8192, d=128, t=256, dtype="bf16", seed=400, kind="peaked",
                     layers=36),
    "cfg5": Workload("cfg5", H=8, G=4, T=131072, d=128, t=1024, dtype="bf16", seed=501,
                     kind="peaked", needles=64),
}


def workload(name: str, **kw) -> Workload:
    """A named workload, optionally with fields replaced (e.g. smaller T)."""
    w = WORKLOADS[name]
    return replace(w, **kw) if kw else w


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """16-bit bfloat16 patterns of float32 values that are already bf16-exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("array is not bf16-exact; call bf16_round first")
    return (u >> 16).astype(np.uint16)


def _peaked_head(rng: np.random.Generator, T: int, n_q: int, d: int):
    K = rng.standard_normal((T, d), dtype=np.float32)
    ch = rng.choice(d, size=min(4, d), replace=False)
    K[:, ch] *= 8.0
    src = rng.integers(0, T, size=n_q)
    Q = 0.5 * K[src] + rng.standard_normal((n_q, d), dtype=np.float32)
    V = rng.standard_normal((T, d), dtype=np.float32)
    return Q, K, V


def _iid_head(rng: np.random.Generator, T: int, n_q: int, d: int):
    Q = rng.standard_normal((n_q, d), dtype=np.float32)
    K = rng.standard_normal((T, d), dtype=np.float32)
    V = rng.standard_normal((T, d), dtype=np.float32)
    return Q, K, V


def _needle_sites(rng, T, n_q, n):
    pos = rng.choice(T, size=n, replace=False)
    rows = rng.choice(n_q, size=n, replace=False)
    return pos.astype(np.int64), rows.astype(np.int64)


def _plant_needles(Q, K, pos, rows, margin, s, rnd):
    """Move the keys at ``pos`` so that query row ``rows[i]`` has a logit on key
    ``pos[i]`` that beats its best other logit by ``margin``: a closed-form shift
    of the key along the query direction, which leaves every other logit of that
    query unchanged.  Needles are planted in order; returns the margins
    re-measured after storage rounding and after all needles are in place."""
    K64 = K.astype(np.float64)
    Q64 = Q[rows].astype(np.float64)
    for i, p in enumerate(pos):
        q = Q64[i]
        logits = s * (K64 @ q)
        logits[p] = -np.inf
        best = logits.max()
        k = K64[p]
        k = k + ((best + margin) / s - q @ k) / (q @ q) * q
        K[p] = rnd(k.astype(np.float32)[None])[0]
        K64[p] = K[p]
    got = []
    for i, p in enumerate(pos):
        logits = s * (K64 @ Q64[i])
        own = logits[p]
        logits[p] = -np.inf
        got.append(own - logits.max())
    return np.array(got)


def make(w: Workload, heads=None):
    """Draw one layer of ``w``.

    Returns a dict with float32 arrays ``Q [h, n_q, d]``, ``K [h, T, d]``,
    ``V [h, T, d]`` (bf16-exact for bf16 workloads) for the requested heads
    (default all), and for needle workloads ``needle_pos``, ``needle_rows`` and
    ``needle_margin`` per head.  Heads are drawn in order from one PCG64 stream
    seeded with ``w.seed``, so a subset of heads equals the same heads of the
    full draw.
    """
    if w.layers != 1:
        raise ValueError("draw multi-layer workloads one layer at a time with w.layer(l)")
    heads = list(range(w.H)) if heads is None else list(heads)
    rng = np.random.Generator(np.random.PCG64(w.seed))
    rnd = bf16_round if w.dtype == "bf16" else (lambda a: np.asarray(a, np.float32))
    out = {"Q": [], "K": [], "V": [], "needle_pos": [], "needle_rows": [], "needle_margin": []}
    for h in range(max(heads) + 1):
        gen = _peaked_head if w.kind == "peaked" else _iid_head
        Q, K, V = gen(rng, w.T, w.n_q, w.d)
        Q, K, V = rnd(Q), rnd(K), rnd(V)
        if w.needles:
            npos, nrows = _needle_sites(rng, w.T, w.n_q, w.needles)
        if h in heads:
            if w.needles:
                marg = _plant_needles(Q, K, npos, nrows, w.needle_margin, w.softmax_scale, rnd)
            out["Q"].append(Q)
            out["K"].append(K)
            out["V"].append(V)
            if w.needles:
                out["needle_pos"].append(npos)
                out["needle_rows"].append(nrows)
                out["needle_margin"].append(marg)
    res = {k: np.stack(out[k]) for k in ("Q", "K", "V")}
    if w.needles:
        for k in ("needle_pos", "needle_rows", "needle_margin"):
            res[k] = np.stack(out[k])
    return res


def heldout_queries(w: Workload, K: np.ndarray, n: int, seed: int) -> np.ndarray:
    """Held-out queries for the keys K [h, T, d] of a drawn layer, from the
    workload's own query recipe (peaked: 0.5 * a random key of the head plus
    N(0, 1) noise; iid: N(0, 1)) with a separate seed.  -> [h, n, d]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rnd = bf16_round if w.dtype == "bf16" else (lambda a: np.asarray(a, np.float32))
    out = []
    for Kh in np.asarray(K, np.float32):
        if w.kind == "peaked":
            src = rng.integers(0, Kh.shape[0], size=n)
            q = 0.5 * Kh[src] + rng.standard_normal((n, Kh.shape[1]), dtype=np.float32)
        else:
            q = rng.standard_normal((n, Kh.shape[1]), dtype=np.float32)
        out.append(rnd(q))
    return np.stack(out)


def appended_tokens(w: Workload, n_new: int, seed: int):
    """Keys and values of tokens appended after compaction (question and
    generated tokens), N(0, 1), bf16-exact for bf16 workloads.
    -> (K_new, V_new), each [H, n_new, d]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rnd = bf16_round if w.dtype == "bf16" else (lambda a: np.asarray(a, np.float32))
    Kn = rnd(rng.standard_normal((w.H, n_new, w.d), dtype=np.float32))
    Vn = rnd(rng.standard_normal((w.H, n_new, w.d), dtype=np.float32))
    return Kn, Vn


def tie_heavy_scores(n_heads: int, T: int, seed: int, levels=(0.0, -1.0, -2.0)) -> np.ndarray:
    """Score arrays whose values come from a small set, so many keys tie."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.asarray(rng.choice(np.asarray(levels, np.float32), size=(n_heads, T)), np.float32)


def continuous_scores(n_heads: int, T: int, seed: int) -> np.ndarray:
    """Log-probability-like score arrays (all <= 0), with an exact duplicate and
    a negative zero planted in each row to exercise tie and sign handling."""
    rng = np.random.Generator(np.random.PCG64(seed))
    u = -np.abs(rng.standard_normal((n_heads, T)).astype(np.float32)) * 4.0
    if T >= 4:
        u[:, T // 2] = u[:, T // 3]
        u[:, 1] = np.float32(-0.0)
        u[:, 2] = np.float32(0.0)
    return u
