"""Write ``cfg5_head<h>.npz``: the float64 oracle's compaction of head h of the
long-context workload (131072 cached keys, 524288 reference queries, d = 128,
t = 1024, bf16 inputs with 64 planted needles).

Calls only the oracle and the seeded input generator.  One run takes a little
over an hour on 8 host cores (about 75 minutes), which is why the result is
stored rather than recomputed by the GPU test that reads it.  Stored:

* ``u`` (float32): the key scores, log of each key's largest attention
  probability ("Latent Compaction with Test-Time Training" Eq. (6));
* ``idx``, ``w``, ``beta`` and ``Cv`` (float32): the selection and the fitted
  biases and values ("KV compaction" blog, "Fast KV Compaction via Attention
  Matching");
* ``rows``, ``m``, ``lse``: the oracle's row statistics of a seeded sample of
  query rows (every needle row included);
* ``inputs_sha256``: a digest of head 0's bf16 inputs, so that the test can
  tell whether the generator on its machine drew the same layer.

Usage: ``python tests/golden/make_cfg5_head.py [h]`` from the repository root
(h = 0 by default).
"""
from __future__ import annotations

import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

def inputs_digest(d) -> str:
    h = hashlib.sha256()
    for k in ("Q", "K", "V"):
        h.update(synth.bf16_bits(d[k][0]).tobytes())
    return h.hexdigest()


def main(head: int):
    out = os.path.join(HERE, f"cfg5_head{head}.npz")
    w = synth.workload("cfg5")
    d = synth.make(w, heads=[head])
    Q, K, V = d["Q"][0], d["K"][0], d["V"][0]
    t0 = time.time()
    r = oracle.compact_head(Q, K, V, w.t, w.softmax_scale)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([np.asarray(d["needle_rows"][0]),
                                     rng.choice(w.n_q, 448, replace=False)]))
    np.savez_compressed(
        out, u=r["u"].astype(np.float32), idx=r["idx"].astype(np.int32), w=r["w"],
        beta=r["beta"], Cv=r["Cv"].astype(np.float32), rows=rows.astype(np.int64),
        m=r["m"][rows], lse=r["lse"][rows], nnls_status=np.int32(r["nnls"]["status"]),
        ols_status=np.int32(r["ols_status"]), inputs_sha256=np.array(inputs_digest(d)))
    print(f"wrote {out} in {time.time() - t0:.0f} s; NNLS {r['nnls']}, "
          f"{int(np.sum(r['w'] > 0))} positive weights")


if __name__ == "__main__":
    main(int(sys.argv[1]) if len(sys.argv) > 1 else 0)
