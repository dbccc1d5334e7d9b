"""Float64 CPU oracle for attention-matching compaction of one layer's KV cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
leg of the benchmark may import this package.  The library never calls it and
shares no code with it; the two meet only in the seeded input generator
(``synth``), which holds none of the method's arithmetic.

Every function works in float64 on the exact values of its (bf16- or
fp32-valued) inputs, in query-row chunks of at most ``CHUNK`` rows so that the
score matrix never has to be held whole.  Chunking only regroups the sums over
query rows; nothing else is blocked, fused or reordered.

Sources (page title, then section / equation):

* [LC]  "Latent Compaction with Test-Time Training" -- §3 Preliminaries Eq. (1)
  (attention output and normaliser, scale s = 1/sqrt(d)); §3.1 Eq. (2)-(3)
  (biased compact attention: logits s*K_cmp q + b, output V_cmp^T softmax);
  §3.2 Eq. (6) (key score: max over reference queries of the softmax
  probability); Appendix A.2 "Normalizer Computation and Storage".
* [KVC] "KV compaction" (bkal01 blog) -- section "Fast KV Compaction via
  Attention Matching": output- and mass-matching equations, the q = 0 argument
  for beta, the three steps (top keys by attention, beta by NNLS on the mass
  equation, C_v by OLS on the output equation), C_k a subset of K; sections
  "Attempt #3: Two-Pass", "Choosing beta", "Choosing C_v" (fast path,
  held-out errors).
* [LC] §3.1 "Handling Subsequent Tokens" Eq. (4)-(5) and Appendix A.2
  (decode-time consumer); §3.2 Eq. (7) (farthest-first diversifiers);
  Appendix A.3 (the Attention Matching baseline: RMS attention key
  selection, two bounded NNLS iterations with bounds [e^-3, e^3]).

Readings taken where the pages leave a step open (each is also listed in the
design notes):

* All reference queries see all T keys (no causal mask).
* The key score is reduced with max (Eq. 6), in the log domain:
  u_j = max_i (S_ij - lse_i) = log a_j.
* Top-t ties go to the lower key index; -0 counts as +0; output ascending.
* NNLS is solved in per-query max-shifted form: A_ij = exp(S_C,ij - m_i),
  b_i = exp(lse_i - m_i) with m_i the full-row max of S; w = exp(beta) >= 0 is
  unbounded above; Lawson-Hanson with tolerance 10*eps*t*max|c|, at most 3t
  outer steps and t inner steps per outer step.
* The OLS design matrix is the compact softmax X = softmax_j(s q.C_kj + beta_j)
  over the keys with w_j > 0; C_v = (X^T X)^-1 X^T O by Cholesky; keys with
  w_j = 0 keep their original value row.
* Singular systems (the pages give no ridge): when a Cholesky factorisation
  of an n x n system breaks down, a ridge of n * 2^-20 * mean(diag) is added
  once and the status says so.  The size scaling is what lets the same rule
  work in single precision: on a rank-deficient system the rounding errors
  of a factorisation add up coherently to about n unit roundoffs of the
  diagonal, which the ridge must exceed.
* A kept key whose vector equals that of a kept key at an earlier position
  has w = 0: its column of A equals the earlier one's, so the NNLS minimiser
  is not unique, and this is the one Lawson-Hanson reaches with argmax ties
  going to the lower index (the later copy never enters the passive set).

* Decode consumer: row r of the queries sees the compacted entries whose
  beta is finite and the first n_vis[r] appended tokens (a causal mask given
  as a count per row); a row that sees nothing has log Z = -inf and output 0.
* Held-out errors: mass error = mean over held-out queries of
  |log Z_cmp - log Z_full|, output error = mean of ||A_cmp - A_full||_2.
* Farthest-first ties go to the lower key index.
* Baseline variant: the RMS is over the group's reference queries; a bounded
  iteration solves over the free weights with the pinned ones at their
  bounds, then pins every free weight outside [lo, hi] at the bound it
  crossed; two iterations from all-free, stopping early if nothing is pinned.

Parity is pinned for every function here by the CPU tests (brute force on tiny
inputs, closed forms, library cross-checks, invariants); see tests/.
"""
from __future__ import annotations

import numpy as np

try:  # scipy is a convenience for triangular solves; numpy alone also works
    from scipy.linalg import solve_triangular as _solve_tri
except Exception:  # pragma: no cover
    _solve_tri = None

CHUNK = 2048

# Status codes, numerically equal to the library's, so that reports compare.
OK = 0
NOT_CONVERGED = 5
SINGULAR = 6


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _chunks(n, size=CHUNK):
    for a in range(0, n, size):
        yield a, min(n, a + size)


# ---------------------------------------------------------------- step 1 ----
def full_stats(Q, K, V, scale):
    """Full-cache statistics of every reference query ([LC] Eq. 1).

    S = scale * Q K^T; m_i = max_j S_ij; lse_i = log sum_j exp(S_ij) (the log
    attention mass, computed as m_i + log sum_j exp(S_ij - m_i));
    O_i = sum_j exp(S_ij - lse_i) V_j (the attention output).
    Q [n_q, d], K [T, d], V [T, d_v] -> m [n_q], lse [n_q], O [n_q, d_v].
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    n_q = Q.shape[0]
    m = np.empty(n_q)
    lse = np.empty(n_q)
    O = np.empty((n_q, V.shape[1]))
    for a, b in _chunks(n_q):
        S = scale * (Q[a:b] @ K.T)
        mm = S.max(axis=1)
        ls = mm + np.log(np.exp(S - mm[:, None]).sum(axis=1))
        P = np.exp(S - ls[:, None])
        m[a:b] = mm
        lse[a:b] = ls
        O[a:b] = P @ V
    return m, lse, O


# ---------------------------------------------------------------- step 2 ----
def key_scores(Q, K, lse, scale):
    """Log of each key's maximum attention probability ([LC] Eq. 6).

    u_j = max_i (scale * q_i . k_j - lse_i), so a_j = exp(u_j) is the largest
    softmax probability any reference query puts on key j.  -> u [T].
    """
    Q, K, lse = _f64(Q), _f64(K), _f64(lse)
    u = np.full(K.shape[0], -np.inf)
    for a, b in _chunks(Q.shape[0]):
        S = scale * (Q[a:b] @ K.T) - lse[a:b, None]
        u = np.maximum(u, S.max(axis=0))
    return u


# ---------------------------------------------------------------- step 3 ----
def select(u, t):
    """Indices of the t highest scores ([KVC]: C_k = the keys with the highest
    attention), ascending.

    tau is the t-th largest value; the result is every j with u_j > tau plus
    the lowest-index keys with u_j == tau until t are taken.  Works on the
    array's own dtype (so an fp32 score array is compared in fp32); -0 is
    treated as +0.
    """
    u = np.asarray(u)
    T = u.shape[0]
    if not (0 < t <= T):
        raise ValueError("need 0 < t <= T")
    u = u + u.dtype.type(0)           # -0 + 0 = +0
    tau = np.sort(u)[::-1][t - 1]
    above = np.flatnonzero(u > tau)
    ties = np.flatnonzero(u == tau)[: t - above.size]
    return np.sort(np.concatenate([above, ties])).astype(np.int64)


# ---------------------------------------------------------------- step 4 ----
def mass_system(Q, Kc, m, lse, scale):
    """Normal equations of the mass-matching fit ([KVC] mass equation), in
    per-query max-shifted form.

    A_ij = exp(scale * q_i . c_j - m_i) (compact unnormalised weights),
    b_i  = exp(lse_i - m_i) (full mass).  Returns G = A^T A [t, t],
    c = A^T b [t] and bb = b^T b, so ||A w - b||^2 = w^T G w - 2 c^T w + bb.
    """
    Q, Kc, m, lse = _f64(Q), _f64(Kc), _f64(m), _f64(lse)
    t = Kc.shape[0]
    G = np.zeros((t, t))
    c = np.zeros(t)
    bb = 0.0
    for a, b in _chunks(Q.shape[0]):
        A = np.exp(scale * (Q[a:b] @ Kc.T) - m[a:b, None])
        bv = np.exp(lse[a:b] - m[a:b])
        G += A.T @ A
        c += A.T @ bv
        bb += bv @ bv
    return G, c, bb


def _chol_solve(M, r):
    """Solve M x = r for symmetric positive definite M by Cholesky; None if the
    factorisation breaks down."""
    try:
        L = np.linalg.cholesky(M)
    except np.linalg.LinAlgError:
        return None
    if _solve_tri is not None:
        y = _solve_tri(L, r, lower=True)
        return _solve_tri(L.T, y, lower=False)
    return np.linalg.solve(L.T, np.linalg.solve(L, r))


def ridge(M):
    """The ridge added to an n x n system whose Cholesky factorisation broke
    down: n * 2^-20 times the mean of its diagonal."""
    return M.shape[0] * 2.0 ** -20 * float(np.mean(np.diag(M))) if M.size else 0.0


def nnls_tolerance(c, t, eps=np.finfo(np.float64).eps):
    return 10.0 * eps * t * float(np.max(np.abs(c))) if c.size else 0.0


def nnls_lh(G, c, max_outer=0, max_inner=0, tol=None):
    """min_{w >= 0} ||A w - b||^2 given G = A^T A and c = A^T b, by the
    Lawson-Hanson active-set method ([KVC]: beta is fitted by NNLS on the mass
    equation; w = exp(beta)).

    Steps: start with an empty passive set P and w = 0.  Each outer step
    computes the descent direction g = c - G w; it stops when P holds every
    index or no index outside P has g_j > tol; otherwise the index with the
    largest g_j (lowest index on ties) joins P.  The inner loop solves the
    unconstrained problem on P (G_PP z = c_P); if every z_j > 0 it becomes w;
    otherwise w moves toward z by the largest step that keeps w >= 0 and the
    indices that reach zero leave P.  Should the index that just joined get
    z_j <= 0 (no progress possible in exact arithmetic, so a rounding effect)
    it leaves again and is not retried until w changes.  A passive system
    whose factorisation breaks down is solved with the ridge of ``ridge``
    added and the status is SINGULAR.

    Returns (w, info) with info = {"outer", "inner", "status"}.
    """
    G, c = _f64(G), _f64(c)
    t = c.shape[0]
    max_outer = max_outer or 3 * t
    max_inner = max_inner or t
    tol = nnls_tolerance(c, t) if tol is None else tol
    w = np.zeros(t)
    P = np.zeros(t, dtype=bool)
    blocked = np.zeros(t, dtype=bool)
    status = NOT_CONVERGED
    singular = False
    outer = inner_total = 0
    while outer < max_outer:
        g = c - G @ w
        cand = np.where(~P & ~blocked, g, -np.inf)
        if P.all() or not (cand.max() > tol):
            status = OK
            break
        j = int(np.argmax(cand))
        P[j] = True
        outer += 1
        first = True
        for _ in range(max_inner):
            inner_total += 1
            idx = np.flatnonzero(P)
            GP = G[np.ix_(idx, idx)]
            zP = _chol_solve(GP, c[idx])
            if zP is None:
                singular = True
                zP = _chol_solve(GP + ridge(GP) * np.eye(idx.size), c[idx])
                if zP is None:
                    return w, {"outer": outer, "inner": inner_total, "status": SINGULAR}
            z = np.zeros(t)
            z[idx] = zP
            if np.all(zP > 0):
                w = z
                blocked[:] = False
                break
            if first and z[j] <= 0:
                P[j] = False
                blocked[j] = True
                break
            first = False
            # largest step toward z that keeps w >= 0: the smallest
            # w_j / (w_j - z_j) over the indices of P with z_j <= 0
            neg = idx[zP <= 0]
            den = w[neg] - z[neg]
            ratio = np.where(den > 0, w[neg] / np.where(den > 0, den, 1.0), 0.0)
            k = int(np.argmin(ratio))
            w = w + ratio[k] * (z - w)
            w[neg[k]] = 0.0
            P &= w > 0
            w[~P] = 0.0
            blocked[:] = False
        else:
            return w, {"outer": outer, "inner": inner_total, "status": NOT_CONVERGED}
    if singular and status == OK:
        status = SINGULAR
    return w, {"outer": outer, "inner": inner_total, "status": status}


# ---------------------------------------------------------------- step 5 ----
def compact_weights(Q, Kc, beta, scale):
    """Compact attention probabilities ([LC] Eq. 2-3): X = softmax_j(scale *
    q . c_j + beta_j) over the given keys.  Q [n, d], Kc [p, d] -> X [n, p]."""
    L = scale * (_f64(Q) @ _f64(Kc).T) + _f64(beta)[None, :]
    L = L - L.max(axis=1, keepdims=True)
    E = np.exp(L)
    return E / E.sum(axis=1, keepdims=True)


def output_system(Q, Kc, w, O, scale):
    """Normal equations of the output-matching fit ([KVC] output equation).

    On the support P = {j : w_j > 0}: X = compact softmax with beta = log w;
    returns (support indices, H = X^T X, R = X^T O)."""
    w = _f64(w)
    sup = np.flatnonzero(w > 0)
    Q, O = _f64(Q), _f64(O)
    Kp = _f64(Kc)[sup]
    bp = np.log(w[sup])
    p = sup.size
    H = np.zeros((p, p))
    R = np.zeros((p, O.shape[1]))
    for a, b in _chunks(Q.shape[0]):
        X = compact_weights(Q[a:b], Kp, bp, scale)
        H += X.T @ X
        R += X.T @ O[a:b]
    return sup, H, R


def ols(H, R):
    """C = H^-1 R by Cholesky; on breakdown the ridge of ``ridge`` (n * 2^-20
    * mean(diag H)) is added once.  Returns (C, status)."""
    H, R = _f64(H), _f64(R)
    C = _chol_solve(H, R)
    if C is not None:
        return C, OK
    C = _chol_solve(H + ridge(H) * np.eye(H.shape[0]), R)
    if C is None:
        C = np.zeros_like(R)
    return C, SINGULAR


# ------------------------------------------------------------ one head ------
def later_duplicates(Kc):
    """True for each kept key whose vector equals (value for value; -0 equals
    +0) the vector of a kept key at an earlier position."""
    Kc = np.asarray(Kc)
    dup = np.zeros(Kc.shape[0], dtype=bool)
    for j in range(1, Kc.shape[0]):
        dup[j] = bool(np.any(np.all(Kc[:j] == Kc[j], axis=1)))
    return dup


def fit_head(Q, K, V, idx, m, lse, O, scale, max_outer=0, max_inner=0):
    """Steps 4-5 for one head given the selected keys and the full statistics:
    returns dict(w, beta, Cv, nnls=info, ols_status)."""
    idx = np.asarray(idx, np.int64)
    Kc = _f64(K)[idx]
    G, c, bb = mass_system(Q, Kc, m, lse, scale)
    keep = np.flatnonzero(~later_duplicates(Kc))
    w = np.zeros(idx.size)
    w[keep], info = nnls_lh(G[np.ix_(keep, keep)], c[keep], max_outer, max_inner)
    with np.errstate(divide="ignore"):
        beta = np.log(w)
    sup, H, R = output_system(Q, Kc, w, O, scale)
    Cv = _f64(V)[idx].copy()
    C, st = ols(H, R)
    Cv[sup] = C
    return {"w": w, "beta": beta, "Cv": Cv, "nnls": info, "ols_status": st,
            "G": G, "c": c, "bb": bb, "H": H, "R": R, "support": sup}


def compact_head(Q, K, V, t, scale, max_outer=0, max_inner=0):
    """All five steps for one KV head.  Q [n_q, d] holds the reference queries
    of every query head in the group; K, V [T, d]."""
    m, lse, O = full_stats(Q, K, V, scale)
    u = key_scores(Q, K, lse, scale)
    idx = select(u, t)
    res = fit_head(Q, K, V, idx, m, lse, O, scale, max_outer, max_inner)
    res.update({"m": m, "lse": lse, "O": O, "u": u, "idx": idx})
    return res


def compact_layer(Q, K, V, t, scale, max_outer=0, max_inner=0):
    """``compact_head`` for each KV head of a layer: Q [H, n_q, d], K, V
    [H, T, d] -> list of per-head result dicts."""
    return [compact_head(Q[h], K[h], V[h], t, scale, max_outer, max_inner)
            for h in range(Q.shape[0])]


# ------------------------------------------------------------ fast path -----
# [KVC] "Attempt #3: Two-Pass", "Choosing beta" (uniform redistribution) and
# "Choosing C_v" (direct selection): a compaction that never forms the full
# n_q x T score matrix.  Readings (also in the design notes): the query subset
# Q' is given as row indices (the random draw is an input); first-pass scores
# are the key scores of Q' under full attention over all T keys (Q' is small,
# so its exact lse is cheap); the second pass normalises each full query over
# the k*t shortlist keys only, which is all QK'^T provides; the redistribution
# takes n = all reference queries and the shortlist as the total mass; the
# softmax scale s is applied as in [LC] Eq. (1).

def lse_over(Q, K, scale):
    """log sum_j exp(scale * q_i . k_j) for every row of Q over the rows of K
    (the log attention mass of each query over those keys)."""
    Q, K = _f64(Q), _f64(K)
    out = np.empty(Q.shape[0])
    for a, b in _chunks(Q.shape[0]):
        S = scale * (Q[a:b] @ K.T)
        mm = S.max(axis=1)
        out[a:b] = mm + np.log(np.exp(S - mm[:, None]).sum(axis=1))
    return out


def two_pass_select(Q, K, qsel, t, k, scale):
    """Two-pass key selection ([KVC] "Attempt #3: Two-Pass").

    Pass 1: the query subset Q' = Q[qsel] scores every key,
    u'_j = max_{i in Q'} (s q_i.k_j - lse_i) with lse_i over all T keys; the
    k*t best keys (capped at T) form the shortlist K'.  Pass 2: every query
    scores the shortlist normalised over the shortlist,
    u_j = max_i (s q_i.k'_j - lse'_i), lse'_i = log sum_{l in K'} exp(s q_i.k'_l);
    the t best shortlist keys are C_k.  Ties go to the lower key index.
    Returns dict(short, u1, u2, idx) with idx ascending original key indices.
    """
    Q, K = _f64(Q), _f64(K)
    Qs = Q[np.asarray(qsel, np.int64)]
    u1 = key_scores(Qs, K, lse_over(Qs, K, scale), scale)
    kt = min(k * t, K.shape[0])
    short = select(u1, kt)
    Ks = K[short]
    u2 = key_scores(Q, Ks, lse_over(Q, Ks, scale), scale)
    pos = select(u2, t)
    return {"short": short, "u1": u1, "u2": u2, "idx": short[pos]}


def redistribute_beta(Q, K, short, idx, scale):
    """Uniform redistribution of the missing mass ([KVC] "Choosing beta").

    Over the n reference queries: m_j = (1/n) sum_i exp(s q_i.c_j) for each
    selected key, Delta = (1/n) sum_i [sum_{l in K'} exp(s q_i.k'_l) -
    sum_{j in C_k} exp(s q_i.c_j)], and beta_j = log((m_j + Delta/t) / m_j).
    C_k is a subset of K' (the page notes this), so the bracket equals the
    sum over the dropped shortlist keys K' \\ C_k term by term; it is
    evaluated that way, which has no cancellation when the dropped keys carry
    little of the mass (no dropped key gives Delta = 0 and beta = 0 exactly).
    Every exponent is shifted by one common constant (beta is invariant
    under it).  -> beta [t]."""
    Q, K = _f64(Q), _f64(K)
    short = np.asarray(short, np.int64)
    idx = np.asarray(idx, np.int64)
    if not np.all(np.isin(idx, short)):
        raise ValueError("the selected keys must be shortlist keys")
    dropped = np.setdiff1d(short, idx)
    t = idx.size
    n = Q.shape[0]
    M = lse_over(Q, K[short], scale).max()  # >= every exponent below
    m = np.zeros(t)
    delta = 0.0
    for a, b in _chunks(n):
        m += np.exp(scale * (Q[a:b] @ K[idx].T) - M).sum(axis=0)
        if dropped.size:
            delta += np.exp(scale * (Q[a:b] @ K[dropped].T) - M).sum()
    m /= n
    delta /= n
    return np.log((m + delta / t) / m)


def direct_values(V, idx):
    """C_v = V[idx] ([KVC] "Choosing C_v", direct selection)."""
    return _f64(V)[np.asarray(idx, np.int64)].copy()


def compact_head_fast(Q, K, V, qsel, t, k, scale):
    """Two-pass selection, redistributed beta, direct C_v for one KV head."""
    r = two_pass_select(Q, K, qsel, t, k, scale)
    r["beta"] = redistribute_beta(Q, K, r["short"], r["idx"], scale)
    r["Cv"] = direct_values(V, r["idx"])
    return r


# ------------------------------------------------------ decode consumer -----
# [LC] §3.1 "Handling Subsequent Tokens", Eq. (4)-(5), and Appendix A.2
# "Normalizer Computation and Storage": the compacted document branch (biased
# logits, padded slots excluded) and the branch of tokens appended after
# compaction (no bias, causal visibility) are each reduced to an output and a
# log-normaliser, then merged with the shared normaliser in log space.
def branch_attention(Q, K, V, bias, valid, scale):
    """Output and log-normaliser of one branch for every row of Q.

    scores = s q.k_j (+ bias_j), entries with valid_j = False excluded.
    Returns (out [n, d_v], log_z [n]); a row with no valid entry has
    log_z = -inf and out = 0 (its branch carries no mass)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    n = Q.shape[0]
    valid = np.broadcast_to(np.asarray(valid, bool), (n, K.shape[0]))
    out = np.zeros((n, V.shape[1]))
    log_z = np.full(n, -np.inf)
    for a, b in _chunks(n):
        S = scale * (Q[a:b] @ K.T)
        if bias is not None:
            S = S + _f64(bias)[None, :]
        S = np.where(valid[a:b], S, -np.inf)
        mm = S.max(axis=1) if S.shape[1] else np.full(b - a, -np.inf)
        has = np.isfinite(mm)
        E = np.zeros_like(S)
        E[has] = np.exp(S[has] - mm[has, None])
        z = E.sum(axis=1)
        log_z[a:b][has] = mm[has] + np.log(z[has])
        out[a:b][has] = (E[has] @ V) / z[has, None]
    return out, log_z


def combine_attention(Q, Ck, beta, Cv, Knew, Vnew, n_vis, scale):
    """Attention of queries over a compacted cache plus appended tokens
    ([LC] Eq. (4)-(5)).  Row r sees the compacted entries with finite beta
    and the first n_vis[r] appended tokens.  Z_cmp and Z_new are the
    branches' normalisers; A = (Z_cmp A_cmp + Z_new A_new) / (Z_cmp + Z_new)
    with the weights formed from log-normalisers.  -> (A [n, d_v], log_z)."""
    beta = _f64(beta)
    n = np.asarray(Q).shape[0]
    doc_out, doc_lz = branch_attention(Q, Ck, Cv, np.where(np.isfinite(beta), beta, 0.0),
                                       np.isfinite(beta)[None, :], scale)
    n_new = np.asarray(Knew).shape[0]
    vis = np.arange(n_new)[None, :] < np.asarray(n_vis)[:, None]
    new_out, new_lz = branch_attention(Q, Knew, Vnew, None, vis, scale)
    tot = np.logaddexp(doc_lz, new_lz)
    A = np.zeros_like(doc_out)
    ok = np.isfinite(tot)
    wd = np.exp(doc_lz[ok] - tot[ok])
    wn = np.exp(new_lz[ok] - tot[ok])
    A[ok] = wd[:, None] * doc_out[ok] + wn[:, None] * new_out[ok]
    assert A.shape[0] == n
    return A, tot


def heldout_errors(Qh, K, V, Ck, beta, Cv, scale):
    """Quality of a compaction on held-out queries ([KVC] "Choosing beta" and
    "Choosing C_v": the mass and the attention-output reconstruction errors).

    Per query, the full cache gives (A_full, log Z_full) and the compacted
    cache (no appended tokens) gives (A_cmp, log Z_cmp).  Returns
    (mass_err, out_err) = (mean_i |log Z_cmp - log Z_full|,
                           mean_i ||A_cmp - A_full||_2)."""
    Qh = _f64(Qh)
    _, lse, O = full_stats(Qh, K, V, scale)
    beta = _f64(beta)
    A, lz = branch_attention(Qh, Ck, Cv, np.where(np.isfinite(beta), beta, 0.0),
                             np.isfinite(beta)[None, :], scale)
    return float(np.mean(np.abs(lz - lse))), float(np.mean(np.linalg.norm(A - O, axis=1)))


# ------------------------------------------------ farthest-first traversal --
def farthest_first(K, seeds, M):
    """Diversifier selection by farthest-first traversal ([LC] §3.2 Eq. (7),
    after Gonzalez 1985): starting from the index set S = seeds, repeatedly add
    i* = argmax_{i not in S} min_{j in S} ||k_i - k_j||^2 until |S| = M.
    Ties go to the lower index.  Returns the added indices in the order
    chosen (M - |seeds| of them; fewer if the keys run out)."""
    K = _f64(K)
    S = [int(s) for s in seeds]
    if not S:
        raise ValueError("farthest-first traversal needs at least one seed")
    N = K.shape[0]
    taken = np.zeros(N, bool)
    taken[S] = True
    mind = np.full(N, np.inf)
    for j in S:
        mind = np.minimum(mind, ((K - K[j]) ** 2).sum(axis=1))
    added = []
    while len(S) < M and not taken.all():
        cand = np.where(taken, -np.inf, mind)
        i = int(np.argmax(cand))  # first maximum = lowest index
        added.append(i)
        S.append(i)
        taken[i] = True
        mind = np.minimum(mind, ((K - K[i]) ** 2).sum(axis=1))
    return np.asarray(added, np.int64)


# ------------------------------------------------- baseline AM variant -----
# [LC] Appendix A.3 "Baselines and Budgets": the Attention Matching baseline
# selects keys by RMS attention and fits the biases with two bounded
# non-negative least-squares iterations, bounds [e^-3, e^3], then fits the
# values by least squares.  Readings: the RMS runs over the reference queries
# of the group; one bounded iteration solves the normal equations over the
# free weights with the pinned ones held at their bounds and then pins every
# free weight that left [lo, hi] at the bound it crossed (the first steps of
# an active-set method for bound constraints), starting with every weight
# free.
def rms_key_scores(Q, K, lse, scale):
    """u_j = log sqrt((1/n) sum_i p_ij^2), p_ij = exp(s q_i.k_j - lse_i): the
    log of key j's RMS attention probability over the n queries."""
    Q, K, lse = _f64(Q), _f64(K), _f64(lse)
    n = Q.shape[0]
    mx = np.full(K.shape[0], -np.inf)
    for a, b in _chunks(n):
        mx = np.maximum(mx, (2.0 * (scale * (Q[a:b] @ K.T) - lse[a:b, None])).max(axis=0))
    acc = np.zeros(K.shape[0])
    for a, b in _chunks(n):
        acc += np.exp(2.0 * (scale * (Q[a:b] @ K.T) - lse[a:b, None]) - mx[None, :]).sum(axis=0)
    return 0.5 * (mx + np.log(acc) - np.log(n))


def bounded_ls(G, c, lo, hi, iters):
    """Bounded least squares from the normal equations (G = A^T A, c = A^T b):
    `iters` iterations of [solve G_FF w_F = c_F - G_FB w_B over the free set
    F with the pinned set B at its bounds; pin every free w_j outside
    [lo, hi] at the bound it crossed], starting with F = all.  Stops early
    when an iteration pins nothing.  -> (w, iterations run)."""
    G, c = _f64(G), _f64(c)
    t = c.size
    w = np.zeros(t)
    free = np.ones(t, bool)
    it = 0
    while it < iters and free.any():
        it += 1
        F = np.flatnonzero(free)
        B = np.flatnonzero(~free)
        rhs = c[F] - G[np.ix_(F, B)] @ w[B]
        x = _chol_solve(G[np.ix_(F, F)], rhs)
        if x is None:  # not positive definite: the same ridge as the OLS fallback
            M = G[np.ix_(F, F)]
            x = _chol_solve(M + ridge(M) * np.eye(F.size), rhs)
        w[F] = x
        low = free & (w < lo)
        high = free & (w > hi)
        w[low] = lo
        w[high] = hi
        if not (low.any() or high.any()):
            break
        free &= ~(low | high)
    return w, it


def compact_head_variant(Q, K, V, t, scale, iters=2, lo=np.exp(-3.0), hi=np.exp(3.0)):
    """The baseline AM variant for one KV head: full statistics, RMS key
    scores, top-t selection, bounded biases (two iterations, [e^-3, e^3]),
    least-squares values over all t keys (every w_j > 0)."""
    m, lse, O = full_stats(Q, K, V, scale)
    u = rms_key_scores(Q, K, lse, scale)
    idx = select(u, t)
    Kc = _f64(K)[idx]
    G, c, bb = mass_system(Q, Kc, m, lse, scale)
    w, it = bounded_ls(G, c, lo, hi, iters)
    beta = np.log(w)
    sup, H, R = output_system(Q, Kc, w, O, scale)
    C, st = ols(H, R)
    Cv = _f64(V)[idx].copy()
    Cv[sup] = C
    return {"m": m, "lse": lse, "O": O, "u": u, "idx": idx, "w": w, "beta": beta, "Cv": Cv,
            "iters": it, "ols_status": st, "G": G, "c": c}
