"""Pins for the float64 oracle: checks against things other than the oracle
itself -- brute-force loops on tiny inputs, closed forms, library routines
(scipy's Lawson-Hanson NNLS, numpy's SVD least squares, a stable sort), and
invariants of the method.

Each ``check_*`` takes the oracle module as an argument and raises
AssertionError on a mismatch, so that ``test_oracle_mutants`` can show that a
plausible mistake planted in a copy of the oracle fails at least one pin.

Sources of the closed forms: "Latent Compaction with Test-Time Training" §3
Eq. (1)-(3) and (6); "KV compaction" (bkal01 blog), section "Fast KV
Compaction via Attention Matching" (the mass/output equations; with q = 0 an
unbiased compact cache has mass t instead of T, which is why beta exists).
"""
from __future__ import annotations

import decimal
import itertools
import math

import numpy as np


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _close(a, b, tol, what):
    a, b = np.asarray(a, float), np.asarray(b, float)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert a.shape == b.shape and err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# ----------------------------------------------------------------- step 1 ---
def check_full_stats_brute(o):
    """m, lse, O against plain loops over the definition (Eq. 1)."""
    rng = _rng(11)
    for n_q, T, d, dv in [(5, 7, 3, 2), (3, 1, 4, 3), (4, 64, 8, 2)]:
        Q = rng.standard_normal((n_q, d))
        K = rng.standard_normal((T, d))
        V = rng.standard_normal((T, dv))
        s = 0.37
        m, lse, O = o.full_stats(Q, K, V, s)
        for i in range(n_q):
            logit = [s * sum(Q[i, k] * K[j, k] for k in range(d)) for j in range(T)]
            Z = sum(math.exp(x) for x in logit)
            _close(m[i], max(logit), 1e-12, "rowmax")
            _close(lse[i], math.log(Z), 1e-12, "lse")
            for c in range(dv):
                _close(O[i, c], sum(math.exp(x) / Z * V[j, c] for j, x in enumerate(logit)),
                       1e-12, "O")


def check_full_stats_closed_forms(o):
    rng = _rng(12)
    T, d = 9, 5
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, 3))
    # q = 0: every key equally likely
    m, lse, O = o.full_stats(np.zeros((2, d)), K, V, 0.5)
    _close(m, [0, 0], 0, "q=0 rowmax")
    _close(lse, [math.log(T)] * 2, 1e-14, "q=0 lse = log T")
    _close(O, np.tile(V.mean(0), (2, 1)), 1e-14, "q=0 O = mean V")
    # a single key: lse is its logit, the output its value
    q = rng.standard_normal((1, d))
    m, lse, O = o.full_stats(q, K[:1], V[:1], 0.5)
    _close(lse, [0.5 * float(q[0] @ K[0])], 1e-14, "T=1 lse")
    _close(O, V[:1], 1e-14, "T=1 O")
    # identical huge logits: lse = L + log T without overflow
    Kb = np.tile(np.array([[1.0, 0, 0, 0, 0]]), (T, 1))
    qb = np.array([[4000.0, 0, 0, 0, 0]])
    m, lse, O = o.full_stats(qb, Kb, V, 0.5)
    _close(lse, [2000.0 + math.log(T)], 1e-10, "huge logits")
    assert np.all(np.isfinite(O))


# ----------------------------------------------------------------- step 2 ---
def check_key_scores_brute(o):
    """u_j = log max_i softmax_i,j against loops (Eq. 6)."""
    rng = _rng(21)
    n_q, T, d = 6, 10, 4
    Q = rng.standard_normal((n_q, d)) * 2
    K = rng.standard_normal((T, d))
    s = 0.6
    _, lse, _ = o.full_stats(Q, K, np.zeros((T, 1)), s)
    u = o.key_scores(Q, K, lse, s)
    for j in range(T):
        best = 0.0
        for i in range(n_q):
            logit = [s * float(Q[i] @ K[l]) for l in range(T)]
            p = math.exp(logit[j]) / sum(math.exp(x) for x in logit)
            best = max(best, p)
        _close(u[j], math.log(best), 1e-12, "key score")
    assert np.all(u <= 1e-12), "a probability above 1"
    # q = 0: every probability is 1/T
    _, lse0, _ = o.full_stats(np.zeros((3, d)), K, np.zeros((T, 1)), s)
    _close(o.key_scores(np.zeros((3, d)), K, lse0, s), [-math.log(T)] * T, 1e-14, "q=0 scores")
    # the log-domain order is the probability order
    a = np.exp(u)
    assert list(np.argsort(-u, kind="stable")) == list(np.argsort(-a, kind="stable"))


# ----------------------------------------------------------------- step 3 ---
def _select_by_sort(u, t):
    u = [0.0 if x == 0 else float(x) for x in u]
    order = sorted(range(len(u)), key=lambda j: (-u[j], j))
    return sorted(order[:t])


def check_select(o):
    import synth
    cases = [synth.continuous_scores(3, 97, 31), synth.tie_heavy_scores(3, 200, 32),
             synth.tie_heavy_scores(2, 64, 33, levels=(0.0, -0.0))]
    for arr in cases:
        for row in arr:
            for t in (1, 2, 7, len(row) // 2, len(row)):
                got = list(o.select(row, t))
                assert got == _select_by_sort(row, t), f"select t={t}"
    # fp32 input is compared in fp32: two keys equal in fp32 tie
    u = np.array([-1.0, np.float32(-1.0 + 1e-9), -2.0], dtype=np.float32)
    assert list(o.select(u, 1)) == [0]
    try:
        o.select(np.zeros(4), 5)
    except ValueError:
        pass
    else:
        raise AssertionError("t > T accepted")


# ----------------------------------------------------------------- step 4 ---
def _nnls_by_supports(A, b):
    """Exhaustive NNLS for tiny t: the best feasible unconstrained fit over all
    supports (the minimiser is the unconstrained fit on its own support)."""
    t = A.shape[1]
    best_w, best_r = np.zeros(t), float(b @ b)
    for k in range(1, t + 1):
        for S in itertools.combinations(range(t), k):
            S = list(S)
            x, *_ = np.linalg.lstsq(A[:, S], b, rcond=None)
            if np.all(x > 0):
                w = np.zeros(t)
                w[S] = x
                r = float(np.sum((A @ w - b) ** 2))
                if r < best_r - 1e-12:
                    best_w, best_r = w, r
    return best_w


def _random_problem(rng, n, t):
    A = np.exp(rng.standard_normal((n, t)))
    b = A @ np.abs(rng.standard_normal(t)) - 0.8 * A[:, 0] * rng.uniform(0, 2) \
        + rng.standard_normal(n) * 3
    return A, b


def check_mass_system_brute(o):
    """G = A^T A, c = A^T b and b.b in per-query max-shifted form, against
    loops: A_ij = exp(s q_i.c_j - m_i), b_i = exp(lse_i - m_i) with m_i the
    full-row max and lse_i the full log mass; and the residual ||A w - b||^2
    = w^T G w - 2 c^T w + b.b at an arbitrary w."""
    rng = _rng(45)
    n_q, T, d, t = 5, 8, 3, 3
    Q = rng.standard_normal((n_q, d)) * 3
    K = rng.standard_normal((T, d))
    s = 0.9
    m, lse, _ = o.full_stats(Q, K, np.zeros((T, 1)), s)
    idx = [1, 4, 6]
    G, c, bb = o.mass_system(Q, K[idx], m, lse, s)
    for j in range(t):
        for k in range(t):
            ref = 0.0
            for i in range(n_q):
                logit = [s * float(Q[i] @ K[l]) for l in range(T)]
                mx = max(logit)
                ref += math.exp(logit[idx[j]] - mx) * math.exp(logit[idx[k]] - mx)
            _close(G[j, k], ref, 1e-12, "mass Gram")
        ref = 0.0
        for i in range(n_q):
            logit = [s * float(Q[i] @ K[l]) for l in range(T)]
            mx = max(logit)
            ref += math.exp(logit[idx[j]] - mx) * sum(math.exp(x - mx) for x in logit)
        _close(c[j], ref, 1e-11, "mass right-hand side")
    ref = 0.0
    for i in range(n_q):
        logit = [s * float(Q[i] @ K[l]) for l in range(T)]
        mx = max(logit)
        ref += sum(math.exp(x - mx) for x in logit) ** 2
    _close(bb, ref, 1e-11, "mass b.b")
    # the residual identity the three terms exist for, at an arbitrary w
    w = np.array([0.3, 1.7, 0.05])
    A = np.array([[math.exp(s * float(Q[i] @ K[l]) - m[i]) for l in idx] for i in range(n_q)])
    b = np.array([math.exp(lse[i] - m[i]) for i in range(n_q)])
    _close(w @ G @ w - 2 * c @ w + bb, float(np.sum((A @ w - b) ** 2)), 1e-10, "mass residual")


def check_nnls_bruteforce(o):
    rng = _rng(41)
    for _ in range(12):
        A, b = _random_problem(rng, 14, 6)
        w, info = o.nnls_lh(A.T @ A, A.T @ b)
        assert info["status"] == o.OK
        _close(w, _nnls_by_supports(A, b), 1e-8, "NNLS vs support enumeration")


def check_nnls_scipy(o):
    from scipy.optimize import nnls as scipy_nnls
    rng = _rng(42)
    for t in (5, 12, 30):
        A, b = _random_problem(rng, 3 * t, t)
        w, info = o.nnls_lh(A.T @ A, A.T @ b)
        ws, _ = scipy_nnls(A, b)
        assert info["status"] == o.OK
        _close(w, ws, 1e-8 * max(1.0, np.abs(ws).max()), "NNLS vs scipy")


def check_nnls_planted_and_kkt(o):
    rng = _rng(43)
    t = 10
    A = np.exp(rng.standard_normal((40, t)))
    ws = np.abs(rng.standard_normal(t))
    ws[[1, 4, 7]] = 0.0
    w, _ = o.nnls_lh(A.T @ A, A.T @ (A @ ws))
    _close(w, ws, 1e-9, "planted NNLS solution")
    # KKT on a problem with active bounds
    A, b = _random_problem(rng, 60, 20)
    G, c = A.T @ A, A.T @ b
    w, info = o.nnls_lh(G, c)
    g = c - G @ w
    tol = 1e-9 * np.abs(c).max()
    assert np.all(w >= 0), "negative weight"
    assert np.all(g[w == 0] <= tol), "a zero weight could still lower the residual"
    assert np.all(np.abs(g[w > 0]) <= tol), "gradient not zero on the support"
    assert np.any(w == 0), "problem has no active bound (test is not testing)"


def check_nnls_q_zero_and_caps(o):
    """All queries at q = 0: A = 1, b = T (the pages' argument for beta): an
    unbiased compact cache (w = 1) has mass t, the fit restores sum w = T."""
    n, t, T = 7, 4, 50
    A = np.ones((n, t))
    b = np.full(n, float(T))
    w, info = o.nnls_lh(A.T @ A, A.T @ b)
    _close(w.sum(), T, 1e-9, "q=0: compact mass sum(w) = T")
    assert abs(np.ones(t).sum() - T) > 1, "unbiased mass equals T (test is not testing)"
    rng = _rng(44)
    A, b = _random_problem(rng, 30, 10)
    _, info = o.nnls_lh(A.T @ A, A.T @ b, max_outer=1)
    assert info["status"] == o.NOT_CONVERGED, "iteration cap not reported"


# ----------------------------------------------------------------- step 5 ---
def check_compact_weights(o):
    rng = _rng(51)
    Q = rng.standard_normal((5, 3))
    Kc = rng.standard_normal((4, 3))
    beta = rng.standard_normal(4)
    s = 0.8
    X = o.compact_weights(Q, Kc, beta, s)
    for i in range(5):
        e = [math.exp(s * float(Q[i] @ Kc[j]) + beta[j]) for j in range(4)]
        _close(X[i], np.array(e) / sum(e), 1e-14, "compact softmax (Eq. 2-3)")
    _close(X.sum(1), np.ones(5), 1e-14, "rows sum to 1")
    _close(o.compact_weights(Q, Kc, beta + 7.0, s), X, 1e-14, "shift invariance")


def check_ols(o):
    rng = _rng(52)
    n, t, d = 80, 9, 4
    X = o.compact_weights(rng.standard_normal((n, 3)) * 2, rng.standard_normal((t, 3)),
                          rng.standard_normal(t), 1.0)
    Ot = rng.standard_normal((n, d))
    C, st = o.ols(X.T @ X, X.T @ Ot)
    Cref, *_ = np.linalg.lstsq(X, Ot, rcond=None)
    assert st == o.OK
    _close(C, Cref, 1e-8 * max(1, np.abs(Cref).max()), "OLS vs SVD least squares")
    H, R = X.T @ X, X.T @ Ot
    res = np.linalg.norm(H @ C - R) / (np.linalg.norm(H) * np.linalg.norm(C) + np.linalg.norm(R))
    assert res <= 1e-12, f"normal-equation residual {res:.2e}"
    Cs = rng.standard_normal((t, d))
    C2, _ = o.ols(X.T @ X, X.T @ (X @ Cs))
    _close(C2, Cs, 1e-7, "planted OLS solution")
    # duplicated column: singular, ridge fallback; the ridge solution tends to
    # the minimum-norm least-squares solution (SVD) as the ridge shrinks, which
    # splits the coefficient evenly between the two equal columns
    Xd = np.concatenate([X, X[:, :1]], axis=1)
    C3, st = o.ols(Xd.T @ Xd, Xd.T @ Ot)
    assert st == o.SINGULAR and np.all(np.isfinite(C3))
    # In the SVD basis a ridge lam scales the coefficient along singular value
    # sv by sv^2 / (sv^2 + lam), so both the coefficients and the fitted
    # outputs move by at most lam / sv_min^2 (smallest nonzero sv) relative.
    Cmn, *_ = np.linalg.lstsq(Xd, Ot, rcond=None)
    sv = np.linalg.svd(Xd, compute_uv=False)
    lam = Xd.shape[1] * 2.0 ** -20 * float(np.mean(np.diag(Xd.T @ Xd)))
    bound = lam / sv[sv > 1e-10 * sv[0]].min() ** 2
    assert bound < 0.1, "ridge bound too loose (test is not testing)"
    assert np.linalg.norm(C3 - Cmn) <= 1.01 * bound * np.linalg.norm(Cmn), \
        "ridge fallback vs minimum-norm least squares"
    assert np.linalg.norm(Xd @ (C3 - Cmn)) <= 1.01 * bound * np.linalg.norm(Xd @ Cmn), \
        "ridge fallback: fitted outputs"
    _close(C3[0], C3[t], 1e-9 * np.abs(C3).max(), "equal columns share the coefficient")


# ------------------------------------------------------------ end to end ----
def check_t_equals_T(o):
    """Keeping every key (t = T) matches the full cache exactly: w = 1,
    C_v = V, and for every query the compact mass and output equal the full
    ones."""
    rng = _rng(61)
    T, d, n_q = 12, 6, 40
    K = rng.standard_normal((T, d))
    Q = 0.5 * K[rng.integers(0, T, n_q)] + rng.standard_normal((n_q, d))
    V = rng.standard_normal((T, 3))
    s = 1 / math.sqrt(d)
    r = o.compact_head(Q, K, V, T, s)
    assert list(r["idx"]) == list(range(T))
    _close(r["w"], np.ones(T), 1e-8, "t=T: w = 1")
    _close(r["Cv"], V, 1e-6, "t=T: C_v = V")
    logit = s * Q @ K.T + r["beta"][None, :]
    mass = np.log(np.exp(logit).sum(1))
    _close(mass, r["lse"], 1e-8, "t=T: compact log mass = full")
    X = o.compact_weights(Q, K, r["beta"], s)
    _close(X @ r["Cv"], r["O"], 1e-6, "t=T: compact output = full")


def _softmax_rows(L):
    L = L - L.max(axis=1, keepdims=True)
    E = np.exp(L)
    return E / E.sum(axis=1, keepdims=True)


def check_fit_zero_weight_branch(o):
    """Steps 4-5 through ``fit_head`` on a planted problem whose NNLS solution
    has zeros: the mass targets are b = A w* with w* >= 0 and three zero
    weights, the output targets O = X C* with X the compact softmax over the
    keys with w*_j > 0 ("KV compaction" blog, output equation; "Latent
    Compaction with Test-Time Training" Eq. (2)-(3)).  Then w = w*, beta is
    -inf exactly on the zeros, C_v on the support is the least-squares fit of
    O on X restricted to the support (numpy's SVD solver, = C*), and every row
    off the support is the key's original value row, bit for bit."""
    rng = _rng(62)
    T, d, dv, n_q, t = 16, 4, 3, 60, 8
    K = rng.standard_normal((T, d))
    Q = 1.5 * rng.standard_normal((n_q, d))
    V = rng.standard_normal((T, dv))
    s = 0.7
    idx = np.array([0, 2, 3, 5, 8, 9, 12, 14])
    logit = s * Q @ K[idx].T
    m = logit.max(axis=1) + 0.3          # any per-row shift defines the same fit
    A = np.exp(logit - m[:, None])
    ws = np.abs(rng.standard_normal(t)) + 0.2
    off = np.array([1, 4, 6])
    ws[off] = 0.0
    lse = m + np.log(A @ ws)
    sup = np.flatnonzero(ws > 0)
    X = _softmax_rows(logit[:, sup] + np.log(ws[sup])[None, :])
    Cs = rng.standard_normal((sup.size, dv))
    O = X @ Cs
    r = o.fit_head(Q, K, V, idx, m, lse, O, s)
    _close(r["w"], ws, 1e-9, "planted weights with zeros")
    assert np.all(r["w"][off] == 0.0), "a zero weight came back nonzero"
    assert np.all(np.isneginf(r["beta"][off])), "beta of a zero weight is not -inf"
    Cref, *_ = np.linalg.lstsq(X, O, rcond=None)
    _close(r["Cv"][sup], Cref, 1e-8, "C_v on the support vs SVD least squares")
    _close(Cref, Cs, 1e-8, "planted values (test is not testing)")
    assert np.array_equal(r["Cv"][off], V[idx[off]]), "off-support rows are not V[idx]"


def check_fit_duplicate_keys(o):
    """Two kept keys with equal vectors give equal columns of A, so the NNLS
    minimiser is not unique.  Lawson-Hanson with argmax ties going to the
    lower index never lets the later copy into the passive set: on a system
    whose rows and columns are duplicated by index (bitwise equal) it returns
    w = 0 there and the distinct-column solution elsewhere.  ``fit_head``
    gives the same: w = 0 and beta = -inf at the later copy, its C_v row the
    original value row, the other weights equal to the exhaustive NNLS over
    supports of the distinct columns and C_v on the support equal to SVD
    least squares."""
    rng = _rng(63)
    A, b = _random_problem(rng, 14, 5)
    G0, c0 = A.T @ A, A.T @ b
    p = [0, 1, 2, 1, 3, 4]
    w, info = o.nnls_lh(G0[np.ix_(p, p)], c0[p])
    assert w[3] == 0.0, "the later copy entered the passive set"
    _close(w[[0, 1, 2, 4, 5]], _nnls_by_supports(A, b), 1e-8, "duplicated system vs distinct")

    T, d, dv, n_q = 10, 3, 2, 40
    K = rng.standard_normal((T, d))
    K[7] = K[2]
    Q = 0.5 * K[rng.integers(0, T, n_q)] + rng.standard_normal((n_q, d))
    V = rng.standard_normal((T, dv))
    s = 0.8
    idx = np.array([1, 2, 4, 7, 9])
    m, lse, O = o.full_stats(Q, K, V, s)
    r = o.fit_head(Q, K, V, idx, m, lse, O, s)
    assert r["w"][3] == 0.0 and np.isneginf(r["beta"][3]), "later copy has a weight"
    assert np.array_equal(r["Cv"][3], V[7]), "later copy's value row changed"
    keep = [0, 1, 2, 4]
    Ad = np.array([[math.exp(s * float(Q[i] @ K[j]) - m[i]) for j in idx[keep]]
                   for i in range(n_q)])
    bd = np.exp(lse - m)
    _close(r["w"][keep], _nnls_by_supports(Ad, bd), 1e-8 * max(1.0, r["w"].max()),
           "weights vs exhaustive NNLS on the distinct keys")
    sup = np.flatnonzero(r["w"] > 0)
    X = _softmax_rows(s * Q @ K[idx[sup]].T + np.log(r["w"][sup])[None, :])
    Cref, *_ = np.linalg.lstsq(X, O, rcond=None)
    _close(r["Cv"][sup], Cref, 1e-7 * max(1.0, np.abs(Cref).max()), "C_v with a duplicate")


def check_fit_reduces_error(o):
    """With t < T the fitted beta and C_v match mass and output better than
    keeping the selected keys unchanged (beta = 0, C_v = V[idx])."""
    import synth
    w = synth.workload("cfg2", H=1, T=256, t=16)
    dd = synth.make(w)
    Q, K, V = dd["Q"][0], dd["K"][0], dd["V"][0]
    s = w.softmax_scale
    r = o.compact_head(Q, K, V, w.t, s)
    Kc = K[r["idx"]].astype(float)
    base_mass = np.log(np.exp(s * Q.astype(float) @ Kc.T).sum(1))
    fit_mass = np.log(np.exp(s * Q.astype(float) @ Kc.T + r["beta"]).sum(1))
    assert np.mean((fit_mass - r["lse"]) ** 2) < np.mean((base_mass - r["lse"]) ** 2)
    Xb = o.compact_weights(Q, Kc, np.zeros(w.t), s)
    Xf = o.compact_weights(Q, Kc, r["beta"], s)
    assert np.sum((Xf @ r["Cv"] - r["O"]) ** 2) < np.sum((Xb @ V[r["idx"]] - r["O"]) ** 2)


# ------------------------------------------------------------ fast path -----
def check_two_pass_brute(o):
    """Two-pass selection on a tiny head against plain loops: per-row log
    masses, first-pass key scores of the query subset, shortlist by a stable
    sort, second-pass scores normalised over the shortlist, final top-t."""
    rng = _rng(41)
    n_q, T, d, t, k = 9, 13, 4, 3, 2
    Q = rng.normal(size=(n_q, d))
    K = rng.normal(size=(T, d))
    qsel = np.array([1, 4, 7])
    s = 0.6

    def lse_row(q, keys):
        return math.log(sum(math.exp(s * float(q @ kk)) for kk in keys))

    u1 = np.array([max(s * float(Q[i] @ K[j]) - lse_row(Q[i], K) for i in qsel) for j in range(T)])
    short = np.array(_select_by_sort(u1, k * t))
    Ks = K[short]
    u2 = np.array([max(s * float(Q[i] @ Ks[j]) - lse_row(Q[i], Ks) for i in range(n_q))
                   for j in range(len(short))])
    idx = short[np.array(_select_by_sort(u2, t))]
    r = o.two_pass_select(Q, K, qsel, t, k, s)
    _close(r["u1"], u1, 1e-12, "first-pass scores")
    assert np.array_equal(r["short"], short), "shortlist"
    _close(r["u2"], u2, 1e-12, "second-pass scores")
    assert np.array_equal(r["idx"], np.sort(idx)), "selection"


def check_two_pass_full_shortlist(o):
    """With k*t >= T the shortlist is every key and the second pass is the
    full method's key scoring: same scores, same selection."""
    rng = _rng(42)
    Q = rng.normal(size=(40, 8))
    K = rng.normal(size=(24, 8))
    s = 1 / math.sqrt(8)
    r = o.two_pass_select(Q, K, np.arange(0, 40, 5), 6, 4, s)
    _, lse, _ = o.full_stats(Q, K, np.zeros((24, 1)), s)
    u = o.key_scores(Q, K, lse, s)
    assert np.array_equal(r["short"], np.arange(24))
    _close(r["u2"], u, 1e-12, "second pass = full key scores")
    assert np.array_equal(r["idx"], o.select(u, 6))


def check_redistribute(o):
    """Uniform redistribution: against loops on a tiny head; the compact mass
    with beta reproduces the shortlist mass on average over the queries (the
    missing mass is redistributed, not lost); no missing mass gives beta = 0;
    queries at q = 0 give beta_j = log(k t / t)."""
    rng = _rng(43)
    n, T, d = 7, 10, 3
    Q = rng.normal(size=(n, d))
    K = rng.normal(size=(T, d))
    s = 0.8
    short = np.array([0, 2, 3, 5, 8, 9])
    idx = np.array([2, 5, 9])
    t = idx.size
    m = np.array([sum(math.exp(s * float(Q[i] @ K[j])) for i in range(n)) / n for j in idx])
    tot = sum(math.exp(s * float(Q[i] @ K[j])) for i in range(n) for j in short) / n
    delta = tot - m.sum()
    beta = o.redistribute_beta(Q, K, short, idx, s)
    _close(beta, np.log((m + delta / t) / m), 1e-12, "beta vs loops")
    _close(np.sum(m * np.exp(beta)), tot, 1e-12, "mass conserved")
    _close(o.redistribute_beta(Q, K, idx, idx, s), np.zeros(t), 1e-12, "no missing mass")
    Z = np.zeros((5, d))
    _close(o.redistribute_beta(Z, K, short, idx, s), np.full(t, math.log(short.size / t)),
           1e-12, "q = 0")
    assert np.array_equal(o.direct_values(K, idx), K[idx])
    # dropped keys carrying ~1e-14 of the mass: the definition evaluated in
    # 50-digit decimal arithmetic (a float64 difference of the two sums
    # loses most of Delta's digits here)
    sc = 0.5
    Q3 = np.array([[1.0, 0.3], [1.0, -0.7], [1.0, 2.0]])
    K3 = np.array([[0.0, 0.0], [-70.0, 0.0], [-66.0, 0.1], [-64.0, -0.1]])
    sh3, id3 = np.array([0, 1, 2, 3]), np.array([0, 1])
    with decimal.localcontext() as ctx:
        ctx.prec = 50
        ex = [[(decimal.Decimal(sc) * (decimal.Decimal(float(Q3[i, 0])) * decimal.Decimal(float(K3[j, 0]))
                + decimal.Decimal(float(Q3[i, 1])) * decimal.Decimal(float(K3[j, 1])))).exp()
               for j in range(4)] for i in range(3)]
        nD = decimal.Decimal(3)
        mD = [sum(ex[i][j] for i in range(3)) / nD for j in id3]
        totD = sum(ex[i][j] for i in range(3) for j in sh3) / nD
        dD = totD - sum(mD)
        ref = np.array([float(((mj + dD / 2) / mj).ln()) for mj in mD])
    _close(o.redistribute_beta(Q3, K3, sh3, id3, sc), ref, 1e-12, "beta, tiny dropped mass")


# ------------------------------------------------------- decode consumer ---
def check_combine_single_softmax(o):
    """[LC] Eq. (5) is one softmax over the compacted entries (with their
    biases) and the visible appended tokens (without): against loops over
    that single softmax; no appended token gives the document branch alone;
    every compacted entry dropped (beta = -inf) gives the appended branch
    alone; a row that sees nothing has log Z = -inf."""
    rng = _rng(51)
    n, t, n_new, d, dv = 5, 4, 3, 3, 2
    Q = rng.normal(size=(n, d))
    Ck = rng.normal(size=(t, d))
    Cv = rng.normal(size=(t, dv))
    beta = np.array([0.3, -np.inf, -1.2, 2.0])
    Kn = rng.normal(size=(n_new, d))
    Vn = rng.normal(size=(n_new, dv))
    n_vis = np.array([0, 1, 2, 3, 3])
    s = 0.7
    A, lz = o.combine_attention(Q, Ck, beta, Cv, Kn, Vn, n_vis, s)
    for i in range(n):
        logits, vals = [], []
        for j in range(t):
            if np.isfinite(beta[j]):
                logits.append(s * float(Q[i] @ Ck[j]) + beta[j])
                vals.append(Cv[j])
        for m in range(n_vis[i]):
            logits.append(s * float(Q[i] @ Kn[m]))
            vals.append(Vn[m])
        ex = [math.exp(x) for x in logits]
        z = sum(ex)
        _close(lz[i], math.log(z), 1e-12, "combined log Z")
        _close(A[i], sum(e * v for e, v in zip(ex, vals)) / z, 1e-12, "combined output")
    A0, lz0 = o.combine_attention(Q, Ck, beta, Cv, Kn, Vn, np.zeros(n, int), s)
    Ab, lzb = o.branch_attention(Q, Ck, Cv, np.where(np.isfinite(beta), beta, 0.0),
                                 np.isfinite(beta)[None, :], s)
    _close(A0, Ab, 1e-12, "no appended token: document branch")
    _close(lz0, lzb, 1e-12, "no appended token: document log Z")
    An, lzn = o.combine_attention(Q, Ck, np.full(t, -np.inf), Cv, Kn, Vn, n_vis, s)
    assert np.isneginf(lzn[0]) and np.all(An[0] == 0), "empty row"
    Bn, lzbn = o.branch_attention(Q[1:], Kn, Vn, None,
                                  np.arange(n_new)[None, :] < n_vis[1:, None], s)
    _close(An[1:], Bn, 1e-12, "all entries dropped: appended branch")
    _close(lzn[1:], lzbn, 1e-12, "all entries dropped: appended log Z")


def check_heldout_errors(o):
    """Held-out mass and output errors: zero for the identity compaction
    (C_k = K, beta = 0, C_v = V); against loops on a tiny head otherwise."""
    rng = _rng(52)
    n, T, d = 6, 7, 3
    Q = rng.normal(size=(n, d))
    K = rng.normal(size=(T, d))
    V = rng.normal(size=(T, 2))
    s = 0.9
    me, oe = o.heldout_errors(Q, K, V, K, np.zeros(T), V, s)
    _close([me, oe], [0.0, 0.0], 1e-12, "identity compaction")
    idx = np.array([1, 4, 6])
    beta = np.array([0.5, -0.25, 1.0])
    Cv = rng.normal(size=(3, 2))
    me, oe = o.heldout_errors(Q, K, V, K[idx], beta, Cv, s)
    mref, oref = 0.0, 0.0
    for i in range(n):
        ef = [math.exp(s * float(Q[i] @ K[j])) for j in range(T)]
        ec = [math.exp(s * float(Q[i] @ K[j]) + b) for j, b in zip(idx, beta)]
        Af = sum(e * V[j] for e, j in zip(ef, range(T))) / sum(ef)
        Ac = sum(e * c for e, c in zip(ec, Cv)) / sum(ec)
        mref += abs(math.log(sum(ec)) - math.log(sum(ef))) / n
        oref += float(np.linalg.norm(Ac - Af)) / n
    _close([me, oe], [mref, oref], 1e-12, "held-out errors vs loops")


# ------------------------------------------------ farthest-first traversal -
def check_farthest_first(o):
    """Farthest-first traversal against a from-scratch recomputation of every
    step; the chosen distances never increase; on tiny sets the result is
    within the traversal's factor-2 bound of the exhaustive optimum of the
    k-center problem it approximates (Gonzalez 1985); exact distance ties go
    to the lowest index."""
    rng = _rng(53)
    K = rng.normal(size=(40, 3))
    seeds = [5, 17]
    added = o.farthest_first(K, seeds, 12)
    S = list(seeds)
    prev = np.inf
    for i in added:
        best, arg = -1.0, -1
        for c in range(K.shape[0]):
            if c in S:
                continue
            dmin = min(float(((K[c] - K[j]) ** 2).sum()) for j in S)
            if dmin > best:
                best, arg = dmin, c
        assert i == arg, f"step chose {i}, expected {arg}"
        assert best <= prev + 1e-12, "chosen distance increased"
        prev = best
        S.append(i)
    assert len(added) == 10 and len(set(S)) == 12
    # factor-2 bound on the k-center radius (radius in plain distance)
    P = rng.normal(size=(11, 2))
    k = 3
    sel = [0] + list(o.farthest_first(P, [0], k))
    rad = max(min(np.linalg.norm(P[c] - P[j]) for j in sel) for c in range(len(P)))
    opt = min(max(min(np.linalg.norm(P[c] - P[j]) for j in comb) for c in range(len(P)))
              for comb in itertools.combinations(range(len(P)), k))
    assert rad <= 2 * opt + 1e-12, f"radius {rad} > 2 x optimum {opt}"
    # all keys taken: the traversal stops
    assert len(o.farthest_first(K[:4], [0], 10)) == 3
    # exact ties (integer points, so every squared distance is exact): the
    # lowest index wins.  From the seed at the origin, (2,0), (-2,0), (0,2)
    # tie at 4 and are taken in index order; then the four unit points tie
    # at 1 and the lowest two follow.
    P = np.array([[0, 0], [1, 0], [-1, 0], [0, 1], [0, -1], [2, 0], [-2, 0], [0, 2]], float)
    assert list(o.farthest_first(P, [0], 6)) == [5, 6, 7, 1, 2]


# ------------------------------------------------- baseline AM variant -----
def check_rms_scores(o):
    """RMS key scores against loops over the softmax probabilities; the RMS
    lies between the largest probability / sqrt(n) and the largest."""
    rng = _rng(81)
    n, T, d = 9, 7, 3
    Q = rng.normal(size=(n, d)) * 2
    K = rng.normal(size=(T, d))
    s = 0.6
    _, lse, _ = o.full_stats(Q, K, np.zeros((T, 1)), s)
    u = o.rms_key_scores(Q, K, lse, s)
    for j in range(T):
        ps = []
        for i in range(n):
            z = sum(math.exp(s * float(Q[i] @ K[l])) for l in range(T))
            ps.append(math.exp(s * float(Q[i] @ K[j])) / z)
        rms = math.sqrt(sum(p * p for p in ps) / n)
        _close(u[j], math.log(rms), 1e-12, "RMS score vs loops")
        assert max(ps) / math.sqrt(n) - 1e-15 <= rms <= max(ps) + 1e-15


def check_bounded_ls(o):
    """Bounded least squares: one iteration is the clipped unconstrained
    solution (numpy lstsq on the design matrix); two iterations re-solve the
    free weights with the pinned ones at their bounds (lstsq again); an
    interior solution is returned unchanged; when the two iterations reach
    the optimum it equals scipy's bounded-variable least squares and
    satisfies the bound-constrained KKT conditions."""
    from scipy.optimize import lsq_linear
    rng = _rng(82)
    lo, hi = math.exp(-3), math.exp(3)
    for trial in range(20):
        A = np.abs(rng.normal(size=(30, 5)))
        wtrue = np.exp(rng.uniform(-5, 5, size=5))
        b = A @ wtrue + 0.1 * rng.normal(size=30)
        G, c = A.T @ A, A.T @ b
        x0 = np.linalg.lstsq(A, b, rcond=None)[0]
        w1, _ = o.bounded_ls(G, c, lo, hi, 1)
        _close(w1, np.clip(x0, lo, hi), 1e-8 * max(1, np.abs(x0).max()), "one iteration")
        pinned = (x0 < lo) | (x0 > hi)
        w2, it = o.bounded_ls(G, c, lo, hi, 2)
        if pinned.any() and not pinned.all():
            F = ~pinned
            wp = np.clip(x0, lo, hi)
            xf = np.linalg.lstsq(A[:, F], b - A[:, pinned] @ wp[pinned], rcond=None)[0]
            ref = wp.copy()
            ref[F] = np.clip(xf, lo, hi)
            _close(w2, ref, 1e-7 * max(1, np.abs(xf).max()), "two iterations")
            g = G @ w2 - c
            inside = (w2 > lo) & (w2 < hi)
            kkt = (np.all(np.abs(g[inside]) <= 1e-6 * np.abs(c).max())
                   and np.all(g[w2 == lo] >= -1e-6 * np.abs(c).max())
                   and np.all(g[w2 == hi] <= 1e-6 * np.abs(c).max()))
            if kkt:
                ws = lsq_linear(A, b, bounds=(lo, hi), method="bvls", tol=1e-14).x
                _close(w2, ws, 1e-6 * max(1, np.abs(ws).max()), "optimum vs BVLS")
        if not pinned.any():
            _close(w2, x0, 1e-8 * max(1, np.abs(x0).max()), "interior solution")
            assert it == 1
    # an exact interior solution comes back after one iteration
    A = np.abs(rng.normal(size=(30, 4)))
    wi = np.exp(rng.uniform(-1, 1, size=4))
    w, it = o.bounded_ls(A.T @ A, A.T @ (A @ wi), lo, hi, 2)
    _close(w, wi, 1e-9, "interior solution")
    assert it == 1
    # every weight pushed below the lower bound: all pinned there
    w, it = o.bounded_ls(np.eye(3), -np.ones(3), lo, hi, 2)
    _close(w, np.full(3, lo), 0.0, "all at the lower bound")


def check_variant_t_equals_T(o):
    """The baseline variant keeping every key: w = 1 lies inside [e^-3, e^3],
    so beta = 0 and C_v = V."""
    rng = _rng(83)
    T, d, n_q = 10, 4, 30
    K = rng.standard_normal((T, d))
    Q = 0.5 * K[rng.integers(0, T, n_q)] + rng.standard_normal((n_q, d))
    V = rng.standard_normal((T, 2))
    r = o.compact_head_variant(Q, K, V, T, 1 / math.sqrt(d))
    assert list(r["idx"]) == list(range(T))
    _close(r["w"], np.ones(T), 1e-8, "variant t=T: w = 1")
    _close(r["Cv"], V, 1e-6, "variant t=T: C_v = V")


def check_chunk_boundaries(o):
    """The oracle forms its sums over query rows in chunks of o.CHUNK rows.
    With n = 2 CHUNK + 37 rows, every chunked function must agree with the
    same function evaluated on groups of rows that straddle the chunk
    boundaries, each group shorter than a chunk: row-wise results row by
    row, sums over rows as the sum over the groups, maxima as the maximum
    over the groups, the mean-square score through its group means.  A
    dropped, repeated or misplaced chunk breaks one of these."""
    rng = _rng(97)
    n, T, d, s = 2 * o.CHUNK + 37, 24, 8, 0.35
    Q = rng.normal(size=(n, d))
    K = rng.normal(size=(T, d))
    V = rng.normal(size=(T, 5))
    cuts = [0, 700, o.CHUNK - 3, o.CHUNK + 5, 2 * o.CHUNK - 1, 2 * o.CHUNK + 20, n]
    groups = list(zip(cuts[:-1], cuts[1:]))
    assert all(0 < b - a < o.CHUNK for a, b in groups)

    def close(x, y):
        assert np.allclose(x, y, rtol=1e-12, atol=1e-14), float(np.max(np.abs(np.asarray(x) - y)))

    m, lse, O = o.full_stats(Q, K, V, s)
    parts = [o.full_stats(Q[a:b], K, V, s) for a, b in groups]
    for k, full in enumerate((m, lse, O)):
        close(full, np.concatenate([p[k] for p in parts]))
    close(o.lse_over(Q, K, s), np.concatenate([o.lse_over(Q[a:b], K, s) for a, b in groups]))
    bias = rng.normal(size=T)
    valid = rng.random((n, T)) < 0.7
    out, lz = o.branch_attention(Q, K, V, bias, valid, s)
    bp = [o.branch_attention(Q[a:b], K, V, bias, valid[a:b], s) for a, b in groups]
    close(out, np.concatenate([p[0] for p in bp]))
    close(lz, np.concatenate([p[1] for p in bp]))
    close(o.key_scores(Q, K, lse, s),
          np.max([o.key_scores(Q[a:b], K, lse[a:b], s) for a, b in groups], axis=0))
    u = o.rms_key_scores(Q, K, lse, s)
    ms = sum((b - a) * np.exp(2.0 * o.rms_key_scores(Q[a:b], K, lse[a:b], s)) for a, b in groups)
    close(u, 0.5 * np.log(ms / n))
    Kc = K[:6]
    G, c, bb = o.mass_system(Q, Kc, m, lse, s)
    gp = [o.mass_system(Q[a:b], Kc, m[a:b], lse[a:b], s) for a, b in groups]
    close(G, sum(p[0] for p in gp))
    close(c, sum(p[1] for p in gp))
    close(bb, sum(p[2] for p in gp))
    w = np.array([0.5, 0.0, 1.5, 2.0, 0.0, 0.25])
    sup, H, R = o.output_system(Q, Kc, w, O, s)
    op = [o.output_system(Q[a:b], Kc, w, O[a:b], s) for a, b in groups]
    assert all(np.array_equal(sup, p[0]) for p in op)
    close(H, sum(p[1] for p in op))
    close(R, sum(p[2] for p in op))


ALL_CHECKS = [
    check_full_stats_brute, check_full_stats_closed_forms, check_key_scores_brute,
    check_select, check_mass_system_brute, check_nnls_bruteforce, check_nnls_scipy, check_nnls_planted_and_kkt,
    check_nnls_q_zero_and_caps, check_compact_weights, check_ols, check_t_equals_T,
    check_fit_zero_weight_branch, check_fit_duplicate_keys,
    check_fit_reduces_error, check_two_pass_brute, check_two_pass_full_shortlist,
    check_redistribute, check_combine_single_softmax, check_heldout_errors,
    check_farthest_first, check_rms_scores, check_bounded_ls, check_variant_t_equals_T,
    check_chunk_boundaries,
]
