"""Planted mistakes in a private copy of the oracle (CPU only): each plausible
slip -- a dropped scale, a flipped sign, a wrong reduction, a tie broken the
wrong way, a missing normalisation, a skipped step-back in the active set --
must fail at least one pin.  The real oracle is never modified."""
import importlib.util
import os

import numpy as np
import pytest

from oracle_pins import ALL_CHECKS

ORACLE_FILE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "__init__.py")


def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_mutant", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _no_scale(o):
    orig = o.full_stats
    o.full_stats = lambda Q, K, V, scale: orig(Q, K, V, 1.0)


def _unnormalised_output(o):
    orig = o.full_stats

    def f(Q, K, V, scale):
        m, lse, O = orig(Q, K, V, scale)
        return m, lse, O * np.exp(lse - m)[:, None]
    o.full_stats = f


def _score_plus_lse(o):
    orig = o.key_scores
    o.key_scores = lambda Q, K, lse, scale: orig(Q, K, -np.asarray(lse, float), scale)


def _score_min(o):
    def f(Q, K, lse, scale):
        S = scale * (np.asarray(Q, float) @ np.asarray(K, float).T) - np.asarray(lse)[:, None]
        return S.min(axis=0)
    o.key_scores = f


def _ties_high(o):
    def f(u, t):
        u = np.asarray(u)
        order = sorted(range(len(u)), key=lambda j: (-float(u[j]), -j))
        return np.sort(np.array(order[:t]))
    o.select = f


def _no_stepback(o):
    def f(G, c, max_outer=0, max_inner=0, tol=None):
        w = np.linalg.solve(np.asarray(G, float), np.asarray(c, float))
        return w, {"outer": 1, "inner": 1, "status": o.OK}
    o.nnls_lh = f


def _mass_unshifted(o):
    orig = o.mass_system
    o.mass_system = lambda Q, Kc, m, lse, scale: orig(Q, Kc, np.zeros_like(m), lse, scale)


def _weights_no_bias(o):
    orig = o.compact_weights
    o.compact_weights = lambda Q, Kc, beta, scale: orig(Q, Kc, np.zeros_like(beta), scale)


def _ols_diag(o):
    o.ols = lambda H, R: (np.asarray(R) / np.diag(H)[:, None], o.OK)


def _second_pass_full_lse(o):
    # the second pass normalised over every key instead of the shortlist
    def f(Q, K, qsel, t, k, scale):
        Q, K = np.asarray(Q, float), np.asarray(K, float)
        Qs = Q[np.asarray(qsel)]
        u1 = o.key_scores(Qs, K, o.lse_over(Qs, K, scale), scale)
        short = o.select(u1, min(k * t, K.shape[0]))
        u2 = o.key_scores(Q, K[short], o.lse_over(Q, K, scale), scale)
        return {"short": short, "u1": u1, "u2": u2, "idx": short[o.select(u2, t)]}
    o.two_pass_select = f


def _delta_not_shared(o):
    # the whole missing mass given to every key instead of Delta / t
    orig = o.redistribute_beta

    def f(Q, K, short, idx, scale):
        b = orig(Q, K, short, idx, scale)
        t = len(idx)
        return np.log(1 + t * np.expm1(b))
    o.redistribute_beta = f


def _delta_by_difference(o):
    # Delta as the float64 difference of the shortlist and selected sums
    def f(Q, K, short, idx, scale):
        Q, K = np.asarray(Q, float), np.asarray(K, float)
        S_all = scale * (Q @ K[np.asarray(short)].T)
        S_sel = scale * (Q @ K[np.asarray(idx)].T)
        M = S_all.max()
        m = np.exp(S_sel - M).mean(axis=0)
        delta = np.exp(S_all - M).sum(axis=1).mean() - m.sum()
        return np.log((m + delta / len(idx)) / m)
    o.redistribute_beta = f


def _combine_unbiased(o):
    # the compacted branch without its biases
    orig = o.combine_attention

    def f(Q, Ck, beta, Cv, Knew, Vnew, n_vis, scale):
        b = np.asarray(beta, float)
        return orig(Q, Ck, np.where(np.isfinite(b), 0.0, b), Cv, Knew, Vnew, n_vis, scale)
    o.combine_attention = f


def _mass_error_signed(o):
    # the mean log-mass difference without the absolute value
    def f(Qh, K, V, Ck, beta, Cv, scale):
        _, lse, O = o.full_stats(Qh, K, V, scale)
        b = np.asarray(beta, float)
        A, lz = o.branch_attention(Qh, Ck, Cv, b, np.ones((1, len(b)), bool), scale)
        return float(np.mean(lz - lse)), float(np.mean(np.linalg.norm(A - O, axis=1)))
    o.heldout_errors = f


def _farthest_by_sum(o):
    # farthest from the sum of distances to the set instead of the nearest
    def f(K, seeds, M):
        K = np.asarray(K, float)
        S = [int(x) for x in seeds]
        out = []
        while len(S) < M and len(S) < K.shape[0]:
            tot = sum(((K - K[j]) ** 2).sum(axis=1) for j in S)
            tot[S] = -np.inf
            i = int(np.argmax(tot))
            out.append(i)
            S.append(i)
        return np.asarray(out, np.int64)
    o.farthest_first = f


def _rms_as_mean(o):
    # mean attention probability instead of its root mean square
    def f(Q, K, lse, scale):
        Q, K, lse = np.asarray(Q, float), np.asarray(K, float), np.asarray(lse, float)
        P = np.exp(scale * (Q @ K.T) - lse[:, None])
        return np.log(P.mean(axis=0))
    o.rms_key_scores = f


def _bounded_pins_at_zero(o):
    # the re-solve holds the pinned weights at 0 instead of their bounds
    def f(G, c, lo, hi, iters):
        G, c = np.asarray(G, float), np.asarray(c, float)
        w = np.zeros(c.size)
        free = np.ones(c.size, bool)
        it = 0
        while it < iters and free.any():
            it += 1
            F = np.flatnonzero(free)
            w[F] = np.linalg.solve(G[np.ix_(F, F)], c[F])
            low, high = free & (w < lo), free & (w > hi)
            if not (low.any() or high.any()):
                break
            w[low], w[high] = 0.0, 0.0
            free &= ~(low | high)
        return np.clip(w, lo, hi), it
    o.bounded_ls = f


def _off_support_zeroed(o):
    # rows of C_v off the support set to 0 instead of the original values
    orig = o.fit_head

    def f(Q, K, V, idx, m, lse, O, scale, max_outer=0, max_inner=0):
        r = orig(Q, K, V, idx, m, lse, O, scale, max_outer, max_inner)
        r["Cv"][~(r["w"] > 0)] = 0.0
        return r
    o.fit_head = f


def _support_ignored(o):
    # zero weights replaced by a small positive weight before the output fit,
    # so every kept key enters the least squares
    orig = o.output_system

    def f(Q, Kc, w, O, scale):
        w = np.asarray(w, float)
        return orig(Q, Kc, np.where(w > 0, w, 1e-3), O, scale)
    o.output_system = f


def _duplicate_keeps_later(o):
    # of two equal kept keys, the earlier one dropped instead of the later one
    def later(Kc):
        Kc = np.asarray(Kc)
        dup = np.zeros(Kc.shape[0], dtype=bool)
        for j in range(Kc.shape[0] - 1):
            dup[j] = bool(np.any(np.all(Kc[j + 1:] == Kc[j], axis=1)))
        return dup
    o.later_duplicates = later


def _no_ridge(o):
    # a failed factorisation gives zeros instead of the ridge solution
    orig = o.ols

    def f(H, R):
        C, st = orig(H, R)
        return (np.zeros_like(C), st) if st == o.SINGULAR else (C, st)
    o.ols = f


def _farthest_ties_high(o):
    # distance ties in farthest-first broken towards the higher index
    def f(K, seeds, M):
        K = np.asarray(K, float)
        S = [int(s) for s in seeds]
        N = K.shape[0]
        taken = np.zeros(N, bool)
        taken[S] = True
        mind = np.full(N, np.inf)
        for j in S:
            mind = np.minimum(mind, ((K - K[j]) ** 2).sum(axis=1))
        added = []
        while len(S) < M and not taken.all():
            cand = np.where(taken, -np.inf, mind)
            i = int(N - 1 - np.argmax(cand[::-1]))  # last maximum
            added.append(i)
            S.append(i)
            taken[i] = True
            mind = np.minimum(mind, ((K - K[i]) ** 2).sum(axis=1))
        return np.asarray(added, np.int64)
    o.farthest_first = f


def _lse_is_max(o):
    # the log-normaliser replaced by the row maximum
    orig = o.full_stats

    def f(Q, K, V, scale):
        m, lse, O = orig(Q, K, V, scale)
        return m, m.copy(), O
    o.full_stats = f


def _select_by_score(o):
    # the kept keys returned in score order instead of ascending index order
    orig = o.select

    def f(u, t):
        idx = orig(u, t)
        return idx[np.argsort(-np.asarray(u)[idx], kind="stable")]
    o.select = f


def _nnls_clipped(o):
    # the unconstrained least-squares solution clipped at zero in place of NNLS
    def f(G, c, max_outer=0, max_inner=0, tol=None):
        w = np.linalg.lstsq(np.asarray(G, float), np.asarray(c, float), rcond=None)[0]
        return np.maximum(w, 0.0), {"outer": 1, "inner": 1, "status": o.OK}
    o.nnls_lh = f


def _weights_over_queries(o):
    # the compact softmax normalised over the queries instead of the keys
    def f(Q, Kc, beta, scale):
        L = scale * (np.asarray(Q, float) @ np.asarray(Kc, float).T) + np.asarray(beta, float)[None, :]
        E = np.exp(L - L.max(axis=0, keepdims=True))
        return E / E.sum(axis=0, keepdims=True)
    o.compact_weights = f


def _ridge_too_large(o):
    # the singular-system ridge a thousand times too large
    orig = o.ridge
    o.ridge = lambda M: 1000.0 * orig(M)


def _redistribute_over_T(o):
    # the dropped mass shared over all T keys instead of the t kept ones
    orig = o.redistribute_beta

    def f(Q, K, short, idx, scale):
        b = orig(Q, K, short, idx, scale)
        return np.log1p(np.expm1(b) * len(idx) / np.asarray(K).shape[0])
    o.redistribute_beta = f


def _combine_drops_appended(o):
    # tokens appended after compaction left out of the attention
    def f(Q, Ck, beta, Cv, Knew, Vnew, n_vis, scale):
        beta = np.asarray(beta, float)
        return o.branch_attention(Q, Ck, Cv, np.where(np.isfinite(beta), beta, 0.0),
                                  np.isfinite(beta)[None, :], scale)
    o.combine_attention = f


def _bounded_opposite_bound(o):
    # a weight that leaves [lo, hi] pinned at the opposite bound
    def f(G, c, lo, hi, iters):
        G, c = np.asarray(G, float), np.asarray(c, float)
        w = np.zeros(c.size)
        free = np.ones(c.size, bool)
        it = 0
        while it < iters and free.any():
            it += 1
            F, B = np.flatnonzero(free), np.flatnonzero(~free)
            w[F] = np.linalg.solve(G[np.ix_(F, F)], c[F] - G[np.ix_(F, B)] @ w[B])
            low, high = free & (w < lo), free & (w > hi)
            w[low], w[high] = hi, lo
            if not (low.any() or high.any()):
                break
            free &= ~(low | high)
        return w, it
    o.bounded_ls = f


def _chunk_tail_dropped(o):
    # the last, partial chunk of query rows never visited
    def ch(n, size=o.CHUNK):
        return [(a, a + size) for a in range(0, n - size + 1, size)] or [(0, n)]
    o._chunks = ch


def _chunks_overlap(o):
    # each chunk after the first starting one row early (that row counted twice)
    def ch(n, size=o.CHUNK):
        return [(max(0, a - 1), min(n, a + size)) for a in range(0, n, size)]
    o._chunks = ch


def _bb_dropped(o):
    # the constant term b.b of the mass residual left at zero
    orig = o.mass_system

    def f(Q, Kc, m, lse, scale):
        G, c, _ = orig(Q, Kc, m, lse, scale)
        return G, c, 0.0
    o.mass_system = f


MUTANTS = [_no_scale, _unnormalised_output, _score_plus_lse, _score_min, _ties_high,
           _no_stepback, _mass_unshifted, _weights_no_bias, _ols_diag, _second_pass_full_lse,
           _delta_not_shared, _delta_by_difference, _combine_unbiased, _mass_error_signed,
           _farthest_by_sum, _rms_as_mean, _bounded_pins_at_zero, _off_support_zeroed,
           _support_ignored, _duplicate_keeps_later, _no_ridge, _farthest_ties_high, _lse_is_max,
           _select_by_score, _nnls_clipped, _weights_over_queries, _ridge_too_large,
           _redistribute_over_T, _combine_drops_appended, _bounded_opposite_bound,
           _chunk_tail_dropped, _chunks_overlap, _bb_dropped]


@pytest.mark.parametrize("mutate", MUTANTS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutate):
    o = _fresh_oracle()
    mutate(o)
    caught = []
    for check in ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(o)
        except (AssertionError, np.linalg.LinAlgError) as e:
            caught.append((check.__name__, type(e).__name__))
    assert caught, f"no pin catches {mutate.__name__}"
