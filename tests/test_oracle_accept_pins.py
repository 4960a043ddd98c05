"""Pins of the oracle's stochastic acceptance: ``accept_stochastic`` (the
ratio test, the residual and the bonus draw) and ``race_sample`` (the
exponential race), the two functions the GPU accept kernel is compared with.

What fixes them (none re-types the oracle's code):
  * the lossless theorem (DFlash Guide, "The Cost Breakdown of Speculative
    Rounds", verification phase; "DFlash: Diffusion Drafts the Block", the
    lossless rule: the emitted stream is distributed exactly as the target's):
    an exact enumeration of the rule's emitted-stream distribution, with no
    random numbers, must equal the target's to 1e-12, for sampled drafts with
    their full q and for argmax drafts with the point-mass q;
  * the same rule's per-round outcome probabilities (accept a prefix, then a
    residual or bonus token), written out in closed form, against the
    empirical outcome frequencies of ``accept_stochastic`` itself (chi-square),
    and the lossless multi-round stream run through ``accept_stochastic``;
  * the exponential race's defining property (v wins with probability
    r(v)/sum r) against ``race_sample`` itself;
  * the S = 2 reading: with sampled drafts whose earlier positions are drawn
    after (and conditioned on) later committed ones, the per-position ratio
    test is not exactly lossless (the enumeration shows a nonzero gap), while
    argmax drafts with the point-mass q stay exact.
"""
import itertools

import numpy as np
import pytest
import scipy.stats

from oracle import dflash_oracle as O


# ---------------------------------------------------------------- the rule, enumerated

def _residual(p, q_row, d):
    """norm(max(0, p - q)); the point-mass q (q_row None) zeroes p at d; a
    residual without mass falls back to p."""
    if q_row is None:
        r = p.copy()
        r[d] = 0.0
    else:
        r = np.maximum(0.0, p - q_row)
    s = r.sum()
    return p if s <= 0 else r / s


def _outcomes_fixed_drafts(P, Q, d):
    """Exact outcome distribution of one round with fixed drafts d [K]:
    {(tau, emitted tuple): probability}.  P [K+1, V] target rows, Q [K, V]
    draft rows or None (point mass at d).  Accept d_i with probability
    a_i = min(1, P_i(d_i)/Q_i(d_i)); on the first reject emit a residual
    token; after K accepts emit a token of P_K."""
    K, V = len(d), P.shape[1]
    out = {}
    reach = 1.0
    for i in range(K):
        qd = 1.0 if Q is None else Q[i, d[i]]
        a = 1.0 if qd <= 0 else min(1.0, P[i, d[i]] / qd)
        res = _residual(P[i], None if Q is None else Q[i], d[i])
        for v in range(V):
            w = reach * (1.0 - a) * res[v]
            if w > 0:
                out[(i, tuple(d[:i]) + (v,))] = w
        reach *= a
    for v in range(V):
        if reach * P[K, v] > 0:
            out[(K, tuple(d) + (v,))] = reach * P[K, v]
    return out


class _Model:
    """A target p(. | prefix) and a draft q(. | prefix) over vocab V, each an
    independent Dirichlet draw per prefix (so both depend on the context)."""

    def __init__(self, V, seed, q_conc=0.7):
        self.V, self.seed, self.q_conc = V, seed, q_conc
        self._p, self._q = {}, {}

    def p(self, prefix):
        if prefix not in self._p:
            g = np.random.default_rng([self.seed, 1, len(prefix)] + list(prefix))
            self._p[prefix] = g.dirichlet(np.ones(self.V))
        return self._p[prefix]

    def q(self, prefix):
        if prefix not in self._q:
            g = np.random.default_rng([self.seed, 2, len(prefix)] + list(prefix))
            self._q[prefix] = g.dirichlet(np.ones(self.V) * self.q_conc)
        return self._q[prefix]


def _round_dist(m, s, K, sampled):
    """Emitted-token distribution of one round from context s: {emitted: prob}.

    sampled: d_i ~ q(. | s + d_<i) and the full q enters the ratio and the
    residual; otherwise d_i = argmax q(. | s + d_<i) with the point-mass q.
    The target rows are p(. | s + d_<i), as a verify pass over the drafts
    gives them.  The walk descends only through accepted drafts: drafts after
    the first reject do not change what is emitted, and their probabilities
    sum to one."""
    out = {}

    def walk(dp, w):
        i = len(dp)
        P = m.p(s + dp)
        if i == K:
            for y in range(m.V):
                out[dp + (y,)] = out.get(dp + (y,), 0.0) + w * P[y]
            return
        qrow = m.q(s + dp)
        cands = range(m.V) if sampled else [int(np.argmax(qrow))]
        for d in cands:
            wq = w * (qrow[d] if sampled else 1.0)
            qd = qrow[d] if sampled else 1.0
            a = 1.0 if qd <= 0 else min(1.0, P[d] / qd)
            res = _residual(P, qrow if sampled else None, d)
            for y in range(m.V):
                if res[y] > 0:
                    out[dp + (y,)] = out.get(dp + (y,), 0.0) + wq * (1.0 - a) * res[y]
            if a > 0:
                walk(dp + (d,), wq * a)

    walk((), 1.0)
    return out


def _stream_dist(m, K, n, sampled):
    """Distribution of the first n emitted tokens over as many rounds as
    needed, each round starting from the tokens emitted so far."""
    memo = {}

    def f(s):
        if s in memo:
            return memo[s]
        res = {}
        for em, w in _round_dist(m, s, K, sampled).items():
            s2 = s + em
            if len(s2) >= n:
                c = s2[len(s):n]
                res[c] = res.get(c, 0.0) + w
            else:
                for c2, w2 in f(s2).items():
                    c = em + c2
                    res[c] = res.get(c, 0.0) + w * w2
        memo[s] = res
        return res

    return f(())


@pytest.mark.parametrize("K,n,sampled", [(2, 3, True), (2, 3, False), (3, 4, True), (3, 4, False)])
def test_lossless_theorem_exact_enumeration(K, n, sampled):
    """The rule's emitted stream equals the target's: every sequence of the
    first n tokens has probability prod_j p(y_j | y_<j), to 1e-12."""
    V = 8
    m = _Model(V, seed=40 + K + 10 * sampled)
    got = _stream_dist(m, K, n, sampled)
    worst = 0.0
    for y in itertools.product(range(V), repeat=n):
        want = 1.0
        for j in range(n):
            want *= m.p(y[:j])[y[j]]
        worst = max(worst, abs(got.get(y, 0.0) - want))
    assert worst < 1e-12, worst
    assert abs(sum(got.values()) - 1.0) < 1e-12


def test_s2_sampled_drafts_are_not_exactly_lossless():
    """The S = 2 counterexample (K = 2, vocab 3): position 1 is committed in
    the first pass, d_1 ~ q_1, and position 0 is drafted in the second pass
    conditioned on it, d_0 ~ q_0(. | d_1).  The per-position ratio test with
    those draft distributions leaves a nonzero gap in the two-token stream
    (after accepting d_0, the conditional of d_1 is no longer q_1), while
    argmax drafts with the point-mass q stay exact."""
    V = 3
    g = np.random.default_rng(5)
    p0 = g.dirichlet(np.ones(V))
    p1 = g.dirichlet(np.ones(V), size=V)          # p1[y0] = p(. | y0)
    q1 = g.dirichlet(np.ones(V))
    q0 = g.dirichlet(np.ones(V), size=V)          # q0[d1] = q(d0 | d1)
    target = p0[:, None] * p1

    def stream(sampled):
        P = np.zeros((V, V))
        d1s = range(V) if sampled else [int(np.argmax(q1))]
        for d1 in d1s:
            w1 = q1[d1] if sampled else 1.0
            d0s = range(V) if sampled else [int(np.argmax(q0[d1]))]
            for d0 in d0s:
                w = w1 * (q0[d1][d0] if sampled else 1.0)
                qa = q0[d1] if sampled else None
                a0 = min(1.0, p0[d0] / (qa[d0] if sampled else 1.0))
                # reject at 0: y0 from the residual, y1 from an exact target step
                r0 = _residual(p0, qa, d0)
                P += w * (1 - a0) * r0[:, None] * p1
                # accept d0, then the test at position 1 against p(. | d0)
                qb = q1 if sampled else None
                a1 = min(1.0, p1[d0][d1] / (qb[d1] if sampled else 1.0))
                P[d0, d1] += w * a0 * a1
                P[d0] += w * a0 * (1 - a1) * _residual(p1[d0], qb, d1)
        return P

    gap_sampled = np.abs(stream(True) - target).max()
    gap_argmax = np.abs(stream(False) - target).max()
    assert gap_sampled > 1e-3, gap_sampled
    assert gap_argmax < 1e-12, gap_argmax


# ---------------------------------------------------------------- the oracle's code

def _rows(V, K, rng):
    """Target logits rows (one set shared by every sequence), draft rows q
    and drafts d: q_i(d_i) = 0.6 and p_i(d_i) = 0.35, the rest of each row
    spread at random over the other tokens, so every position both accepts
    and rejects with fair probability under either q."""
    d = rng.integers(0, V, size=K)
    Q = np.zeros((K, V))
    P = np.zeros((K + 1, V))
    for i in range(K):
        others = np.arange(V) != d[i]
        Q[i, d[i]], Q[i, others] = 0.6, 0.4 * rng.dirichlet(np.ones(V - 1))
        P[i, d[i]], P[i, others] = 0.35, 0.65 * rng.dirichlet(np.ones(V - 1))
    P[K] = rng.dirichlet(np.ones(V))
    return np.log(P), Q, d


@pytest.mark.parametrize("point_mass", [True, False])
def test_accept_stochastic_equals_vectorised_trials(point_mass):
    """accept_stochastic (one sequence at a time) and accept_stochastic_trials
    (all trials at once) take the same decisions on the same Philox counters:
    tau and every emitted token, rejects and bonus draws included."""
    V, K, N = 8, 4, 1200
    rng = np.random.default_rng(31 + point_mass)
    z, Q, _ = _rows(V, K, rng)
    d = np.stack([[rng.choice(V, p=Q[i]) for i in range(K)] for _ in range(N)])
    P = np.stack([O.softmax(z[i]) for i in range(K + 1)])
    zz = np.broadcast_to(z, (N, K + 1, V)).copy()
    qq = None if point_mass else np.broadcast_to(Q, (N, K, V)).copy()
    tau_a, em_a, n_a = O.accept_stochastic(zz, d, qq, 1.0, 77, 5)
    tau_b, em_b = O.accept_stochastic_trials(P, None if point_mass else Q, d, 77, 5)
    np.testing.assert_array_equal(tau_a, tau_b)
    np.testing.assert_array_equal(em_a, em_b)
    np.testing.assert_array_equal(n_a, tau_a + 1)
    assert set(np.unique(tau_a)) >= {0, 1, K}          # early rejects and the bonus path occur


def _chi_square_outcomes(counts, probs, N):
    """Chi-square p-value of outcome counts against probabilities, pooling
    outcomes with expected count below 5 into one cell."""
    keys = sorted(set(probs) | set(counts))
    exp = np.array([N * probs.get(k, 0.0) for k in keys])
    obs = np.array([counts.get(k, 0) for k in keys], float)
    assert obs[exp == 0].sum() == 0, "an outcome of probability 0 occurred"
    small = exp < 5
    e = np.append(exp[~small], exp[small].sum())
    o = np.append(obs[~small], obs[small].sum())
    if e[-1] == 0:
        e, o = e[:-1], o[:-1]
    return scipy.stats.chisquare(o, e * o.sum() / e.sum()).pvalue


@pytest.mark.parametrize("point_mass", [True, False])
def test_accept_stochastic_outcome_frequencies(point_mass):
    """accept_stochastic's (tau, emitted) frequencies over many sequences with
    the same rows and drafts (each its own Philox sequence index) match the
    rule's outcome probabilities, residual and bonus tokens included."""
    V, K, N = 8, 3, 12000
    rng = np.random.default_rng(17 + point_mass)
    z, Q, d = _rows(V, K, rng)
    P = np.stack([O.softmax(z[i]) for i in range(K + 1)])
    probs = _outcomes_fixed_drafts(P, None if point_mass else Q, d)
    assert {k[0] for k in probs} == set(range(K + 1))
    zz = np.broadcast_to(z, (N, K + 1, V)).copy()
    qq = None if point_mass else np.broadcast_to(Q, (N, K, V)).copy()
    tau, em, _ = O.accept_stochastic(zz, np.broadcast_to(d, (N, K)), qq, 1.0, 1234, 9)
    counts = {}
    for t, e in zip(tau, em):
        k = (int(t), tuple(int(x) for x in e[:t + 1]))
        counts[k] = counts.get(k, 0) + 1
    assert _chi_square_outcomes(counts, probs, N) > 1e-3
    # every branch of the rule is exercised
    assert {k[0] for k in counts} == set(range(K + 1))


@pytest.mark.parametrize("point_mass", [True, False])
def test_lossless_stream_monte_carlo_through_accept_stochastic(point_mass):
    """The spec check run through accept_stochastic itself: vocab 8,
    K = 4, position-dependent target and draft rows; rounds chained until
    each stream holds 3 tokens; each token's distribution and the first two
    tokens' joint distribution equal the target's (chi-square, TV bound)."""
    V, K, n_tok, N = 8, 4, 3, 16000
    rng = np.random.default_rng(60 + point_mass)
    P = rng.dirichlet(np.ones(V), size=n_tok + K + 1)
    Q = rng.dirichlet(np.ones(V) * 0.7, size=n_tok + K + 1)
    logP = np.log(P)
    pos = np.zeros(N, int)
    toks = np.full((N, n_tok), -1)
    step = 0
    while (pos < n_tok).any():
        for s in np.unique(pos[pos < n_tok]):
            idx = np.flatnonzero(pos == s)
            rows_q = Q[s:s + K]
            if point_mass:
                d = np.broadcast_to(np.argmax(rows_q, axis=1), (idx.size, K))
                qq = None
            else:
                d = np.stack([[rng.choice(V, p=rows_q[i]) for i in range(K)] for _ in idx])
                qq = np.broadcast_to(rows_q, (idx.size, K, V))
            zz = np.broadcast_to(logP[s:s + K + 1], (idx.size, K + 1, V))
            tau, em, _ = O.accept_stochastic(zz, d, qq, 1.0, 99 + point_mass, 500 + step)
            for j in range(K + 1):
                tgt = pos[idx] + j
                ok = (tau >= j) & (tgt < n_tok)
                toks[idx[ok], tgt[ok]] = em[ok, j]
            pos[idx] += tau + 1
            step += 1
    for j in range(n_tok):
        cnt = np.bincount(toks[:, j], minlength=V)
        assert scipy.stats.chisquare(cnt, N * P[j]).pvalue > 1e-3, (j, cnt / N, P[j])
    cells = np.bincount(toks[:, 0] * V + toks[:, 1], minlength=V * V)
    expect = N * np.outer(P[0], P[1]).ravel()
    assert scipy.stats.chisquare(cells, expect).pvalue > 1e-3
    assert 0.5 * np.abs(cells - expect).sum() / N < 3 * np.sqrt(V * V / N)


def test_race_sample_frequencies():
    """race_sample(r) returns v with probability r(v)/sum r: one call per
    sequence index b, zero-mass entries never win."""
    V, N = 8, 30000
    rng = np.random.default_rng(23)
    r = rng.dirichlet(np.ones(V)) * 3.7               # unnormalised on purpose
    r[5] = 0.0
    got = np.array([O.race_sample(r, 11, 4, b, 2) for b in range(N)])
    cnt = np.bincount(got, minlength=V)
    assert cnt[5] == 0
    keep = r > 0
    assert scipy.stats.chisquare(cnt[keep], N * r[keep] / r.sum()).pvalue > 1e-3


def test_race_sample_uses_the_race_stream_uniforms():
    """The race's winner is the argmax of r(v) / -ln U_v with U_v the
    race-stream uniform at (seed, round, b, i, v): with r uniform the winner
    is the v whose uniform is largest (E_v smallest), which the Philox
    known-answer vectors fix independently of the race code."""
    V = 16
    r = np.ones(V)
    for b in range(50):
        u = O.rng_uniform(7, 3, b, 1, O.STREAM_RACE, np.arange(V))
        assert O.race_sample(r, 7, 3, b, 1) == int(np.argmax(u))
