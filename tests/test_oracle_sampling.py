"""Pins of the oracle's sampling walk and rejection-sampling verification
against closed forms, a limiting case and the distribution-preservation
property of rejection sampling (no GPU)."""
import math

import numpy as np

import oracle


def test_two_candidate_walk_matches_the_logistic_closed_form():
    for s0, s1, T in [(1.0, 0.0, 1.0), (0.25, 0.75, 0.5), (-2.0, 1.0, 2.0)]:
        P = np.array([[[s0, s1], [-np.inf, -np.inf]]])
        q0 = 1.0 / (1.0 + math.exp((s1 - s0) / T))  # P(rank 0) for two options
        ranks, q, mg = oracle.sample_walk(P, T, [0.5])
        assert abs(q[0, 0] - q0) < 1e-12 and abs(q[0, 1] - (1 - q0)) < 1e-12
        assert oracle.sample_walk(P, T, [q0 - 1e-9])[0][0] == 0
        assert oracle.sample_walk(P, T, [q0 + 1e-9])[0][0] == 1
        assert abs(oracle.sample_walk(P, T, [q0 - 1e-6])[2][0] - 1e-6) < 1e-9


def test_zero_temperature_limit_is_the_greedy_walk():
    rng = np.random.default_rng(3)
    for _ in range(20):
        L, K = 5, 7
        P = rng.normal(size=(L, K, K))
        P[0, 1:] = -np.inf
        g, _, _, _ = oracle.greedy(P)
        for u in (rng.random(L), np.full(L, 0.999), np.zeros(L)):
            r, _, _ = oracle.sample_walk(P, 1e-6, u)
            assert r.tolist() == g.tolist()


def _random_case(rng, V=8, K=3, L=2):
    P = rng.normal(size=(L, K, K))
    P[0, 1:] = -np.inf
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(L)]).astype(np.int32)
    p = rng.dirichlet(np.ones(V), size=L + 1)
    return P, ids, p


def test_rejection_sampling_preserves_the_target_distribution():
    """The first emitted token is distributed as the target's p_0 whatever the
    draft distribution (the property that makes sampling lossless)."""
    rng = np.random.default_rng(7)
    V, K, L, T = 8, 3, 2, 0.7
    P, ids, p = _random_case(rng, V, K, L)
    draws = 60000
    counts = np.zeros(V)
    accepted0 = 0
    q0 = None
    for _ in range(draws):
        u = rng.random(2 * L + 1)
        ranks, q, _ = oracle.sample_walk(P, T, u[:L])
        q0 = q[0]
        path = ids[np.arange(L), ranks]
        n, emitted, _, _ = oracle.verify_rejection(path, ids, q, p, u[L:2 * L], u[2 * L])
        counts[emitted[0]] += 1
        accepted0 += n >= 1
    freq = counts / draws
    sigma = np.sqrt(p[0] * (1 - p[0]) / draws)
    assert np.all(np.abs(freq - p[0]) < 5 * sigma + 1e-4), (freq, p[0])
    # acceptance rate of the first draft: sum_j min(q(j), p(c_j))
    rate = sum(min(q0[j], p[0][ids[0, j]]) for j in range(K))
    assert abs(accepted0 / draws - rate) < 5 * math.sqrt(rate * (1 - rate) / draws) + 1e-4


def test_rejection_special_cases():
    rng = np.random.default_rng(9)
    V, K, L = 10, 4, 3
    P, ids, _ = _random_case(rng, V, K, L)
    for _ in range(50):
        u = rng.random(2 * L + 1)
        ranks, q, _ = oracle.sample_walk(P, 1.0, u[:L])
        path = ids[np.arange(L), ranks]
        # target equal to the draft on the candidates: every draft is accepted
        p = np.zeros((L + 1, V))
        for t in range(L):
            p[t, ids[t]] = q[t]
        p[L] = rng.dirichlet(np.ones(V))
        n, emitted, _, _ = oracle.verify_rejection(path, ids, q, p, u[L:2 * L], u[2 * L])
        assert n == L and emitted[:L].tolist() == path.tolist() and p[L, emitted[L]] > 0
        # target with no mass on the candidates of t = 0: immediate rejection, draw from p_0
        p2 = rng.dirichlet(np.ones(V), size=L + 1)
        p2[0, ids[0]] = 0.0
        p2[0] /= p2[0].sum()
        n, emitted, _, _ = oracle.verify_rejection(path, ids, q, p2, u[L:2 * L], u[2 * L])
        assert n == 0 and emitted[0] not in ids[0].tolist() and (emitted[1:] == -1).all()


def test_hand_worked_rejection_and_draw():
    """One draft rejected, worked by hand: p_0 = (0.1, 0.2, 0.3, 0.4), the only
    candidate is token 2 with q = 1. Acceptance min(1, 0.3/1) = 0.3 < u = 0.5, so
    it is rejected; the residual is (0.1, 0.2, 0, 0.4) with Z = 0.7; u_res = 0.2
    gives the target 0.14, crossed in vocabulary order at token 1 (running sums
    0.1, 0.3). With u_acc = 0.25 the draft is kept and the bonus comes from p_1."""
    ids = np.array([[2]], np.int32)
    path = np.array([2], np.int32)
    q = np.array([[1.0]])
    p = np.array([[0.1, 0.2, 0.3, 0.4], [0.5, 0.25, 0.125, 0.125]])
    n, emitted, am, rm = oracle.verify_rejection(path, ids, q, p, [0.5], 0.2)
    assert n == 0 and emitted.tolist() == [1, -1]
    assert abs(am[0] - 0.2) < 1e-12
    assert abs(rm - (0.14 - 0.1) / 0.7) < 1e-12  # the nearest CDF boundary is 0.1 (0.3 is farther)
    for u_res, tok in [(0.1, 0), (0.5, 3), (0.99, 3)]:  # targets 0.07, 0.35, 0.693
        assert oracle.verify_rejection(path, ids, q, p, [0.5], u_res)[1][0] == tok
    n, emitted, _, _ = oracle.verify_rejection(path, ids, q, p, [0.25], 0.6)  # bonus: target 0.6 in (0.5, 0.75]
    assert n == 1 and emitted.tolist() == [2, 1]
