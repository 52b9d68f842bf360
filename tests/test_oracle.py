"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-worked examples, the acceptance-length closed form from the pages' recall
table, brute-force path enumeration, library routines (fp64 matmul, stable
sort, einsum) and invariants of the walk. No GPU is needed."""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from speculative_decoding_draft_tcgen05_gb300 import workloads


def bits(x):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.as_tensor(np.asarray(x, dtype=np.float32))), "example must be exact in bf16"
    return workloads.bf16_bits(t)


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def run_example(ex, walk, zero_gate=False):
    WH = np.zeros_like(np.asarray(ex["W_H"], dtype=np.float32)) if zero_gate else ex["W_H"]
    return oracle.select(bits(ex["W"]), bits(ex["E"]), bits(ex["W_A"]), bits(ex["W_B"]), bits(WH),
                         bits(ex["hidden"]), ex["anchor"], ex["K"], walk=walk)


@pytest.mark.parametrize("name", ["hand_example_2pos.json", "hand_example_3pos.json"])
def test_hand_examples(golden_dir, name):
    ex = load(golden_dir, name)
    x = ex["expect"]
    r = run_example(ex, oracle.WALK_VITERBI)
    assert r["ids"].tolist() == x["ids"]
    assert r["vals"].tolist() == x["vals"]
    assert r["topk_margin"].tolist() == x["topk_margin"]
    # t = 0: only the anchor row exists
    assert r["P"][0, 0].tolist() == x["P_row0_t0"]
    assert np.all(np.isneginf(r["P"][0, 1:]))
    assert r["P"][1].tolist() == x["P_t1"]
    if "P_t2" in x:
        assert r["P"][2].tolist() == x["P_t2"]
    assert r["tokens"].tolist() == x["viterbi_tokens"]
    assert r["score"] == x["viterbi_score"]
    if "viterbi_ranks" in x:
        assert r["ranks"].tolist() == x["viterbi_ranks"]
        sm = [None if np.isinf(v) else v for v in r["step_margin"].tolist()]
        assert sm == x["viterbi_step_margin"]
        assert r["final_margin"] == x["viterbi_final_margin"]
    g = run_example(ex, oracle.WALK_GREEDY)
    assert g["tokens"].tolist() == x["greedy_tokens"]
    assert g["score"] == x["greedy_score"]
    if "greedy_step_margin" in x:
        assert g["step_margin"].tolist() == x["greedy_step_margin"]
    if "top1_tokens" in x:
        assert r["ids"][:, 0].tolist() == x["top1_tokens"]
        assert brute.path_score(r["P"], [0] * ex["L"]) == x["top1_score"]
    z = run_example(ex, oracle.WALK_VITERBI, zero_gate=True)
    assert z["tokens"].tolist() == x["no_gate_viterbi_tokens"]
    assert z["score"] == x["no_gate_viterbi_score"]
    n, emitted = oracle.verify(r["tokens"], x["target"])
    assert n == x["accept"]
    assert emitted.tolist() == x["emitted"]


def test_acceptance_length_closed_form(golden_dir):
    """The pages print per-position recall rates and an acceptance length per
    row. Enumerating every match pattern of the seven positions, weighting it
    by the product of the rates, and counting the oracle's accepted prefix plus
    the bonus token must reproduce the printed length. Counting all matches
    (not the leading prefix), or leaving out the bonus token, misses it."""
    g = load(golden_dir, "recall_tau.json")
    L = 7
    path = np.arange(1, L + 1, dtype=np.int32)
    for row in g["rows"]:
        r = row["rates"]
        tau = 0.0
        tau_all_matches = 0.0
        for pattern in itertools.product([0, 1], repeat=L):
            p = 1.0
            for t in range(L):
                p *= r[t] if pattern[t] else 1.0 - r[t]
            target = np.array([path[t] if pattern[t] else 1000 + t for t in range(L)] + [999], np.int32)
            n, emitted = oracle.verify(path, target)
            assert emitted[n] == target[n]
            tau += p * (n + 1)
            tau_all_matches += p * (sum(pattern) + 1)
        assert abs(tau - row["tau"]) <= g["tolerance"], (row["name"], tau)
        assert abs(tau_all_matches - row["tau"]) > 10 * g["tolerance"]
        assert abs((tau - 1) - row["tau"]) > 10 * g["tolerance"]


def _rand_bits(rng, shape, std=1.0):
    return workloads.bf16_bits(torch.from_numpy(rng.normal(0, std, size=shape).astype(np.float32)).to(torch.bfloat16))


def _f64(b):
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def test_logits_and_topk_against_library():
    rng = np.random.default_rng(11)
    V, d, N, K = 1000, 96, 5, 16
    Wb = _rand_bits(rng, (V, d), 0.05)
    # duplicated rows give exactly equal logits: the tie rule (smaller id first) must hold
    Wb[700] = Wb[3]
    Wb[701] = Wb[3]
    Hb = _rand_bits(rng, (N, d))
    U = oracle.logits(Wb, Hb, nthreads=2)
    ref = _f64(Hb) @ _f64(Wb).T
    np.testing.assert_allclose(U, ref, rtol=1e-12, atol=1e-12)
    for n in range(N):
        ids, vals, m = oracle.topk(U[n], K)
        order = torch.sort(torch.from_numpy(-U[n]), stable=True).indices.numpy()
        assert ids.tolist() == order[:K].tolist()
        assert vals.tolist() == U[n][order[:K]].tolist()
        assert m == U[n][order[K - 1]] - U[n][order[K]]
        rest = np.setdiff1d(np.arange(V), ids)
        assert U[n][rest].max() <= vals.min()
    # an exact three-way tie inside the list keeps ascending ids
    Ut = np.zeros(10)
    Ut[[7, 2, 5]] = 3.0
    ids, vals, m = oracle.topk(Ut, 2)
    assert ids.tolist() == [2, 5] and m == 0.0


def test_projection_and_pair_scores_against_library():
    rng = np.random.default_rng(12)
    e, d, K = 8, 64, 5
    P = _rand_bits(rng, (e, d), 0.1)
    x = _rand_bits(rng, (d,))
    np.testing.assert_allclose(oracle.project(P, x), _f64(P) @ _f64(x[None])[0], rtol=1e-12, atol=1e-14)
    A = rng.normal(size=(K, e))
    B = rng.normal(size=(K, e))
    g = rng.normal(size=e)
    U = rng.normal(size=K)
    S = oracle.pair_scores(A, g, B, U)
    np.testing.assert_allclose(S, U[None, :] + np.einsum("ik,k,jk->ij", A, g, B), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L,K,seed", [(1, 16, 1), (2, 16, 2), (3, 16, 3), (5, 3, 4), (4, 5, 5)])
def test_viterbi_against_brute_force(L, K, seed):
    rng = np.random.default_rng(seed)
    P = rng.normal(size=(L, K, K))
    P[0, 1:] = -np.inf
    ranks, score, sm, fm = oracle.viterbi(P)
    best, bscore, runner = brute.best_path(P)
    assert ranks.tolist() == best.tolist()
    assert abs(score - bscore) < 1e-12
    assert abs(fm - 0) >= 0  # defined
    # the greedy walk and the independent top-1 path never beat the max-sum path
    gr, gscore, _, _ = oracle.greedy(P)
    assert gscore <= score + 1e-12
    assert abs(brute.path_score(P, gr.tolist()) - gscore) < 1e-12
    top1 = [int(np.argmax(P[0, 0]))] + [0] * (L - 1)
    assert brute.path_score(P, top1) <= score + 1e-12


def test_viterbi_tie_rules():
    # equal incoming values: the smaller predecessor rank wins; equal finals: the smaller rank
    P = np.zeros((2, 3, 3))
    P[0, 0] = [1.0, 1.0, 0.0]
    P[0, 1:] = -np.inf
    P[1] = [[0.0, 2.0, 0.0], [0.0, 2.0, 0.0], [5.0, 0.0, 0.0]]
    ranks, score, sm, fm = oracle.viterbi(P)
    # delta0 = [1, 1, 0]; delta1 = [max(1,1,5)=5 from 2, max(3,3,0)=3 from 0, 1 from 0]
    assert ranks.tolist() == [2, 0] and score == 5.0
    P[1, 2, 0] = 2.0  # now delta1 = [2 (from 2, tie 1 vs 1 vs 2), 3, 1] -> final rank 1 from pred 0
    ranks, score, sm, fm = oracle.viterbi(P)
    assert ranks.tolist() == [0, 1] and score == 3.0 and sm[1] == 0.0
    Q = np.zeros((1, 4, 4))
    Q[0, 0] = [1.0, 3.0, 3.0, 2.0]
    Q[0, 1:] = -np.inf
    ranks, score, sm, fm = oracle.viterbi(Q)
    assert ranks.tolist() == [1] and fm == 0.0
    ranks, score, sm, fm = oracle.greedy(Q)
    assert ranks.tolist() == [1] and sm[0] == 0.0


def _tiny_inputs(seed, V=300, d=64, e=16, L=3, K=4, zero_gate=False):
    rng = np.random.default_rng(seed)
    W = _rand_bits(rng, (V, d), 0.1)
    E = _rand_bits(rng, (V, d), 0.3)
    WA = _rand_bits(rng, (e, d), 0.3)
    WB = _rand_bits(rng, (e, d), 0.3)
    WH = np.zeros((e, d), np.uint16) if zero_gate else _rand_bits(rng, (e, d), 0.3)
    h = _rand_bits(rng, (L, d))
    anchor = int(rng.integers(0, V))
    return W, E, WA, WB, WH, h, anchor, K


@pytest.mark.parametrize("seed", [21, 22, 23])
def test_whole_selector_against_library_and_brute_force(seed):
    """The oracle's whole pipeline against a composition of library routines
    (fp64 matmul, stable sort, einsum) and brute-force path enumeration."""
    W, E, WA, WB, WH, h, anchor, K = _tiny_inputs(seed)
    L = h.shape[0]
    r = oracle.select(W, E, WA, WB, WH, h, anchor, K)
    Wf, Ef, WAf, WBf, WHf, hf = map(_f64, (W, E, WA, WB, WH, h))
    U = hf @ Wf.T
    P = np.full((L, K, K), -np.inf)
    ids = np.zeros((L, K), np.int64)
    for t in range(L):
        ids[t] = torch.sort(torch.from_numpy(-U[t]), stable=True).indices.numpy()[:K]
    g = hf @ WHf.T
    for t in range(L):
        prev = [anchor] if t == 0 else ids[t - 1]
        A = Ef[prev] @ WAf.T
        Bm = Ef[ids[t]] @ WBf.T
        P[t, : len(prev)] = U[t, ids[t]][None, :] + np.einsum("ik,k,jk->ij", A, g[t], Bm)
    assert r["ids"].tolist() == ids.tolist()
    np.testing.assert_allclose(r["P"][np.isfinite(P)], P[np.isfinite(P)], rtol=1e-12, atol=1e-12)
    best, bscore, runner = brute.best_path(P)
    assert bscore - runner > 1e-9
    assert r["ranks"].tolist() == best.tolist()
    assert r["tokens"].tolist() == [int(ids[t, best[t]]) for t in range(L)]
    assert abs(r["score"] - bscore) < 1e-9
    assert abs(r["final_margin"]) > 0
    # the same through the given-candidates entry
    s = oracle.select_given(W, E, WA, WB, WH, h, anchor, r["ids"])
    assert s["tokens"].tolist() == r["tokens"].tolist()
    np.testing.assert_array_equal(s["P"], r["P"])


def test_zero_gate_gives_independent_top1():
    W, E, WA, WB, WH, h, anchor, K = _tiny_inputs(31, L=5, K=6, zero_gate=True)
    r = oracle.select(W, E, WA, WB, WH, h, anchor, K)
    assert r["ranks"].tolist() == [0] * 5
    assert r["tokens"].tolist() == r["ids"][:, 0].tolist()


def test_verify_planted_prefix_and_bounds():
    rng = np.random.default_rng(5)
    L, V = 7, 1000
    for _ in range(200):
        path = rng.integers(0, V, L).astype(np.int32)
        n0 = int(rng.integers(0, L + 1))
        tgt = workloads.plant_targets(torch.from_numpy(path[None]), torch.from_numpy(
            rng.integers(0, V, (1, L + 1)).astype(np.int32)), torch.tensor([n0], dtype=torch.int32), V)[0].numpy()
        n, emitted = oracle.verify(path, tgt)
        assert n == n0 and 0 <= n <= L
        assert emitted[:n].tolist() == path[:n].tolist() and emitted[n] == tgt[n]
        assert (emitted[n + 1:] == -1).all()
