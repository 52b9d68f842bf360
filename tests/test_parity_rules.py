"""The parity rules themselves, on the CPU: a stand-in for the GPU's outputs
built from the oracle's own results (values rounded to fp32) must pass
``parity.compare``, and each planted mistake in it must fail. This checks the
comparison code that the GPU tests rely on, without a GPU."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl


def fake_gpu(inp, orc, walk=0, targets=None, chosen=None):
    """GPU-shaped outputs from oracle results ``chosen`` (default ``orc``)."""
    chosen = chosen or orc
    w = inp.wl
    B = w.B
    out = dict(topk_ids=np.zeros((B, w.L, w.K), np.int32), topk_vals=np.zeros((B, w.L, w.K), np.float32),
               pair_scores=np.zeros((B, w.L, w.K, w.K), np.float32), path=np.zeros((B, w.L), np.int32),
               path_score=np.zeros(B, np.float32), tie_flags=np.zeros((B, w.L), np.uint8),
               accept=np.zeros(B, np.int32), emitted=np.zeros((B, w.L + 1), np.int32))
    for s, r in chosen.items():
        out["topk_ids"][s] = r["ids"]
        out["topk_vals"][s] = r["vals"]
        out["pair_scores"][s] = r["P"]
        out["path"][s] = r["tokens"]
        out["path_score"][s] = r["score"]
        for t in range(w.L):
            m = r["step_margin"][t]
            if np.isfinite(m) and m < parity.TIE_EPS:
                out["tie_flags"][s, t] |= 1
        if walk == 0 and r["final_margin"] < parity.TIE_EPS:
            out["tie_flags"][s, w.L - 1] |= 2
        if targets is not None:
            n, em = oracle.verify(r["tokens"], targets[s])
            out["accept"][s] = n
            out["emitted"][s] = em
    return out


@pytest.fixture(scope="module")
def tiny():
    inp = parity.inputs_for("tiny")
    orc = parity.run_oracle(inp, range(inp.wl.B))
    targets = {s: inp.target_rand[s].numpy() for s in range(inp.wl.B)}
    return inp, orc, targets


def test_oracle_outputs_pass(tiny):
    inp, orc, targets = tiny
    rep = parity.compare(inp, fake_gpu(inp, orc, targets=targets), orc, targets=targets)
    assert rep["path_equal"] == inp.wl.B and rep["accept_checked"] == inp.wl.B
    assert rep["flags_checked"] == inp.wl.B * inp.wl.L  # L-1 step flags and the final flag per sequence


@pytest.mark.parametrize("mistake", ["path", "flag", "set", "logit", "table", "accept"])
def test_planted_mistakes_fail(tiny, mistake):
    inp, orc, targets = tiny
    g = fake_gpu(inp, orc, targets=targets)
    s, t = 1, 3
    if mistake == "path":
        g["path"][s, t] = g["topk_ids"][s, t, 5]
    elif mistake == "flag":
        g["tie_flags"][s, t] ^= 1
    elif mistake == "set":  # a token far below the boundary replaces the K-th candidate
        U = oracle.logits(wl.bf16_bits(inp.W), wl.bf16_bits(inp.hidden[s][t:t + 1]))[0]
        g["topk_ids"][s, t, -1] = int(np.argmin(U))
    elif mistake == "logit":
        g["topk_vals"][s, t, 2] += 0.05
    elif mistake == "table":
        g["pair_scores"][s, t, 4, 7] += 0.05
    elif mistake == "accept":
        g["accept"][s] = (g["accept"][s] + 1) % (inp.wl.L + 1)
    with pytest.raises(AssertionError):
        parity.compare(inp, g, orc, targets=targets)


def test_own_table_optimality_check(tiny):
    """The property check on the GPU's own tables accepts the best path and
    rejects a worse one, for both walks."""
    inp, orc, _ = tiny
    for walk in (0, 1):
        r = parity.run_oracle(inp, [0], walk=walk)[0]
        P = r["P"].astype(np.float32)
        parity.optimal_on_own_tables(P, list(r["ranks"]), walk)
        worse = list(r["ranks"])
        worse[-1] = int(np.argsort(P[-1, worse[-2]])[0])  # the lowest successor at the last step
        with pytest.raises(AssertionError):
            parity.optimal_on_own_tables(P, worse, walk)


def test_valid_swap_at_a_tied_boundary_is_followed():
    """Two vocabulary rows with equal weights tie exactly at the top-K
    boundary: either may be kept. A stand-in that keeps the other one passes
    (its path is compared against the oracle run on that set); a swap with a
    token that is not tied fails."""
    w = wl.custom(name="tied", B=1, L=3, K=16, V=40, d=64, seed=3, std_w=0.05)
    inp = wl.make_inputs(w)
    h = inp.hidden[0].float()
    U = (inp.W.float() @ h.T)  # [V, L], only to find the boundary tokens of this fixture
    order = torch.argsort(U[:, 1], descending=True)
    kth, nxt = int(order[15]), int(order[16])
    inp.W[nxt] = inp.W[kth]  # the two tokens now tie exactly at every position
    orc = parity.run_oracle(inp, [0])
    r = orc[0]
    assert r["topk_margin"][1] == 0.0
    ids = r["ids"].copy()
    other = nxt if kth in ids[1] else kth
    ids[1][ids[1] == (kth if other == nxt else nxt)] = other
    alt = oracle.select_given(*parity._bits(inp), wl.bf16_bits(inp.hidden[0]), int(inp.anchor[0]),
                              np.ascontiguousarray(ids))
    alt["ids"] = ids
    g = fake_gpu(inp, orc, chosen={0: alt})
    rep = parity.compare(inp, g, orc)
    assert rep["topk_swapped"] >= 1
    bad = fake_gpu(inp, orc, chosen={0: alt})
    far = int(order[-1])
    bad["topk_ids"][0, 1][bad["topk_ids"][0, 1] == other] = far
    with pytest.raises(AssertionError):
        parity.compare(inp, bad, orc)


def _tables(rng, L, K):
    P = rng.normal(size=(L, K, K))
    P[0, 1:] = -np.inf
    return P


def test_viterbi_open_decision_takes_valid_alternatives():
    """A planted near-tie at one node of the max-sum walk: the path through the
    other predecessor (with the best prefix ending there) is accepted, a path
    that also changes a decided position or goes through a clearly worse
    predecessor is not."""
    rng = np.random.default_rng(5)
    L, K = 5, 4
    P = _tables(rng, L, K)
    ranks = list(oracle.viterbi(P)[0])
    bi, j = ranks[2], ranks[3]
    gi, worse = [i for i in range(K) if i != bi][:2]
    s_b = oracle.viterbi(parity._force_end(P[:3], bi))[1]
    s_g = oracle.viterbi(parity._force_end(P[:3], gi))[1]
    P[3, gi, j] = s_b + P[3, bi, j] - s_g - 1e-5  # via gi: 1e-5 below the best incoming value
    s_w = oracle.viterbi(parity._force_end(P[:3], worse))[1]
    P[3, worse, j] = s_b + P[3, bi, j] - s_w - 0.5  # via `worse`: clearly below
    assert list(oracle.viterbi(P)[0]) == ranks and oracle.viterbi(P)[2][3] < parity.TIE_EPS
    assert parity.check_viterbi_path(P, ranks, 0.0) >= 1
    alt = list(oracle.viterbi(parity._force_end(P[:3], gi))[0]) + ranks[3:]
    assert alt != ranks
    assert parity.check_viterbi_path(P, alt, 0.0) >= 1
    wrong = list(alt)
    wrong[4] = (wrong[4] + 1) % K  # a decided position
    with pytest.raises(AssertionError):
        parity.check_viterbi_path(P, wrong, 0.0)
    bad = list(oracle.viterbi(parity._force_end(P[:3], worse))[0]) + ranks[3:]
    with pytest.raises(AssertionError):
        parity.check_viterbi_path(P, bad, 0.0)


def test_greedy_open_step_takes_valid_alternatives():
    rng = np.random.default_rng(6)
    L, K = 5, 4
    P = _tables(rng, L, K)
    ranks = list(oracle.greedy(P)[0])
    row = P[2, ranks[1]]
    other = [k for k in range(K) if k != ranks[2]]
    row[other[0]] = row[ranks[2]] - 1e-5  # a near-tied successor at step 2
    row[other[1]] = row[ranks[2]] - 0.5
    row[other[2]] = row[ranks[2]] - 0.7
    assert list(oracle.greedy(P)[0]) == ranks
    assert parity.check_greedy_path(P, ranks, 0.0) >= 1
    # continuing from the near-tied successor with the best successors from there on
    alt = ranks[:2] + [other[0]]
    prev = other[0]
    for t in range(3, L):
        prev = int(np.argmax(P[t, prev]))
        alt.append(prev)
    assert parity.check_greedy_path(P, alt, 0.0) >= 1
    bad = ranks[:2] + [other[1]] + alt[3:]
    with pytest.raises(AssertionError):
        parity.check_greedy_path(P, bad, 0.0)
