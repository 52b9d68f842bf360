"""Shared helpers of the parity tests: run the CUDA path and the CPU oracle on
the same seeded inputs and compare them under the stated rules.

Rules (bf16 inputs, fp32 accumulation on the GPU, fp64 in the oracle):
  - top-K id sets are bit-exact at every position whose oracle boundary gap
    U_(K) - U_(K+1) is at least TIE_EPS. Where it is smaller, several sets are
    correct: the GPU's set must then be a valid one (every token it swapped
    in or out lies within TIE_EPS of the boundary in the oracle's own fp64
    logits);
  - the later stages are compared against the oracle run on that valid set
    (the "conditional" reference: the oracle's own candidates, with the
    swapped tokens of excused positions, ordered by the oracle's logits).
    Its logits, every pair-table entry, the walk and the accept check follow;
  - paths and accept lengths are bit-exact, except at walk decisions whose
    oracle margin is below TIE_EPS (reported, not failed). There the GPU's
    choice must score within TIE_EPS of the best, and the rest of its path is
    compared with the oracle's walk continued from that choice, so every
    position of every path is checked (``check_viterbi_path``,
    ``check_greedy_path``). A path that took another valid choice has its
    accept length checked on its own tokens;
  - the GPU's tie flags agree bit for bit with (oracle margin < TIE_EPS),
    except inside a band around TIE_EPS that covers how far fp32 tables and
    an fp32 recursion can move a margin (see ``tie_band``);
  - the GPU's path is an optimal path of the GPU's own tables (a property that
    holds for every sequence, including excused ones);
  - logits and pair scores agree within |gpu - ref| <= ATOL + RTOL * |ref|.
No input of the oracle comes from the GPU: targets are planted on the
oracle's own path, and the conditional reference only takes from the GPU
which of the oracle's valid alternatives it chose.
"""
from __future__ import annotations

import functools
import os

import numpy as np
import torch

import oracle
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl

RTOL = 2e-2
ATOL = 2e-3
TIE_EPS = 1e-3
F32_HALF_ULP = 2.0 ** -24  # relative rounding error of one fp32 addition


@functools.lru_cache(maxsize=1)
def inputs_for(name: str):
    return wl.make_inputs(wl.WORKLOADS[name])


def oracle_threads() -> int:
    return max(1, min(len(os.sched_getaffinity(0)), 64))


def close(gpu, ref, rtol=RTOL, atol=ATOL):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(gpu - ref) <= atol + rtol * np.abs(ref)


def to_device(inp: wl.Inputs, dev):
    return {k: getattr(inp, k).to(dev) for k in ("W", "E", "W_A", "W_B", "W_H", "hidden", "anchor")}


def run_gpu(inp: wl.Inputs, dev="cuda", walk=0, max_batch=None, dtensors=None, targets=None, tables=False,
            dedup=False):
    """Runs the whole selector through the C ABI (and, given target tokens
    [B, L+1], the accept check); returns CPU numpy outputs."""
    import speculative_decoding_draft_tcgen05_gb300 as pkg
    w = inp.wl
    d = dtensors if dtensors is not None else to_device(inp, dev)
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K,
                      max_batch=max_batch or w.B, walk=walk, tie_eps=TIE_EPS, tables=tables, dedup=dedup) as sel:
        out = sel.run(d["hidden"], d["anchor"])
        if targets is not None:
            out["accept"] = torch.empty(w.B, dtype=torch.int32, device=dev)
            out["emitted"] = torch.empty(w.B, w.L + 1, dtype=torch.int32, device=dev)
            pkg.dflash_verify_prefix(out["path"], torch.as_tensor(targets).to(dev), out["accept"], out["emitted"])
        pkg.dflash_select_sync_status(sel.h)
        torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _bits(inp: wl.Inputs):
    b = wl.bf16_bits
    return b(inp.W), b(inp.E), b(inp.W_A), b(inp.W_B), b(inp.W_H)


def run_oracle(inp: wl.Inputs, seqs, walk=0, nthreads=None):
    nthreads = nthreads or oracle_threads()
    Wb, Eb, WAb, WBb, WHb = _bits(inp)
    b = wl.bf16_bits
    return {s: oracle.select(Wb, Eb, WAb, WBb, WHb, b(inp.hidden[s]), int(inp.anchor[s]), inp.wl.K, walk=walk,
                             nthreads=nthreads) for s in seqs}


def walk_near(r, walk=0) -> bool:
    """Whether any walk decision of oracle result ``r`` has a margin below TIE_EPS."""
    sm = r["step_margin"] if walk == 1 else r["step_margin"][1:]
    return bool((sm < TIE_EPS).any() or r["final_margin"] < TIE_EPS)


def is_near_tie(r, walk=0) -> bool:
    """Any oracle margin below TIE_EPS: a top-K boundary or a walk decision."""
    return bool((r["topk_margin"] < TIE_EPS).any()) or walk_near(r, walk)


def oracle_topk_rows(inp: wl.Inputs, H_bits: np.ndarray, K: int):
    """The oracle's top-K of positions H_bits [N, d] (bf16 bits): a list of
    (ids, vals, boundary margin), one per position."""
    U = oracle.logits(wl.bf16_bits(inp.W), H_bits, nthreads=oracle_threads())
    return [oracle.topk(U[n], K) for n in range(U.shape[0])]


def compare_topk(inp: wl.Inputs, H_bits: np.ndarray, g_ids: np.ndarray, g_vals, ref) -> dict:
    """Top-K of positions H_bits [N, d] against the oracle's rows ``ref``
    (from ``oracle_topk_rows``): sorted values, distinct ids, the exact set at
    clear boundaries and a valid swap at near-tied ones, and every logit within
    tolerance of the oracle's."""
    Wb = wl.bf16_bits(inp.W)
    rep = dict(positions=len(ref), excused=0, swapped=0)
    for n, (ids, vals, margin) in enumerate(ref):
        G = set(g_ids[n].tolist())
        O = set(ids.tolist())
        assert len(G) == len(g_ids[n]), f"position {n}: repeated candidate"
        by_id = dict(zip(ids.tolist(), vals.tolist()))
        if margin < TIE_EPS:
            rep["excused"] += 1
        if G != O:
            assert margin < TIE_EPS, f"position {n}: top-K set differs at a clear boundary"
            extra = sorted(G - O)
            u_extra = oracle.project(np.ascontiguousarray(Wb[extra]), H_bits[n])
            assert max(by_id[tok] for tok in O - G) - float(u_extra.min()) < TIE_EPS, f"position {n}: invalid swap"
            by_id.update(zip(extra, u_extra.tolist()))
            rep["swapped"] += 1
        if g_vals is not None:
            assert np.all(np.diff(g_vals[n]) <= 0), f"position {n}: values not sorted"
            for j, tok in enumerate(g_ids[n].tolist()):
                assert close(g_vals[n][j], by_id[tok]), f"position {n}: logit of {tok}"
    return rep


def conditional_reference(inp: wl.Inputs, s: int, r: dict, g_ids: np.ndarray, walk=0):
    """The oracle's result on the GPU's choice among the valid top-K sets.

    Where the GPU's candidate set of a position differs from the oracle's,
    the position must be an excused near-tie and the swap must be valid: the
    oracle's fp64 logits of the tokens the GPU dropped exceed those of the
    tokens it took by less than TIE_EPS. The reference then runs the oracle's
    later stages (projections, tables, walk) on the oracle's candidates with
    those swaps, ordered by the oracle's own logits (value descending, id
    ascending). Returns (reference, number of positions with a swap)."""
    w = inp.wl
    differs = [set(g_ids[t].tolist()) != set(r["ids"][t].tolist()) for t in range(w.L)]
    if not any(differs):
        return r, 0
    Wb, Eb, WAb, WBb, WHb = _bits(inp)
    hb = wl.bf16_bits(inp.hidden[s])
    alt = r["ids"].copy()
    for t in range(w.L):
        if not differs[t]:
            continue
        assert r["topk_margin"][t] < TIE_EPS, f"seq {s} t {t}: top-K set differs at a clear boundary"
        O = set(r["ids"][t].tolist())
        G = set(g_ids[t].tolist())
        extra = sorted(G - O)
        by_id = dict(zip(r["ids"][t].tolist(), r["vals"][t].tolist()))
        u_extra = oracle.project(np.ascontiguousarray(Wb[extra]), hb[t])
        dropped = [by_id[tok] for tok in O - G]
        assert max(dropped) - float(u_extra.min()) < TIE_EPS, \
            f"seq {s} t {t}: the GPU's candidate set is not a valid top-K (swap of {max(dropped) - u_extra.min():.3g})"
        by_id.update(zip(extra, u_extra.tolist()))
        alt[t] = np.array(sorted(G, key=lambda tok: (-by_id[tok], tok)), dtype=np.int32)
    c = oracle.select_given(Wb, Eb, WAb, WBb, WHb, hb, int(inp.anchor[s]), alt, walk=walk)
    c["topk_margin"] = r["topk_margin"]
    return c, sum(differs)


def gpu_ranks(g_ids: np.ndarray, path: np.ndarray) -> list:
    """Rank of each path token in the GPU's own candidate list."""
    return [int(np.nonzero(g_ids[t] == path[t])[0][0]) for t in range(len(path))]


def optimal_on_own_tables(P: np.ndarray, ranks, walk: int) -> float:
    """Checks that the GPU's path is the walk's result over the GPU's own fp32
    tables P [L, K, K]: for the max-sum walk its fp64 score is the maximum over
    all paths (dynamic programming) up to the fp32 rounding of the GPU's
    recursion; for the greedy walk every step takes the largest entry of its
    row with the smallest rank on ties (exact, the same fp32 values). Returns
    the shortfall of the max-sum path (0 for greedy)."""
    L, K, _ = P.shape
    P = P.astype(np.float64)
    if walk == 1:
        prev = 0
        for t in range(L):
            row = P[t, prev]
            assert ranks[t] == int(np.argmax(row)), f"greedy step {t} is not the best successor"
            prev = ranks[t]
        return 0.0
    delta = P[0, 0].copy()
    for t in range(1, L):
        delta = (delta[:, None] + P[t]).max(axis=0)
    best = float(delta.max())
    mine = float(P[0, 0, ranks[0]] + sum(P[t, ranks[t - 1], ranks[t]] for t in range(1, L)))
    bound = 2 * L * F32_HALF_ULP * float(np.abs(P[np.isfinite(P)]).max()) * L
    assert mine >= best - bound, f"GPU path scores {mine} on its own tables, best is {best}"
    return best - mine


def _force_end(P: np.ndarray, rank: int) -> np.ndarray:
    """Tables P [T, K, K] whose last step may only end at candidate ``rank``."""
    P2 = np.array(P, dtype=np.float64, copy=True)
    keep = np.full(P2.shape[2], -np.inf)
    keep[rank] = 0.0
    P2[-1] = P2[-1] + keep[None, :]
    return P2


def check_viterbi_path(P: np.ndarray, g_ranks, band: float, s=None) -> int:
    """Compares a path (candidate ranks ``g_ranks`` in the order of the oracle
    tables P [L, K, K]) with the oracle's max-sum walk over P, position by
    position. Backtracking from the end, the stretch after the last open
    decision (a chosen node whose best and second-best incoming values differ
    by less than TIE_EPS, or an open final choice) must equal the oracle's path
    exactly. At an open decision the path's own choice must score within
    TIE_EPS (+ ``band``, the fp32 slack) of the best; the part before it is then
    compared with the oracle's best path ending at that choice (the walk over
    the leading tables with the last step restricted to it), and so on.
    Returns the number of open decisions met."""
    L = P.shape[0]
    end, forced, opened = L, None, 0
    while end > 0:
        ranks, score, sm, fm = oracle.viterbi(P[:end] if forced is None else _force_end(P[:end], forced))
        if forced is None and fm < TIE_EPS:  # the final choice is open
            g = int(g_ranks[end - 1])
            ranks, score_g, sm, fm = oracle.viterbi(_force_end(P[:end], g))
            assert score - score_g <= TIE_EPS + band, f"seq {s}: final choice scores {score - score_g:.3g} below best"
            opened += 1
        open_t = [t for t in range(1, end) if sm[t] < TIE_EPS]
        t0 = open_t[-1] if open_t else 0
        assert list(g_ranks[t0:end]) == [int(x) for x in ranks[t0:end]], \
            f"seq {s} t {t0}..{end - 1}: path differs from the oracle"
        if t0 == 0:
            break
        gi, bi, j = int(g_ranks[t0 - 1]), int(ranks[t0 - 1]), int(ranks[t0])
        if gi != bi:  # the predecessor taken at the open node must be within TIE_EPS of the best
            s_b = oracle.viterbi(_force_end(P[:t0], bi))[1] + P[t0, bi, j]
            s_g = oracle.viterbi(_force_end(P[:t0], gi))[1] + P[t0, gi, j]
            assert s_b - s_g <= TIE_EPS + band, f"seq {s} t {t0}: predecessor scores {s_b - s_g:.3g} below best"
        opened += 1
        end, forced = t0, gi
    return opened


def check_greedy_path(P: np.ndarray, g_ranks, band: float, s=None) -> int:
    """The greedy walk's counterpart of ``check_viterbi_path``: forward from
    x0, the stretch before the first open step (best and second-best successor
    within TIE_EPS) equals the oracle's walk; at an open step the path's choice
    must be within TIE_EPS (+ ``band``) of the best successor, and the walk is
    compared again from that choice. Returns the number of open steps met."""
    L, K, _ = P.shape
    start, prev, opened = 0, 0, 0
    while start < L:
        seg = np.array(P[start:], dtype=np.float64, copy=True)
        if start > 0:  # the segment starts from the previous choice's successor row
            row = seg[0, prev].copy()
            seg[0] = -np.inf
            seg[0, 0] = row
        ranks, _, sm, _ = oracle.greedy(seg)
        open_t = [t for t in range(len(ranks)) if sm[t] < TIE_EPS]
        t1 = open_t[0] if open_t else len(ranks)
        assert list(g_ranks[start:start + t1]) == [int(x) for x in ranks[:t1]], \
            f"seq {s} t {start}..{start + t1 - 1}: path differs from the oracle"
        if t1 == len(ranks):
            break
        row = seg[t1, int(ranks[t1 - 1]) if t1 > 0 else 0]
        g = int(g_ranks[start + t1])
        assert row.max() - row[g] <= TIE_EPS + band, f"seq {s} t {start + t1}: successor {row.max() - row[g]:.3g} below best"
        opened += 1
        start, prev = start + t1 + 1, g
    return opened


def tie_band(L: int, table_dev: float, P_ref: np.ndarray) -> float:
    """How far the GPU's margins can sit from the oracle's: every path sum over
    the GPU's tables is within L * table_dev of the oracle's, and a margin is a
    difference of two maxima of such sums (2 L table_dev); the GPU adds in fp32,
    each of the L additions off by at most half an ulp of a sum bounded by
    L * max|P| (twice, for the two sides of a margin)."""
    pmax = float(np.abs(P_ref[np.isfinite(P_ref)]).max())
    return 2 * L * table_dev + 2 * L * F32_HALF_ULP * L * pmax


def compare(inp: wl.Inputs, gpu: dict, orc: dict, walk=0, targets=None):
    """Asserts the parity rules on the sequences in ``orc``; returns a report.

    ``targets`` maps a sequence to its target tokens; the GPU's accept length
    (``gpu["accept"]``) is then checked against the oracle's."""
    w = inp.wl
    L, K = w.L, w.K
    rep = dict(seqs=len(orc), positions=0, topk_excused=0, topk_swapped=0, near_tie_seqs=0, path_equal=0,
               path_alternative=0, path_positions=0, decisions_open=0, tables_checked=0, accept_checked=0,
               accept_on_gpu_path=0, flags_checked=0, flags_raised=0, flags_in_band=0, max_table_dev=0.0,
               max_own_shortfall=0.0)
    for s, r in orc.items():
        g_ids = gpu["topk_ids"][s]
        g_vals = gpu["topk_vals"][s]
        for t in range(L):
            rep["positions"] += 1
            assert np.all(np.diff(g_vals[t]) <= 0), f"seq {s} t {t}: values not sorted"
            assert len(set(g_ids[t].tolist())) == K, f"seq {s} t {t}: repeated candidate"
            if r["topk_margin"][t] < TIE_EPS:
                rep["topk_excused"] += 1
            else:
                assert set(g_ids[t].tolist()) == set(r["ids"][t].tolist()), f"seq {s} t {t}: top-K set differs"
        c, swapped = conditional_reference(inp, s, r, g_ids, walk)
        rep["topk_swapped"] += swapped
        # logits and every table entry, ranks aligned by token id
        dev = 0.0
        P = gpu["pair_scores"][s]
        for t in range(L):
            ref_by_id = dict(zip(c["ids"][t].tolist(), c["vals"][t].tolist()))
            for j, tok in enumerate(g_ids[t].tolist()):
                assert close(g_vals[t][j], ref_by_id[tok]), f"seq {s} t {t}: logit of {tok}"
            rank_c = {tok: k for k, tok in enumerate(c["ids"][t].tolist())}
            jmap = [rank_c[tok] for tok in g_ids[t].tolist()]
            if t == 0:
                assert np.all(np.isneginf(P[0, 1:])), f"seq {s}: rows 1.. at t=0 must be -inf"
                ref = c["P"][0, 0, jmap]
                assert close(P[0, 0], ref).all(), f"seq {s} t 0: pair scores"
                dev = max(dev, float(np.abs(P[0, 0] - ref).max()))
            else:
                prev_c = {tok: k for k, tok in enumerate(c["ids"][t - 1].tolist())}
                imap = [prev_c[tok] for tok in g_ids[t - 1].tolist()]
                ref = c["P"][t][np.ix_(imap, jmap)]
                bad = ~close(P[t], ref)
                assert not bad.any(), f"seq {s} t {t}: {bad.sum()} pair scores out of tolerance"
                dev = max(dev, float(np.abs(P[t] - ref).max()))
            rep["tables_checked"] += 1
        rep["max_table_dev"] = max(rep["max_table_dev"], dev)
        # the GPU's path is the walk's result over its own tables
        g_path = gpu["path"][s]
        ranks = gpu_ranks(g_ids, g_path)
        rep["max_own_shortfall"] = max(rep["max_own_shortfall"], optimal_on_own_tables(P, ranks, walk))
        # the path, position by position, against the conditional reference:
        # decided stretches exactly, open decisions as valid choices
        band = tie_band(L, dev, c["P"])
        g_ranks_c = [int(np.nonzero(c["ids"][t] == g_path[t])[0][0]) for t in range(L)]
        check = check_greedy_path if walk == 1 else check_viterbi_path
        rep["decisions_open"] += check(c["P"], g_ranks_c, band, s)
        rep["path_positions"] += L
        same_path = g_path.tolist() == c["tokens"].tolist()
        if walk_near(c, walk):
            rep["near_tie_seqs"] += 1
        if same_path:
            assert close(gpu["path_score"][s], c["score"], atol=ATOL * L), f"seq {s}: path score"
            rep["path_equal"] += 1
        else:
            rep["path_alternative"] += 1
        if targets is not None and s in targets:
            if same_path:
                n_o, em_o = oracle.verify(c["tokens"], targets[s])
                rep["accept_checked"] += 1
            else:  # the path is one of several correct ones: its accept check must still be right
                n_o, em_o = oracle.verify(g_path, targets[s])
                rep["accept_on_gpu_path"] += 1
            assert int(gpu["accept"][s]) == n_o, f"seq {s}: accept length"
            assert gpu["emitted"][s].tolist() == em_o.tolist(), f"seq {s}: emitted tokens"
        sm, fm = c["step_margin"], c["final_margin"]
        # tie flags along the path, where the path is the oracle's
        if "tie_flags" in gpu and same_path:
            flags = gpu["tie_flags"][s]
            checks = [(t, 1, sm[t]) for t in range(L) if np.isfinite(sm[t])]
            if walk == 0:
                checks.append((L - 1, 2, fm))
            for t, bit, m in checks:
                if abs(m - TIE_EPS) <= band:
                    rep["flags_in_band"] += 1
                    continue
                raised = bool(flags[t] & bit)
                assert raised == (m < TIE_EPS), f"seq {s} t {t}: tie flag bit {bit} is {raised}, margin {m:.3g}"
                rep["flags_checked"] += 1
                rep["flags_raised"] += int(raised)
    return rep
