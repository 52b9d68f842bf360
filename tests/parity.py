"""Shared helpers of the parity tests: run the CUDA path and the CPU oracle on
the same seeded inputs and compare them under the stated rules.

Rules (bf16 inputs, fp32 accumulation on the GPU, fp64 in the oracle):
  - top-K id sets, paths and accept lengths are bit-exact, except where the
    oracle's own margin is below TIE_EPS (reported, not failed);
  - logits and pair scores agree within |gpu - ref| <= ATOL + RTOL * |ref|.
No input of the oracle and no expected value comes from the GPU: targets are
planted on the oracle's own path.
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


def run_gpu(inp: wl.Inputs, dev="cuda", walk=0, max_batch=None, dtensors=None, targets=None, tables=False):
    """Runs the whole selector through the C ABI (and, given target tokens
    [B, L+1], the accept check); returns CPU numpy outputs."""
    import speculative_decoding_draft_tcgen05_gb300 as pkg
    w = inp.wl
    d = dtensors if dtensors is not None else to_device(inp, dev)
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K,
                      max_batch=max_batch or w.B, walk=walk, tie_eps=TIE_EPS, tables=tables) as sel:
        out = sel.run(d["hidden"], d["anchor"])
        if targets is not None:
            out["accept"] = torch.empty(w.B, dtype=torch.int32, device=dev)
            out["emitted"] = torch.empty(w.B, w.L + 1, dtype=torch.int32, device=dev)
            pkg.dflash_verify_prefix(out["path"], torch.as_tensor(targets).to(dev), out["accept"], out["emitted"])
        pkg.dflash_select_sync_status(sel.h)
        torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_oracle(inp: wl.Inputs, seqs, walk=0, nthreads=None):
    nthreads = nthreads or oracle_threads()
    b = wl.bf16_bits
    Wb, Eb, WAb, WBb, WHb = b(inp.W), b(inp.E), b(inp.W_A), b(inp.W_B), b(inp.W_H)
    return {s: oracle.select(Wb, Eb, WAb, WBb, WHb, b(inp.hidden[s]), int(inp.anchor[s]), inp.wl.K, walk=walk,
                             nthreads=nthreads) for s in seqs}


def is_near_tie(r, walk=0) -> bool:
    if (r["topk_margin"] < TIE_EPS).any():
        return True
    sm = r["step_margin"] if walk == 1 else r["step_margin"][1:]
    return bool((sm < TIE_EPS).any() or r["final_margin"] < TIE_EPS)


def compare(inp: wl.Inputs, gpu: dict, orc: dict, walk=0, targets=None):
    """Asserts the parity rules on the sequences in ``orc``; returns a report.

    Pair tables are compared entry by entry after aligning ranks by token id
    (the two sides may order near-equal candidates differently), at every
    position whose candidate set and whose predecessor set both match.
    ``targets`` maps a sequence to its target tokens; the GPU's accept length
    (``gpu["accept"]``) is then checked against the oracle's."""
    w = inp.wl
    rep = dict(seqs=len(orc), positions=0, topk_excused=0, near_tie_seqs=0, path_equal=0, tables_checked=0,
               accept_checked=0)
    for s, r in orc.items():
        g_ids = gpu["topk_ids"][s]
        g_vals = gpu["topk_vals"][s]
        same_set = []
        for t in range(w.L):
            rep["positions"] += 1
            assert np.all(np.diff(g_vals[t]) <= 0), f"seq {s} t {t}: values not sorted"
            ok_set = set(g_ids[t].tolist()) == set(r["ids"][t].tolist())
            if r["topk_margin"][t] < TIE_EPS:
                rep["topk_excused"] += 1
            else:
                assert ok_set, f"seq {s} t {t}: top-K set differs"
            same_set.append(ok_set)
            ref_by_id = dict(zip(r["ids"][t].tolist(), r["vals"][t].tolist()))
            for j, tok in enumerate(g_ids[t].tolist()):
                if tok in ref_by_id:
                    assert close(g_vals[t][j], ref_by_id[tok]), f"seq {s} t {t}: logit of {tok}"
        P = gpu["pair_scores"][s]
        for t in range(w.L):
            if not same_set[t] or (t > 0 and not same_set[t - 1]):
                continue
            rank_o = {tok: k for k, tok in enumerate(r["ids"][t].tolist())}
            jmap = [rank_o[tok] for tok in g_ids[t].tolist()]
            if t == 0:
                assert np.all(np.isneginf(P[0, 1:])), f"seq {s}: rows 1.. at t=0 must be -inf"
                ref = r["P"][0, 0, jmap]
                assert close(P[0, 0], ref).all(), f"seq {s} t 0: pair scores"
            else:
                prev_o = {tok: k for k, tok in enumerate(r["ids"][t - 1].tolist())}
                imap = [prev_o[tok] for tok in g_ids[t - 1].tolist()]
                ref = r["P"][t][np.ix_(imap, jmap)]
                bad = ~close(P[t], ref)
                assert not bad.any(), f"seq {s} t {t}: {bad.sum()} pair scores out of tolerance"
            rep["tables_checked"] += 1
        near = is_near_tie(r, walk)
        if near:
            rep["near_tie_seqs"] += 1
        else:
            assert gpu["path"][s].tolist() == r["tokens"].tolist(), f"seq {s}: path differs from oracle"
            assert close(gpu["path_score"][s], r["score"], atol=ATOL * w.L), f"seq {s}: path score"
            rep["path_equal"] += 1
        if targets is not None and s in targets:
            n_o, em_o = oracle.verify(r["tokens"], targets[s])
            if not near:
                assert int(gpu["accept"][s]) == n_o, f"seq {s}: accept length"
                assert gpu["emitted"][s].tolist() == em_o.tolist(), f"seq {s}: emitted tokens"
                rep["accept_checked"] += 1
    return rep
