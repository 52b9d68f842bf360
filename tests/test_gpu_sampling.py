"""GPU parity of the sampling walk and the rejection-sampling verifier against
the CPU oracle (uniform random numbers are inputs to both sides).

Decisions taken by comparing a uniform with a cumulative probability are
compared exactly, except where the oracle's own distance between the uniform
and the decision boundary is below SAMPLE_EPS (reported, not failed), and
where a top-K boundary is a near-tie (the candidate sets may then differ)."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SAMPLE_EPS = 1e-4  # the walk: GPU and oracle tables differ by ~1e-6
EXACT_EPS = 1e-9   # the verifier on identical inputs (double precision on both sides)
DRAW_EPS = 2e-6    # the final draw when the draft probabilities come from the GPU (they
                   # differ from the oracle's by <= ~2e-7 in total, which moves the
                   # residual's CDF by as much)


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_draft_tcgen05_gb300 import build
    build.build()
    import speculative_decoding_draft_tcgen05_gb300 as p
    p.lib()
    return p


def _gpu_sampled(pkg, inp, hidden, anchor, u_walk, T):
    w = inp.wl
    B = anchor.shape[0]
    d = parity.to_device(inp, "cuda")
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=B,
                      walk=pkg.DFLASH_WALK_SAMPLE, temperature=T) as sel:
        out = sel.outputs(B)
        out["draft_probs"] = torch.empty(B, w.L, w.K, dtype=torch.float32, device="cuda")
        pkg.dflash_select_run_sampled(sel.h, hidden.cuda(), anchor.cuda(), torch.from_numpy(u_walk).cuda(), **out)
        pkg.dflash_select_sync_status(sel.h)
        torch.cuda.synchronize()
        launches = pkg.dflash_select_launches_per_run(sel.h, B)
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["fused_tail"] = launches == 2  # lm_head + the clustered tail; else merge, projection, pair tables + walk
    return res


def _target_probs(rng, q_rows, ids_rows, V, L):
    """p_t = half the draft distribution on its candidates + half a random
    distribution over the vocabulary; p_L random. fp32, as the GPU reads it."""
    p = np.empty((L + 1, V), np.float64)
    for t in range(L + 1):
        r = rng.gamma(1.0, size=V)
        p[t] = 0.5 * r / r.sum() if t < L else r / r.sum()
        if t < L:
            p[t, ids_rows[t]] += 0.5 * q_rows[t]
    return p.astype(np.float32)


def _check_walk(inp, gpu, seqs_hidden_idx, u_walk, T):
    """Per replica b (hidden of sequence seqs_hidden_idx[b]): the GPU's sampled
    path and draft distribution against the oracle's sampling walk over the
    oracle's tables on the GPU's (validated) candidate sets; the draws whose
    uniform lies within SAMPLE_EPS of a CDF boundary are excused, and so is
    the rest of the walk after them."""
    w = inp.wl
    orc = parity.run_oracle(inp, sorted(set(seqs_hidden_idx)))
    rep = dict(checked=0, excused=0, steps_checked=0, flags_checked=0)
    for b, s in enumerate(seqs_hidden_idx):
        c, _ = parity.conditional_reference(inp, s, orc[s], gpu["topk_ids"][b])
        ranks, q, mg = oracle.sample_walk(c["P"], T, u_walk[b].astype(np.float64))
        tokens = c["ids"][np.arange(w.L), ranks]
        open_at = [t for t in range(w.L) if mg[t] < SAMPLE_EPS]
        decided = open_at[0] if open_at else w.L
        assert gpu["path"][b][:decided].tolist() == tokens[:decided].tolist(), f"replica {b}: sampled path"
        for t in range(decided + 1 if decided < w.L else w.L):  # the distribution at the first open step is known
            by_id = dict(zip(c["ids"][t].tolist(), q[t].tolist()))
            for j, tok in enumerate(gpu["topk_ids"][b][t].tolist()):
                assert parity.close(gpu["draft_probs"][b][t][j], by_id[tok]), f"replica {b} t {t}: draft prob"
        for t in range(decided):  # the flag marks a uniform within tie_eps of a CDF boundary
            if abs(mg[t] - parity.TIE_EPS) > SAMPLE_EPS:
                assert bool(gpu["tie_flags"][b][t] & 1) == (mg[t] < parity.TIE_EPS), f"replica {b} t {t}: flag"
                rep["flags_checked"] += 1
        rep["steps_checked"] += decided
        if decided == w.L:
            rep["checked"] += 1
        else:
            rep["excused"] += 1
    return rep, orc


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_sampling_walk_tiny(pkg, T):
    inp = parity.inputs_for("tiny")
    rng = np.random.default_rng(41)
    reps = 16
    idx = [b % inp.wl.B for b in range(reps)]
    hidden = inp.hidden[idx].contiguous()
    anchor = inp.anchor[idx].contiguous()
    u_walk = rng.random((reps, inp.wl.L)).astype(np.float32)
    gpu = _gpu_sampled(pkg, inp, hidden, anchor, u_walk, T)
    rep, _ = _check_walk(inp, gpu, idx, u_walk, T)
    print("sampling walk tiny T", T, rep)
    assert rep["checked"] >= reps // 2


def test_sampling_walk_fused_tail(pkg):
    """Eight replicas of the tiny workload fit the clustered small-batch tail
    (the launch configuration of the benchmark's sampling step at batch 1)."""
    inp = parity.inputs_for("tiny")
    rng = np.random.default_rng(44)
    reps = 8
    idx = [b % inp.wl.B for b in range(reps)]
    u_walk = rng.random((reps, inp.wl.L)).astype(np.float32)
    gpu = _gpu_sampled(pkg, inp, inp.hidden[idx].contiguous(), inp.anchor[idx].contiguous(), u_walk, 1.0)
    assert gpu["fused_tail"]
    rep, _ = _check_walk(inp, gpu, idx, u_walk, 1.0)
    print("sampling walk, fused tail", rep)
    assert rep["checked"] >= reps - 1


@pytest.mark.parametrize("reps,fused", [(4, True), (12, False)])
def test_sampling_walk_k32(pkg, reps, fused):
    """K = 32 candidates and 16 positions, on both tail paths."""
    w = wl.custom(name="sample_k32", B=2, L=16, K=32, V=5000, d=192, seed=29, std_w=0.05)
    inp = wl.make_inputs(w)
    rng = np.random.default_rng(45 + reps)
    idx = [b % w.B for b in range(reps)]
    u_walk = rng.random((reps, w.L)).astype(np.float32)
    gpu = _gpu_sampled(pkg, inp, inp.hidden[idx].contiguous(), inp.anchor[idx].contiguous(), u_walk, 1.0)
    assert gpu["fused_tail"] == fused
    rep, _ = _check_walk(inp, gpu, idx, u_walk, 1.0)
    print("sampling walk K=32, fused" if fused else "sampling walk K=32, three kernels", rep)
    assert rep["checked"] >= reps // 2 and rep["steps_checked"] >= 0.75 * reps * w.L


def _verify_case(pkg, inp, orc_seq, rng, reps, T):
    """Rejection verifier in isolation: the oracle's draft (path, candidates,
    fp32-rounded draft distribution) and random target rows, on both sides."""
    w = inp.wl
    L, K, V = w.L, w.K, w.V
    paths, ids, qs, ps, ua, ur = [], [], [], [], [], []
    for b in range(reps):
        r = orc_seq
        u = rng.random(L).astype(np.float32)
        ranks, q, _ = oracle.sample_walk(r["P"], T, u.astype(np.float64))
        paths.append(r["ids"][np.arange(L), ranks].astype(np.int32))
        ids.append(r["ids"].astype(np.int32))
        qs.append(q.astype(np.float32))
        ps.append(_target_probs(rng, q, r["ids"], V, L))
        ua.append(rng.random(L).astype(np.float32))
        ur.append(np.float32(rng.random()))
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(np.stack(a) if isinstance(a, list) else a)).to(dt).cuda()
    acc = torch.empty(reps, dtype=torch.int32, device="cuda")
    em = torch.empty(reps, L + 1, dtype=torch.int32, device="cuda")
    pkg.dflash_verify_rejection(t(paths, torch.int32), t(ids, torch.int32), t(qs, torch.float32),
                                t(ps, torch.float32), t(ua, torch.float32),
                                torch.tensor(ur, dtype=torch.float32).cuda(), acc, em)
    torch.cuda.synchronize()
    acc, em = acc.cpu().numpy(), em.cpu().numpy()
    checked = excused = 0
    ns = []
    for b in range(reps):
        n, e, am, rm = oracle.verify_rejection(paths[b], ids[b], qs[b].astype(np.float64), ps[b].astype(np.float64),
                                               ua[b].astype(np.float64), float(ur[b]))
        ns.append(n)
        if (am[:min(n + 1, L)] < EXACT_EPS).any() or rm < EXACT_EPS:
            excused += 1
            continue
        assert acc[b] == n, f"replica {b}: accept length"
        assert em[b].tolist() == e.tolist(), f"replica {b}: emitted"
        checked += 1
    return checked, excused, ns


@pytest.mark.parametrize("name", ["tiny", "4b_b1"])
def test_rejection_verifier_against_oracle(pkg, name):
    inp = parity.inputs_for(name)
    orc = parity.run_oracle(inp, [0])[0]
    rng = np.random.default_rng(43)
    checked, excused, ns = _verify_case(pkg, inp, orc, rng, reps=48, T=1.0)
    print(name, "rejection verifier: checked", checked, "excused", excused, "accept lengths", np.bincount(ns))
    assert checked >= 46
    assert len(set(ns)) > 2  # both rejections at several depths and full acceptances occur


@pytest.mark.parametrize("B,V,K", [(1, 4099, 16), (3, 40, 16), (80, 4099, 32), (20, 151936, 16), (2, 151936, 32)])
def test_rejection_verifier_shapes(pkg, B, V, K):
    """Random drafts and targets over the launch shapes the verifier takes
    (1 to 16 CTAs per sequence, rows that are not 16-byte aligned, a vocabulary
    smaller than the CTAs' slices), exact against the oracle on the same inputs."""
    rng = np.random.default_rng(B * 7 + V + K)
    L = 7
    ids = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(L)]) for _ in range(B)]).astype(np.int32)
    q = rng.dirichlet(np.ones(K) * 0.5, size=(B, L)).astype(np.float32)
    path = np.take_along_axis(ids, rng.integers(0, K, size=(B, L, 1)), axis=2)[..., 0].astype(np.int32)
    p = rng.gamma(0.3, size=(B, L + 1, V))
    p[:, :L] *= 0.5 / p[:, :L].sum(-1, keepdims=True)
    for b in range(B):  # half of each target row agrees with the draft's candidates
        for t in range(L):
            p[b, t, ids[b, t]] += 0.5 * q[b, t]
    p[:, L] /= p[:, L].sum(-1, keepdims=True)
    p = p.astype(np.float32)
    ua = rng.random((B, L)).astype(np.float32)
    ur = rng.random(B).astype(np.float32)
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    em = torch.empty(B, L + 1, dtype=torch.int32, device="cuda")
    c = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pkg.dflash_verify_rejection(c(path), c(ids), c(q), c(p), c(ua), c(ur), acc, em)
    torch.cuda.synchronize()
    acc, em = acc.cpu().numpy(), em.cpu().numpy()
    checked = 0
    for b in range(B):
        n, e, am, rm = oracle.verify_rejection(path[b], ids[b], q[b].astype(np.float64), p[b].astype(np.float64),
                                               ua[b].astype(np.float64), float(ur[b]))
        if (am[:min(n + 1, L)] < EXACT_EPS).any() or rm < EXACT_EPS:
            continue
        assert acc[b] == n and em[b].tolist() == e.tolist(), f"sequence {b}"
        checked += 1
    assert checked >= B - 1


def test_sampled_step_end_to_end_full_size(pkg):
    """Qwen3-4B-shaped head at full size: GPU sampled walk then GPU verifier,
    against the oracle's walk then the oracle's verifier, 8 uniform draws."""
    inp = parity.inputs_for("4b_b1")
    w = inp.wl
    rng = np.random.default_rng(47)
    reps = 8
    idx = [0] * reps
    hidden = inp.hidden[idx].contiguous()
    anchor = inp.anchor[idx].contiguous()
    u_walk = rng.random((reps, w.L)).astype(np.float32)
    gpu = _gpu_sampled(pkg, inp, hidden, anchor, u_walk, 1.0)
    rep, orc = _check_walk(inp, gpu, idx, u_walk, 1.0)
    r = orc[0]
    ps, ua, ur, onum = [], [], [], []
    for b in range(reps):
        ranks, q, _ = oracle.sample_walk(r["P"], 1.0, u_walk[b].astype(np.float64))
        ps.append(_target_probs(rng, q, r["ids"], w.V, w.L))
        ua.append(rng.random(w.L).astype(np.float32))
        ur.append(np.float32(rng.random()))
    acc = torch.empty(reps, dtype=torch.int32, device="cuda")
    em = torch.empty(reps, w.L + 1, dtype=torch.int32, device="cuda")
    pkg.dflash_verify_rejection(torch.from_numpy(gpu["path"]).cuda(), torch.from_numpy(gpu["topk_ids"]).cuda(),
                                torch.from_numpy(gpu["draft_probs"]).cuda(), torch.from_numpy(np.stack(ps)).cuda(),
                                torch.from_numpy(np.stack(ua)).cuda(), torch.tensor(ur, dtype=torch.float32).cuda(),
                                acc, em)
    torch.cuda.synchronize()
    acc, em = acc.cpu().numpy(), em.cpu().numpy()
    # the verifier on the GPU's own draft, against the oracle's verifier on the same draft: exact
    exact = 0
    for b in range(reps):
        n, e, am, rm = oracle.verify_rejection(gpu["path"][b], gpu["topk_ids"][b],
                                               gpu["draft_probs"][b].astype(np.float64), ps[b].astype(np.float64),
                                               ua[b].astype(np.float64), float(ur[b]))
        if (am[:min(n + 1, w.L)] < EXACT_EPS).any() or rm < EXACT_EPS:
            continue
        assert acc[b] == n and em[b].tolist() == e.tolist(), f"replica {b}: verifier on the GPU's draft"
        exact += 1
    assert exact >= reps - 1
    # the whole sampled step against the oracle's walk and verifier
    checked = draws = 0
    for b in range(reps):
        ranks, q, mg = oracle.sample_walk(r["P"], 1.0, u_walk[b].astype(np.float64))
        path = r["ids"][np.arange(w.L), ranks]
        n, e, am, rm = oracle.verify_rejection(path, r["ids"], q, ps[b].astype(np.float64), ua[b].astype(np.float64),
                                               float(ur[b]))
        if (mg < SAMPLE_EPS).any() or (am[:min(n + 1, w.L)] < SAMPLE_EPS).any():
            continue
        assert acc[b] == n and em[b][:n].tolist() == e[:n].tolist(), f"replica {b}: kept drafts"
        checked += 1
        # the drawn token depends on the draft probabilities, which differ by
        # ~1e-7 between the GPU's fp32 softmax and the oracle's fp64 one
        if rm >= DRAW_EPS:
            assert em[b][n] == e[n], f"replica {b}: drawn token"
            draws += 1
    print("sampled step 4b_b1:", rep, "exact on the GPU draft", exact, "verified", checked, "draws compared", draws)
    assert rep["checked"] >= reps // 2 and checked >= reps // 2


def test_sampling_arguments(pkg):
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    with pytest.raises(pkg.DflashError):
        pkg.dflash_select_init(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=2,
                               walk=pkg.DFLASH_WALK_SAMPLE, temperature=0.0)
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=2,
                      walk=pkg.DFLASH_WALK_SAMPLE) as sel:
        out = sel.outputs(2)
        with pytest.raises(pkg.DflashError) as e:  # a sampling handle needs its uniforms
            pkg.dflash_select_run(sel.h, d["hidden"], d["anchor"], **out)
        assert e.value.status == pkg.DFLASH_ERR_INVALID_ARG
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=2) as sel:
        out = sel.outputs(2)
        q = torch.empty(2, w.L, w.K, dtype=torch.float32, device="cuda")
        u = torch.rand(2, w.L, device="cuda")
        with pytest.raises(pkg.DflashError):  # a max-sum handle does not sample
            pkg.dflash_select_run_sampled(sel.h, d["hidden"], d["anchor"], u, draft_probs=q, **out)
