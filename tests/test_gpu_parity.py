"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, plus boundary behaviour of the C ABI on a GPU."""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_draft_tcgen05_gb300 import build
    build.build()
    import speculative_decoding_draft_tcgen05_gb300 as p
    p.lib()
    return p


def _full_check(inp, walk=0, seqs=None, max_batch=None, tables=False):
    seqs = list(range(inp.wl.B)) if seqs is None else seqs
    orc = parity.run_oracle(inp, seqs, walk=walk)
    # target tokens: planted on the oracle's path for the checked sequences
    # (accept lengths then span 0..L), the seeded uniform draws elsewhere
    tgt = inp.target_rand.clone()
    if inp.wl.planted_targets:
        idx = torch.tensor(seqs, dtype=torch.long)
        path = torch.stack([torch.from_numpy(orc[s]["tokens"]) for s in seqs])
        tgt[idx] = wl.plant_targets(path, inp.target_rand[idx], inp.n0[idx], inp.wl.V)
    gpu = parity.run_gpu(inp, walk=walk, max_batch=max_batch, targets=tgt, tables=tables)
    targets = {s: tgt[s].numpy() for s in seqs}
    rep = parity.compare(inp, gpu, orc, walk=walk, targets=targets)
    print(inp.wl.name, "walk", walk, "tables" if tables else "", rep)
    return gpu, orc, rep


def assert_mostly_exact(rep, frac=0.75):
    """Most sampled sequences have their whole path and accept length compared
    exactly (the rest only at their decided positions)."""
    assert rep["path_equal"] >= frac * rep["seqs"], rep
    assert rep["accept_checked"] >= frac * rep["seqs"], rep


@pytest.mark.parametrize("walk", [0, 1])
def test_tiny_parity(pkg, walk):
    inp = parity.inputs_for("tiny")
    gpu, orc, rep = _full_check(inp, walk=walk)
    assert rep["path_equal"] + rep["path_alternative"] == inp.wl.B
    assert rep["path_equal"] == inp.wl.B and rep["flags_checked"] > 0


EDGE = [
    # ragged vocabulary tail, one draft position
    dict(B=3, L=1, K=16, V=1000, d=64),
    # longest block, K = 32, d not a multiple of 128
    dict(B=2, L=16, K=32, V=5000, d=192),
    # more than 256 positions: several n-tiles of the lm_head kernel
    dict(B=40, L=7, K=16, V=2000, d=128),
    # vocabulary exactly K
    dict(B=2, L=2, K=32, V=32, d=64),
    # one sequence, vocabulary just above one tile
    dict(B=1, L=5, K=16, V=129, d=256),
    # 129 to 256 positions take the CTA-pair lm_head kernel: 200 positions (104
    # per CTA), an odd vocabulary tile count (the pair's last tile is half past V)
    dict(B=25, L=8, K=16, V=20000, d=128),
    # 256 positions at K = 32 with the sampled-threshold pilot pass (258 tiles)
    dict(B=16, L=16, K=32, V=33000, d=192),
    # 135 positions (72 per CTA), odd tile count, pilot, d not a multiple of 128
    dict(B=9, L=15, K=16, V=40000, d=320),
]


@pytest.mark.parametrize("shape", EDGE, ids=[f"B{s['B']}L{s['L']}K{s['K']}V{s['V']}d{s['d']}" for s in EDGE])
def test_edge_shapes(pkg, shape):
    inp = wl.make_inputs(wl.custom(name="edge", seed=17, std_w=0.05, **shape))
    for walk in (0, 1):
        gpu, orc, rep = _full_check(inp, walk=walk, max_batch=shape["B"] + 3)
        assert rep["positions"] == shape["B"] * shape["L"]
        assert rep["path_equal"] >= 0.75 * rep["seqs"], rep


def test_batch_smaller_than_max_and_zero(pkg):
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=7) as sel:
        one = sel.run(d["hidden"][1:2].contiguous(), d["anchor"][1:2].contiguous())
        empty_path = torch.empty(0, w.L, dtype=torch.int32, device="cuda")
        pkg.dflash_select_run(sel.h, d["hidden"][:0], d["anchor"][:0], path=empty_path)
        pkg.dflash_select_sync_status(sel.h)
    full = parity.run_gpu(inp)
    assert one["path"].cpu().numpy().tolist() == full["path"][1:2].tolist()
    assert one["topk_ids"].cpu().numpy().tolist() == full["topk_ids"][1:2].tolist()


def test_invalid_arguments(pkg):
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    bad = [dict(K=8), dict(L=17), dict(L=0), dict(max_batch=0)]
    for kw in bad:
        args = dict(L=w.L, K=w.K, max_batch=2)
        args.update(kw)
        with pytest.raises(pkg.DflashError) as e:
            pkg.dflash_select_init(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], **args)
        assert e.value.status in (pkg.DFLASH_ERR_UNSUPPORTED, pkg.DFLASH_ERR_INVALID_ARG)
    # e != 256
    with pytest.raises(pkg.DflashError) as e:
        pkg.dflash_select_init(d["W"], d["E"], d["W_A"][:128].contiguous(), d["W_B"], d["W_H"], L=w.L, K=w.K,
                               max_batch=2)
    assert e.value.status == pkg.DFLASH_ERR_UNSUPPORTED
    # d not a multiple of 64
    W3 = torch.zeros(w.V, 96 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkg.DflashError) as e:
        pkg.dflash_select_init(W3, W3, W3[:256], W3[:256], W3[:256], L=w.L, K=w.K, max_batch=2)
    assert e.value.status == pkg.DFLASH_ERR_UNSUPPORTED
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=2) as sel:
        out = sel.outputs(3)
        hid3 = torch.zeros(3, w.L, w.d, dtype=torch.bfloat16, device="cuda")
        anc3 = torch.zeros(3, dtype=torch.int32, device="cuda")
        with pytest.raises(pkg.DflashError) as e:  # B > max_batch
            pkg.dflash_select_run(sel.h, hid3, anc3, **out)
        assert e.value.status == pkg.DFLASH_ERR_INVALID_ARG
        flat = torch.zeros(2 * w.L * w.d + 1, dtype=torch.bfloat16, device="cuda")
        misaligned = flat[1:].view(2, w.L, w.d)
        with pytest.raises(pkg.DflashError) as e:
            pkg.dflash_select_run(sel.h, misaligned, anc3[:2], path=out["path"][:2])
        assert e.value.status == pkg.DFLASH_ERR_INVALID_ARG
        # the handle still works after rejected calls
        sel.run(d["hidden"], d["anchor"])
        pkg.dflash_select_sync_status(sel.h)
    with pytest.raises(pkg.DflashError):
        pkg.dflash_verify_prefix(torch.zeros(2, 17, dtype=torch.int32, device="cuda"),
                                 torch.zeros(2, 18, dtype=torch.int32, device="cuda"),
                                 torch.zeros(2, dtype=torch.int32, device="cuda"))


def test_out_of_range_anchor_is_reported(pkg):
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=w.B) as sel:
        anchor = d["anchor"].clone()
        anchor[0] = w.V  # one past the end: the kernel must not read it
        sel.run(d["hidden"], anchor)
        with pytest.raises(pkg.DflashError) as e:
            pkg.dflash_select_sync_status(sel.h)
        assert e.value.status == pkg.DFLASH_ERR_DEVICE_CHECK
        # the error word is cleared and the handle keeps working
        sel.run(d["hidden"], d["anchor"])
        pkg.dflash_select_sync_status(sel.h)


@pytest.mark.parametrize("L", [1, 2, 7, 15, 16])
def test_verify_kernel(pkg, L):
    rng = np.random.default_rng(100 + L)
    B, V = 333, 50
    path = rng.integers(0, V, (B, L)).astype(np.int32)
    n0 = rng.integers(0, L + 1, B).astype(np.int32)
    tgt = wl.plant_targets(torch.from_numpy(path), torch.from_numpy(rng.integers(0, V, (B, L + 1)).astype(np.int32)),
                           torch.from_numpy(n0), V).numpy()
    tgt[::7] = rng.integers(0, 3, (len(tgt[::7]), L + 1))  # some unplanted rows with chance matches
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    em = torch.empty(B, L + 1, dtype=torch.int32, device="cuda")
    pkg.dflash_verify_prefix(torch.from_numpy(path).cuda(), torch.from_numpy(tgt).cuda(), acc, em)
    torch.cuda.synchronize()
    acc, em = acc.cpu().numpy(), em.cpu().numpy()
    for b in range(B):
        n, e = oracle.verify(path[b], tgt[b])
        assert acc[b] == n and em[b].tolist() == e.tolist()


def test_step_from_host_buffers(pkg):
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    full = parity.run_gpu(inp, dtensors=d)
    orc = parity.run_oracle(inp, range(w.B))
    assert not any(parity.is_near_tie(orc[b]) for b in range(w.B))
    opath = torch.stack([torch.from_numpy(orc[b]["tokens"]) for b in range(w.B)])
    tgt = wl.plant_targets(opath, inp.target_rand, torch.tensor([3, 0], dtype=torch.int32), w.V)
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=w.B) as sel:
        hid = inp.hidden.pin_memory()
        anc = inp.anchor.pin_memory()
        tg = tgt.pin_memory()
        path = torch.empty(w.B, w.L, dtype=torch.int32).pin_memory()
        acc = torch.empty(w.B, dtype=torch.int32).pin_memory()
        em = torch.empty(w.B, w.L + 1, dtype=torch.int32).pin_memory()
        for _ in range(2):
            pkg.dflash_select_step_host(sel.h, hid, anc, tg, path, acc, em)
            assert path.numpy().tolist() == full["path"].tolist()
            assert acc.tolist() == [3, 0]
            for b in range(w.B):
                n, e = oracle.verify(orc[b]["tokens"], tgt[b].numpy())
                assert path[b].tolist() == orc[b]["tokens"].tolist() and em[b].tolist() == e.tolist()


def test_step_host_bound_pageable_and_error(pkg):
    """The pre-bound host step equals the plain call, pageable host buffers
    work too, and a latched device error comes back through the one read-back
    (then the handle runs cleanly again)."""
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    full = parity.run_gpu(inp, dtensors=d)
    tgt = wl.plant_targets(torch.from_numpy(full["path"]), inp.target_rand, torch.tensor([2, 7], dtype=torch.int32),
                           w.V)
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=w.B) as sel:
        outs = []
        for pinned in (True, False):
            mk = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
            hid, anc, tg = mk(inp.hidden), mk(inp.anchor), mk(tgt)
            path = mk(torch.full((w.B, w.L), -5, dtype=torch.int32))
            acc = mk(torch.full((w.B,), -5, dtype=torch.int32))
            em = mk(torch.full((w.B, w.L + 1), -5, dtype=torch.int32))
            step = pkg.bind_step_host(sel.h, hid, anc, tg, path, acc, em)
            step()
            outs.append((path.clone(), acc.clone(), em.clone()))
            assert path.numpy().tolist() == full["path"].tolist()
            assert acc.tolist() == [2, 7]
        assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1]))
        bad = inp.anchor.clone()
        bad[1] = w.V
        path = torch.empty(w.B, w.L, dtype=torch.int32)
        acc = torch.empty(w.B, dtype=torch.int32)
        em = torch.empty(w.B, w.L + 1, dtype=torch.int32)
        with pytest.raises(pkg.DflashError) as e:
            pkg.dflash_select_step_host(sel.h, inp.hidden, bad, tgt, path, acc, em)
        assert e.value.status == pkg.DFLASH_ERR_DEVICE_CHECK
        pkg.dflash_select_step_host(sel.h, inp.hidden, inp.anchor, tgt, path, acc, em)
        assert path.numpy().tolist() == full["path"].tolist()


@pytest.mark.parametrize("B", [40, 3])
def test_step_host_equals_run_verify(pkg, B):
    """The host step (anchor and target read from mapped host memory, results
    written there by the walking kernel) equals the device-buffer run with
    the accept check, on the three-kernel tail (B = 40) and the fused one."""
    inp = wl.make_inputs(wl.custom(name="edge", seed=23, std_w=0.05, B=B, L=7, K=16, V=2000, d=128))
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    tgt = torch.randint(0, w.V, (B, w.L + 1), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=B) as sel:
        out = sel.outputs(B, full=False)
        acc_d = torch.empty(B, dtype=torch.int32, device="cuda")
        em_d = torch.empty(B, w.L + 1, dtype=torch.int32, device="cuda")
        step = pkg.bind_step(sel.h, d["hidden"], d["anchor"], out["path"], target=tgt.cuda(), accept_len=acc_d,
                             emitted=em_d)
        step()
        pkg.dflash_select_sync_status(sel.h)
        path_h = torch.empty(B, w.L, dtype=torch.int32).pin_memory()
        acc_h = torch.empty(B, dtype=torch.int32).pin_memory()
        em_h = torch.empty(B, w.L + 1, dtype=torch.int32).pin_memory()
        host = pkg.bind_step_host(sel.h, inp.hidden.pin_memory(), inp.anchor.pin_memory(), tgt.pin_memory(),
                                  path_h, acc_h, em_h)
        for _ in range(3):
            host()
            assert torch.equal(path_h, out["path"].cpu())
            assert torch.equal(acc_h, acc_d.cpu()) and torch.equal(em_h, em_d.cpu())


def test_profile_records_kernels(pkg):
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=w.B) as sel:
        pkg.dflash_select_profile(sel.h, True)
        out = sel.outputs(w.B)
        for _ in range(5):
            sel.run(d["hidden"], d["anchor"], out=out)
        rec = pkg.dflash_select_profile_read(sel.h)
        pkg.dflash_select_profile(sel.h, False)
        per_run = pkg.dflash_select_launches_per_run(sel.h, w.B)
    assert set(rec) == set(pkg.KERNEL_NAMES)
    launched = {name for name, (ms, n) in rec.items() if n}
    # the small batch takes the fused tail; larger ones the three-kernel tail
    assert launched in ({"lmhead_topk", "select_tail"}, {"lmhead_topk", "topk_merge", "projection", "pair_walk"})
    assert per_run == len(launched)
    for name in launched:
        ms, n = rec[name]
        assert n == 5 and ms > 0, name


def test_headline_config_full_size(pkg):
    """Qwen3-4B-shaped head, batch 1, at full size in the benchmark's launch
    configuration: every output against the oracle."""
    inp = parity.inputs_for("4b_b1")
    gpu, orc, rep = _full_check(inp)
    assert rep["positions"] == 7
    assert rep["path_equal"] == 1 and rep["accept_checked"] == 1


@pytest.mark.parametrize("name,seqs", [
    ("4b_b8", None),
    ("4b_b32", [0, 3, 5, 9, 12, 17, 20, 24, 28, 31]),
    ("27b_b1", None),
    ("27b_b8", None),
    ("27b_b32", [1, 4, 8, 13, 19, 22, 26, 30]),
])
def test_larger_configs_sampled(pkg, name, seqs):
    inp = parity.inputs_for(name)
    gpu, orc, rep = _full_check(inp, seqs=seqs)
    assert rep["seqs"] == (len(seqs) if seqs else inp.wl.B)
    assert_mostly_exact(rep)


@pytest.mark.parametrize("name", ["stress_k16", "stress_k32"])
def test_stress_sampled_with_near_ties(pkg, name):
    inp = parity.inputs_for(name)
    planted_seqs = sorted({b for (b, t, v1, v2) in inp.near_tie_pos})
    seqs = planted_seqs[:8]
    seqs += [b for b in range(0, 256, 16) if b not in seqs][:16 - len(seqs)]
    gpu, orc, rep = _full_check(inp, seqs=seqs)
    assert rep["seqs"] == 16
    assert_mostly_exact(rep)
    # the planted near-ties are seen by the oracle and reported, not failed
    planted_here = [(b, t) for (b, t, v1, v2) in inp.near_tie_pos if b in orc]
    gaps = [orc[b]["vals"][t][0] - orc[b]["vals"][t][1] for (b, t) in planted_here]
    print(name, "planted near-ties in sample:", len(planted_here), "achieved gap<1e-3:",
          sum(g < 1e-3 for g in gaps))
    assert planted_here and sum(g < 1e-3 for g in gaps) >= 0.9 * len(gaps)


def test_init_reports_a_failed_device_allocation(pkg):
    """A CUDA failure on the host side comes back as DFLASH_ERR_CUDA: with the
    precomputed tables a vocabulary of 2^31 - 1 tokens asks for a 4 TB table,
    which cudaMalloc refuses (nothing is launched before that request, so the
    small weight tensors are never read as if they had that many rows). The
    process and the device stay usable: a normal handle is created and run
    right after."""
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    cfg = pkg.dflash_select_config(V=2 ** 31 - 1, d=w.d, L=w.L, K=w.K, e=256, max_batch=1, walk=0, tie_eps=1e-3,
                                   temperature=1.0, tables=1)
    h = pkg.ctypes.c_void_p()
    P = lambda t: pkg.ctypes.c_void_p(t.data_ptr())
    st = pkg.lib().dflash_select_init(pkg.ctypes.byref(cfg), P(d["W"]), P(d["E"]), P(d["W_A"]), P(d["W_B"]),
                                      P(d["W_H"]), None, pkg.ctypes.byref(h))
    assert st == pkg.DFLASH_ERR_CUDA, pkg.dflash_last_error()
    assert h.value is None
    assert "cudaMalloc" in pkg.dflash_last_error()
    full = parity.run_gpu(inp, dtensors=d)
    orc = parity.run_oracle(inp, range(w.B))
    assert parity.compare(inp, full, orc)["path_equal"] == w.B


@pytest.mark.parametrize("name,seqs", [("tiny", None), ("4b_b8", None)])
def test_run_verify_equals_run_then_verify(pkg, name, seqs):
    """The fused run + accept check gives the outputs of dflash_select_run
    followed by dflash_verify_prefix, on the small-batch fused tail (tiny) and on
    the pair-table kernel (batch 8), with accept lengths spanning 0..L."""
    inp = parity.inputs_for(name)
    w = inp.wl
    d = parity.to_device(inp, "cuda")
    sel_seqs = list(range(w.B))
    orc = parity.run_oracle(inp, sel_seqs)
    path = torch.stack([torch.from_numpy(orc[s]["tokens"]) for s in sel_seqs])
    n0 = torch.arange(w.B, dtype=torch.int32) % (w.L + 1)
    tgt = wl.plant_targets(path, inp.target_rand, n0, w.V)
    ref = parity.run_gpu(inp, dtensors=d, targets=tgt)
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=w.B,
                      tie_eps=parity.TIE_EPS) as sel:
        out = sel.outputs(w.B)
        acc = torch.full((w.B,), -5, dtype=torch.int32, device="cuda")
        em = torch.full((w.B, w.L + 1), -5, dtype=torch.int32, device="cuda")
        for _ in range(2):
            pkg.dflash_select_run_verify(sel.h, d["hidden"], d["anchor"], tgt.cuda(), accept_len=acc, emitted=em,
                                         **out)
            pkg.dflash_select_sync_status(sel.h)
            got = {k: v.cpu().numpy() for k, v in out.items()}
            for k in ("topk_ids", "topk_vals", "pair_scores", "path", "path_score", "tie_flags"):
                assert np.array_equal(got[k], ref[k]), k
            assert np.array_equal(acc.cpu().numpy(), ref["accept"]) and np.array_equal(em.cpu().numpy(), ref["emitted"])
    got["accept"], got["emitted"] = acc.cpu().numpy(), em.cpu().numpy()
    rep = parity.compare(inp, got, orc, targets={s: tgt[s].numpy() for s in sel_seqs})
    assert rep["accept_checked"] == w.B
    assert sorted(set(got["accept"].tolist())) == sorted(set(n0.tolist()))
