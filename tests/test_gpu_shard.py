"""The vocabulary-sharded selector on one GPU: the lm_head rows are split into
G shards, each shard's handle streams its rows and writes its K best keys per
position, the lists are stacked as an exchange between G GPUs would deliver
them, and one handle finishes the selector from them. The result must equal
the whole-vocabulary run exactly (every logit is computed by the same MMA
sequence, whichever shard holds its row) and match the oracle."""
import numpy as np
import pytest
import torch

from tests import parity
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl
from speculative_decoding_draft_tcgen05_gb300.shard import shard_range

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


def run_sharded(pkg, inp, ranges, walk=0):
    w = inp.wl
    d = parity.to_device(inp, "cuda")
    handles = [pkg.dflash_select_init_shard(d["W"][v0:v1], v0, v1, d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L,
                                            K=w.K, max_batch=w.B, walk=walk, tie_eps=parity.TIE_EPS)
               for v0, v1 in ranges]
    try:
        keys = torch.zeros(len(ranges), w.B, w.L, w.K, dtype=torch.int64, device="cuda")
        for g, h in enumerate(handles):
            pkg.dflash_select_topk_shard(h, d["hidden"], keys[g])
        out = dict(path=torch.empty(w.B, w.L, dtype=torch.int32, device="cuda"),
                   topk_ids=torch.empty(w.B, w.L, w.K, dtype=torch.int32, device="cuda"),
                   topk_vals=torch.empty(w.B, w.L, w.K, dtype=torch.float32, device="cuda"),
                   pair_scores=torch.empty(w.B, w.L, w.K, w.K, dtype=torch.float32, device="cuda"),
                   path_score=torch.empty(w.B, dtype=torch.float32, device="cuda"),
                   tie_flags=torch.empty(w.B, w.L, dtype=torch.uint8, device="cuda"))
        pkg.dflash_select_run_gathered(handles[0], d["anchor"], keys, **out)
        for h in handles:
            pkg.dflash_select_sync_status(h)
        torch.cuda.synchronize()
    finally:
        for h in handles:
            pkg.dflash_select_destroy(h)
    return {k: v.cpu().numpy() for k, v in out.items()}, keys.cpu().numpy()


def key_ids(keys):
    return (~(keys & 0xFFFFFFFF)).astype(np.int64) & 0xFFFFFFFF


CASES = [
    ("tiny", [(0, 4096)]),                    # one shard through the exchange entry points
    ("tiny", [(0, 1000), (1000, 4096)]),      # a boundary inside a 128-row tile
    ("tiny", [shard_range(4096, 3, r) for r in range(3)]),
    ("4b_b1", [shard_range(151936, 2, r) for r in range(2)]),
    ("4b_b8", [shard_range(151936, 4, r) for r in range(4)]),
]


@pytest.mark.parametrize("name,ranges", CASES, ids=[f"{n}-G{len(r)}-{r[0][1]}" for n, r in CASES])
def test_sharded_selector_equals_whole_vocabulary(pkg, name, ranges):
    inp = parity.inputs_for(name)
    w = inp.wl
    whole = parity.run_gpu(inp)
    got, keys = run_sharded(pkg, inp, ranges)
    # every shard's list holds only its own rows, best first
    for g, (v0, v1) in enumerate(ranges):
        ids = key_ids(keys[g])
        assert ((ids >= v0) & (ids < v1)).all(), f"shard {g} returned a token outside [{v0}, {v1})"
        u = keys[g].astype(np.uint64)
        assert (u[..., :-1] > u[..., 1:]).all(), f"shard {g}: keys not sorted best first"
    for k in ("topk_ids", "topk_vals", "pair_scores", "path", "path_score", "tie_flags"):
        assert np.array_equal(got[k], whole[k]), f"{k} differs from the whole-vocabulary run"
    orc = parity.run_oracle(inp, range(min(w.B, 4)))
    rep = parity.compare(inp, got, orc)
    print(name, len(ranges), "shards", rep)
    assert rep["path_equal"] == len(orc)


def test_shard_arguments(pkg):
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    w = inp.wl
    for v0, v1 in [(-1, 10), (10, 10), (0, w.V + 1)]:
        with pytest.raises(pkg.DflashError) as e:
            pkg.lib()  # the binding checks the shape; call the C entry point directly for the range checks
            cfg = pkg.dflash_select_config(V=w.V, d=w.d, L=w.L, K=w.K, e=256, max_batch=2, walk=0, tie_eps=1e-3,
                                           temperature=1.0, tables=0)
            h = pkg.ctypes.c_void_p()
            P = lambda t: pkg.ctypes.c_void_p(t.data_ptr())
            st = pkg.lib().dflash_select_init_shard(pkg.ctypes.byref(cfg), P(d["W"]), v0, v1, P(d["E"]),
                                                    P(d["W_A"]), P(d["W_B"]), P(d["W_H"]), None,
                                                    pkg.ctypes.byref(h))
            pkg._check(st, "dflash_select_init_shard")
        assert e.value.status == pkg.DFLASH_ERR_INVALID_ARG
    h = pkg.dflash_select_init_shard(d["W"][:2048], 0, 2048, d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K,
                                     max_batch=2)
    try:
        path = torch.empty(2, w.L, dtype=torch.int32, device="cuda")
        with pytest.raises(pkg.DflashError) as e:  # a shard handle does not run the whole selector
            pkg.dflash_select_run(h, d["hidden"], d["anchor"], path=path)
        assert e.value.status == pkg.DFLASH_ERR_INVALID_ARG
        keys = torch.zeros(0, 2, w.L, w.K, dtype=torch.int64, device="cuda")
        with pytest.raises(pkg.DflashError):  # G = 0
            pkg.dflash_select_run_gathered(h, d["anchor"], keys, path=path)
    finally:
        pkg.dflash_select_destroy(h)
