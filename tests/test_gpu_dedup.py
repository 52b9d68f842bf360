"""The candidate-deduplication variant (each distinct token of a batch is
projected once, the pair tables read its row) against the per-row
projections and the oracle. A token's A and B rows come from the same MMA
sequence whichever rows share its tile, so every output must be identical to
the run without deduplication."""
import numpy as np
import pytest
import torch

from tests import parity
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

KEYS = ("topk_ids", "topk_vals", "pair_scores", "path", "path_score", "tie_flags")


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_draft_tcgen05_gb300 import build
    build.build()
    import speculative_decoding_draft_tcgen05_gb300 as p
    p.lib()
    return p


def paired_inputs(w):
    """Every odd sequence repeats the even one before it (hidden and anchor):
    half of all gathered rows are duplicates."""
    inp = wl.make_inputs(w)
    inp.hidden[1::2] = inp.hidden[0::2]
    inp.anchor[1::2] = inp.anchor[0::2]
    return inp


CASES = [
    ("small-vocabulary", lambda: wl.make_inputs(wl.custom(name="dd", B=40, L=7, K=16, V=2000, d=128, seed=51,
                                                          std_w=0.05))),
    ("paired-sequences", lambda: paired_inputs(wl.custom(name="dd", B=40, L=7, K=16, V=20000, d=128, seed=52,
                                                         std_w=0.05))),
    ("K32-L16", lambda: wl.make_inputs(wl.custom(name="dd", B=12, L=16, K=32, V=5000, d=192, seed=53, std_w=0.05))),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("walk", [0, 1])
def test_dedup_equals_per_row_projections(pkg, name, make, walk):
    inp = make()
    w = inp.wl
    d = parity.to_device(inp, "cuda")
    ref = parity.run_gpu(inp, dtensors=d, walk=walk)
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=w.L, K=w.K, max_batch=w.B, walk=walk,
                      tie_eps=parity.TIE_EPS, dedup=True) as sel:
        assert pkg.dflash_select_launches_per_run(sel.h, w.B) == 5  # merge, dedup, projection, pair tables
        for call in range(2):  # the marks of the first run must not leak into the second
            out = sel.run(d["hidden"], d["anchor"])
            pkg.dflash_select_sync_status(sel.h)
            got = {k: v.cpu().numpy() for k, v in out.items()}
            for k in KEYS:
                assert np.array_equal(got[k], ref[k]), f"call {call}: {k} differs"
    seqs = list(range(0, w.B, max(1, w.B // 6)))
    orc = parity.run_oracle(inp, seqs, walk=walk)
    rep = parity.compare(inp, got, orc, walk=walk)
    print(name, "walk", walk, rep)
    assert rep["path_equal"] >= 0.75 * len(seqs)


@pytest.mark.parametrize("name,seqs", [("4b_b32", [0, 11, 31]), ("stress_k16", [0, 100, 255])])
def test_dedup_workloads(pkg, name, seqs):
    inp = parity.inputs_for(name)
    d = parity.to_device(inp, "cuda")
    ref = parity.run_gpu(inp, dtensors=d)
    got = parity.run_gpu(inp, dtensors=d, dedup=True)
    for k in KEYS:
        assert np.array_equal(got[k], ref[k]), f"{k} differs"
    orc = parity.run_oracle(inp, seqs)
    rep = parity.compare(inp, got, orc)
    print(name, "dedup", rep)
    assert rep["path_equal"] >= 2


def test_dedup_reports_out_of_range_anchor(pkg):
    inp = wl.make_inputs(wl.custom(name="dd", B=40, L=3, K=16, V=1000, d=128, seed=5, std_w=0.05))
    d = parity.to_device(inp, "cuda")
    anchor = d["anchor"].clone()
    anchor[7] = 1000
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=3, K=16, max_batch=40, dedup=True) as sel:
        sel.run(d["hidden"], anchor)
        with pytest.raises(pkg.DflashError) as e:
            pkg.dflash_select_sync_status(sel.h)
        assert e.value.status == pkg.DFLASH_ERR_DEVICE_CHECK
        sel.run(d["hidden"], d["anchor"])
        pkg.dflash_select_sync_status(sel.h)


def test_dedup_arguments(pkg):
    inp = parity.inputs_for("tiny")
    d = parity.to_device(inp, "cuda")
    with pytest.raises(pkg.DflashError) as e:
        pkg.dflash_select_init(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=7, K=16, max_batch=2, tables=True,
                               dedup=True)
    assert e.value.status == pkg.DFLASH_ERR_INVALID_ARG
