"""GPU parity of the precomputed-tables variant (A|B of every token computed
once at init, table rows gathered in every run) against the CPU oracle, on
both tail paths: the fused small-batch kernel and the pair-table kernel."""
import pytest
import torch

from tests import parity
from tests.test_gpu_parity import _full_check
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


@pytest.mark.parametrize("walk", [0, 1])
def test_tiny_tables(pkg, walk):
    inp = parity.inputs_for("tiny")
    gpu, orc, rep = _full_check(inp, walk=walk, tables=True)
    assert rep["path_equal"] + rep["path_alternative"] == inp.wl.B


@pytest.mark.parametrize("shape", [dict(B=2, L=16, K=32, V=5000, d=192), dict(B=40, L=7, K=16, V=2000, d=128),
                                   dict(B=1, L=5, K=16, V=129, d=256)],
                         ids=["L16K32", "several-n-tiles", "V129"])
def test_edge_shapes_tables(pkg, shape):
    inp = wl.make_inputs(wl.custom(name="edge", seed=17, std_w=0.05, **shape))
    gpu, orc, rep = _full_check(inp, tables=True, max_batch=shape["B"] + 3)
    assert rep["positions"] == shape["B"] * shape["L"]


@pytest.mark.parametrize("name,seqs", [("4b_b1", None), ("4b_b8", None), ("4b_b32", [0, 9, 31]), ("27b_b1", None)])
def test_workloads_tables(pkg, name, seqs):
    inp = parity.inputs_for(name)
    gpu, orc, rep = _full_check(inp, seqs=seqs, tables=True)
    assert rep["seqs"] == (len(seqs) if seqs else inp.wl.B)


def test_stress_tables_sampled(pkg):
    inp = parity.inputs_for("stress_k32")
    seqs = [0, 37, 64, 101, 128, 170, 211, 255]
    gpu, orc, rep = _full_check(inp, seqs=seqs, tables=True)
    assert rep["seqs"] == len(seqs)
    assert rep["path_equal"] >= 0.75 * len(seqs) and rep["accept_checked"] >= 0.75 * len(seqs), rep


@pytest.mark.parametrize("B", [1, 40])
def test_out_of_range_anchor_tables(pkg, B):
    """Both tail paths latch an out-of-range anchor with tables too."""
    inp = wl.make_inputs(wl.custom(name="edge", seed=5, std_w=0.05, B=B, L=3, K=16, V=1000, d=128))
    d = parity.to_device(inp, "cuda")
    anchor = d["anchor"].clone()
    anchor[B - 1] = 1000
    with pkg.Selector(d["W"], d["E"], d["W_A"], d["W_B"], d["W_H"], L=3, K=16, max_batch=B, tables=True) as sel:
        sel.run(d["hidden"], anchor)
        with pytest.raises(pkg.DflashError) as e:
            pkg.dflash_select_sync_status(sel.h)
        assert e.value.status == pkg.DFLASH_ERR_DEVICE_CHECK
