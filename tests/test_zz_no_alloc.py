"""The allocation-free lm_head + top-K entry point against the selector's own.

dflash_lmhead_topk_noalloc serves callers that may not allocate device memory
(engines that own every byte of device memory in their own arena, or code
where an allocation would synchronise the device). It keeps its scratch in a
fixed array inside the library instead of a handle's workspace. Here it is
called twice in a row through the C ABI and must return the same candidates
and logits as dflash_select_run on the same inputs. This file is collected
last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

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


CASES = [
    wl.WORKLOADS["tiny"],
    wl.custom(name="noalloc_k32", B=2, L=16, K=32, V=5000, d=192, seed=23, std_w=0.05),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_selector_twice(pkg, w):
    inp = wl.make_inputs(w)
    d = parity.to_device(inp, "cuda")
    ref = parity.run_gpu(inp, dtensors=d)  # the handle-based entry point
    N = w.B * w.L
    hidden = d["hidden"].reshape(N, w.d).contiguous()
    for call in range(2):
        ids = torch.full((N, w.K), -7, dtype=torch.int32, device="cuda")
        vals = torch.full((N, w.K), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        pkg.dflash_lmhead_topk_noalloc(d["W"], hidden, w.K, ids, vals, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status"
        g_ids = ids.cpu().numpy().reshape(w.B, w.L, w.K)
        g_vals = vals.cpu().numpy().reshape(w.B, w.L, w.K)
        assert np.array_equal(g_ids, ref["topk_ids"]), f"call {call}: candidates differ"
        assert parity.close(g_vals, ref["topk_vals"]).all(), f"call {call}: logits differ"
    # the values output is optional
    ids2 = torch.empty((N, w.K), dtype=torch.int32, device="cuda")
    pkg.dflash_lmhead_topk_noalloc(d["W"], hidden, w.K, ids2)
    torch.cuda.synchronize()
    assert np.array_equal(ids2.cpu().numpy().reshape(w.B, w.L, w.K), ref["topk_ids"])


def test_noalloc_rejects_sizes_beyond_its_scratch(pkg):
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w)
    W = inp.W.cuda()
    too_many = torch.zeros(257, w.d, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(257, w.K, dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.DflashError) as e:
        pkg.dflash_lmhead_topk_noalloc(W, too_many, w.K, ids)
    assert e.value.status == pkg.DFLASH_ERR_UNSUPPORTED
    with pytest.raises(pkg.DflashError) as e:
        pkg.dflash_lmhead_topk_noalloc(W, too_many[:4], 8, ids[:4])
    assert e.value.status == pkg.DFLASH_ERR_UNSUPPORTED
    # a rejected call leaves the entry point usable
    ok_ids = torch.empty(4, w.K, dtype=torch.int32, device="cuda")
    pkg.dflash_lmhead_topk_noalloc(W, inp.hidden.reshape(-1, w.d)[:4].contiguous().cuda(), w.K, ok_ids)
    torch.cuda.synchronize()
