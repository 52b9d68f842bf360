"""The allocation-free lm_head + top-K entry point.

dflash_lmhead_topk_noalloc serves callers that may not allocate device memory
(engines that own every byte of device memory in their own arena, or code
where an allocation would synchronise the device). It keeps its scratch in a
fixed array inside the library instead of a handle's workspace. Here it is
called twice in a row through the C ABI; both calls must return the oracle's
top-K (under the usual near-tie rules) and the same candidates and logits as
dflash_select_run on the same inputs. This file is collected last so that a
run stopping at the first failure has run every other test.
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
    # 200 positions: two position tiles of 112
    wl.custom(name="noalloc_n200", B=25, L=8, K=16, V=20000, d=128, seed=24, std_w=0.05),
    # 256 positions at K = 32: two tiles of 128
    wl.custom(name="noalloc_n256_k32", B=16, L=16, K=32, V=6000, d=64, seed=25, std_w=0.05),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_oracle_and_selector_twice(pkg, w):
    inp = wl.make_inputs(w)
    d = parity.to_device(inp, "cuda")
    ref = parity.run_gpu(inp, dtensors=d)  # the handle-based entry point
    N = w.B * w.L
    H_bits = wl.bf16_bits(inp.hidden.reshape(N, w.d).contiguous())
    orc = parity.oracle_topk_rows(inp, H_bits, w.K)
    hidden = d["hidden"].reshape(N, w.d).contiguous()
    for call in range(2):
        ids = torch.full((N, w.K), -7, dtype=torch.int32, device="cuda")
        vals = torch.full((N, w.K), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        pkg.dflash_lmhead_topk_noalloc(d["W"], hidden, w.K, ids, vals, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status"
        g_ids = ids.cpu().numpy()
        g_vals = vals.cpu().numpy()
        rep = parity.compare_topk(inp, H_bits, g_ids, g_vals, orc)
        print(w.name, "call", call, rep)
        assert np.array_equal(g_ids.reshape(w.B, w.L, w.K), ref["topk_ids"]), f"call {call}: candidates differ"
        assert parity.close(g_vals.reshape(w.B, w.L, w.K), ref["topk_vals"]).all(), f"call {call}: logits differ"
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
    # 256 positions at K = 32 over 8192 rows: 64 CTAs per position tile hold
    # 64 * 256 * 32 * 8 bytes (4 MiB) of partial lists, more than the scratch
    W_big = torch.zeros(8192, 64, dtype=torch.bfloat16, device="cuda")
    h256 = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    ids256 = torch.empty(256, 32, dtype=torch.int32, device="cuda")
    with pytest.raises(pkg.DflashError) as e:
        pkg.dflash_lmhead_topk_noalloc(W_big, h256, 32, ids256)
    assert e.value.status == pkg.DFLASH_ERR_UNSUPPORTED
    assert "scratch" in str(e.value)
    # a rejected call leaves the entry point usable
    ok_ids = torch.empty(4, w.K, dtype=torch.int32, device="cuda")
    pkg.dflash_lmhead_topk_noalloc(W, inp.hidden.reshape(-1, w.d)[:4].contiguous().cuda(), w.K, ok_ids)
    torch.cuda.synchronize()
    ref = parity.oracle_topk_rows(inp, wl.bf16_bits(inp.hidden.reshape(-1, w.d)[:4].contiguous()), w.K)
    parity.compare_topk(inp, wl.bf16_bits(inp.hidden.reshape(-1, w.d)[:4].contiguous()), ok_ids.cpu().numpy(), None,
                        ref)
