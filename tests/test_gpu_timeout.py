"""The bounded pipeline wait of the kernels runs out, reports DEV_ERR_TIMEOUT
(bit 2) and leaves the context usable; no pipeline is broken and the GPU does
not fault: the test kernel waits on an mbarrier that nothing completes."""
import time

import pytest
import torch

from tests import parity

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


def test_wait_runs_out_and_context_survives(pkg):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    pkg.dflash_selftest_wait_timeout(status)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) & 2, "the timeout bit was not latched"
    assert 0.9 < elapsed < 10.0, elapsed  # the wait's bound is 1 s
    # the context still works: a whole selector run after it
    inp = parity.inputs_for("tiny")
    gpu = parity.run_gpu(inp)
    assert gpu["path"].shape == (inp.wl.B, inp.wl.L)
