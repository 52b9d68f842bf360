"""GPU parity of the two-tap dynamic depthwise convolution against the CPU
oracle, through the C ABI (bf16 in and out, fp32 accumulation)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2e-2, 2e-3  # bf16 inputs, fp32 accumulation, bf16 output


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_draft_tcgen05_gb300 import build
    build.build()
    import speculative_decoding_draft_tcgen05_gb300 as p
    p.lib()
    return p


def _run(pkg, ci):
    with pkg.Conv2(ci.base.cuda(), ci.Wc.cuda()) as conv:
        Y = conv(ci.X.cuda())
        pkg.dflash_conv2_sync_status(conv.h)
    torch.cuda.synchronize()
    return Y.float().cpu().numpy()


def _oracle(ci, rows=None):
    X = ci.X if rows is None else ci.X[rows]
    return oracle.conv2(wl.bf16_bits(X), wl.bf16_bits(ci.base), wl.bf16_bits(ci.Wc), nthreads=oracle.max_threads())


def _check(gpu, ref):
    err = np.abs(gpu - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance, worst {err.max():.3g}"


@pytest.mark.parametrize("B,S,d", [
    # up to 8 rows: the CUDA-core kernel
    (1, 8, 128),      # one block, d = 128
    (1, 8, 2560),     # Qwen3-4B width, one block
    (1, 8, 4096),     # the widest d with two 16-byte pieces per thread (one pass)
    (1, 7, 4160),     # the narrowest d with one piece per thread (three passes)
    (1, 8, 5120),     # 27B-class width
    (3, 1, 256),      # S = 1: every row starts a block
    (1, 5, 16384),    # the widest d (64 KB of Wc rows per CTA)
    # more rows: the tcgen05 kernel
    (2, 8, 2560),     # 16 rows: a 16-wide tile, d split over a cluster of 8
    (4, 8, 2560),     # 32 rows
    (3, 11, 1024),    # 33 rows: three 16-wide tiles
    (5, 7, 640),      # ragged rows, 80 Wc rows (one partial Wc tile)
    (40, 8, 2560),    # 320 rows, three Wc tiles (the last ragged): 64-wide tiles, d split over 8
    (32, 8, 5120),    # 256 rows at the 27B-class width: 128-wide tiles, d split over 8
    (1, 300, 64),     # one long block, d = 64 (a single k-block, no split)
])
def test_conv_matches_oracle(pkg, B, S, d):
    ci = wl.make_conv_inputs(B, S, d, seed=B * 131 + S * 7 + d)
    _check(_run(pkg, ci), _oracle(ci))


def test_conv_stress_shape_sampled(pkg):
    """The stress shape (256 blocks of 16 rows at d = 2560) in the launch the
    bench times; the oracle checks a sample of the blocks."""
    ci = wl.make_conv_inputs(256, 16, 2560, seed=11)
    gpu = _run(pkg, ci)
    rows = [0, 1, 77, 128, 255]
    ref = _oracle(ci, rows)
    _check(gpu[rows], ref)


def test_conv_arguments(pkg):
    d = 256
    ci = wl.make_conv_inputs(2, 4, d, seed=3)
    base, Wc = ci.base.cuda(), ci.Wc.cuda()
    with pytest.raises(pkg.DflashError) as e:  # d not a multiple of 64
        pkg.dflash_conv2_init(base[:, :96].contiguous(), Wc[:12, :96].contiguous())
    assert e.value.status == pkg.DFLASH_ERR_UNSUPPORTED
    with pkg.Conv2(base, Wc) as conv:
        X = ci.X.cuda()
        with pytest.raises(pkg.DflashError) as e:  # in place
            pkg.dflash_conv2_run(conv.h, X, X)
        assert e.value.status == pkg.DFLASH_ERR_INVALID_ARG
        empty = torch.empty(0, 4, d, dtype=torch.bfloat16, device="cuda")
        pkg.dflash_conv2_run(conv.h, empty, torch.empty_like(empty))  # B = 0: nothing launched
        # two calls in a row on the same handle give the same result
        Y1, Y2 = conv(X), conv(X)
        pkg.dflash_conv2_sync_status(conv.h)
        assert torch.equal(Y1, Y2)
