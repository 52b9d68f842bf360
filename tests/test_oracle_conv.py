"""Pins of the oracle's two-tap dynamic depthwise convolution (no GPU):
a hand-worked example, the fixed-kernel special case against numpy's
convolution, the pages' parameter count, and block locality."""
import json
import os

import numpy as np
import torch

import oracle
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "conv2_hand_example.json")


def _bits(a):
    return wl.bf16_bits(torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def test_hand_worked_example():
    g = json.load(open(GOLDEN))
    B, S, d = g["B"], g["S"], g["d"]
    X = np.zeros((B, S, d), np.float32)
    for b, t, c, v in g["X_nonzero"]:
        X[b, t, c] = v
    base = np.stack([np.full(d, g["base"]["tap0_all_channels"]), np.full(d, g["base"]["tap1_all_channels"])])
    Wc = np.zeros((2 * d // 16, d), np.float32)
    for r, c, v in g["Wc_nonzero"]:
        Wc[r, c] = v
    want = np.zeros((B, S, d))
    for b, t, c, v in g["Y_nonzero"]:
        want[b, t, c] = v
    Y = oracle.conv2(_bits(X), _bits(base), _bits(Wc))
    assert np.array_equal(Y, want), np.argwhere(Y != want)


def test_fixed_kernel_is_a_causal_depthwise_convolution():
    """Wc = 0 leaves the base kernel: per channel, numpy's full convolution of
    the block with (base0, base1), truncated to the block (x_{-1} = 0)."""
    rng = np.random.default_rng(5)
    B, S, d = 3, 8, 64
    X = _f(rng.normal(size=(B, S, d)))
    base = _f(rng.normal(size=(2, d)))
    Y = oracle.conv2(_bits(X), _bits(base), _bits(np.zeros((2 * d // 16, d))))
    for b in range(B):
        for c in range(d):
            ref = np.convolve(X[b, :, c].astype(np.float64), [base[0, c], base[1, c]])[:S]
            assert np.allclose(Y[b, :, c], ref, rtol=1e-14, atol=1e-14)


def test_correction_shared_by_16_channels_and_taken_from_the_current_row():
    """With a zero base kernel, Y[t, c] / x_t[c] is the tap-0 correction of c's
    group and depends on x_t only; channels of one group share it."""
    rng = np.random.default_rng(6)
    B, S, d = 1, 4, 64
    X = _f(rng.uniform(0.5, 1.5, size=(B, S, d)))
    Wc = _f(rng.normal(size=(2 * d // 16, d)))
    Wc[1::2] = 0.0  # tap 1 off: y_t = corr_{t,0} * x_t
    Y = oracle.conv2(_bits(X), _bits(np.zeros((2, d))), _bits(Wc))
    for t in range(S):
        ratio = Y[0, t] / X[0, t].astype(np.float64)
        for g in range(d // 16):
            expect = float(np.dot(Wc[2 * g].astype(np.float64), X[0, t].astype(np.float64)))
            assert np.allclose(ratio[16 * g:16 * g + 16], expect, rtol=1e-12)


def test_parameter_count_matches_the_pages():
    """Base [2, d] + Wc [2 d/16, d] per convolution, one in front of and one
    behind every attention and every feed-forward sublayer of the five-layer
    drafter (20 in all), at the Qwen3-4B width d = 2560: the pages' 16.5M added parameters."""
    d = 2560
    per_conv = 2 * d + 2 * (d // 16) * d
    total = 5 * 2 * 2 * per_conv
    assert abs(total / 1e6 - 16.5) < 0.05, total


def test_blocks_are_independent():
    rng = np.random.default_rng(7)
    B, S, d = 3, 5, 32
    X = _f(rng.normal(size=(B, S, d)))
    base = _f(rng.normal(size=(2, d)))
    Wc = _f(rng.normal(size=(2 * d // 16, d)) * 0.1)
    Y = oracle.conv2(_bits(X), _bits(base), _bits(Wc))
    X2 = X.copy()
    X2[0] = _f(rng.normal(size=(S, d)))
    X2[2] = _f(rng.normal(size=(S, d)))
    Y2 = oracle.conv2(_bits(X2), _bits(base), _bits(Wc))
    assert np.array_equal(Y[1], Y2[1])


def _f(a):
    """Round to bf16 (the values both sides consume)."""
    return (_bits(a).astype(np.uint32) << 16).view(np.float32)
