"""Seeded synthetic workloads for the DFlash 2 path selector.

This module only draws random inputs; it holds none of the selector's
arithmetic (no logits, no top-K, no pair scores, no walk). Both the CUDA path
and the CPU oracle consume what it returns, so the two always see the same
bf16 values.

Shapes follow the pages' setting (DFlash 2 blog, "A Lightweight Path Selector":
top-16 candidates per draft position, 256-dim token embeddings; dev.to
commentary, "Key facts": block size 8, i.e. seven draft positions after the
last verified token; blog "Putting It Together": 15-position blocks).

Distributions (all seeded, CPU torch generator, drawn in a fixed order):
  W (lm_head) and E (token table): [V, d] ~ N(0, std_w), rounded to bf16
  W_A, W_B, W_H: [e, d] ~ N(0, 1/sqrt(d)), rounded to bf16
  hidden: [B, L, d] ~ N(0, 1), rounded to bf16 (optionally with planted
          near-tied top-2 logits, see ``plant_near_ties``)
  anchor (last verified token x0): [B] uniform in [0, V)
  target_rand: [B, L+1] uniform in [0, V)
  n0 (planted accepted-prefix length): [B] uniform in [0, L]
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

E_DIM = 256  # width of the A/B token embeddings and of the context gate


@dataclass(frozen=True)
class Workload:
    name: str
    label: str
    B: int
    L: int
    K: int
    V: int
    d: int
    seed: int
    std_w: float
    e: int = E_DIM
    planted_targets: bool = True
    near_tie_frac: float = 0.0

    @property
    def N(self) -> int:
        return self.B * self.L


def _w(name, label, **kw):
    return Workload(name=name, label=label, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        _w("tiny", "tiny selector: batch 2, L=7, K=16, V=4096, d=128, e=256",
           B=2, L=7, K=16, V=4096, d=128, seed=0, std_w=0.05, planted_targets=False),
        _w("4b_b1", "Qwen3-4B-shaped drafter head, batch 1: d=2560, V=151936, L=7, K=16, e=256",
           B=1, L=7, K=16, V=151936, d=2560, seed=1, std_w=0.02),
        _w("4b_b8", "Qwen3-4B-shaped drafter head, batch 8: d=2560, V=151936, L=7, K=16, e=256",
           B=8, L=7, K=16, V=151936, d=2560, seed=2, std_w=0.02),
        _w("4b_b32", "Qwen3-4B-shaped drafter head, batch 32: d=2560, V=151936, L=7, K=16, e=256",
           B=32, L=7, K=16, V=151936, d=2560, seed=3, std_w=0.02),
        _w("27b_b1", "27B-class drafter head, batch 1: d=5120, V=151936, L=7, K=16, e=256",
           B=1, L=7, K=16, V=151936, d=5120, seed=4, std_w=0.02),
        _w("27b_b8", "27B-class drafter head, batch 8: d=5120, V=151936, L=7, K=16, e=256",
           B=8, L=7, K=16, V=151936, d=5120, seed=5, std_w=0.02),
        _w("27b_b32", "27B-class drafter head, batch 32: d=5120, V=151936, L=7, K=16, e=256",
           B=32, L=7, K=16, V=151936, d=5120, seed=6, std_w=0.02),
        _w("stress_k16", "stress: d=2560, V=151936, block 16 (L=15), K=16, e=256, batch 256, 10% near-tied top logits",
           B=256, L=15, K=16, V=151936, d=2560, seed=7, std_w=0.02, near_tie_frac=0.10),
        _w("stress_k32", "stress: d=2560, V=151936, block 16 (L=15), K=32, e=256, batch 256, 10% near-tied top logits",
           B=256, L=15, K=32, V=151936, d=2560, seed=8, std_w=0.02, near_tie_frac=0.10),
    ]
}


def custom(name="custom", *, B, L, K, V, d, seed=0, std_w=0.02, planted_targets=False,
           near_tie_frac=0.0) -> Workload:
    """A workload of any shape with the same distributions (used for edge cases)."""
    return Workload(name=name, label=f"{name}: B={B} L={L} K={K} V={V} d={d}", B=B, L=L, K=K, V=V,
                    d=d, seed=seed, std_w=std_w, planted_targets=planted_targets,
                    near_tie_frac=near_tie_frac)


def _randn_bf16(rows: int, cols: int, std: float, g: torch.Generator, chunk: int = 16384) -> torch.Tensor:
    """N(0, std) rows drawn in fixed-size row chunks (bounded peak memory), rounded to bf16."""
    out = torch.empty(rows, cols, dtype=torch.bfloat16)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        out[r0:r1] = torch.randn(r1 - r0, cols, generator=g).mul_(std).to(torch.bfloat16)
    return out


@dataclass
class Inputs:
    wl: Workload
    W: torch.Tensor        # [V, d] bf16 lm_head
    E: torch.Tensor        # [V, d] bf16 token table
    W_A: torch.Tensor      # [e, d] bf16
    W_B: torch.Tensor      # [e, d] bf16
    W_H: torch.Tensor      # [e, d] bf16
    hidden: torch.Tensor   # [B, L, d] bf16
    anchor: torch.Tensor   # [B] int32
    target_rand: torch.Tensor  # [B, L+1] int32
    n0: torch.Tensor       # [B] int32
    near_tie_pos: list = field(default_factory=list)  # planted (b, t, v1, v2)


def make_inputs(wl: Workload) -> Inputs:
    """Draws every input of ``wl`` from its seed, in a fixed order."""
    g = torch.Generator().manual_seed(wl.seed)
    W = _randn_bf16(wl.V, wl.d, wl.std_w, g)
    E = _randn_bf16(wl.V, wl.d, wl.std_w, g)
    s = 1.0 / math.sqrt(wl.d)
    W_A = _randn_bf16(wl.e, wl.d, s, g)
    W_B = _randn_bf16(wl.e, wl.d, s, g)
    W_H = _randn_bf16(wl.e, wl.d, s, g)
    hidden32 = torch.randn(wl.B, wl.L, wl.d, generator=g)
    anchor = torch.randint(0, wl.V, (wl.B,), generator=g, dtype=torch.int64).to(torch.int32)
    target_rand = torch.randint(0, wl.V, (wl.B, wl.L + 1), generator=g, dtype=torch.int64).to(torch.int32)
    n0 = torch.randint(0, wl.L + 1, (wl.B,), generator=g, dtype=torch.int64).to(torch.int32)
    near = []
    hidden = hidden32.to(torch.bfloat16)
    if wl.near_tie_frac > 0:
        hidden, near = plant_near_ties(hidden32, W, wl.near_tie_frac, g)
    return Inputs(wl, W, E, W_A, W_B, W_H, hidden, anchor, target_rand, n0, near)


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    """float64 values of bf16 bit patterns (uint16 array)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_step(bits: np.ndarray, up: np.ndarray) -> np.ndarray:
    """bf16 bit patterns one representable step above (up) or below each entry of ``bits``."""
    b = bits.astype(np.int64)
    zero = (b & 0x7FFF) == 0
    positive = (b & 0x8000) == 0
    step = np.where(positive == up, b + 1, b - 1)
    step = np.where(zero, np.where(up, 0x0001, 0x8001), step)
    return step.astype(np.uint16)


def plant_near_ties(hidden32: torch.Tensor, W: torch.Tensor, frac: float, g: torch.Generator,
                    beta: float = 10.0, gap: float = 5e-4):
    """Gives a fraction ``frac`` of the (b, t) positions two tokens v1 != v2 whose
    rows of W score (almost) the same against the position's hidden state, well
    above the rest of the vocabulary.

    Recipe, in fp64 on the two rows w1, w2 only: take D = w1 - w2 and the part u
    of w1 + w2 orthogonal to D (unit length); remove from h its components along
    D and u, add beta * u, round to bf16; then, while |D . h| >= gap, move by one
    bf16 step the coordinate (among the 64 with the largest |D_i|) that brings
    |D . h| down the most. Returns the bf16 hidden tensor and the planted
    (b, t, v1, v2).
    """
    B, L, d = hidden32.shape
    V = W.shape[0]
    npos = B * L
    nplant = int(round(frac * npos))
    order = torch.randperm(npos, generator=g)[:nplant].tolist()
    toks = torch.randint(0, V, (nplant, 2), generator=g, dtype=torch.int64).tolist()
    h = hidden32.to(torch.float64).reshape(npos, d).numpy()
    out = hidden32.to(torch.bfloat16).reshape(npos, d).clone()
    out_bits = out.view(torch.int16).numpy().view(np.uint16)
    planted = []
    for p, (v1, v2) in zip(order, toks):
        if v1 == v2:
            v2 = (v1 + 1) % V
        w1 = W[v1].to(torch.float64).numpy()
        w2 = W[v2].to(torch.float64).numpy()
        D = w1 - w2
        S = w1 + w2
        u = S - (D @ S) / (D @ D) * D
        u = u / np.linalg.norm(u)
        hp = h[p] - (D @ h[p]) / (D @ D) * D
        hp = hp - (u @ hp) * u + beta * u
        bits = torch.from_numpy(hp).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
        vals = _bf16_values(bits)
        cur = float(D @ vals)
        cand = np.argsort(-np.abs(D))[:64]
        for _ in range(256):
            if abs(cur) < gap:
                break
            up = (cur * D[cand]) < 0  # raising h_i lowers |cur| when D_i and cur differ in sign
            nb = _bf16_step(bits[cand], up)
            new = cur + D[cand] * (_bf16_values(nb) - vals[cand])
            k = int(np.argmin(np.abs(new)))
            if abs(new[k]) >= abs(cur):
                break
            i = cand[k]
            bits[i] = nb[k]
            vals[i] = _bf16_values(nb[k:k + 1])[0]
            cur = float(new[k])
        out_bits[p] = bits
        planted.append((p // L, p % L, v1, v2))
    return out.reshape(B, L, d), planted


def plant_targets(path_tokens: torch.Tensor, target_rand: torch.Tensor, n0: torch.Tensor, V: int) -> torch.Tensor:
    """Target argmax tokens [B, L+1] whose first n0[b] entries equal the given
    path, whose entry n0[b] differs from path[b, n0[b]] (when n0[b] < L), and
    whose remaining entries are the uniform draws ``target_rand``. A greedy
    prefix check then accepts exactly n0[b] draft tokens."""
    B, L = path_tokens.shape
    tgt = target_rand.clone()
    for b in range(B):
        n = int(n0[b])
        tgt[b, :n] = path_tokens[b, :n]
        if n < L and int(tgt[b, n]) == int(path_tokens[b, n]):
            tgt[b, n] = (int(path_tokens[b, n]) + 1) % V
    return tgt


def bf16_bits(t: torch.Tensor):
    """The raw bf16 bit patterns of a CPU tensor as a numpy uint16 array (no copy of values)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")


@dataclass
class ConvInputs:
    """One two-tap dynamic convolution and the blocks it runs over (bf16, CPU)."""
    X: torch.Tensor     # [B, S, d] blocks: the last verified token's row, then the draft rows
    base: torch.Tensor  # [2, d] base kernels (tap 0: current row, tap 1: the row before)
    Wc: torch.Tensor    # [d/8, d] correction weights, row 2g + i = tap i of channel group g


def make_conv_inputs(B: int, S: int, d: int, seed: int) -> ConvInputs:
    """Seeded inputs of the drafter's two-tap convolution at a workload's shape
    (blocks of S = L + 1 rows). Draw order and distributions:
      X    [B, S, d] ~ N(0, 1)               (hidden states)
      base [2, d]:   tap 0 ~ 1 + N(0, 0.1), tap 1 ~ N(0, 0.1)
      Wc   [d/8, d] ~ N(0, 0.1 / sqrt(d))    (a small correction)
    all rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(B, S, d, generator=g).to(torch.bfloat16)
    base = torch.randn(2, d, generator=g) * 0.1
    base[0] += 1.0
    Wc = torch.randn(d // 8, d, generator=g) * (0.1 / math.sqrt(d))
    return ConvInputs(X=X, base=base.to(torch.bfloat16), Wc=Wc.to(torch.bfloat16))
