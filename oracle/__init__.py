"""Plain fp64 CPU oracle of the DFlash 2 path selector (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never calls it and
shares no code with it. The arithmetic lives in ``oracle.c`` (explicit loops,
double precision, a full sort); this module only compiles it with gcc and
marshals numpy arrays. ``brute.py`` holds the brute-force path enumeration
used to pin the walk.

Method source: blog post "DFlash 2: Keep Drafting Parallel", section
"A Lightweight Path Selector" (pair score S_t and the walk), and section
"The Right Tokens Are Already There" (top-16 candidate lists).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

WALK_VITERBI = 0
WALK_GREEDY = 1


def build(force: bool = False) -> str:
    """Compiles oracle.c into liboracle.so (plain -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
                        "-ffp-contract=off", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int
            lib.oracle_logits.argtypes = [P, P, i64, i64, i64, P, i32]
            lib.oracle_topk.argtypes = [P, i64, i32, P, P, P]
            lib.oracle_project.argtypes = [P, i64, i64, P, P]
            lib.oracle_pair_scores.argtypes = [i32, i32, i64, P, P, P, P, P]
            lib.oracle_viterbi.argtypes = [i32, i32, P, P, P, P, P]
            lib.oracle_greedy.argtypes = [i32, i32, P, P, P, P, P]
            lib.oracle_verify.argtypes = [i32, P, P, P]
            lib.oracle_verify.restype = i32
            lib.oracle_select.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, i32, P, ctypes.c_int32,
                                          P, P, P, P, P, P, P, P, P, i32]
            lib.oracle_select_given.argtypes = [P, P, P, P, P, i64, i64, i64, i32, i32, i32, P,
                                                ctypes.c_int32, P, P, P, P, P, P, P, P]
            lib.oracle_max_threads.restype = i32
            lib.oracle_sample_walk.argtypes = [i32, i32, P, ctypes.c_double, P, P, P, P]
            lib.oracle_verify_rejection.argtypes = [i32, i32, i64, P, P, P, P, P, ctypes.c_double, P, P, P]
            lib.oracle_verify_rejection.restype = i32
            lib.oracle_conv2.argtypes = [i64, i64, i64, P, P, P, P, i32]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 inputs are passed as raw uint16 bit patterns"
    return a


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def logits(W_bits, H_bits, nthreads: int = 1) -> np.ndarray:
    """U [N, V] = H W^T in fp64 from bf16 bit patterns W [V, d], H [N, d]."""
    W_bits, H_bits = _u16(W_bits), _u16(H_bits)
    V, d = W_bits.shape
    H2 = H_bits.reshape(-1, d)
    U = np.empty((H2.shape[0], V), dtype=np.float64)
    _load().oracle_logits(_p(W_bits), _p(H2), V, d, H2.shape[0], _p(U), int(nthreads))
    return U


def topk(U_row, K: int):
    """(ids [K] int32, vals [K] fp64, boundary margin U_(K) - U_(K+1))."""
    U_row = np.ascontiguousarray(U_row, dtype=np.float64)
    ids = np.empty(K, dtype=np.int32)
    vals = np.empty(K, dtype=np.float64)
    m = np.empty(1, dtype=np.float64)
    _load().oracle_topk(_p(U_row), U_row.shape[0], K, _p(ids), _p(vals), _p(m))
    return ids, vals, float(m[0])


def project(P_bits, x_bits) -> np.ndarray:
    """P x in fp64 for bf16 P [rows, d] and x [d]."""
    P_bits, x_bits = _u16(P_bits), _u16(x_bits)
    rows, d = P_bits.shape
    out = np.empty(rows, dtype=np.float64)
    _load().oracle_project(_p(P_bits), rows, d, _p(x_bits), _p(out))
    return out


def pair_scores(A, g, B, U) -> np.ndarray:
    """S [n_prev, K] with S[i, j] = U[j] + sum_k A[i,k] g[k] B[j,k] (fp64 inputs)."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    U = np.ascontiguousarray(U, dtype=np.float64)
    n_prev, e = A.shape
    K = B.shape[0]
    S = np.empty((n_prev, K), dtype=np.float64)
    _load().oracle_pair_scores(n_prev, K, e, _p(A), _p(g), _p(B), _p(U), _p(S))
    return S


def _walk(fn, P):
    P = np.ascontiguousarray(P, dtype=np.float64)
    L, K, _ = P.shape
    ranks = np.empty(L, dtype=np.int32)
    score = np.empty(1, dtype=np.float64)
    sm = np.empty(L, dtype=np.float64)
    fm = np.empty(1, dtype=np.float64)
    fn(L, K, _p(P), _p(ranks), _p(score), _p(sm), _p(fm))
    return ranks, float(score[0]), sm, float(fm[0])


def viterbi(P):
    """Max-sum walk over tables P [L, K, K] (row 0 only at t = 0).
    Returns (ranks [L], score, step margins [L], final margin)."""
    return _walk(_load().oracle_viterbi, P)


def greedy(P):
    """Best-successor walk over P [L, K, K]. Returns (ranks, score, step margins, inf)."""
    return _walk(_load().oracle_greedy, P)


def verify(path, target):
    """(accept length n, emitted [L+1]) for path [L] and target argmax tokens [L+1]."""
    path = np.ascontiguousarray(path, dtype=np.int32)
    target = np.ascontiguousarray(target, dtype=np.int32)
    L = path.shape[0]
    assert target.shape[0] == L + 1
    emitted = np.empty(L + 1, dtype=np.int32)
    n = _load().oracle_verify(L, _p(path), _p(target), _p(emitted))
    return int(n), emitted


def select(W_bits, E_bits, WA_bits, WB_bits, WH_bits, h_bits, anchor: int, K: int,
           walk: int = WALK_VITERBI, nthreads: int = 1) -> dict:
    """The whole selector for one sequence (h_bits [L, d])."""
    W_bits, E_bits = _u16(W_bits), _u16(E_bits)
    WA_bits, WB_bits, WH_bits, h_bits = map(_u16, (WA_bits, WB_bits, WH_bits, h_bits))
    V, d = W_bits.shape
    e = WA_bits.shape[0]
    L = h_bits.shape[0]
    out = dict(ids=np.empty((L, K), np.int32), vals=np.empty((L, K), np.float64),
               topk_margin=np.empty(L, np.float64), P=np.empty((L, K, K), np.float64),
               ranks=np.empty(L, np.int32), tokens=np.empty(L, np.int32),
               score=np.empty(1, np.float64), step_margin=np.empty(L, np.float64),
               final_margin=np.empty(1, np.float64))
    _load().oracle_select(_p(W_bits), _p(E_bits), _p(WA_bits), _p(WB_bits), _p(WH_bits), V, d, e,
                          L, K, walk, _p(h_bits), int(anchor), _p(out["ids"]), _p(out["vals"]),
                          _p(out["topk_margin"]), _p(out["P"]), _p(out["ranks"]), _p(out["tokens"]),
                          _p(out["score"]), _p(out["step_margin"]), _p(out["final_margin"]),
                          int(nthreads))
    out["score"] = float(out["score"][0])
    out["final_margin"] = float(out["final_margin"][0])
    return out


def select_given(W_bits, E_bits, WA_bits, WB_bits, WH_bits, h_bits, anchor: int, ids,
                 walk: int = WALK_VITERBI) -> dict:
    """The selector for one sequence with candidate ids [L, K] given."""
    W_bits, E_bits = _u16(W_bits), _u16(E_bits)
    WA_bits, WB_bits, WH_bits, h_bits = map(_u16, (WA_bits, WB_bits, WH_bits, h_bits))
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    V, d = W_bits.shape
    e = WA_bits.shape[0]
    L, K = ids.shape
    out = dict(ids=ids, vals=np.empty((L, K), np.float64), P=np.empty((L, K, K), np.float64),
               ranks=np.empty(L, np.int32), tokens=np.empty(L, np.int32),
               score=np.empty(1, np.float64), step_margin=np.empty(L, np.float64),
               final_margin=np.empty(1, np.float64))
    _load().oracle_select_given(_p(W_bits), _p(E_bits), _p(WA_bits), _p(WB_bits), _p(WH_bits), V, d,
                                e, L, K, walk, _p(h_bits), int(anchor), _p(ids), _p(out["vals"]),
                                _p(out["P"]), _p(out["ranks"]), _p(out["tokens"]), _p(out["score"]),
                                _p(out["step_margin"]), _p(out["final_margin"]))
    out["score"] = float(out["score"][0])
    out["final_margin"] = float(out["final_margin"][0])
    return out


def sample_walk(P, T: float, u):
    """Sampling walk over tables P [L, K, K] with temperature T and uniforms u [L].
    Returns (ranks [L], q [L, K] distributions drawn from, margins [L])."""
    P = np.ascontiguousarray(P, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    L, K, _ = P.shape
    ranks = np.empty(L, np.int32)
    q = np.empty((L, K), np.float64)
    mg = np.empty(L, np.float64)
    _load().oracle_sample_walk(L, K, _p(P), float(T), _p(u), _p(ranks), _p(q), _p(mg))
    return ranks, q, mg


def verify_rejection(path, ids, q, p, u_acc, u_res: float):
    """Rejection-sampling verification. path [L], ids [L, K], q [L, K] draft
    probabilities, p [L+1, V] target probabilities, u_acc [L], u_res.
    Returns (n, emitted [L+1], acceptance margins [L], draw margin)."""
    path = np.ascontiguousarray(path, dtype=np.int32)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    q = np.ascontiguousarray(q, dtype=np.float64)
    p = np.ascontiguousarray(p, dtype=np.float64)
    u_acc = np.ascontiguousarray(u_acc, dtype=np.float64)
    L, K = ids.shape
    V = p.shape[1]
    assert p.shape[0] == L + 1
    emitted = np.empty(L + 1, np.int32)
    am = np.empty(L, np.float64)
    rm = np.empty(1, np.float64)
    n = _load().oracle_verify_rejection(L, K, V, _p(path), _p(ids), _p(q), _p(p), _p(u_acc), float(u_res),
                                        _p(emitted), _p(am), _p(rm))
    return int(n), emitted, am, float(rm[0])


def conv2(X_bits, base_bits, Wc_bits, nthreads: int = 1) -> np.ndarray:
    """Two-tap dynamic depthwise convolution of blocks X [B, S, d] (bf16 bits)
    with base kernels [2, d] and correction weights Wc [2 d/16, d] (bf16 bits):
    Y [B, S, d] in fp64."""
    X_bits, base_bits, Wc_bits = _u16(X_bits), _u16(base_bits), _u16(Wc_bits)
    B, S, d = X_bits.shape
    assert d % 16 == 0 and base_bits.shape == (2, d) and Wc_bits.shape == (2 * (d // 16), d)
    Y = np.empty((B, S, d), dtype=np.float64)
    _load().oracle_conv2(B, S, d, _p(X_bits), _p(base_bits), _p(Wc_bits), _p(Y), int(nthreads))
    return Y
