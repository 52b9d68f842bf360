"""DFlash 2 path selector on one GB300 GPU: Python binding of libdflash_select.

The functions below have the names of the C entry points declared in
``include/dflash_select.h`` and ``include/dflash_conv2.h`` and only marshal
arguments: every step of the
selector runs in the library's CUDA kernels. PyTorch supplies device memory
and streams. If the library has not been built the calls raise; there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdflash_select.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "dflash_select.h")

DFLASH_OK = 0
DFLASH_ERR_INVALID_ARG = 1
DFLASH_ERR_UNSUPPORTED = 2
DFLASH_ERR_CUDA = 3
DFLASH_ERR_DEVICE_CHECK = 4
DFLASH_ERR_TIMEOUT = 5
STATUS_NAMES = {0: "DFLASH_OK", 1: "DFLASH_ERR_INVALID_ARG", 2: "DFLASH_ERR_UNSUPPORTED", 3: "DFLASH_ERR_CUDA",
                4: "DFLASH_ERR_DEVICE_CHECK", 5: "DFLASH_ERR_TIMEOUT"}

DFLASH_WALK_VITERBI = 0
DFLASH_WALK_GREEDY = 1
DFLASH_WALK_SAMPLE = 2

KERNEL_NAMES = ("lmhead_topk", "topk_merge", "projection", "pair_walk", "select_tail", "dedup")


class DflashError(RuntimeError):
    def __init__(self, status: int, func: str, msg: str):
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class dflash_select_config(ctypes.Structure):
    _fields_ = [("V", ctypes.c_int64), ("d", ctypes.c_int32), ("L", ctypes.c_int32), ("K", ctypes.c_int32),
                ("e", ctypes.c_int32), ("max_batch", ctypes.c_int32), ("walk", ctypes.c_int32),
                ("tie_eps", ctypes.c_float), ("temperature", ctypes.c_float), ("tables", ctypes.c_int32),
                ("dedup", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -m "
                                   "speculative_decoding_draft_tcgen05_gb300.build)")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.dflash_select_init.argtypes = [ctypes.POINTER(dflash_select_config), P, P, P, P, P, P,
                                             ctypes.POINTER(P)]
            L.dflash_select_run.argtypes = [P, P, P, i32, P, P, P, P, P, P, P]
            L.dflash_verify_prefix.argtypes = [P, P, i32, i32, P, P, P]
            L.dflash_select_run_sampled.argtypes = [P, P, P, i32, P, P, P, P, P, P, P, P, P]
            L.dflash_verify_rejection.argtypes = [P, P, P, P, P, P, i32, i32, i32, i64, P, P, P]
            L.dflash_select_step_host.argtypes = [P, P, P, P, i32, P, P, P, P]
            L.dflash_select_sync_status.argtypes = [P, P]
            L.dflash_select_profile.argtypes = [P, i32]
            L.dflash_select_profile_read.argtypes = [P, P, P, i32, P]
            L.dflash_select_launches_per_run.argtypes = [P, i32]
            L.dflash_select_launches_per_run.restype = i32
            L.dflash_select_destroy.argtypes = [P]
            L.dflash_select_init_shard.argtypes = [ctypes.POINTER(dflash_select_config), P, i64, i64, P, P, P, P, P,
                                                   ctypes.POINTER(P)]
            L.dflash_select_topk_shard.argtypes = [P, P, i32, P, P]
            L.dflash_select_run_gathered.argtypes = [P, P, i32, P, i32, P, P, P, P, P, P, P]
            L.dflash_select_run_verify.argtypes = [P, P, P, i32, P, P, P, P, P, P, P, P, P, P]
            L.dflash_lmhead_topk_noalloc.argtypes = [P, i64, i32, P, i32, i32, P, P, P, P]
            L.dflash_selftest_wait_timeout.argtypes = [P, P]
            L.dflash_conv2_init.argtypes = [P, P, i32, ctypes.POINTER(P)]
            L.dflash_conv2_run.argtypes = [P, P, i32, i32, P, P]
            L.dflash_conv2_sync_status.argtypes = [P, P]
            L.dflash_conv2_destroy.argtypes = [P]
            L.dflash_last_error.restype = ctypes.c_char_p
            for f in ("dflash_select_init", "dflash_select_run", "dflash_verify_prefix", "dflash_select_step_host",
                      "dflash_select_sync_status", "dflash_select_profile", "dflash_select_profile_read",
                      "dflash_select_destroy", "dflash_lmhead_topk_noalloc", "dflash_select_run_sampled",
                      "dflash_verify_rejection", "dflash_conv2_init", "dflash_conv2_run", "dflash_conv2_sync_status",
                      "dflash_conv2_destroy", "dflash_selftest_wait_timeout", "dflash_select_init_shard",
                      "dflash_select_topk_shard", "dflash_select_run_gathered", "dflash_select_run_verify"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def dflash_last_error() -> str:
    return lib().dflash_last_error().decode(errors="replace")


def _check(status: int, func: str):
    if status != DFLASH_OK:
        raise DflashError(status, func, dflash_last_error())


def _ptr(t, dtype=None, name="tensor", device=True):
    """Device (or host) address of a contiguous tensor; None stays NULL."""
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not device and t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def dflash_select_init(W, E, W_A, W_B, W_H, *, L: int, K: int, max_batch: int, walk: int = DFLASH_WALK_VITERBI,
                       tie_eps: float = 1e-3, temperature: float = 1.0, tables: bool = False, dedup: bool = False,
                       stream=None):
    """Creates a selector handle over device bf16 weights W [V, d], E [V, d], W_A/W_B/W_H [256, d]
    (tables=True: precompute A|B for every token at init and gather table rows in every run;
    dedup=True: project each distinct token of a batch once on the larger-batch path)."""
    import torch
    V, d = W.shape
    cfg = dflash_select_config(V=V, d=d, L=L, K=K, e=W_A.shape[0], max_batch=max_batch, walk=walk,
                               tie_eps=tie_eps, temperature=temperature, tables=1 if tables else 0,
                               dedup=1 if dedup else 0)
    h = ctypes.c_void_p()
    _check(lib().dflash_select_init(ctypes.byref(cfg), _ptr(W, torch.bfloat16, "W"), _ptr(E, torch.bfloat16, "E"),
                                    _ptr(W_A, torch.bfloat16, "W_A"), _ptr(W_B, torch.bfloat16, "W_B"),
                                    _ptr(W_H, torch.bfloat16, "W_H"), _stream(stream), ctypes.byref(h)),
           "dflash_select_init")
    return h


def dflash_select_init_shard(W_shard, v0, v1, E, W_A, W_B, W_H, *, L: int, K: int, max_batch: int,
                             walk: int = DFLASH_WALK_VITERBI, tie_eps: float = 1e-3, tables: bool = False,
                             stream=None):
    """A handle that streams the lm_head rows [v0, v1) only: W_shard [v1 - v0, d] holds those rows, E [V, d] the
    whole token table (V = E's rows)."""
    import torch
    V, d = E.shape
    if tuple(W_shard.shape) != (v1 - v0, d):
        raise ValueError(f"W_shard must be [{v1 - v0}, {d}], got {tuple(W_shard.shape)}")
    cfg = dflash_select_config(V=V, d=d, L=L, K=K, e=W_A.shape[0], max_batch=max_batch, walk=walk,
                               tie_eps=tie_eps, temperature=1.0, tables=1 if tables else 0)
    h = ctypes.c_void_p()
    _check(lib().dflash_select_init_shard(ctypes.byref(cfg), _ptr(W_shard, torch.bfloat16, "W_shard"), v0, v1,
                                          _ptr(E, torch.bfloat16, "E"), _ptr(W_A, torch.bfloat16, "W_A"),
                                          _ptr(W_B, torch.bfloat16, "W_B"), _ptr(W_H, torch.bfloat16, "W_H"),
                                          _stream(stream), ctypes.byref(h)), "dflash_select_init_shard")
    return h


def dflash_select_topk_shard(handle, hidden, shard_keys, stream=None):
    """The handle's vocabulary shard of the lm_head pass: hidden [B, L, d] bf16 into shard_keys [B, L, K] (int64
    tensor holding the uint64 keys)."""
    import torch
    B = hidden.shape[0]
    _check(lib().dflash_select_topk_shard(handle, _ptr(hidden, torch.bfloat16, "hidden"), B,
                                          _ptr(shard_keys, torch.int64, "shard_keys"), _stream(stream)),
           "dflash_select_topk_shard")


def dflash_select_run_gathered(handle, anchor, all_keys, *, path, topk_ids=None, topk_vals=None, pair_scores=None,
                               path_score=None, tie_flags=None, stream=None):
    """The selector after the exchange: all_keys [G, B, L, K] (int64 tensor of uint64 keys) from every shard."""
    import torch
    B = anchor.shape[0]
    G = all_keys.shape[0]
    _check(lib().dflash_select_run_gathered(handle, _ptr(anchor, torch.int32, "anchor"), B,
                                            _ptr(all_keys, torch.int64, "all_keys"), G,
                                            _ptr(topk_ids, torch.int32, "topk_ids"),
                                            _ptr(topk_vals, torch.float32, "topk_vals"),
                                            _ptr(pair_scores, torch.float32, "pair_scores"),
                                            _ptr(path, torch.int32, "path"),
                                            _ptr(path_score, torch.float32, "path_score"),
                                            _ptr(tie_flags, torch.uint8, "tie_flags"), _stream(stream)),
           "dflash_select_run_gathered")


def dflash_select_run(handle, hidden, anchor, *, path, topk_ids=None, topk_vals=None, pair_scores=None,
                      path_score=None, tie_flags=None, stream=None):
    """Runs the selector for hidden [B, L, d] bf16 and anchor [B] int32 into the given device outputs."""
    import torch
    B = anchor.shape[0]
    _check(lib().dflash_select_run(handle, _ptr(hidden, torch.bfloat16, "hidden"), _ptr(anchor, torch.int32, "anchor"),
                                   B, _ptr(topk_ids, torch.int32, "topk_ids"),
                                   _ptr(topk_vals, torch.float32, "topk_vals"),
                                   _ptr(pair_scores, torch.float32, "pair_scores"), _ptr(path, torch.int32, "path"),
                                   _ptr(path_score, torch.float32, "path_score"),
                                   _ptr(tie_flags, torch.uint8, "tie_flags"), _stream(stream)), "dflash_select_run")


def dflash_select_run_verify(handle, hidden, anchor, target, *, path, accept_len, emitted=None, topk_ids=None,
                             topk_vals=None, pair_scores=None, path_score=None, tie_flags=None, stream=None):
    """dflash_select_run and dflash_verify_prefix in one call: target [B, L+1] int32 in, path [B, L],
    accept_len [B] and emitted [B, L+1] out (the walking kernel checks the path)."""
    import torch
    B = anchor.shape[0]
    _check(lib().dflash_select_run_verify(handle, _ptr(hidden, torch.bfloat16, "hidden"),
                                          _ptr(anchor, torch.int32, "anchor"), B, _ptr(target, torch.int32, "target"),
                                          _ptr(path, torch.int32, "path"), _ptr(accept_len, torch.int32, "accept_len"),
                                          _ptr(emitted, torch.int32, "emitted"),
                                          _ptr(topk_ids, torch.int32, "topk_ids"),
                                          _ptr(topk_vals, torch.float32, "topk_vals"),
                                          _ptr(pair_scores, torch.float32, "pair_scores"),
                                          _ptr(path_score, torch.float32, "path_score"),
                                          _ptr(tie_flags, torch.uint8, "tie_flags"), _stream(stream)),
           "dflash_select_run_verify")


def dflash_select_run_sampled(handle, hidden, anchor, u_walk, *, path, draft_probs, topk_ids=None, topk_vals=None,
                              pair_scores=None, path_score=None, tie_flags=None, stream=None):
    """The selector with the sampling walk: u_walk [B, L] fp32 uniforms in, draft_probs [B, L, K] out."""
    import torch
    B = anchor.shape[0]
    _check(lib().dflash_select_run_sampled(handle, _ptr(hidden, torch.bfloat16, "hidden"),
                                           _ptr(anchor, torch.int32, "anchor"), B, _ptr(u_walk, torch.float32, "u_walk"),
                                           _ptr(topk_ids, torch.int32, "topk_ids"),
                                           _ptr(topk_vals, torch.float32, "topk_vals"),
                                           _ptr(pair_scores, torch.float32, "pair_scores"),
                                           _ptr(path, torch.int32, "path"), _ptr(draft_probs, torch.float32, "draft_probs"),
                                           _ptr(path_score, torch.float32, "path_score"),
                                           _ptr(tie_flags, torch.uint8, "tie_flags"), _stream(stream)),
           "dflash_select_run_sampled")


def dflash_verify_rejection(path, topk_ids, draft_probs, target_probs, u_acc, u_res, accept_len, emitted, stream=None):
    """Rejection-sampling verification: path [B, L], topk_ids / draft_probs [B, L, K], target_probs [B, L+1, V],
    u_acc [B, L], u_res [B] (device) into accept_len [B] and emitted [B, L+1]."""
    import torch
    B, L = path.shape
    K = topk_ids.shape[2]
    V = target_probs.shape[2]
    _check(lib().dflash_verify_rejection(_ptr(path, torch.int32, "path"), _ptr(topk_ids, torch.int32, "topk_ids"),
                                         _ptr(draft_probs, torch.float32, "draft_probs"),
                                         _ptr(target_probs, torch.float32, "target_probs"),
                                         _ptr(u_acc, torch.float32, "u_acc"), _ptr(u_res, torch.float32, "u_res"), B, L,
                                         K, V, _ptr(accept_len, torch.int32, "accept_len"),
                                         _ptr(emitted, torch.int32, "emitted"), _stream(stream)),
           "dflash_verify_rejection")


def dflash_verify_prefix(path, target, accept_len, emitted=None, stream=None):
    """Greedy accept lengths of path [B, L] against target [B, L+1] (int32, device)."""
    import torch
    B, L = path.shape
    _check(lib().dflash_verify_prefix(_ptr(path, torch.int32, "path"), _ptr(target, torch.int32, "target"), B, L,
                                      _ptr(accept_len, torch.int32, "accept_len"),
                                      _ptr(emitted, torch.int32, "emitted"), _stream(stream)), "dflash_verify_prefix")


def dflash_select_step_host(handle, hidden_host, anchor_host, target_host, path_host, accept_host, emitted_host,
                            stream=None):
    """Whole step from host buffers (pinned for asynchronous copies); returns when results are on the host."""
    import torch
    B = anchor_host.shape[0]
    _check(lib().dflash_select_step_host(handle, _ptr(hidden_host, torch.bfloat16, "hidden_host", device=False),
                                         _ptr(anchor_host, torch.int32, "anchor_host", device=False),
                                         _ptr(target_host, torch.int32, "target_host", device=False), B,
                                         _ptr(path_host, torch.int32, "path_host", device=False),
                                         _ptr(accept_host, torch.int32, "accept_host", device=False),
                                         _ptr(emitted_host, torch.int32, "emitted_host", device=False),
                                         _stream(stream)), "dflash_select_step_host")


def bind_step_host(handle, hidden_host, anchor_host, target_host, path_host, accept_host, emitted_host,
                   stream=None):
    """Marshals the arguments of dflash_select_step_host once and returns a
    zero-argument callable that makes the same call again; for tight loops
    over fixed host buffers."""
    import torch
    B = anchor_host.shape[0]
    args = (handle, _ptr(hidden_host, torch.bfloat16, "hidden_host", device=False),
            _ptr(anchor_host, torch.int32, "anchor_host", device=False),
            _ptr(target_host, torch.int32, "target_host", device=False), B,
            _ptr(path_host, torch.int32, "path_host", device=False),
            _ptr(accept_host, torch.int32, "accept_host", device=False),
            _ptr(emitted_host, torch.int32, "emitted_host", device=False), _stream(stream))
    fn = lib().dflash_select_step_host

    def step():
        st = fn(*args)
        if st:
            _check(st, "dflash_select_step_host")
    return step


def dflash_select_sync_status(handle, stream=None) -> int:
    """Waits for the stream; returns the latched device status (raises on error)."""
    st = lib().dflash_select_sync_status(handle, _stream(stream))
    _check(st, "dflash_select_sync_status")
    return st


def dflash_select_profile(handle, enable: bool):
    _check(lib().dflash_select_profile(handle, int(bool(enable))), "dflash_select_profile")


def dflash_select_profile_read(handle):
    """{kernel name: (total ms, launches)} over the recorded runs."""
    n = len(KERNEL_NAMES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    nk = ctypes.c_int32()
    _check(lib().dflash_select_profile_read(handle, ms, cnt, n, ctypes.byref(nk)), "dflash_select_profile_read")
    return {KERNEL_NAMES[i]: (ms[i], cnt[i]) for i in range(nk.value)}


def dflash_select_launches_per_run(handle, B: int) -> int:
    return int(lib().dflash_select_launches_per_run(handle, B))


def bind_step(handle, hidden, anchor, path, target=None, accept_len=None, emitted=None, stream=None, **outs):
    """Marshals the arguments of dflash_select_run (with target given,
    dflash_select_run_verify: the run and the accept check in one call) once and
    returns a zero-argument callable that makes the same call again; for tight
    loops over fixed buffers."""
    import torch
    L_ = lib()
    B = anchor.shape[0]
    run_args = (handle, _ptr(hidden, torch.bfloat16, "hidden"), _ptr(anchor, torch.int32, "anchor"), B,
                _ptr(outs.get("topk_ids"), torch.int32, "topk_ids"), _ptr(outs.get("topk_vals"), torch.float32,
                                                                          "topk_vals"),
                _ptr(outs.get("pair_scores"), torch.float32, "pair_scores"), _ptr(path, torch.int32, "path"),
                _ptr(outs.get("path_score"), torch.float32, "path_score"),
                _ptr(outs.get("tie_flags"), torch.uint8, "tie_flags"), _stream(stream))
    run = L_.dflash_select_run
    if target is None:
        def step():
            st = run(*run_args)
            if st:
                _check(st, "dflash_select_run")
        return step
    # with targets: the fused run + accept check (one launch fewer than the two calls)
    rv_args = (handle, _ptr(hidden, torch.bfloat16, "hidden"), _ptr(anchor, torch.int32, "anchor"), B,
               _ptr(target, torch.int32, "target"), _ptr(path, torch.int32, "path"),
               _ptr(accept_len, torch.int32, "accept_len"), _ptr(emitted, torch.int32, "emitted"),
               _ptr(outs.get("topk_ids"), torch.int32, "topk_ids"),
               _ptr(outs.get("topk_vals"), torch.float32, "topk_vals"),
               _ptr(outs.get("pair_scores"), torch.float32, "pair_scores"),
               _ptr(outs.get("path_score"), torch.float32, "path_score"),
               _ptr(outs.get("tie_flags"), torch.uint8, "tie_flags"), _stream(stream))
    rv = L_.dflash_select_run_verify

    def step():
        st = rv(*rv_args)
        if st:
            _check(st, "dflash_select_run_verify")
    return step


def dflash_lmhead_topk_noalloc(W, hidden, K, topk_ids, topk_vals=None, device_status=None, stream=None):
    """lm_head + top-K of hidden [N, d] against W [V, d] (bf16, device) into
    topk_ids [N, K] (and topk_vals) without any device allocation: the library
    keeps a fixed scratch array per GPU. Calls on one GPU must not overlap."""
    import torch
    V, d = W.shape
    N = hidden.shape[0]
    if hidden.dim() != 2 or hidden.shape[1] != d:
        raise ValueError("hidden must be [N, d]")
    _check(lib().dflash_lmhead_topk_noalloc(_ptr(W, torch.bfloat16, "W"), V, d, _ptr(hidden, torch.bfloat16, "hidden"),
                                            N, K, _ptr(topk_ids, torch.int32, "topk_ids"),
                                            _ptr(topk_vals, torch.float32, "topk_vals"),
                                            _ptr(device_status, torch.int32, "device_status"), _stream(stream)),
           "dflash_lmhead_topk_noalloc")


def bind_sampled_step(handle, hidden, anchor, u_walk, topk_ids, path, draft_probs, target_probs, u_acc, u_res,
                      accept_len, emitted, stream=None):
    """Marshals one dflash_select_run_sampled + dflash_verify_rejection pair
    once; returns a zero-argument callable that makes both calls again."""
    import torch
    L_ = lib()
    B, L = path.shape
    K = topk_ids.shape[2]
    V = target_probs.shape[2]
    st = _stream(stream)
    run_args = (handle, _ptr(hidden, torch.bfloat16, "hidden"), _ptr(anchor, torch.int32, "anchor"), B,
                _ptr(u_walk, torch.float32, "u_walk"), _ptr(topk_ids, torch.int32, "topk_ids"), None, None,
                _ptr(path, torch.int32, "path"), _ptr(draft_probs, torch.float32, "draft_probs"), None, None, st)
    ver_args = (_ptr(path, torch.int32, "path"), _ptr(topk_ids, torch.int32, "topk_ids"),
                _ptr(draft_probs, torch.float32, "draft_probs"), _ptr(target_probs, torch.float32, "target_probs"),
                _ptr(u_acc, torch.float32, "u_acc"), _ptr(u_res, torch.float32, "u_res"), B, L, K, V,
                _ptr(accept_len, torch.int32, "accept_len"), _ptr(emitted, torch.int32, "emitted"), st)
    run, ver = L_.dflash_select_run_sampled, L_.dflash_verify_rejection

    def step():
        r = run(*run_args)
        if r:
            _check(r, "dflash_select_run_sampled")
        r = ver(*ver_args)
        if r:
            _check(r, "dflash_verify_rejection")
    return step


def dflash_select_destroy(handle):
    _check(lib().dflash_select_destroy(handle), "dflash_select_destroy")


class Selector:
    """Owns a handle and the output tensors of one batch size (convenience only)."""

    def __init__(self, W, E, W_A, W_B, W_H, *, L, K, max_batch, walk=DFLASH_WALK_VITERBI, tie_eps=1e-3,
                 temperature=1.0, tables=False, dedup=False):
        import torch
        self.L, self.K, self.max_batch = L, K, max_batch
        self.device = W.device
        self.h = dflash_select_init(W, E, W_A, W_B, W_H, L=L, K=K, max_batch=max_batch, walk=walk, tie_eps=tie_eps,
                                    temperature=temperature, tables=tables, dedup=dedup)
        self._weights = (W, E, W_A, W_B, W_H)  # the handle borrows them: keep them alive with it
        self._torch = torch

    def outputs(self, B, full=True):
        t = self._torch
        dev = self.device
        out = dict(path=t.empty(B, self.L, dtype=t.int32, device=dev))
        if full:
            out.update(topk_ids=t.empty(B, self.L, self.K, dtype=t.int32, device=dev),
                       topk_vals=t.empty(B, self.L, self.K, dtype=t.float32, device=dev),
                       pair_scores=t.empty(B, self.L, self.K, self.K, dtype=t.float32, device=dev),
                       path_score=t.empty(B, dtype=t.float32, device=dev),
                       tie_flags=t.empty(B, self.L, dtype=t.uint8, device=dev))
        return out

    def run(self, hidden, anchor, out=None, stream=None):
        if out is None:
            out = self.outputs(anchor.shape[0])
        dflash_select_run(self.h, hidden, anchor, stream=stream, **out)
        return out

    def close(self):
        if self.h is not None:
            dflash_select_destroy(self.h)
            self.h = None
            self._weights = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def dflash_conv2_init(base, Wc):
    """Handle of one two-tap dynamic convolution: base [2, d] and Wc [d/8, d] bf16 device weights (borrowed)."""
    import torch
    d = base.shape[1]
    if tuple(base.shape) != (2, d) or tuple(Wc.shape) != (d // 8, d):
        raise ValueError(f"base must be [2, d] and Wc [d/8, d], got {tuple(base.shape)} and {tuple(Wc.shape)}")
    h = ctypes.c_void_p()
    _check(lib().dflash_conv2_init(_ptr(base, torch.bfloat16, "base"), _ptr(Wc, torch.bfloat16, "Wc"), d,
                                   ctypes.byref(h)), "dflash_conv2_init")
    return h


def dflash_conv2_run(handle, X, Y, stream=None):
    """Y [B, S, d] = the convolution of the blocks X [B, S, d] (bf16, device)."""
    import torch
    B, S, d = X.shape
    if tuple(Y.shape) != (B, S, d):
        raise ValueError("Y must have X's shape")
    _check(lib().dflash_conv2_run(handle, _ptr(X, torch.bfloat16, "X"), B, S, _ptr(Y, torch.bfloat16, "Y"),
                                  _stream(stream)), "dflash_conv2_run")


def dflash_conv2_sync_status(handle, stream=None):
    _check(lib().dflash_conv2_sync_status(handle, _stream(stream)), "dflash_conv2_sync_status")


def dflash_conv2_destroy(handle):
    _check(lib().dflash_conv2_destroy(handle), "dflash_conv2_destroy")


class Conv2:
    """Owns a convolution handle (convenience only)."""

    def __init__(self, base, Wc):
        self.h = dflash_conv2_init(base, Wc)
        self._weights = (base, Wc)  # the handle borrows them: keep them alive with it

    def __call__(self, X, Y=None, stream=None):
        import torch
        if Y is None:
            Y = torch.empty_like(X)
        dflash_conv2_run(self.h, X, Y, stream=stream)
        return Y

    def close(self):
        if self.h is not None:
            dflash_conv2_destroy(self.h)
            self.h = None
            self._weights = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def dflash_selftest_wait_timeout(device_status, stream=None):
    """Launches a kernel whose bounded wait runs out (about 1 s); bit 2 of device_status [1] int32 gets set."""
    import torch
    _check(lib().dflash_selftest_wait_timeout(_ptr(device_status, torch.int32, "device_status"), _stream(stream)),
           "dflash_selftest_wait_timeout")
