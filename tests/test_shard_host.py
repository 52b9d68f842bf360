"""Host side of the vocabulary-sharded selector, without a GPU: the row
partition, and the exchange of the ranks' top-K lists between two gloo ranks
on CPU. Each rank takes the oracle's logits of its own rows, keeps its K best
as keys in the library's documented format (fp32 logit mapped to an
order-preserving unsigned word, then ~id), all-gathers the lists, and merges
them by key; the merged candidates must be the oracle's top-K over the whole
vocabulary."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl
from speculative_decoding_draft_tcgen05_gb300.shard import all_gather_keys, shard_range


@pytest.mark.parametrize("V,G", [(4096, 2), (4096, 3), (151936, 8), (129, 2), (100, 1), (1000, 7)])
def test_shard_ranges_partition_the_vocabulary(V, G):
    ranges = [shard_range(V, G, r) for r in range(G)]
    assert ranges[0][0] == 0 and ranges[-1][1] == V
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0  # contiguous, disjoint
    for v0, v1 in ranges:
        assert v0 % 128 == 0 and v1 >= v0
    sizes = [(v1 - v0 + 127) // 128 for v0, v1 in ranges]
    assert max(sizes) - min(sizes) <= 1


def encode_keys(vals32: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """The documented key of (fp32 logit, token id) as int64 bit patterns."""
    u = vals32.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = np.where(vals32 == 0, np.uint64(0), u)  # -0 taken as +0
    neg = (u & np.uint64(0x80000000)) != 0
    hi = np.where(neg, ~u & np.uint64(0xFFFFFFFF), u | np.uint64(0x80000000))
    lo = ~ids.astype(np.uint64) & np.uint64(0xFFFFFFFF)
    return ((hi << np.uint64(32)) | lo).view(np.int64)


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = wl.make_inputs(wl.WORKLOADS["tiny"])
    w = inp.wl
    v0, v1 = shard_range(w.V, world, rank)
    H = wl.bf16_bits(inp.hidden.reshape(-1, w.d).contiguous())
    U = oracle.logits(np.ascontiguousarray(wl.bf16_bits(inp.W)[v0:v1]), H)  # [N, rows]
    K = w.K
    local = np.zeros((U.shape[0], K), np.int64)
    for n in range(U.shape[0]):
        ids, vals, _ = oracle.topk(U[n], K)
        local[n] = encode_keys(vals.astype(np.float32), ids + v0)
    gathered = all_gather_keys(torch.from_numpy(local.reshape(w.B, w.L, K)))
    q.put((rank, gathered.numpy()))
    dist.destroy_process_group()


def test_exchange_and_merge_give_the_global_top_k():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert np.array_equal(out[0], out[1])  # every rank holds the same [G, B, L, K], in rank order
    gathered = out[0]
    inp = wl.make_inputs(wl.WORKLOADS["tiny"])
    w = inp.wl
    assert gathered.shape == (world, w.B, w.L, w.K)
    for g in range(world):
        v0, v1 = shard_range(w.V, world, g)
        ids = (~gathered[g].view(np.uint64) & np.uint64(0xFFFFFFFF)).astype(np.int64)
        assert ((ids >= v0) & (ids < v1)).all()
    U = oracle.logits(wl.bf16_bits(inp.W), wl.bf16_bits(inp.hidden.reshape(-1, w.d).contiguous()))
    union = gathered.view(np.uint64).transpose(1, 2, 0, 3).reshape(w.B * w.L, world * w.K)
    for n in range(w.B * w.L):
        best = np.sort(union[n])[::-1][:w.K]
        ids = (~best & np.uint64(0xFFFFFFFF)).astype(np.int64)
        o_ids, _, margin = oracle.topk(U[n], w.K)
        if margin >= 1e-3:
            assert ids.tolist() == o_ids.tolist(), f"position {n}"
