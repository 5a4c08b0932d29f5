"""The N > 1 path of indexer context parallelism on CPU, as two gloo ranks.

"[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (ROCm/ATOM #2744),
review thread on the unused page-16 tables: every rank scores its share of a
request's index keys, the ranks exchange candidate keys and merge them into the
top-k. Each rank here holds a contiguous share of the blocks of every row (its
block scores drawn, with ties, so the lower-id rule is exercised); it encodes its
oracle candidates in the library's documented key format, the ranks exchange
them through cp.exchange_candidates (an all-gather), and the decoded union,
merged by the oracle, must be the top-k of the whole row on every rank.
"""

import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
R, TOPK, NB = 6, 16, 300


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ordered(x: np.float32) -> int:
    """The order-preserving map of an fp32's bits (-0 as +0)."""
    if x == 0:
        x = np.float32(0.0)
    b = int(np.array([x], dtype=np.float32).view(np.uint32)[0])
    return (b | 0x80000000) if b < 0x80000000 else (~b & 0xFFFFFFFF)


def encode(rec) -> int:
    """An oracle rank record (class, value, id) as the library's uint64 key, read as int64."""
    cls, val, i = rec
    if cls == 2:
        k = (0xFFFFFFFF << 32) | (0xFFFFFFFF - i)
    elif cls == 1:
        k = (0xFFFFFFFE << 32) | i
    else:
        k = (_ordered(np.float32(val)) << 32) | (0xFFFFFFFF - i)
    return k - (1 << 64) if k >= 1 << 63 else k


def decode(k: int, scores: np.ndarray):
    """The record of a key (0 = an empty slot -> None)."""
    if k == 0:
        return None
    u = k & 0xFFFFFFFFFFFFFFFF
    hi, lo = u >> 32, u & 0xFFFFFFFF
    if hi == 0xFFFFFFFE:
        return (1, float(lo), lo)
    i = 0xFFFFFFFF - lo
    if hi == 0xFFFFFFFF:
        return (2, -float(i), i)
    return (0, float(scores[i]), i)


def _scores(seed: int) -> np.ndarray:
    """fp32 block scores [R, NB] with many exact ties (a coarse grid)."""
    rng = np.random.default_rng(seed)
    return (rng.integers(-40, 40, size=(R, NB)) / 8.0).astype(np.float32)


def _rank_main(rank, world, port, cuts, forced, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from nvfp4_block_sparse_m3s_gb300 import cp
    from oracle import m3s_oracle as O
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        init, local = forced
        sc = _scores(5)
        lo, hi = cuts[rank], cuts[rank + 1]
        mine = np.zeros((R, TOPK), dtype=np.int64)
        for r in range(R):
            recs = O.slice_candidates(sc[r].astype(np.float64), lo, hi, TOPK, init, local)
            mine[r, : len(recs)] = [encode(x) for x in recs]
        allk = cp.exchange_candidates(torch.from_numpy(mine)).numpy()
        assert allk.shape == (world, R, TOPK)
        assert np.array_equal(allk[rank], mine)
        merged = np.zeros((R, TOPK), dtype=np.int32)
        for r in range(R):
            lists = [[rec for rec in (decode(int(k), sc[r]) for k in allk[s, r]) if rec is not None]
                     for s in range(world)]
            merged[r] = O.merge_candidates(lists, TOPK)
        out[rank] = merged
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(cuts, forced):
    world = len(cuts) - 1
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, cuts, forced, out), nprocs=world, join=True)
        return dict(out)


def _expected(forced):
    sys.path.insert(0, ROOT)
    from oracle import m3s_oracle as O
    sc = _scores(5)
    return np.stack([O.topk_ids(sc[r].astype(np.float64), TOPK, *forced) for r in range(R)])


def test_two_gloo_ranks_exchange_and_merge_to_the_whole_rows_top_k():
    res = _run([0, 37, NB], (0, 0))   # an uneven split
    want = _expected((0, 0))
    for rank in range(2):
        np.testing.assert_array_equal(res[rank], want)


def test_two_gloo_ranks_with_forced_blocks():
    res = _run([0, 298, NB], (2, 3))   # the local blocks all on rank 1, init on rank 0
    want = _expected((2, 3))
    for rank in range(2):
        np.testing.assert_array_equal(res[rank], want)


def test_key_encoding_orders_like_the_oracle():
    """The documented key order is the oracle's rank order: sorting records by
    key gives the oracle's best-first order (ties to the lower id, forced first)."""
    sys.path.insert(0, ROOT)
    from oracle import m3s_oracle as O
    sc = _scores(9)[0].astype(np.float64)
    sc[[3, 4, 5]] = [-0.0, 0.0, -1e-30]
    recs = O.rank_records(sc, range(NB), NB, 2, 3)
    by_key = sorted(recs, key=lambda x: encode(x) & 0xFFFFFFFFFFFFFFFF, reverse=True)
    ref = O.slice_candidates(sc, 0, NB, NB, 2, 3)
    assert [x[2] for x in by_key] == [x[2] for x in ref]
