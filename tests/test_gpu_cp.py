"""GPU parity of indexer context parallelism.

"[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (ROCm/ATOM #2744),
review thread on the unused page-16 tables: one request's index keys are split
over ranks, each rank scores its share, and the ranks' candidate keys are merged
into the top-k. Here the blocks of a skewed decode batch (one long request,
several shorter ones) are cut into contiguous slices at uneven points, each
slice scored on its own shifted block table (m3s_index_score_candidates), and
the slices' candidates merged (m3s_merge_candidates). Because each block of a
row's top-k is among its own slice's top-k, the merge must give exactly the ids
of the unsplit call; the slices' own candidates must be their oracle top-k,
in the documented key format.
"""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import DeviceCache, OracleCache, check_topk, check_topk_forced, i32

pytestmark = pytest.mark.gpu

CTX = (46080,) + (15360,) * 3 + (2000, 700, 129, 5000)


def _cuts(nb_max: int, n: int, seed: int) -> np.ndarray:
    """n + 1 ascending cut points 0 = c0 <= ... <= cn = nb_max, uneven (some
    slices empty, one holding most of the blocks)."""
    u = W.uniform(seed, "cp_cuts", 0, n - 1) ** 3 * nb_max
    return np.concatenate([[0], np.sort(np.floor(u).astype(np.int64)), [nb_max]])


def _slice_tables(bt: np.ndarray, nb: np.ndarray, cuts: np.ndarray):
    """Per slice: (block table [B, max count] holding the slice's pages, blk_begin,
    blk_count); slice s holds blocks cuts[s] .. cuts[s+1] - 1 of every request
    (clipped to the request's blocks)."""
    out = []
    for s in range(len(cuts) - 1):
        begin = np.minimum(cuts[s], nb).astype(np.int32)
        count = (np.minimum(cuts[s + 1], nb) - begin).astype(np.int32)
        width = max(1, int(count.max()))
        t = np.zeros((len(nb), width), dtype=np.int32)
        for b in range(len(nb)):
            t[b, : count[b]] = bt[b, begin[b]: begin[b] + count[b]]
        out.append((t, begin, count))
    return out


def _key_parts(k: np.ndarray):
    """(high word, low word) of int64 keys read as uint64."""
    u = k.astype(np.int64).view(np.uint64)
    return (u >> np.uint64(32)).astype(np.uint64), (u & np.uint64(0xFFFFFFFF)).astype(np.uint64)


def _ordered_to_f32(hi: np.ndarray) -> np.ndarray:
    """Inverse of the documented order-preserving map of a float's bits."""
    hi = hi.astype(np.uint32)
    bits = np.where(hi & 0x80000000, hi & 0x7FFFFFFF, ~hi).astype(np.uint32)
    return bits.view(np.float32)


def _decode_ids(keys: np.ndarray) -> np.ndarray:
    hi, lo = _key_parts(keys)
    ids = np.where(hi == 0xFFFFFFFE, lo, np.uint64(0xFFFFFFFF) - lo).astype(np.int64)
    return np.where(keys == 0, -1, ids)


def _run(init: int, local: int, n: int, seed: int):
    wl = W.make("skewed", ctx=CTX, q_rows=(1,) * len(CTX))
    s = wl.spec
    dev = DeviceCache(wl)
    dev.store_all()
    R = s.rows
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, R)
    bscores = torch.full((R, wl.bt_stride), float("nan"), device="cuda")
    whole = M.m3s_index_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, row_req,
                                   row_len, s.topk, block_scores=bscores, err=dev.err,
                                   init_blocks=init, local_blocks=local)
    nb = (wl.seq_len.astype(np.int64) + 127) // 128
    slices = _slice_tables(wl.block_table, nb, _cuts(int(nb.max()), n, seed))
    cands = []
    for t, begin, count in slices:
        cands.append(M.m3s_index_score_candidates(
            dev.q_idx, dev.w, dev.ic, dev.is_, i32(t), i32(begin), i32(count), row_req, row_len,
            s.topk, err=dev.err, init_blocks=init, local_blocks=local))
    stacked = torch.stack(cands).contiguous()
    merged = M.m3s_merge_candidates(stacked)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    return wl, nb, slices, bscores.cpu().numpy(), whole.cpu().numpy(), stacked.cpu().numpy(), \
        merged.cpu().numpy()


@pytest.mark.parametrize("n", [1, 2, 3, 7])
def test_slices_merge_to_the_unsplit_ids(lib, n):
    wl, nb, slices, gbs, whole, keys, merged = _run(0, 0, n, 40 + n)
    s = wl.spec
    np.testing.assert_array_equal(merged, whole)
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, s.rows)
    _, ref_bs, e = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl, s.topk)
    assert e == 0
    check_topk(merged, ref_bs, s.topk, range(s.rows), gbs)
    # each slice's candidates: descending keys, zero-padded, the documented
    # format (the high word is the GPU's own block score), its oracle top-k
    for (t, begin, count), k in zip(slices, keys):
        for r in range(s.rows):
            b = int(wl.cu_q.searchsorted(r, side="right") - 1)
            u = k[r].astype(np.int64).view(np.uint64)
            live = u != 0
            nlive = int(live.sum())
            assert live[:nlive].all()
            assert np.all(u[:nlive][:-1] > u[:nlive][1:]), (r, u)
            lo, hi = int(begin[b]), int(begin[b] + count[b])
            assert nlive == min(s.topk, hi - lo), (r, nlive, lo, hi)
            if nlive == 0:
                continue
            ids = _decode_ids(k[r, :nlive])
            assert ((ids >= lo) & (ids < hi)).all()
            hw, _ = _key_parts(k[r, :nlive])
            np.testing.assert_array_equal(_ordered_to_f32(hw), gbs[r, ids].astype(np.float32))
            sub = np.asarray(ref_bs[r][lo:hi])
            fake = np.full((1, s.topk), -1, dtype=np.int32)
            fake[0, :nlive] = np.sort(ids - lo)
            check_topk(fake, [sub], s.topk, [0])


def test_forced_blocks_follow_the_rows_own_block_count(lib):
    init, local = 2, 3
    wl, nb, slices, gbs, whole, keys, merged = _run(init, local, 3, 7)
    s = wl.spec
    np.testing.assert_array_equal(merged, whole)
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, s.rows)
    _, ref_bs, e = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl, s.topk)
    check_topk_forced(merged, ref_bs, s.topk, range(s.rows), init, local)
    # forced keys carry the class words whatever slice holds the block
    for k in keys:
        hw, lw = _key_parts(k)
        ids = _decode_ids(k)
        for r in range(s.rows):
            for j in range(s.topk):
                if ids[r, j] < 0:
                    continue
                if ids[r, j] < init:
                    assert hw[r, j] == 0xFFFFFFFF
                elif ids[r, j] >= nb[r] - local:
                    assert hw[r, j] == 0xFFFFFFFE and lw[r, j] == ids[r, j]


def test_empty_slice_and_merge_edges(lib):
    wl = W.make("skewed", ctx=(3000, 129), q_rows=(1, 1))
    s = wl.spec
    dev = DeviceCache(wl)
    dev.store_all()
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, s.rows)
    # a slice that holds no block of either request, and one past the short row's end
    t = i32(np.zeros((2, 1), dtype=np.int32))
    empty = M.m3s_index_score_candidates(dev.q_idx, dev.w, dev.ic, dev.is_, t,
                                         i32(np.array([0, 0], np.int32)),
                                         i32(np.array([0, 0], np.int32)), row_req, row_len, s.topk,
                                         err=dev.err)
    t2 = i32(wl.block_table[:, 5:6].copy())
    past = M.m3s_index_score_candidates(dev.q_idx, dev.w, dev.ic, dev.is_, t2,
                                        i32(np.array([5, 5], np.int32)),
                                        i32(np.array([1, 1], np.int32)), row_req, row_len, s.topk,
                                        err=dev.err)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    assert (empty.cpu().numpy() == 0).all()
    p = past.cpu().numpy()
    assert (p[1] == 0).all() and (_decode_ids(p[0, :1]) == 5).all() and (p[0, 1:] == 0).all()
    # merging only empty lists gives -1 rows; zero lists too
    ids = M.m3s_merge_candidates(torch.stack([empty, empty]).contiguous())
    ids0 = M.m3s_merge_candidates(torch.zeros((0, 2, s.topk), dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert (ids.cpu().numpy() == -1).all() and (ids0.cpu().numpy() == -1).all()
    with pytest.raises(RuntimeError):
        M.m3s_merge_candidates(torch.zeros((257, 2, s.topk), dtype=torch.int64, device="cuda"))
