"""GPU parity of the streaming block top-k: the form score + top-k calls take
with more query tiles than the scorer has CTAs ("[MiniMax-M3.1] FP4 index cache
and NVFP4 sparse KV cache" (#2744), Fused verify top-k: a streaming top-k per
chunk, then a merge). Every warp keeps a running top-k of packed (score, id)
keys, each CTA leaves its share of a tile as candidates, and the CTA that scores
a tile's last block merges them. The ids must equal the oracle's outside the
tie band, ties to the lower id, forced blocks exactly."""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import (DeviceCache, OracleCache, check_block_scores, check_topk, check_topk_forced,
                          i32)

pytestmark = pytest.mark.gpu

MAX_GRID = 256   # the scorers' CTA bound: more tiles than this stream


def _decode_rows(B, seed):
    ctx = tuple(int(129 + (v % 1900)) for v in W.u64(seed, "ctx_stream", 0, B))
    return W.make("decode", ctx=ctx, q_rows=(1,) * B)


@pytest.mark.parametrize("forced", [(0, 0), (2, 3)], ids=["plain", "forced"])
def test_index_path_streams_many_rows(lib, forced):
    init, local = forced
    wl = _decode_rows(300, 31)
    s = wl.spec
    assert s.rows > MAX_GRID
    dev = DeviceCache(wl)
    dev.store_all()
    R = s.rows
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, R)
    bscores = torch.full((R, wl.bt_stride), float("nan"), device="cuda")
    ids = M.m3s_index_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, row_req, row_len,
                                 s.topk, block_scores=bscores, err=dev.err, init_blocks=init,
                                 local_blocks=local)
    # a second call on the same (zeroed once) workspace: the tickets were reset
    ws = torch.zeros(M.m3s_workspace_bytes(M.OP_INDEX_SCORE_TOPK, R, *wl.block_table.shape, 0, 0, s.hi,
                                           s.topk), dtype=torch.uint8, device="cuda")
    ids2 = [M.m3s_index_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, row_req, row_len,
                                   s.topk, ws=ws, err=dev.err, init_blocks=init, local_blocks=local)
            for _ in range(2)]
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    assert torch.equal(ids2[0], ids) and torch.equal(ids2[1], ids)
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    _, ref_bs, e = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl, s.topk)
    assert e == 0
    gbs = bscores.cpu().numpy()
    check_block_scores(gbs, ref_bs, range(R))
    if init or local:
        check_topk_forced(ids.cpu().numpy(), ref_bs, s.topk, range(R), init, local)
        for r in range(R):   # exactly the oracle's selection on the GPU's own scores
            own = O.topk_ids(gbs[r, : len(ref_bs[r])].astype(np.float64), s.topk, init, local)
            assert np.array_equal(own, ids[r].cpu().numpy()), r
    else:
        check_topk(ids.cpu().numpy(), ref_bs, s.topk, range(R), gbs)


def test_index_streaming_ties_take_the_lower_id(lib):
    """Every score 0 (zero queries): the streamed selection keeps blocks 0 .. k-1."""
    wl = _decode_rows(280, 33)
    wl.q_idx = np.zeros_like(wl.q_idx)
    dev = DeviceCache(wl)
    dev.store_all()
    _, _, ids, _, _, _ = dev.step(False)
    torch.cuda.synchronize()
    k = wl.spec.topk
    for r, L in enumerate(wl.seq_len):
        nb = (int(L) + 127) // 128
        assert ids[r].tolist() == list(range(min(k, nb))) + [-1] * (k - min(k, nb)), r


def test_verify_path_streams_many_tiles(lib):
    B = 100
    ctx = tuple(int(300 + (v % 1500)) for v in W.u64(35, "ctx_vstream", 0, B))
    q_rows = tuple(int(17 + v % 8) for v in W.u64(35, "q_vstream", 0, B))   # 3 tiles a request
    wl = W.make("verify", ctx=ctx, q_rows=q_rows)
    s = wl.spec
    assert B * ((max(q_rows) + 7) // 8) > MAX_GRID
    dev = DeviceCache(wl)
    dev.store_all()
    R = s.rows
    _, row_len, ids, _, _, _ = dev.step(True)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    _, ref_bs, e = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl, s.topk)
    assert e == 0
    check_topk(ids.cpu().numpy(), ref_bs, s.topk, range(R))
