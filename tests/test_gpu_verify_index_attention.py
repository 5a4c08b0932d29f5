"""GPU parity of m3s_verify_index_attention: the fused verify scoring, top-k and
block-sparse attention of verify rows in two launches ("[MiniMax-M3.1] FP4 index
cache and NVFP4 sparse KV cache" (#2744), Fused verify top-k and Design /
Attention: a request's rows are scored together, the top-k is kept per chunk and
merged, and each row attends over its top-k blocks).

The verify scorer leaves each CTA's top-k candidates of every row it scores and
the attention merges a row's lists before it reads the row's pages; the result
must be exactly that of m3s_verify_score_topk followed by m3s_sparse_attention
(ids, BF16 outputs and lse bit for bit), and the ids the oracle's top-k outside
the tie band.
"""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import SM_SCALE, DeviceCache, OracleCache, check_topk, check_topk_forced

pytestmark = pytest.mark.gpu


def _both(dev: DeviceCache, R: int, topk: int, init: int = 0, local: int = 0):
    """(fused ids, out, lse), (separate ids, out, lse) on the same inputs."""
    s = dev.wl.spec
    max_q = max(s.q_rows)
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, R)
    lse_f = torch.full((R, s.hq), float("nan"), dtype=torch.float32, device="cuda")
    ids_f, out_f = M.m3s_verify_index_attention(dev.q_idx, dev.w, dev.ic, dev.is_, dev.q, s.hkv, dev.kc, dev.ks,
                                                dev.vc, dev.vs, dev.block_table, dev.cu_q, row_req, row_len,
                                                max_q, topk, SM_SCALE, lse=lse_f, err=dev.err,
                                                init_blocks=init, local_blocks=local)
    ids_s = M.m3s_verify_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, dev.cu_q, row_len,
                                    max_q, topk, err=dev.err, init_blocks=init, local_blocks=local)
    lse_s = torch.full((R, s.hq), float("nan"), dtype=torch.float32, device="cuda")
    out_s = M.m3s_sparse_attention(dev.q, s.hkv, dev.kc, dev.ks, dev.vc, dev.vs, dev.block_table, row_req,
                                   row_len, ids_s, SM_SCALE, lse=lse_s, err=dev.err)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0, f"device error bits {int(dev.err.item())}"
    return (ids_f, out_f, lse_f), (ids_s, out_s, lse_s)


def _same(f, s):
    np.testing.assert_array_equal(f[0].cpu().numpy(), s[0].cpu().numpy())
    assert torch.equal(f[1].view(torch.int16), s[1].view(torch.int16)), "outputs differ"
    np.testing.assert_array_equal(f[2].cpu().numpy(), s[2].cpu().numpy())


CASES = {
    "three_requests": dict(ctx=(3000, 1500, 900), q_rows=(8, 5, 3)),
    "multi_tile_request": dict(ctx=(5000, 2500), q_rows=(20, 3)),   # 3 tiles, the last partial
    "long_and_short": dict(ctx=(46080, 700, 129, 15360), q_rows=(8, 8, 2, 6)),
    "one_row": dict(ctx=(3000,), q_rows=(1,)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fused_equals_verify_score_topk_then_attention(lib, case):
    c = CASES[case]
    wl = W.make("verify", ctx=c["ctx"], q_rows=c["q_rows"])
    dev = DeviceCache(wl)
    dev.store_all()
    f, s = _both(dev, wl.spec.rows, wl.spec.topk)
    _same(f, s)


def test_oracle_top_k_of_the_fused_ids(lib):
    c = CASES["long_and_short"]
    wl = W.make("verify", ctx=c["ctx"], q_rows=c["q_rows"])
    dev = DeviceCache(wl)
    dev.store_all()
    f, _ = _both(dev, wl.spec.rows, wl.spec.topk)
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, wl.spec.rows)
    _, ref_bs, e = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl, wl.spec.topk)
    assert e == 0
    check_topk(f[0].cpu().numpy(), ref_bs, wl.spec.topk, range(wl.spec.rows))


def test_forced_blocks_and_pad_rows(lib):
    c = CASES["three_requests"]
    wl = W.make("verify", ctx=c["ctx"], q_rows=c["q_rows"])
    dev = DeviceCache(wl)
    dev.store_all()
    R = wl.spec.rows + 3   # three pad rows past cu_q[B]: no ids, zero outputs
    dev.q_idx = torch.cat([dev.q_idx, dev.q_idx[:3]]).contiguous()
    dev.w = torch.cat([dev.w, dev.w[:3]]).contiguous()
    dev.q = torch.cat([dev.q, dev.q[:3]]).contiguous()
    f, s = _both(dev, R, wl.spec.topk, init=2, local=3)
    _same(f, s)
    ids = f[0].cpu().numpy()
    assert (ids[-3:] == -1).all() and (f[1][-3:].float() == 0).all()
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, wl.spec.rows)
    _, ref_bs, _ = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl, wl.spec.topk)
    check_topk_forced(ids, ref_bs, wl.spec.topk, range(wl.spec.rows), 2, 3)


@pytest.mark.parametrize("mx", [(True, False), (False, True), (True, True)], ids=["mx_kv", "mx_index", "mx_both"])
def test_mxfp4_planes(lib, mx):
    c = CASES["three_requests"]
    wl = W.make("verify", ctx=c["ctx"], q_rows=c["q_rows"])
    dev = DeviceCache(wl, mx_kv=mx[0], mx_index=mx[1])
    dev.store_all()
    f, s = _both(dev, wl.spec.rows, wl.spec.topk)
    _same(f, s)


def test_more_tiles_than_scorer_ctas_and_top_k_widths(lib):
    """300 one-row requests (300 tiles, above the 256 slots of one wave), and
    top-k 1, 40 and 64."""
    B = 300
    ctx = tuple(int(129 + (v % 2500)) for v in W.u64(78, "ctx_via", 0, B))
    wl = W.make("verify", ctx=ctx, q_rows=(1,) * B)
    dev = DeviceCache(wl)
    dev.store_all()
    for topk in (wl.spec.topk, 1, 40, 64):
        f, s = _both(dev, B, topk)
        _same(f, s)


def test_workspace_and_top_k_zero(lib):
    wl = W.make("verify", ctx=(1000, 300), q_rows=(3, 2))
    dev = DeviceCache(wl)
    dev.store_all()
    s = wl.spec
    R = s.rows
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, R)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.M3SError, match="WORKSPACE"):
        M.m3s_verify_index_attention(dev.q_idx, dev.w, dev.ic, dev.is_, dev.q, 1, dev.kc, dev.ks, dev.vc, dev.vs,
                                     dev.block_table, dev.cu_q, row_req, row_len, 3, 16, SM_SCALE, ws=small)
    _, out = M.m3s_verify_index_attention(dev.q_idx, dev.w, dev.ic, dev.is_, dev.q, 1, dev.kc, dev.ks, dev.vc,
                                          dev.vs, dev.block_table, dev.cu_q, row_req, row_len, 3, 0, SM_SCALE)
    torch.cuda.synchronize()
    assert (out.float() == 0).all()


def test_no_requests_every_row_padding(lib):
    """B = 0 (an empty block table, cu_q = [0]): the verify call launches no
    scorer tile and every row gets no id, a zero output and lse -inf; the
    decode call (one tile per row) gives the same; R = 0 is a no-op."""
    dev = torch.device("cuda")
    R, Hq, Hi, topk = 5, 16, 16, 16
    ic, is_ = M.new_plane(4, 1, dev)
    kc, ks = M.new_plane(4, 1, dev)
    vc, vs = M.new_plane(4, 1, dev)
    bt = torch.empty((0, 8), dtype=torch.int32, device=dev)
    cu_q = torch.zeros(1, dtype=torch.int32, device=dev)
    row_req = torch.full((R,), -1, dtype=torch.int32, device=dev)
    row_len = torch.zeros(R, dtype=torch.int32, device=dev)
    q_idx = torch.randn((R, Hi, 128), device=dev).to(torch.bfloat16)
    w = torch.ones((R, Hi), device=dev)
    q = torch.randn((R, Hq, 128), device=dev).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for fused in ("verify", "decode"):
        lse = torch.zeros((R, Hq), dtype=torch.float32, device=dev)
        ids = torch.zeros((R, topk), dtype=torch.int32, device=dev)
        out = torch.full((R, Hq, 128), 1.0, dtype=torch.bfloat16, device=dev)
        if fused == "verify":
            M.m3s_verify_index_attention(q_idx, w, ic, is_, q, 1, kc, ks, vc, vs, bt, cu_q, row_req, row_len,
                                         4, topk, SM_SCALE, topk_ids=ids, out=out, lse=lse, err=err)
        else:
            M.m3s_index_attention(q_idx, w, ic, is_, q, 1, kc, ks, vc, vs, bt, row_req, row_len, topk,
                                  SM_SCALE, topk_ids=ids, out=out, lse=lse, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"{fused}: device error bits {int(err.item())}"
        assert (ids == -1).all(), fused
        assert (out.float() == 0).all() and torch.isneginf(lse).all(), fused
    ids0, out0 = M.m3s_verify_index_attention(q_idx[:0], w[:0], ic, is_, q[:0], 1, kc, ks, vc, vs, bt, cu_q,
                                              row_req[:0], row_len[:0], 4, topk, SM_SCALE, err=err)
    torch.cuda.synchronize()
    assert ids0.shape == (0, topk) and out0.shape == (0, Hq, 128) and int(err.item()) == 0
