"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by
element, on seeded inputs small enough for the oracle (several tiles, ragged
tails). Acceptance: planes and row maps bit-exact; block scores within 1e-4
relative; top-k sets equal except inside the 1e-5 tie band with ties to the
lower id; attention max relative error <= 1e-2."""

import math

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import (ATTN_RTOL, SM_SCALE, DeviceCache, OracleCache, attention_rel_err,
                          bf16_dev, bf16_np, check_block_scores, check_topk, i32, i64)

pytestmark = pytest.mark.gpu


def _planes_equal(dev_c, dev_s, ref_c, ref_s):
    assert np.array_equal(dev_c.cpu().numpy(), ref_c)
    assert np.array_equal(dev_s.cpu().numpy(), ref_s)


def test_store_bit_exact_heads_pads_and_bad_slot(lib):
    T, H, P = 700, 3, 8
    src = W.bf16_tensor(5, "store", (T, H, 128), 4, 20.0)
    slots = W.permutation(5, "slots", P * 128)[:T].astype(np.int64)
    slots[[3, 100, 699]] = -1
    slots[50] = P * 128 + 5        # out of range: reported, skipped
    ref_c, ref_s = O.new_planes(P, H)
    ref_c[:] = 0xA5
    ref_s[:] = 0x5A
    assert O.nvfp4_store(src, slots, ref_c, ref_s) == O.ERR_SLOT
    dc, ds = M.new_plane(P, H)
    dc.fill_(0xA5)
    ds.fill_(0x5A)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # strided source rows: pad every row to 3*128 + 64 elements
    big = torch.zeros((T, H * 128 + 64), dtype=torch.bfloat16, device="cuda")
    big[:, : H * 128] = bf16_dev(src).reshape(T, H * 128)
    view = big[:, : H * 128].view(T, H, 128)
    M.m3s_nvfp4_store(view, i64(slots), dc, ds, err)
    torch.cuda.synchronize()
    _planes_equal(dc, ds, ref_c, ref_s)
    assert int(err.item()) == M.DEVERR_SLOT


def test_store_hand_worked_and_random_bit_patterns(lib):
    """The golden groups, plus BF16 bit patterns drawn over the whole finite range."""
    from test_oracle_pins import _block, _golden_cases
    rows = [_block(c["x"]) for c in _golden_cases()]
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 1 << 16, size=(4096, 128), dtype=np.uint64).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    bits[exp == 0xFF] &= 0x807F            # no inf / NaN: keep the mantissa, zero exponent
    # also groups with every element in a narrow exponent band (all scale codes hit)
    for e in range(0, 255, 2):
        row = rng.integers(0, 1 << 7, size=128).astype(np.uint16) | np.uint16(min(e, 254) << 7)
        rows.append(row | (rng.integers(0, 2, size=128).astype(np.uint16) << 15))
    src = np.concatenate([np.stack(rows), bits])[:, None, :]
    T = src.shape[0]
    P = (T + 127) // 128
    slots = np.arange(T, dtype=np.int64)
    ref_c, ref_s = O.new_planes(P, 1)
    O.nvfp4_store(src, slots, ref_c, ref_s)
    dc, ds = M.new_plane(P, 1)
    M.m3s_nvfp4_store(bf16_dev(src), i64(slots), dc, ds)
    torch.cuda.synchronize()
    _planes_equal(dc, ds, ref_c, ref_s)


def test_decode_rows_bit_exact(lib):
    rng = np.random.default_rng(4)
    for trial in range(20):
        B = int(rng.integers(0, 40))
        qb = rng.integers(0, 12, B)
        if trial % 4 == 0 and B:
            qb[rng.integers(0, B)] = 0           # an empty request
        seq = (qb + rng.integers(0, 300000, B)).astype(np.int32)
        cu = np.concatenate([[0], np.cumsum(qb)]).astype(np.int32)
        R = int(cu[-1] + rng.integers(0, 5))     # trailing pad rows
        if R == 0:
            continue
        rr, rl = M.m3s_decode_rows(i32(cu), i32(seq), R)
        er, el = O.decode_rows(cu, seq, R)
        assert np.array_equal(rr.cpu().numpy(), er) and np.array_equal(rl.cpu().numpy(), el)


def _small(name, ctx, q_rows, **over):
    wl = W.make(name, ctx=ctx, q_rows=q_rows)
    if over:
        import dataclasses
        wl.spec = dataclasses.replace(wl.spec, **over)
    return wl


CASES = [
    # (spec, contexts, rows per request, fused verify path)
    ("tiny", (4096,), (1,), False),
    ("decode", (1000, 3000, 129, 128, 5000, 257), (1,) * 6, False),
    ("verify", (700, 2500, 1300, 999), (8, 3, 8, 1), True),
    # 20 + 3 rows: three 8-row tiles per request, two of the second request's empty
    ("verify-uneven", (1500, 2200), (20, 3), True),
    ("skewed", (9000, 3000, 3000, 3000), (1, 1, 1, 1), False),
    ("prefill", (2000,), (40,), True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_step_small_vs_oracle(lib, case):
    name, ctx, qr, fused = case
    wl = W.make(name.split("-")[0], ctx=ctx, q_rows=qr)
    s = wl.spec
    dev = DeviceCache(wl)
    dev.store_all()
    row_req, row_len, ids, bscores, out, lse = dev.step(fused)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    ref = OracleCache(wl)
    _planes_equal(dev.ic, dev.is_, ref.ic, ref.is_)
    _planes_equal(dev.kc, dev.ks, ref.kc, ref.ks)
    _planes_equal(dev.vc, dev.vs, ref.vc, ref.vs)
    R = s.rows
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    assert np.array_equal(row_req.cpu().numpy(), rr) and np.array_equal(row_len.cpu().numpy(), rl)
    ref_ids, ref_bs, err = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr,
                                              rl, s.topk)
    assert err == 0
    gids = ids.cpu().numpy()
    gbs = None
    if bscores is not None:
        gbs = bscores.cpu().numpy()
        check_block_scores(gbs, ref_bs, range(R))
    check_topk(gids, ref_bs, s.topk, range(R), gbs)
    # attention over the GPU's own selection (identical to the oracle's outside tie bands)
    o_ref, lse_ref, err = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs,
                                             wl.block_table, rr, rl, gids, SM_SCALE)
    assert err == 0
    e = attention_rel_err(bf16_np(out), o_ref, range(R))
    assert e <= ATTN_RTOL, e
    np.testing.assert_allclose(lse.cpu().numpy(), lse_ref, rtol=1e-4, atol=1e-4)


def test_verify_path_and_index_path_agree(lib):
    """Rows of one request scored together (the fused verify path) select what
    row-by-row scoring selects: both against the oracle's scores, identical
    outside the tie band."""
    wl = W.make("verify", ctx=(3000, 1800, 4000), q_rows=(8, 5, 8))
    s = wl.spec
    dev = DeviceCache(wl)
    dev.store_all()
    R = s.rows
    _, _, ids_v, _, _, _ = dev.step(True)
    _, _, ids_i, _, _, _ = dev.step(False)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0, int(dev.err.item())
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    _, ref_bs, _ = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl,
                                      s.topk)
    check_topk(ids_v.cpu().numpy(), ref_bs, s.topk, range(R))
    check_topk(ids_i.cpu().numpy(), ref_bs, s.topk, range(R))


def test_zero_queries_pick_lowest_ids(lib):
    """Every score 0: ties break to the lower block id (the pages' zero-query tie test)."""
    wl = W.make("decode", ctx=(5000, 3000, 700), q_rows=(1, 1, 1))
    wl.q_idx[:] = 0
    dev = DeviceCache(wl)
    dev.store_all()
    _, _, ids, bs, _, _ = dev.step(False)
    _, _, ids_v, _, _, _ = dev.step(True)
    torch.cuda.synchronize()
    k = wl.spec.topk
    for r, L in enumerate(wl.seq_len):
        nb = (int(L) + 127) // 128
        exp = list(range(min(k, nb))) + [-1] * (k - min(k, nb))
        assert ids[r].tolist() == exp and ids_v[r].tolist() == exp


def test_attention_bad_ids_are_reported_not_wrapped(lib):
    wl = W.make("decode", ctx=(1000, 600), q_rows=(1, 1))
    s = wl.spec
    dev = DeviceCache(wl)
    dev.store_all()
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, 2)
    ids = torch.tensor([[0, 3, 7, 8, 500] + [-1] * 11, [4, 1, 5, 9, -1] + [-1] * 11],
                       dtype=torch.int32, device="cuda")   # 8, 500 / 5, 9 are beyond the rows
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = M.m3s_sparse_attention(dev.q, s.hkv, dev.kc, dev.ks, dev.vc, dev.vs, dev.block_table,
                                 row_req, row_len, ids, SM_SCALE, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == M.DEVERR_BLOCK_ID
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, 2)
    o_ref, _, oerr = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs,
                                        wl.block_table, rr, rl, ids.cpu().numpy(), SM_SCALE)
    assert oerr == O.ERR_BLOCK_ID
    assert attention_rel_err(bf16_np(out), o_ref, range(2)) <= ATTN_RTOL


def test_attention_detects_one_dropped_token(lib):
    """The measured error must sit far below the change that dropping one causal
    token makes (a 2% bound can hide an off-by-one mask; ours cannot)."""
    wl = W.make("decode", ctx=(2000, 1500), q_rows=(1, 1))
    s = wl.spec
    dev = DeviceCache(wl)
    dev.store_all()
    row_req, row_len, ids, _, out, _ = dev.step(False)
    torch.cuda.synchronize()
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, 2)
    gids = ids.cpu().numpy()
    o_ref, _, _ = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs, wl.block_table,
                                     rr, rl, gids, SM_SCALE)
    o_drop, _, _ = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs,
                                      wl.block_table, rr, rl - 1, gids, SM_SCALE)
    e_gpu = attention_rel_err(bf16_np(out), o_ref, range(2))
    e_drop = attention_rel_err(o_drop, o_ref, range(2))
    assert e_gpu * 4 < e_drop, (e_gpu, e_drop)


def test_attention_full_cover_and_gqa_shapes(lib):
    """top-k covering every block, G = 4 and Hkv = 2, against the oracle."""
    import dataclasses
    spec = dataclasses.replace(W.SPECS["tiny"], ctx=(900, 128, 1), q_rows=(1, 1, 1), hq=8, hkv=2,
                               topk=8)
    wl = W.make(spec)
    dev = DeviceCache(wl)
    dev.store_all()
    _, _, ids, _, out, lse = dev.step(False)
    torch.cuda.synchronize()
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, 3)
    gids = ids.cpu().numpy()
    assert gids[0].tolist() == list(range(8)) and gids[2].tolist() == [0] + [-1] * 7
    o_ref, lse_ref, _ = O.sparse_attention(wl.q, 2, ref.kc, ref.ks, ref.vc, ref.vs,
                                           wl.block_table, rr, rl, gids, SM_SCALE)
    assert attention_rel_err(bf16_np(out), o_ref, range(3)) <= ATTN_RTOL
    np.testing.assert_allclose(lse.cpu().numpy(), lse_ref, rtol=1e-4, atol=1e-4)


def test_pad_rows_and_empty_inputs(lib):
    wl = W.make("decode", ctx=(900, 300), q_rows=(1, 1))
    dev = DeviceCache(wl)
    dev.store_all()
    R = 5                                 # rows 2..4 are padding
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, R)
    q_idx = torch.zeros((R, 16, 128), dtype=torch.bfloat16, device="cuda")
    q_idx[:2] = dev.q_idx
    w = torch.ones((R, 16), device="cuda")
    ids = M.m3s_index_score_topk(q_idx, w, dev.ic, dev.is_, dev.block_table, row_req, row_len, 16)
    q = torch.randn((R, 16, 128), device="cuda").to(torch.bfloat16)
    lse = torch.empty((R, 16), device="cuda")
    out = M.m3s_sparse_attention(q, 1, dev.kc, dev.ks, dev.vc, dev.vs, dev.block_table, row_req,
                                 row_len, ids, lse=lse)
    torch.cuda.synchronize()
    assert (ids[2:] == -1).all()
    assert (out[2:] == 0).all() and torch.isneginf(lse[2:]).all()
    # zero-sized calls are no-ops
    M.m3s_nvfp4_store(torch.zeros((0, 1, 128), dtype=torch.bfloat16, device="cuda"),
                      torch.zeros(0, dtype=torch.int64, device="cuda"), dev.ic, dev.is_)


def test_store_batch_equals_single_stores(lib):
    T, P = 300, 4
    srcs = [W.bf16_tensor(9, n, (T, h, 128), 3, 10.0) for n, h in (("bk", 2), ("bv", 2), ("bi", 1))]
    slots = W.permutation(9, "bslots", P * 128)[:T].astype(np.int64)
    slots[7] = -1
    sl = i64(slots)
    single, batch = [], []
    for src in srcs:
        c1, s1 = M.new_plane(P, src.shape[1])
        M.m3s_nvfp4_store(bf16_dev(src), sl, c1, s1)
        single.append((c1, s1))
        batch.append((bf16_dev(src),) + M.new_plane(P, src.shape[1]))
    M.m3s_nvfp4_store_batch(batch, sl)
    torch.cuda.synchronize()
    for (c1, s1), (_, c2, s2) in zip(single, batch):
        assert torch.equal(c1, c2) and torch.equal(s1, s2)


def test_block_topk_direct_against_oracle(lib):
    """m3s_block_topk on given fp32 block scores == the oracle's selection exactly:
    ties (lower id wins), +-0, negatives, rows narrower than k, and rows on
    every path of the selection (keys in registers, in shared memory, re-read)."""
    rng = np.random.default_rng(11)
    # 8192 / 8193: the edge of the keys-in-registers path (8 a thread);
    # 10000: keys kept in shared memory; 20000: keys read again from memory
    widths = [1, 5, 16, 17, 300, 3600, 8192, 8193, 10000, 20000]
    bt_stride = max(widths)
    R = len(widths) * 4
    scores = np.zeros((R, bt_stride), dtype=np.float32)
    lens = np.zeros(R, dtype=np.int32)
    for i, nb in enumerate(widths):
        for v in range(4):
            r = 4 * i + v
            lens[r] = nb * 128 - int(rng.integers(0, 128))
            x = rng.standard_normal(nb).astype(np.float32)
            if v == 1:
                x = np.round(x * 2).astype(np.float32)          # many exact ties
            if v == 2:
                x[:] = 0.0
                x[rng.integers(0, nb, size=max(1, nb // 3))] = -0.0
            if v == 3:
                x = -np.abs(x)                                  # all negative
            scores[r, :nb] = x
            scores[r, nb:] = np.nan                             # never read
    for topk in (1, 8, 16, 64):
        ids = M.m3s_block_topk(torch.from_numpy(scores).cuda(), None, i32(lens), 1, bt_stride, topk)
        torch.cuda.synchronize()
        got = ids.cpu().numpy()
        for r in range(R):
            nb = (int(lens[r]) + 127) // 128
            exp = O.topk_ids(scores[r, :nb].astype(np.float64), topk)
            assert np.array_equal(got[r], exp), (topk, r, got[r], exp)


@pytest.mark.parametrize("fused", [False, True], ids=["index", "verify"])
def test_many_short_rows_cross_tile_ranges(lib, fused):
    """Hundreds of short rows: every CTA's block range spans several query tiles, so
    the pipelines restart at arbitrary block counts (a regression guard for the
    block-to-warpgroup routing across segments)."""
    B = 120
    ctx = tuple(int(129 + (v % 1900)) for v in W.u64(21, "ctx_many", 0, B))
    q_rows = tuple(int(1 + v % 8) if fused else 1 for v in W.u64(21, "q_many", 0, B))
    wl = W.make("decode", ctx=ctx, q_rows=q_rows)
    s = wl.spec
    dev = DeviceCache(wl)
    dev.store_all()
    R = s.rows
    _, row_len, ids, bscores, _, _ = dev.step(fused)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0, int(dev.err.item())
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    _, ref_bs, _ = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl,
                                      s.topk)
    gbs = None
    if bscores is not None:
        gbs = bscores.cpu().numpy()
        check_block_scores(gbs, ref_bs, range(R))
    check_topk(ids.cpu().numpy(), ref_bs, s.topk, range(R), gbs)


def test_block_topk_forced_blocks_direct(lib):
    """m3s_block_topk with forced init / local blocks == the oracle exactly, on
    every selection path, including init + local beyond k."""
    rng = np.random.default_rng(12)
    widths = [3, 16, 40, 300, 3600, 10000, 20000]
    bt_stride = max(widths)
    R = len(widths)
    scores = np.full((R, bt_stride), np.nan, dtype=np.float32)
    lens = np.zeros(R, dtype=np.int32)
    for r, nb in enumerate(widths):
        lens[r] = nb * 128 - int(rng.integers(0, 128))
        scores[r, :nb] = np.round(rng.standard_normal(nb), 1)     # ties
    for topk, init, local in ((16, 0, 0), (16, 2, 3), (16, 4, 16), (8, 10, 2), (64, 1, 64)):
        ids = M.m3s_block_topk(torch.from_numpy(scores).cuda(), None, i32(lens), 1, bt_stride, topk,
                               init_blocks=init, local_blocks=local)
        torch.cuda.synchronize()
        got = ids.cpu().numpy()
        for r in range(R):
            nb = (int(lens[r]) + 127) // 128
            exp = O.topk_ids(scores[r, :nb].astype(np.float64), topk, init, local)
            assert np.array_equal(got[r], exp), (topk, init, local, r, got[r], exp)


@pytest.mark.parametrize("fused", [False, True], ids=["index", "verify"])
@pytest.mark.parametrize("init,local", [(2, 3), (4, 16)], ids=["fit", "over_k"])
def test_step_with_forced_blocks(lib, fused, init, local):
    """Score + top-k with forced blocks through both paths against the oracle:
    forced blocks exact (with 4 + 16 > k = 16, the row's newest blocks are the
    ones kept), the rest by score; attention over the selection."""
    from step_helpers import check_topk_forced
    wl = W.make("verify", ctx=(6000, 1800, 300, 4500), q_rows=(3, 2, 1, 4) if fused else (1, 1, 1, 1))
    s = wl.spec
    dev = DeviceCache(wl)
    dev.store_all()
    R = s.rows
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, R)
    if fused:
        ids = M.m3s_verify_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, dev.cu_q,
                                      row_len, max(s.q_rows), s.topk, err=dev.err,
                                      init_blocks=init, local_blocks=local)
    else:
        ids = M.m3s_index_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, row_req,
                                     row_len, s.topk, err=dev.err, init_blocks=init,
                                     local_blocks=local)
    lse = torch.empty((R, s.hq), dtype=torch.float32, device="cuda")
    out = M.m3s_sparse_attention(dev.q, s.hkv, dev.kc, dev.ks, dev.vc, dev.vs, dev.block_table,
                                 row_req, row_len, ids, SM_SCALE, lse=lse, err=dev.err)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    _, ref_bs, _ = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl,
                                      s.topk)
    gids = ids.cpu().numpy()
    check_topk_forced(gids, ref_bs, s.topk, range(R), init, local)
    if (init, local) == (4, 16):
        for r in range(R):
            nb = (int(rl[r]) + 127) // 128
            if nb > s.topk:
                assert gids[r][-1] == nb - 1      # the current token's block is kept
    o_ref, _, err = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs,
                                       wl.block_table, rr, rl, gids, SM_SCALE)
    assert err == 0
    assert attention_rel_err(bf16_np(out), o_ref, range(R)) <= ATTN_RTOL
