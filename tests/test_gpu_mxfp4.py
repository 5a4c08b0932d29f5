"""GPU parity of the MXFP4 path (e2m1 + one E8M0 scale per 32 elements) against
the fp64 oracle: "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache"
(#2744), Follow-up: MXFP4 caches, and "MXFP4 KV cache for MiniMax-M3.1 on
gfx950" (vllm #64198), Overview. The acceptance rules are the NVFP4 ones:
planes bit-exact; block scores within 1e-4 relative; top-k sets equal outside
the 1e-5 tie band (ties to the lower id); attention within 1e-2."""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import (ATTN_RTOL, SM_SCALE, DeviceCache, OracleCache, attention_rel_err,
                          bf16_dev, bf16_np, check_block_scores, check_topk, i64)

pytestmark = pytest.mark.gpu


def _planes_equal(dev_c, dev_s, ref_c, ref_s):
    assert np.array_equal(dev_c.cpu().numpy(), ref_c)
    assert np.array_equal(dev_s.cpu().numpy(), ref_s)


def test_mx_store_hand_worked_and_random_bit_patterns(lib):
    """The golden MXFP4 groups, BF16 bit patterns over the whole finite range
    (subnormals included), and groups confined to one exponent each (every
    clamped and unclamped shared exponent is hit)."""
    from test_oracle_pins import _mx_golden_cases, _mx_row
    rows = [_mx_row(c)[0] for c in _mx_golden_cases()]
    rng = np.random.default_rng(13)
    bits = rng.integers(0, 1 << 16, size=(4096, 128), dtype=np.uint64).astype(np.uint16)
    bits[((bits >> 7) & 0xFF) == 0xFF] &= 0x807F      # no inf / NaN
    for e in range(0, 255):
        row = rng.integers(0, 1 << 7, size=128).astype(np.uint16) | np.uint16(e << 7)
        rows.append(row | (rng.integers(0, 2, size=128).astype(np.uint16) << 15))
    src = np.concatenate([np.stack(rows), bits])[:, None, :]
    T = src.shape[0]
    P = (T + 127) // 128 + 1
    slots = np.arange(T, dtype=np.int64)
    slots[7] = -1                       # a pad row: its slot stays untouched
    ref_c, ref_s = O.new_planes(P, 1, mx=True)
    ref_c[:] = 0xA5
    ref_s[:] = 0x5A
    assert O.nvfp4_store(src, slots, ref_c, ref_s) == 0
    dc, ds = M.new_plane(P, 1, mx=True)
    dc.fill_(0xA5)
    ds.fill_(0x5A)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.m3s_nvfp4_store(bf16_dev(src), i64(slots), dc, ds, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _planes_equal(dc, ds, ref_c, ref_s)
    # a slot past the planes is reported and skipped
    bad = slots.copy()
    bad[3] = P * 128
    err.zero_()
    M.m3s_nvfp4_store(bf16_dev(src), i64(bad), dc, ds, err)
    torch.cuda.synchronize()
    assert int(err.item()) == M.DEVERR_SLOT


def test_batch_store_mixed_formats(lib):
    """One launch writing MXFP4 K / V planes and an NVFP4 index plane equals the
    single stores (the jobs of a batch may differ in format)."""
    T, H = 300, 2
    k = W.bf16_tensor(21, "mk", (T, H, 128), 3, 10.0)
    v = W.bf16_tensor(21, "mv", (T, H, 128), 3, 10.0)
    ik = W.bf16_tensor(21, "mi", (T, 1, 128), 3, 10.0)
    P = 4
    slots = W.permutation(21, "ms", P * 128)[:T].astype(np.int64)
    kc, ks = M.new_plane(P, H, mx=True)
    vc, vs = M.new_plane(P, H, mx=True)
    ic, is_ = M.new_plane(P, 1)
    M.m3s_nvfp4_store_batch([(bf16_dev(k), kc, ks), (bf16_dev(v), vc, vs), (bf16_dev(ik), ic, is_)],
                            i64(slots))
    torch.cuda.synchronize()
    for src, dc, ds, mx in ((k, kc, ks, True), (v, vc, vs, True), (ik, ic, is_, False)):
        rc, rs = O.new_planes(P, src.shape[1], mx=mx)
        O.nvfp4_store(src, slots, rc, rs)
        _planes_equal(dc, ds, rc, rs)


CASES = [
    # (spec, contexts, rows per request, MXFP4 index plane, MXFP4 K/V planes, fused verify)
    ("tiny", (4096,), (1,), True, True, False),
    ("decode", (1000, 3000, 129, 128, 5000, 257), (1,) * 6, True, True, False),
    ("skewed", (9000, 3000, 3000, 3000), (1, 1, 1, 1), True, True, False),
    ("decode", (2000, 700, 4100), (1, 1, 1), False, True, False),   # NVFP4 index, MXFP4 K/V
    ("decode", (2000, 700, 4100), (1, 1, 1), True, False, False),   # MXFP4 index, NVFP4 K/V
    ("verify", (700, 2500, 1300, 999), (8, 3, 8, 1), True, True, True),
    ("prefill", (2000,), (40,), True, True, True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{'mx' if c[3] else 'nv'}idx-{'mx' if c[4] else 'nv'}kv"
                                              for c in CASES])
def test_mx_step_small_vs_oracle(lib, case):
    name, ctx, qr, mx_index, mx_kv, fused = case
    wl = W.make(name, ctx=ctx, q_rows=qr)
    s = wl.spec
    dev = DeviceCache(wl, mx_kv=mx_kv, mx_index=mx_index)
    dev.store_all()
    row_req, row_len, ids, bscores, out, lse = dev.step(fused)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    ref = OracleCache(wl, mx_kv=mx_kv, mx_index=mx_index)
    _planes_equal(dev.ic, dev.is_, ref.ic, ref.is_)
    _planes_equal(dev.kc, dev.ks, ref.kc, ref.ks)
    _planes_equal(dev.vc, dev.vs, ref.vc, ref.vs)
    R = s.rows
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    ref_ids, ref_bs, err = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr,
                                              rl, s.topk)
    assert err == 0
    gids = ids.cpu().numpy()
    gbs = None
    if bscores is not None:
        gbs = bscores.cpu().numpy()
        check_block_scores(gbs, ref_bs, range(R))
    check_topk(gids, ref_bs, s.topk, range(R), gbs)
    o_ref, lse_ref, err = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs,
                                             wl.block_table, rr, rl, gids, SM_SCALE)
    assert err == 0
    e = attention_rel_err(bf16_np(out), o_ref, range(R))
    assert e <= ATTN_RTOL, e
    np.testing.assert_allclose(lse.cpu().numpy(), lse_ref, rtol=1e-4, atol=1e-4)


def test_mx_extreme_scales_stay_exact(lib):
    """Keys whose four groups span a wide exponent range, K near the smallest E8M0
    exponents and V near the largest, V growing 2^4 per block (the running V
    reference rises block by block), index queries at 2^-100 and attention
    queries at 2^110: the scorer and the attention, both exact while the
    exponents they normalise against span <= 23, match the oracle."""
    rng = np.random.default_rng(17)
    L, hi, hq = 700, 16, 16
    nb = (L + 127) // 128
    P = nb + 1

    def keys(spread):
        x = rng.standard_normal((L, 1, 128)).astype(np.float32)
        for g in range(4):
            x[:, :, 32 * g: 32 * g + 32] *= np.float32(2.0 ** (spread * g / 3.0))
        return W.f32_to_bf16_bits(x)

    ik = keys(20.0)                                           # group exponents 20 apart
    kv = W.f32_to_bf16_bits((rng.standard_normal((L, 1, 128)) * 2.0 ** -120).astype(np.float32))
    vgrow = 2.0 ** (100 + 4 * (np.arange(L) // 128))[:, None, None]
    vv = W.f32_to_bf16_bits((rng.standard_normal((L, 1, 128)) * vgrow).astype(np.float32))
    # queries at both ends of the BF16 range (the kernels scale each head into f16's)
    q_idx = W.f32_to_bf16_bits(rng.standard_normal((1, hi, 128)).astype(np.float32) * np.float32(2.0 ** -100))
    w = rng.random((1, hi)).astype(np.float32)
    q = W.f32_to_bf16_bits(rng.standard_normal((1, hq, 128)).astype(np.float32) * np.float32(2.0 ** 110))
    bt = np.zeros((1, nb), dtype=np.int32)
    bt[0] = rng.permutation(P)[:nb]
    slots = (bt[0][np.arange(L) // 128].astype(np.int64) * 128 + np.arange(L) % 128)
    rr, rl = np.array([0], dtype=np.int32), np.array([L], dtype=np.int32)

    ref = {}
    for name, src, h in (("i", ik, 1), ("k", kv, 1), ("v", vv, 1)):
        c, sc = O.new_planes(P, h, mx=True)
        assert O.nvfp4_store(src, slots, c, sc) == 0
        ref[name] = (c, sc)
    dev = {}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for name, src in (("i", ik), ("k", kv), ("v", vv)):
        c, sc = M.new_plane(P, 1, mx=True)
        M.m3s_nvfp4_store(bf16_dev(src), i64(slots), c, sc, err)
        dev[name] = (c, sc)
    torch.cuda.synchronize()
    for name in dev:
        _planes_equal(*dev[name], *ref[name])
    bt_d = torch.from_numpy(bt).cuda()
    rr_d, rl_d = torch.from_numpy(rr).cuda(), torch.from_numpy(rl).cuda()
    bs = torch.full((1, nb), float("nan"), device="cuda")
    ids = M.m3s_index_score_topk(bf16_dev(q_idx), torch.from_numpy(w).cuda(), *dev["i"], bt_d, rr_d,
                                 rl_d, 4, block_scores=bs, err=err)
    lse = torch.empty((1, hq), dtype=torch.float32, device="cuda")
    out = M.m3s_sparse_attention(bf16_dev(q), 1, *dev["k"], *dev["v"], bt_d, rr_d, rl_d, ids, SM_SCALE,
                                 lse=lse, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _, ref_bs, e = O.index_score_topk(q_idx, w, *ref["i"], bt, rr, rl, 4)
    assert e == 0
    check_block_scores(bs.cpu().numpy(), ref_bs, [0])
    gids = ids.cpu().numpy()
    o_ref, lse_ref, e = O.sparse_attention(q, 1, *ref["k"], *ref["v"], bt, rr, rl, gids, SM_SCALE)
    assert e == 0
    assert attention_rel_err(bf16_np(out), o_ref, [0]) <= ATTN_RTOL
    np.testing.assert_allclose(lse.cpu().numpy(), lse_ref, rtol=1e-4, atol=1e-4)


def test_mx_skewed_full_size_sampled_rows(lib):
    """The skewed batch (1 x 450K + 7 x 150K) with MXFP4 index and K/V planes, in
    the bench's launch configuration, checked on the first and last request's rows."""
    wl = W.make("skewed")
    s = wl.spec
    dev = DeviceCache(wl, mx_kv=True, mx_index=True)
    dev.store_all()
    row_req, row_len, ids, bscores, out, lse = dev.step(False)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    reqs = (0, 7)
    ref = OracleCache(wl, requests=reqs, mx_kv=True, mx_index=True)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, s.rows)
    rows = sorted({int(wl.cu_q[b]) for b in reqs})
    _, ref_bs, err = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl,
                                        s.topk, rows=rows)
    assert err == 0
    gbs = bscores.cpu().numpy()
    check_block_scores(gbs, ref_bs, rows)
    gids = ids.cpu().numpy()
    check_topk(gids, ref_bs, s.topk, rows, gbs)
    o_ref, lse_ref, err = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs,
                                             wl.block_table, rr, rl, gids, SM_SCALE, rows=rows)
    assert err == 0
    assert attention_rel_err(bf16_np(out), o_ref, rows) <= ATTN_RTOL
