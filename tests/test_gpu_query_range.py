"""GPU parity over the whole BF16 query range.

The pages' inputs are BF16 rows ("NVFP4 sparse KV" (ROCm/ATOM #2746), Summary;
"[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (#2744), Design /
Index), whose range (2^-133 .. 2^128) is far wider than the f16 operands of
the tensor-core products. Every kernel scales each (row, head) of the queries
by a power of two before the conversion and undoes it exactly in fp32. These
cases put rows at 2^-126 .. 2^110, heads 2^120 apart inside one row, a head of
BF16 subnormals, and a head of zeros through both scorers and the attention,
against the fp64 oracle with the acceptance tolerances. Only inf / NaN may
raise the query-range error bit.
"""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import (ATTN_RTOL, SCORE_RTOL, SM_SCALE, DeviceCache, OracleCache,
                          attention_rel_err, bf16_np, check_topk)

pytestmark = pytest.mark.gpu

HI = 16
# per row: an exponent applied to every head, or a named per-head pattern
ROWS = [0, -20, -100, 20, 110, -126, "spread", "subnormal-head",
        60, -60, 100, -110, "alternate", 5, "zero-head", -5]


def _head_factors():
    """float64 [16 rows, 16 heads] powers of two (0 = the head is zeroed)."""
    f = np.ones((len(ROWS), HI))
    for r, p in enumerate(ROWS):
        if p == "spread":                       # heads 2^-60 .. 2^60, 2^120 apart end to end
            f[r] = 2.0 ** (-60 + 8 * np.arange(HI))
        elif p == "subnormal-head":            # head 3 replaced by BF16 subnormals (below)
            pass
        elif p == "alternate":                 # 2^-40 and 2^40 heads interleaved
            f[r] = np.where(np.arange(HI) % 2 == 0, 2.0 ** -40, 2.0 ** 40)
        elif p == "zero-head":                 # one head all zero (excluded from the row's scale)
            f[r, 5] = 0.0
        else:
            f[r] = 2.0 ** p
    return f


def _scale_bits(bits, f):
    """BF16 bits [R, H, 128] times per-(row, head) factors, rounded to BF16."""
    x = W.bf16_bits_to_f32(bits).astype(np.float64) * f[:, :, None]
    return W.f32_to_bf16_bits(x.astype(np.float32))


def _workload():
    wl = W.make("verify", ctx=(2500, 1300), q_rows=(8, 8))
    f = _head_factors()
    wl.q_idx = _scale_bits(wl.q_idx, f)
    wl.q = _scale_bits(wl.q, f)
    wl.w = wl.w.copy()
    # head 3 of that row: BF16 subnormals m * 2^-133 (m in 1 .. 127, random signs)
    r_sub = ROWS.index("subnormal-head")
    rng = np.random.default_rng(11)
    for arr in (wl.q_idx, wl.q):
        mant = rng.integers(1, 128, size=128).astype(np.uint16)
        arr[r_sub, 3] = mant | (rng.integers(0, 2, size=128).astype(np.uint16) << 15)
    keep = np.zeros(HI, dtype=bool)
    keep[3] = True
    wl.w[r_sub, ~keep] = 0.0                   # that row's score is the subnormal head's alone
    sub = W.bf16_bits_to_f32(wl.q_idx[r_sub, 3])
    assert np.all(np.abs(sub) < 2.0 ** -126) and np.all(sub != 0)
    return wl


def _check_scores_row_relative(gpu, ref, rows):
    """Block scores within 1e-4 of the oracle's, relative to each score with a
    floor of 1e-6 of its row's largest (so tiny rows are held to the same bar)."""
    worst = 0.0
    for r in rows:
        ref_r = np.asarray(ref[r], dtype=np.float64)
        g = gpu[r, : len(ref_r)].astype(np.float64)
        floor = 1e-6 * float(np.abs(ref_r).max(initial=0.0))
        den = np.maximum(np.abs(ref_r), floor)
        rel = np.where(den > 0, np.abs(g - ref_r) / np.where(den > 0, den, 1.0), np.abs(g))
        worst = max(worst, float(rel.max(initial=0.0)))
    assert worst <= SCORE_RTOL, f"block score relative error {worst:.3g}"
    return worst


def test_scorers_and_attention_over_the_bf16_query_range(lib):
    wl = _workload()
    s = wl.spec
    R = s.rows
    dev = DeviceCache(wl)
    dev.store_all()
    _, row_len, ids_i, bscores, out_i, lse_i = dev.step(False)
    _, _, ids_v, _, out_v, lse_v = dev.step(True)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0, f"device error bits {int(dev.err.item())}"

    ref = OracleCache(wl)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    _, ref_bs, e = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl, s.topk)
    assert e == 0
    gbs = bscores.cpu().numpy()
    _check_scores_row_relative(gbs, ref_bs, range(R))
    check_topk(ids_i.cpu().numpy(), ref_bs, s.topk, range(R), gbs)
    check_topk(ids_v.cpu().numpy(), ref_bs, s.topk, range(R))

    for ids, out, lse in ((ids_i, out_i, lse_i), (ids_v, out_v, lse_v)):
        gids = ids.cpu().numpy()
        o_ref, lse_ref, e = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs,
                                               wl.block_table, rr, rl, gids, SM_SCALE)
        assert e == 0
        err = attention_rel_err(bf16_np(out), o_ref, range(R))
        assert err <= ATTN_RTOL, err
        np.testing.assert_allclose(lse.cpu().numpy(), lse_ref, rtol=1e-4, atol=1e-4)


def test_big_rows_no_longer_flagged_only_inf_and_nan_are(lib):
    """A row at 2^100 (beyond f16's 65504) computes; an inf or NaN element raises
    M3S_DEVERR_QRANGE in each kernel that reads it, and nothing else does."""
    wl = W.make("verify", ctx=(900, 700), q_rows=(8, 8))
    f = np.ones((wl.spec.rows, HI))
    f[2] = 2.0 ** 100
    wl.q_idx = _scale_bits(wl.q_idx, f)
    wl.q = _scale_bits(wl.q, f)
    dev = DeviceCache(wl)
    dev.store_all()
    dev.step(False)
    dev.step(True)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0
    for bad_bits in (0x7F80, 0xFFC1):           # +inf, a NaN
        for which in ("q_idx-index", "q_idx-verify", "q"):
            wl2 = W.make("verify", ctx=(900, 700), q_rows=(8, 8))
            if which.startswith("q_idx"):
                wl2.q_idx[5, 7, 33] = bad_bits
            else:
                wl2.q[5, 7, 33] = bad_bits
            d2 = DeviceCache(wl2)
            d2.store_all()
            torch.cuda.synchronize()
            assert int(d2.err.item()) == 0
            if which == "q":
                R = wl2.spec.rows
                row_req, row_len = M.m3s_decode_rows(d2.cu_q, d2.seq_len, R)
                ids = torch.zeros((R, wl2.spec.topk), dtype=torch.int32, device="cuda")
                M.m3s_sparse_attention(d2.q, 1, d2.kc, d2.ks, d2.vc, d2.vs, d2.block_table, row_req,
                                       row_len, ids, SM_SCALE, err=d2.err)
            else:
                d2.step(which.endswith("verify"))
            torch.cuda.synchronize()
            assert int(d2.err.item()) & M.DEVERR_QRANGE, (which, hex(bad_bits))
