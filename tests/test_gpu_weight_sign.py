"""GPU parity with index-head weights of either sign.

The lightning indexer's token score is sum_h w_h * ReLU(q_h . k_t)
("[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (#2744), Design /
Index), with no sign placed on w_h. A head with a negative weight can only
lower a token's score, and a row whose weights are all negative has block
scores at or below zero. The workloads draw weights from (0, 1), so these
cases change the sign of two heads' weights in every row and of every weight
in row 0 (one sign per row there, so no cancellation blurs the comparison).
The block scores must match the oracle within the 1e-4 rule. The top-k ids of
every scorer path must be the oracle's outside the tie band. Each two-launch
entry must give the ids of its separate calls bit for bit.
"""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import SM_SCALE, DeviceCache, OracleCache, check_block_scores, check_topk

pytestmark = pytest.mark.gpu


def _signed_weights(w: np.ndarray) -> np.ndarray:
    w = w.copy()
    w[:, [1, 5]] *= -1.0
    w[0] = -np.abs(w[0])
    return w


CASES = [
    # (spec, contexts, rows per request, MXFP4 index plane)
    ("decode", (5000, 3000, 129, 700, 2000), (1, 1, 1, 1, 1), False),
    ("decode", (4000, 900, 2600), (1, 1, 1), True),
    ("verify", (2500, 1300, 999), (8, 3, 5), False),
    ("verify", (1800, 3100), (6, 8), True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{'mx' if c[3] else 'nv'}-{len(c[1])}req")
def test_signed_index_weights_vs_oracle(lib, case):
    name, ctx, qr, mx = case
    wl = W.make(name, ctx=ctx, q_rows=qr)
    s = wl.spec
    R, topk = s.rows, s.topk
    w = _signed_weights(wl.w)
    dev = DeviceCache(wl, mx_index=mx)
    dev.w = torch.from_numpy(w).to("cuda")
    dev.store_all()
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, R)

    ref = OracleCache(wl, mx_index=mx)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    _, ref_bs, err = O.index_score_topk(wl.q_idx, w, ref.ic, ref.is_, wl.block_table, rr, rl, topk)
    assert err == 0
    assert (ref_bs[0] <= 0).all() and any((b < 0).any() for b in ref_bs)

    bscores = torch.full((R, wl.bt_stride), float("nan"), device="cuda")
    M.m3s_index_block_scores(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, row_req, row_len, bscores,
                             dev.err)
    ids_i = M.m3s_index_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, row_req, row_len,
                                   topk, err=dev.err)
    ids_a, _ = M.m3s_index_attention(dev.q_idx, dev.w, dev.ic, dev.is_, dev.q, s.hkv, dev.kc, dev.ks, dev.vc,
                                     dev.vs, dev.block_table, row_req, row_len, topk, SM_SCALE, err=dev.err)
    max_q = max(qr)
    ids_v = M.m3s_verify_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table, dev.cu_q, row_len,
                                    max_q, topk, err=dev.err)
    ids_va, _ = M.m3s_verify_index_attention(dev.q_idx, dev.w, dev.ic, dev.is_, dev.q, s.hkv, dev.kc, dev.ks,
                                             dev.vc, dev.vs, dev.block_table, dev.cu_q, row_req, row_len, max_q,
                                             topk, SM_SCALE, err=dev.err)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0, f"device error bits {int(dev.err.item())}"

    gbs = bscores.cpu().numpy()
    check_block_scores(gbs, ref_bs, range(R))
    check_topk(ids_i.cpu().numpy(), ref_bs, topk, range(R), gbs)
    np.testing.assert_array_equal(ids_a.cpu().numpy(), ids_i.cpu().numpy())
    check_topk(ids_v.cpu().numpy(), ref_bs, topk, range(R))
    np.testing.assert_array_equal(ids_va.cpu().numpy(), ids_v.cpu().numpy())
