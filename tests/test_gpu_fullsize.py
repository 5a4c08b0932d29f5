"""GPU parity at the full sizes the benchmark times (decode bs8 x 32K, verify 16 x 8
rows on 64K-192K contexts, skewed 450K + 7 x 150K, prefill 8192 rows on 256K), in
the same launch configuration, checked on what the oracle can compute one by one:

* the row map of every row, bit-exact;
* the planes of the sampled requests (K, V and index-K of every one of their
  tokens, stored by the CUDA path), bit-exact at their slots;
* for the first and last row of each sampled request: block scores within 1e-4
  relative (index path), the top-k set (tie band 1e-5, ties to the lower id) and
  attention over the selected blocks within 1e-2;
* decode rows, the benchmark's step as it launches it: the batched store of the
  step's new rows with the row map in the same launch (the row map of every row
  bit-exact), then m3s_index_attention, whose ids, BF16 outputs and lse equal
  the separate calls' above on every row, bit for bit.

The oracle quantises only the sampled requests (its inputs are the workload's
own seeded BF16 rows, never the device's planes)."""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import (ATTN_RTOL, SM_SCALE, DeviceCache, OracleCache, attention_rel_err,
                          bf16_np, check_block_scores, check_topk)

pytestmark = pytest.mark.gpu

# workload, sampled requests (the longest and the last request where they differ)
FULL = [
    ("decode", (0, 7)),
    ("verify", (int(np.argmax(W.SPECS["verify"].ctx)), 15)),
    ("skewed", (0, 7)),
    ("prefill", (0,)),
]


def _gather(plane: torch.Tensor, pages: np.ndarray, offs: np.ndarray) -> np.ndarray:
    p = torch.from_numpy(pages).to(plane.device)
    o = torch.from_numpy(offs).to(plane.device)
    return plane[p, :, o].cpu().numpy()


@pytest.mark.parametrize("name,reqs", FULL, ids=[f[0] for f in FULL])
def test_full_size_sampled_rows(lib, name, reqs):
    wl = W.make(name)
    s = wl.spec
    fused = name in ("verify", "prefill")
    dev = DeviceCache(wl)
    dev.store_all()
    row_req, row_len, ids, bscores, out, lse = dev.step(fused)
    torch.cuda.synchronize()
    assert int(dev.err.item()) == 0, int(dev.err.item())
    R = s.rows

    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    assert np.array_equal(row_req.cpu().numpy(), rr)
    assert np.array_equal(row_len.cpu().numpy(), rl)

    ref = OracleCache(wl, requests=reqs)
    tok = np.concatenate([np.arange(wl.tok_off[b], wl.tok_off[b + 1]) for b in reqs])
    slots = wl.slot_all[tok]
    pages, offs = (slots // 128).astype(np.int64), (slots % 128).astype(np.int64)
    for dc, ds, rc, rs in ((dev.kc, dev.ks, ref.kc, ref.ks), (dev.vc, dev.vs, ref.vc, ref.vs),
                           (dev.ic, dev.is_, ref.ic, ref.is_)):
        assert np.array_equal(_gather(dc, pages, offs), rc[pages, :, offs])
        assert np.array_equal(_gather(ds, pages, offs), rs[pages, :, offs])

    rows = sorted({int(wl.cu_q[b]) for b in reqs} | {int(wl.cu_q[b + 1]) - 1 for b in reqs})
    _, ref_bs, err = O.index_score_topk(wl.q_idx, wl.w, ref.ic, ref.is_, wl.block_table, rr, rl,
                                        s.topk, rows=rows)
    assert err == 0
    gids = ids.cpu().numpy()
    gbs = None
    if bscores is not None:
        gbs = bscores.cpu().numpy()
        check_block_scores(gbs, ref_bs, rows)
    check_topk(gids, ref_bs, s.topk, rows, gbs)

    o_ref, lse_ref, err = O.sparse_attention(wl.q, s.hkv, ref.kc, ref.ks, ref.vc, ref.vs,
                                             wl.block_table, rr, rl, gids, SM_SCALE, rows=rows)
    assert err == 0
    e = attention_rel_err(bf16_np(out), o_ref, rows)
    assert e <= ATTN_RTOL, e
    got_lse = lse.cpu().numpy()
    np.testing.assert_allclose(got_lse[rows], lse_ref[rows], rtol=1e-4, atol=1e-4)

    if not fused:
        # the two-launch decode step: re-storing the step's new rows writes the
        # same bytes, so the planes checked above are unchanged
        new = torch.from_numpy(np.asarray(wl.new_tok, dtype=np.int64)).to(dev.kc.device)
        rr2, rl2 = M.m3s_nvfp4_store_batch_rows(
            [(dev.k_src[new].contiguous(), dev.kc, dev.ks), (dev.v_src[new].contiguous(), dev.vc, dev.vs),
             (dev.ik_src[new].contiguous(), dev.ic, dev.is_)],
            dev.slot_all[new].contiguous(), dev.cu_q, dev.seq_len, R, err=dev.err)
        lse2 = torch.full((R, s.hq), float("nan"), dtype=torch.float32, device=dev.kc.device)
        ids2, out2 = M.m3s_index_attention(dev.q_idx, dev.w, dev.ic, dev.is_, dev.q, s.hkv, dev.kc, dev.ks,
                                           dev.vc, dev.vs, dev.block_table, rr2, rl2, s.topk, SM_SCALE,
                                           lse=lse2, err=dev.err)
        torch.cuda.synchronize()
        assert int(dev.err.item()) == 0, int(dev.err.item())
        assert np.array_equal(rr2.cpu().numpy(), rr) and np.array_equal(rl2.cpu().numpy(), rl)
        assert np.array_equal(ids2.cpu().numpy(), gids)
        assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
        np.testing.assert_array_equal(lse2.cpu().numpy(), got_lse)
