"""Helpers shared by the GPU parity tests: run the step through the C ABI and
the oracle on the same seeded inputs, and compare with the acceptance rules."""

from __future__ import annotations

import math

import numpy as np
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O

SM_SCALE = 1.0 / math.sqrt(128)
SCORE_RTOL = 1e-4      # block scores, relative (acceptance rule)
TIE_BAND = 1e-5        # top-k: sets may differ only inside this band around the k-th score
ATTN_RTOL = 1e-2       # attention: max over (row, head) of |o - o_ref|_inf / |o_ref|_inf


def bf16_dev(bits: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def i32(x, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev)


def i64(x, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int64)).to(dev)


class DeviceCache:
    """The workload's paged K / V / index-K planes on the device, filled by the CUDA store.

    ``mx_kv`` / ``mx_index``: MXFP4 K/V or index planes (else NVFP4)."""

    def __init__(self, wl: W.Workload, dev="cuda", mx_kv: bool = False, mx_index: bool = False):
        s = wl.spec
        self.wl = wl
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.kc, self.ks = M.new_plane(wl.num_pages, s.hkv, dev, mx=mx_kv)
        self.vc, self.vs = M.new_plane(wl.num_pages, s.hkv, dev, mx=mx_kv)
        self.ic, self.is_ = M.new_plane(wl.num_pages, 1, dev, mx=mx_index)
        self.k_src = bf16_dev(wl.k_src, dev)
        self.v_src = bf16_dev(wl.v_src, dev)
        self.ik_src = bf16_dev(wl.ik_src, dev)
        self.slot_all = i64(wl.slot_all, dev)
        self.block_table = i32(wl.block_table, dev)
        self.seq_len = i32(wl.seq_len, dev)
        self.cu_q = i32(wl.cu_q, dev)
        self.q = bf16_dev(wl.q, dev)
        self.q_idx = bf16_dev(wl.q_idx, dev)
        self.w = torch.from_numpy(wl.w).to(dev)

    def store_all(self):
        for src, c, s in ((self.k_src, self.kc, self.ks), (self.v_src, self.vc, self.vs),
                          (self.ik_src, self.ic, self.is_)):
            M.m3s_nvfp4_store(src, self.slot_all, c, s, self.err)

    def step(self, fused_verify: bool):
        """Row map -> score + top-k (index or fused verify path) -> attention."""
        wl, s = self.wl, self.wl.spec
        R = s.rows
        row_req, row_len = M.m3s_decode_rows(self.cu_q, self.seq_len, R)
        if fused_verify:
            ids = M.m3s_verify_score_topk(self.q_idx, self.w, self.ic, self.is_, self.block_table,
                                          self.cu_q, row_len, max(s.q_rows), s.topk, err=self.err)
            bscores = None
        else:
            bscores = torch.full((R, wl.bt_stride), float("nan"), device=self.q.device)
            ids = M.m3s_index_score_topk(self.q_idx, self.w, self.ic, self.is_, self.block_table,
                                         row_req, row_len, s.topk, block_scores=bscores,
                                         err=self.err)
        lse = torch.empty((R, s.hq), dtype=torch.float32, device=self.q.device)
        out = M.m3s_sparse_attention(self.q, s.hkv, self.kc, self.ks, self.vc, self.vs,
                                     self.block_table, row_req, row_len, ids, SM_SCALE, lse=lse,
                                     err=self.err)
        return row_req, row_len, ids, bscores, out, lse


class OracleCache:
    """Oracle planes of the workload, quantised by the oracle (optionally only some requests)."""

    def __init__(self, wl: W.Workload, requests=None, mx_kv: bool = False, mx_index: bool = False):
        s = wl.spec
        self.wl = wl
        self.kc, self.ks = O.new_planes(wl.num_pages, s.hkv, mx=mx_kv)
        self.vc, self.vs = O.new_planes(wl.num_pages, s.hkv, mx=mx_kv)
        self.ic, self.is_ = O.new_planes(wl.num_pages, 1, mx=mx_index)
        if requests is None:
            tok = np.arange(wl.ntok)
        else:
            tok = np.concatenate([np.arange(wl.tok_off[b], wl.tok_off[b + 1]) for b in requests])
        slots = wl.slot_all[tok]
        for src, c, sc in ((wl.k_src, self.kc, self.ks), (wl.v_src, self.vc, self.vs),
                           (wl.ik_src, self.ic, self.is_)):
            assert O.nvfp4_store(src[tok], slots, c, sc) == 0


def check_block_scores(gpu: np.ndarray, ref: list, rows) -> float:
    """Relative error of the block scores (valid blocks only); asserts the 1e-4 rule."""
    worst = 0.0
    for r in rows:
        ref_r = ref[r]
        g = gpu[r, : len(ref_r)].astype(np.float64)
        floor = 1e-6 * max(1.0, float(np.abs(ref_r).max(initial=0.0)))
        rel = np.abs(g - ref_r) / np.maximum(np.abs(ref_r), floor)
        worst = max(worst, float(rel.max(initial=0.0)))
    assert worst <= SCORE_RTOL, f"block score relative error {worst:.3g} > {SCORE_RTOL}"
    return worst


def check_topk(gpu_ids: np.ndarray, ref_scores: list, topk: int, rows, gpu_scores=None) -> int:
    """Top-k sets equal the oracle's except inside the tie band around the k-th score.

    Also: ids ascending, -1 padded; with the GPU's own block scores given, the
    selection must be exactly their top-k with ties to the lower id.
    Returns the number of rows whose set differs from the oracle's (all in-band).
    """
    differing = 0
    for r in rows:
        sc = np.asarray(ref_scores[r], dtype=np.float64)
        nb = len(sc)
        ids = gpu_ids[r]
        cnt = min(topk, nb)
        assert (ids[cnt:] == -1).all(), (r, ids)
        sel = ids[:cnt]
        assert (np.diff(sel) > 0).all(), f"row {r}: ids not strictly ascending {sel}"
        if cnt == 0:
            continue
        assert sel.min() >= 0 and sel.max() < nb
        ref = O.topk_ids(sc, topk)[:cnt]
        if set(sel.tolist()) != set(ref.tolist()):
            differing += 1
            tau = np.sort(sc)[::-1][cnt - 1]
            band = TIE_BAND * max(abs(tau), 1e-30)
            above = set(np.nonzero(sc > tau + band)[0].tolist())
            inband = set(np.nonzero(np.abs(sc - tau) <= band)[0].tolist())
            s = set(sel.tolist())
            assert above <= s, f"row {r}: a block above the tie band is missing"
            assert s <= above | inband, f"row {r}: a block below the tie band was selected"
        if gpu_scores is not None:
            own = O.topk_ids(gpu_scores[r, :nb].astype(np.float64), topk)[:cnt]
            assert np.array_equal(own, sel), f"row {r}: not the top-k of the GPU's own scores"
    return differing


def attention_rel_err(out: np.ndarray, ref: np.ndarray, rows) -> float:
    worst = 0.0
    for r in rows:
        for h in range(ref.shape[1]):
            den = np.abs(ref[r, h]).max()
            num = np.abs(out[r, h].astype(np.float64) - ref[r, h]).max()
            if den == 0:
                assert num == 0, (r, h)
                continue
            worst = max(worst, num / den)
    return worst


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def check_topk_forced(gpu_ids: np.ndarray, ref_scores: list, topk: int, rows, init_blocks: int,
                      local_blocks: int) -> None:
    """Top-k with forced blocks: the forced part of the selection must be exactly
    the oracle's; the rest comes from the scored blocks under the tie-band rule."""
    for r in rows:
        sc = np.asarray(ref_scores[r], dtype=np.float64)
        nb = len(sc)
        cnt = min(topk, nb)
        ids = gpu_ids[r]
        assert (ids[cnt:] == -1).all(), (r, ids)
        sel = ids[:cnt]
        assert (np.diff(sel) > 0).all(), f"row {r}: ids not strictly ascending {sel}"
        blocks = np.arange(nb)
        forced = (blocks < init_blocks) | (blocks >= nb - local_blocks)
        # which forced blocks are kept does not depend on the scores at all
        kept_forced = set(O.topk_ids(np.zeros(nb), topk, init_blocks, local_blocks)[:cnt].tolist()) & \
            set(np.nonzero(forced)[0].tolist())
        assert set(sel.tolist()) & set(np.nonzero(forced)[0].tolist()) == kept_forced, (r, sel)
        # the scored remainder: the best of the unforced blocks, ties inside the band
        free = np.nonzero(~forced)[0]
        kk = cnt - len(kept_forced)
        rest = np.array(sorted(set(sel.tolist()) - kept_forced), dtype=np.int64)
        assert len(rest) == kk, (r, sel)
        if kk == 0:
            continue
        sub = sc[free]
        pos = {int(b): j for j, b in enumerate(free)}
        sub_ids = np.array([pos[int(b)] for b in rest], dtype=np.int32)
        fake = np.full((1, kk), -1, dtype=np.int32)
        fake[0, :] = np.sort(sub_ids)
        check_topk(fake, [sub], kk, [0])
