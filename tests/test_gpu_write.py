"""GPU parity of quantise-at-write (m3s_qk_norm_rope_store) against the oracle:
"[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (#2744), Follow-up:
MXFP4 caches -- the quantisation inside the kernel that normalises, rotates and
writes the step's rows. Planes and BF16 outputs must be bit-exact."""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import bf16_dev, i64

pytestmark = pytest.mark.gpu


def _tables(T, half, pos0=7):
    t = (pos0 + np.arange(T))[:, None] * (10000.0 ** (-np.arange(half) / half))[None, :]
    return np.cos(t).astype(np.float32), np.sin(t).astype(np.float32)


def _case(seed, T, P, rd, mx_kv, mx_idx, eps=1e-6):
    """Q (16 heads, out), K (2 heads, plane), V (2 heads, plane, no norm / rope),
    index-Q (16 heads, out, rope only), index-K (1 head, plane) in one launch."""
    rng = np.random.default_rng(seed)
    src = {n: W.bf16_tensor(seed, n, (T, h, 128), 3, 10.0)
           for n, h in (("q", 16), ("k", 2), ("v", 2), ("iq", 16), ("ik", 1))}
    wts = {n: (rng.random(128) + 0.5).astype(np.float32) for n in ("q", "k", "ik")}
    cos, sin = _tables(T, rd // 2)
    slots = rng.permutation(P * 128)[:T].astype(np.int64)
    if T > 5:
        slots[5] = -1
    spec = [("q", wts["q"], True, None), ("k", wts["k"], True, mx_kv), ("v", None, False, mx_kv),
            ("iq", None, True, None), ("ik", wts["ik"], True, mx_idx)]
    # oracle
    ref_jobs, ref_dst = [], {}
    for n, w, rope, mx in spec:
        if mx is None:
            ref_dst[n] = np.zeros((T, src[n].shape[1], 128), dtype=np.uint16)
        else:
            ref_dst[n] = O.new_planes(P, src[n].shape[1], mx=mx)
        ref_jobs.append((src[n], w, rope, ref_dst[n]))
    assert O.qk_norm_rope_store(ref_jobs, slots, cos, sin, rd, eps) == 0
    # device
    dev_jobs, dev_dst = [], {}
    for n, w, rope, mx in spec:
        if mx is None:
            dev_dst[n] = torch.zeros((T, src[n].shape[1], 128), dtype=torch.bfloat16, device="cuda")
        else:
            dev_dst[n] = M.new_plane(P, src[n].shape[1], mx=mx)
        dev_jobs.append((bf16_dev(src[n]), None if w is None else torch.from_numpy(w).cuda(), rope,
                         dev_dst[n]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.m3s_qk_norm_rope_store(dev_jobs, i64(slots), torch.from_numpy(cos).cuda(),
                             torch.from_numpy(sin).cuda(), rd, eps, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return ref_dst, dev_dst, (src, wts, cos, sin, slots, dev_jobs)


@pytest.mark.parametrize("rd", [64, 128, 8])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mixed"])
def test_quantise_at_write_bit_exact(lib, rd, fmt):
    mx_kv = fmt == "mxfp4"
    mx_idx = fmt in ("mxfp4", "mixed")
    ref, dev, _ = _case(31 + rd, 300, 4, rd, mx_kv, mx_idx)
    for n in ref:
        if isinstance(ref[n], tuple):
            assert np.array_equal(dev[n][0].cpu().numpy(), ref[n][0]), n
            assert np.array_equal(dev[n][1].cpu().numpy(), ref[n][1]), n
        else:
            got = dev[n].view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got, ref[n]), n


def test_fused_write_equals_staging_then_store(lib):
    """On the device: the fused write's planes equal the unfused path's (the same
    call writing BF16 staging rows, then m3s_nvfp4_store)."""
    ref, dev, (src, wts, cos, sin, slots, _) = _case(5, 200, 3, 64, False, True)
    cos_d, sin_d = torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda()
    for n, mx in (("k", False), ("ik", True)):
        staging = torch.zeros((200, src[n].shape[1], 128), dtype=torch.bfloat16, device="cuda")
        M.m3s_qk_norm_rope_store([(bf16_dev(src[n]), torch.from_numpy(wts[n]).cuda(), True, staging)],
                                 None, cos_d, sin_d, 64, 1e-6)
        c, s = M.new_plane(3, src[n].shape[1], mx=mx)
        M.m3s_nvfp4_store(staging, i64(slots), c, s)
        torch.cuda.synchronize()
        assert torch.equal(c, dev[n][0]) and torch.equal(s, dev[n][1]), n


def test_quantise_at_write_bad_slot_reported(lib):
    T, P = 40, 1
    src = W.bf16_tensor(2, "bk", (T, 1, 128), 0, 1.0)
    slots = np.arange(T, dtype=np.int64)
    slots[9] = P * 128 + 3
    c, s = M.new_plane(P, 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.m3s_qk_norm_rope_store([(bf16_dev(src), None, False, (c, s))], i64(slots), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == M.DEVERR_SLOT
    rc, rs = O.new_planes(P, 1)
    keep = slots < P * 128
    O.nvfp4_store(src[keep], slots[keep], rc, rs)
    assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_fused_planes_checked_without_the_kernels_reduction_order(lib, fmt):
    """The check of the fused write that does not lean on the oracle restating the
    kernel's float32 steps: (1) the same call in its BF16-rows mode gives the rows
    the kernel quantises, and the oracle's own store of those rows equals the fused
    planes bit for bit; (2) those rows lie within BF16 rounding (plus a float32
    allowance) of the unrounded fp64 RMSNorm and rotation, and almost all of them
    are exactly the fp64 value rounded to BF16."""
    mx = fmt == "mxfp4"
    T, P, rd, eps = 300, 4, 64, 1e-6
    ref, dev, (src, wts, cos, sin, slots, _) = _case(71, T, P, rd, mx, mx)
    cos_d, sin_d = torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda()
    for n, w, rope in (("k", wts["k"], True), ("v", None, False), ("ik", wts["ik"], True)):
        H = src[n].shape[1]
        rows = torch.zeros((T, H, 128), dtype=torch.bfloat16, device="cuda")
        M.m3s_qk_norm_rope_store([(bf16_dev(src[n]), None if w is None else torch.from_numpy(w).cuda(),
                                   rope, rows)], None, cos_d, sin_d, rd, eps)
        torch.cuda.synchronize()
        gpu_rows = rows.view(torch.int16).cpu().numpy().view(np.uint16)
        c, sc = O.new_planes(P, H, mx=mx)
        assert O.nvfp4_store(gpu_rows, slots, c, sc) == 0
        assert np.array_equal(dev[n][0].cpu().numpy(), c), n
        assert np.array_equal(dev[n][1].cpu().numpy(), sc), n
        exact = O.norm_rope_rows_f64(src[n], w, cos if rope else None, sin if rope else None, rd, eps)
        # float32 allowance: relative to the terms each output is made of
        y = O.norm_rope_rows_f64(src[n], w, None, None, rd, eps)
        mag = np.abs(y).copy()
        if rope:
            h = rd // 2
            c32, s32 = np.abs(cos[:, None, :h].astype(np.float64)), np.abs(sin[:, None, :h].astype(np.float64))
            mag[..., :h] = np.abs(y[..., :h]) * c32 + np.abs(y[..., h:rd]) * s32
            mag[..., h:rd] = np.abs(y[..., h:rd]) * c32 + np.abs(y[..., :h]) * s32
        got = O.bf16_to_f64(gpu_rows)
        assert np.all(np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact) + 2.0 ** -16 * mag), n
        nearest = O.f32_to_bf16_bits(exact.astype(np.float32))
        same = float(np.mean(nearest == gpu_rows))
        assert same >= 0.99, (n, same)
