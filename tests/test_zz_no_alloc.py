"""m3s_index_score_topk_static (block-score scratch in a file-scope device array,
no caller workspace) against m3s_index_score_topk with a caller workspace.

This file is named to be collected last: the static variant's first call on a
device does its one-time set-up, and the test must pass both alone and after
every other test has used the library."""

import ctypes

import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W

STATIC_SCRATCH_FLOATS = (4 << 20) // 4


def test_static_variant_rejects_oversized_scratch_before_launch():
    """R x bt_stride block scores beyond the fixed scratch: M3S_ERR_WORKSPACE,
    decided on the host before any device call (runs without a GPU)."""
    try:
        lib = M.load()
    except Exception as e:  # no toolchain to build the library here
        pytest.skip(f"library unavailable: {e}")
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the call returns first
    plane = M.Plane(fake, fake, 8, 1)
    R, bt_stride = 4096, STATIC_SCRATCH_FLOATS // 4096 + 1
    rc = lib.m3s_index_score_topk_static(fake, fake, 16, plane, fake, bt_stride, fake, fake, R, 1,
                                         16, fake, None, None)
    assert rc == M.ERR_WORKSPACE
    # null outputs are still invalid arguments, not a workspace problem
    rc = lib.m3s_index_score_topk_static(fake, fake, 16, plane, fake, 8, fake, fake, 4, 1, 16,
                                         None, None, None)
    assert rc == M.ERR_INVALID


def _case(ctx):
    from step_helpers import DeviceCache
    wl = W.make("decode", ctx=ctx, q_rows=(1,) * len(ctx))
    dev = DeviceCache(wl)
    dev.store_all()
    R = wl.spec.rows
    row_req, row_len = M.m3s_decode_rows(dev.cu_q, dev.seq_len, R)
    return wl, dev, row_req, row_len


@pytest.mark.gpu
def test_static_variant_equals_workspace_variant_two_calls_in_a_row():
    """Two different batches back to back through the static variant (the second
    has fewer, shorter rows, so stale scores from the first would show) give the
    same ids as the caller-workspace entry point, bit for bit."""
    cases = [(40000, 129, 9000, 128 * 37, 70000, 300, 5000, 12345),
             (2000, 700, 128, 3000)]
    prepared = [_case(ctx) for ctx in cases]
    refs = []
    for wl, dev, row_req, row_len in prepared:
        refs.append(M.m3s_index_score_topk(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table,
                                           row_req, row_len, wl.spec.topk, err=dev.err))
    torch.cuda.synchronize()
    # the two static calls, back to back on one stream
    gots = [M.m3s_index_score_topk_static(dev.q_idx, dev.w, dev.ic, dev.is_, dev.block_table,
                                          row_req, row_len, wl.spec.topk, err=dev.err)
            for wl, dev, row_req, row_len in prepared]
    torch.cuda.synchronize()
    for (wl, dev, _, _), ref, got in zip(prepared, refs, gots):
        assert int(dev.err.item()) == 0, int(dev.err.item())
        assert torch.equal(ref.cpu(), got.cpu()), (ref, got)
    # the two batches really differ (the second call is not a replay of the first)
    assert refs[0].shape != refs[1].shape
