"""GPU parity of m3s_nvfp4_store_batch_rows: the batched store and the row map in
one launch ("NVFP4 sparse KV" (ROCm/ATOM #2746), Summary: the step's rows are
quantised into the pages; "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV
cache" (#2744), Design / Attention: the row map on device). The planes must equal
those of m3s_nvfp4_store_batch and the row map that of m3s_decode_rows, bit for
bit, and the row map the oracle's closed form."""

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import binding as M
from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O
from step_helpers import bf16_dev, i32, i64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [((3000, 129, 700), (1, 1, 1), 0),
                                   ((5000, 2000), (8, 5), 3),
                                   ((4096,), (1,), 300)],
                         ids=["decode", "verify_pad_rows", "many_pad_rows"])
@pytest.mark.parametrize("mx", [False, True], ids=["nvfp4", "mxfp4"])
def test_store_and_row_map_in_one_launch(lib, shape, mx):
    ctx, q_rows, pad = shape
    wl = W.make("decode", ctx=ctx, q_rows=q_rows)
    s = wl.spec
    R = s.rows + pad
    new = wl.new_tok
    slots = i64(wl.slot_all[new].copy())
    srcs = [bf16_dev(np.ascontiguousarray(x[new])) for x in (wl.k_src, wl.v_src, wl.ik_src)]
    heads = (s.hkv, s.hkv, 1)
    a = [M.new_plane(wl.num_pages, h, "cuda", mx=mx) for h in heads]
    b = [M.new_plane(wl.num_pages, h, "cuda", mx=mx) for h in heads]
    for (c, sc) in a + b:
        c.fill_(0x5A)
        sc.fill_(0x3C)
    cu_q, seq_len = i32(wl.cu_q), i32(wl.seq_len)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rr1, rl1 = M.m3s_nvfp4_store_batch_rows([(src, c, sc) for src, (c, sc) in zip(srcs, a)], slots, cu_q,
                                            seq_len, R, err=err)
    M.m3s_nvfp4_store_batch([(src, c, sc) for src, (c, sc) in zip(srcs, b)], slots, err)
    rr2, rl2 = M.m3s_decode_rows(cu_q, seq_len, R)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for (c1, s1), (c2, s2) in zip(a, b):
        assert torch.equal(c1, c2) and torch.equal(s1, s2)
    assert torch.equal(rr1, rr2) and torch.equal(rl1, rl2)
    ref_req, ref_len = O.decode_rows(wl.cu_q, wl.seq_len, R)
    np.testing.assert_array_equal(rr1.cpu().numpy(), ref_req)
    np.testing.assert_array_equal(rl1.cpu().numpy(), ref_len)


def test_row_map_alone_and_store_alone(lib):
    wl = W.make("decode", ctx=(900, 300), q_rows=(1, 1))
    cu_q, seq_len = i32(wl.cu_q), i32(wl.seq_len)
    rr, rl = M.m3s_nvfp4_store_batch_rows([], torch.zeros(0, dtype=torch.int64, device="cuda"), cu_q, seq_len, 5)
    torch.cuda.synchronize()
    ref_req, ref_len = O.decode_rows(wl.cu_q, wl.seq_len, 5)
    np.testing.assert_array_equal(rr.cpu().numpy(), ref_req)
    np.testing.assert_array_equal(rl.cpu().numpy(), ref_len)
