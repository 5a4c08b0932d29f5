"""Thin ctypes binding of libm3s (argument marshalling only).

The functions carry the C-ABI names and call straight into the CUDA library;
every step of the computation runs in its kernels. Torch is used for device
memory and streams: tensors are passed by ``data_ptr()``, the stream is
``torch.cuda.current_stream()`` unless given. Missing outputs are allocated
with torch on the inputs' device. A nonzero status raises ``M3SError``;
loading fails loudly when the library has not been built.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_LAUNCH = 0, 1, 2, 3, 4
STATUS = {1: "M3S_ERR_INVALID", 2: "M3S_ERR_UNSUPPORTED", 3: "M3S_ERR_WORKSPACE",
          4: "M3S_ERR_LAUNCH"}
DEVERR_SLOT, DEVERR_BLOCK_ID, DEVERR_PAGE, DEVERR_ROW, DEVERR_QRANGE, DEVERR_TIMEOUT = \
    1, 2, 4, 8, 16, 32
OP_INDEX_SCORE_TOPK, OP_VERIFY_SCORE_TOPK, OP_SPARSE_ATTENTION, OP_INDEX_CANDIDATES = 1, 2, 3, 4
OP_INDEX_ATTENTION = 5
OP_VERIFY_INDEX_ATTENTION = 6
FMT_NVFP4, FMT_MXFP4 = 0, 1
HEAD_DIM = PAGE = 128


class M3SError(RuntimeError):
    pass


class Plane(ctypes.Structure):
    """m3s_fp4_plane: codes [P, H, 128, 64] and scales [P, H, 128, 8] (NVFP4) or
    [P, H, 128, 4] (MXFP4), uint8 device tensors; ``format`` is FMT_*."""

    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("format", ctypes.c_int32)]


class StoreJob(ctypes.Structure):
    """m3s_store_job: one tensor of a batched store."""

    _fields_ = [("src", ctypes.c_void_p), ("src_row_stride", ctypes.c_int64),
                ("H", ctypes.c_int32), ("dst", Plane)]


class WriteJob(ctypes.Structure):
    """m3s_write_job: one tensor of a quantise-at-write launch."""

    _fields_ = [("src", ctypes.c_void_p), ("src_row_stride", ctypes.c_int64),
                ("H", ctypes.c_int32), ("norm_weight", ctypes.c_void_p), ("rope", ctypes.c_int32),
                ("dst", Plane), ("out", ctypes.c_void_p), ("out_row_stride", ctypes.c_int64)]


_P, _I32, _I64, _F32, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
_SIGS = {
    "m3s_workspace_bytes": (_SZ, [ctypes.c_int, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "m3s_nvfp4_store": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, Plane, _P, _P]),
    "m3s_nvfp4_store_batch": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P]),
    "m3s_decode_rows": (ctypes.c_int, [_P, _P, _I32, _I32, _P, _P, _P]),
    "m3s_qk_norm_rope_store": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _I32, _F32, _P, _P]),
    "m3s_index_score_topk": (ctypes.c_int, [_P, _P, _I32, Plane, _P, _I32, _P, _P, _I32, _I32,
                                            _I32, _I32, _I32, _P, _P, _P, _SZ, _P, _P]),
    "m3s_index_score_topk_static": (ctypes.c_int, [_P, _P, _I32, Plane, _P, _I32, _P, _P, _I32,
                                                   _I32, _I32, _P, _P, _P]),
    "m3s_index_block_scores": (ctypes.c_int, [_P, _P, _I32, Plane, _P, _I32, _P, _P, _I32, _I32,
                                              _P, _I32, _P, _P]),
    "m3s_block_topk": (ctypes.c_int, [_P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P,
                                      _P]),
    "m3s_verify_score_topk": (ctypes.c_int, [_P, _P, _I32, Plane, _P, _I32, _P, _P, _I32, _I32,
                                             _I32, _I32, _I32, _I32, _P, _P, _SZ, _P, _P]),
    "m3s_sparse_attention": (ctypes.c_int, [_P, _I32, _I32, Plane, Plane, _P, _I32, _I32, _P, _P,
                                            _P, _I32, _I32, _F32, _P, _P, _P, _SZ, _P, _P]),
    "m3s_index_score_candidates": (ctypes.c_int, [_P, _P, _I32, Plane, _P, _I32, _P, _P, _P, _P, _I32,
                                                  _I32, _I32, _I32, _I32, _P, _P, _SZ, _P, _P]),
    "m3s_merge_candidates": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P]),
    "m3s_index_attention": (ctypes.c_int, [_P, _P, _I32, Plane, _P, _I32, _I32, Plane, Plane, _P, _I32,
                                           _I32, _P, _P, _I32, _I32, _I32, _I32, ctypes.c_float, _P, _P,
                                           _P, _P, _SZ, _P, _P]),
    "m3s_verify_index_attention": (ctypes.c_int, [_P, _P, _I32, Plane, _P, _I32, _I32, Plane, Plane, _P,
                                                  _I32, _I32, _P, _P, _P, _I32, _I32, _I32, _I32, _I32,
                                                  ctypes.c_float, _P, _P, _P, _P, _SZ, _P, _P]),
    "m3s_nvfp4_store_batch_rows": (ctypes.c_int, [ctypes.c_void_p, _I32, _I32, _P, _P, _P, _I32, _I32, _P,
                                                  _P, _P, _P]),
    "m3s_version": (ctypes.c_char_p, []),
}

_lib = None


def load(build_if_stale: bool = True) -> ctypes.CDLL:
    """Load libm3s.so (building it first when its sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_stale and _build.stale():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise M3SError(f"libm3s.so is missing ({_build.LIB}); run build() first")
    lib = ctypes.CDLL(_build.LIB)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int, name: str) -> None:
    if rc != OK:
        raise M3SError(f"{name} returned {STATUS.get(rc, rc)}")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def plane(codes: torch.Tensor, scales: torch.Tensor) -> Plane:
    """The C plane of a (codes, scales) pair; its format follows the scale records'
    width (8 bytes: NVFP4, 4 bytes: MXFP4)."""
    cs, ss = codes.shape, scales.shape
    if (codes.dtype is not torch.uint8 or scales.dtype is not torch.uint8 or len(cs) != 4 or len(ss) != 4
            or cs[2] != PAGE or cs[3] != HEAD_DIM // 2 or ss[0] != cs[0] or ss[1] != cs[1] or ss[2] != PAGE
            or (ss[3] != HEAD_DIM // 16 and ss[3] != HEAD_DIM // 32)
            or not codes.is_contiguous() or not scales.is_contiguous()):
        raise TypeError("a plane is contiguous uint8 codes [P, H, 128, 64] and scales [P, H, 128, 8] "
                        "(NVFP4) or [P, H, 128, 4] (MXFP4)")
    return Plane(codes.data_ptr(), scales.data_ptr(), cs[0], cs[1],
                 FMT_MXFP4 if ss[3] == HEAD_DIM // 32 else FMT_NVFP4)


def new_plane(num_pages: int, heads: int, device="cuda", mx: bool = False
              ) -> tuple[torch.Tensor, torch.Tensor]:
    """Zeroed planes: codes [P, H, 128, 64], scales [P, H, 128, 8] (or 4 with ``mx``)."""
    return (torch.zeros((num_pages, heads, PAGE, HEAD_DIM // 2), dtype=torch.uint8, device=device),
            torch.zeros((num_pages, heads, PAGE, HEAD_DIM // (32 if mx else 16)), dtype=torch.uint8,
                        device=device))


def m3s_workspace_bytes(op: int, R: int, B: int, max_blocks: int, Hq: int = 0, Hkv: int = 0,
                        Hi: int = 0, topk: int = 0, max_q: int = 1) -> int:
    return int(load().m3s_workspace_bytes(op, R, B, max_blocks, Hq, Hkv, Hi, topk, max_q))


def m3s_nvfp4_store(src: torch.Tensor, slot_mapping: torch.Tensor, codes: torch.Tensor,
                    scales: torch.Tensor, err: torch.Tensor | None = None, stream=None) -> None:
    """src bf16 [T, H, 128] (rows may be strided), slot_mapping int64 [T]."""
    if slot_mapping.dtype is not torch.int64:
        raise TypeError("slot_mapping must be int64")
    T = src.shape[0] if src.dim() == 3 else -1
    job = _store_job(src, T, codes, scales)
    rc = load().m3s_nvfp4_store(_ptr(src), src.stride(0), T, src.shape[1], _ptr(slot_mapping),
                                job.dst, _ptr(err), _stream(stream))
    _check(rc, "m3s_nvfp4_store")


def _store_job(src: torch.Tensor, T: int, codes: torch.Tensor, scales: torch.Tensor) -> StoreJob:
    """One job of the batched stores: src bf16 [T, H, 128] (rows may be strided)."""
    sh = src.shape
    if (src.dtype is not torch.bfloat16 or len(sh) != 3 or sh[0] != T or sh[2] != HEAD_DIM
            or src.stride(2) != 1 or (sh[1] != 1 and src.stride(1) != HEAD_DIM)):
        raise TypeError("a store job's rows are bfloat16 [T, H, 128] with unit element and head strides")
    return StoreJob(src.data_ptr(), src.stride(0), sh[1], plane(codes, scales))


def m3s_nvfp4_store_batch(jobs, slot_mapping: torch.Tensor, err: torch.Tensor | None = None,
                          stream=None) -> None:
    """jobs: sequence of (src bf16 [T, H, 128], codes, scales) sharing ``slot_mapping``."""
    if slot_mapping.dtype is not torch.int64:
        raise TypeError("slot_mapping must be int64")
    arr = (StoreJob * max(1, len(jobs)))()
    T = slot_mapping.shape[0]
    for i, (src, codes, scales) in enumerate(jobs):
        arr[i] = _store_job(src, T, codes, scales)
    rc = load().m3s_nvfp4_store_batch(arr, len(jobs), T, _ptr(slot_mapping), _ptr(err),
                                      _stream(stream))
    _check(rc, "m3s_nvfp4_store_batch")


def m3s_nvfp4_store_batch_rows(jobs, slot_mapping: torch.Tensor, cu_q: torch.Tensor, seq_len: torch.Tensor,
                               R: int, row_req=None, row_len=None, err=None, stream=None):
    """m3s_nvfp4_store_batch and m3s_decode_rows in one launch; returns (row_req, row_len)."""
    if slot_mapping.dtype is not torch.int64:
        raise TypeError("slot_mapping must be int64")
    arr = (StoreJob * max(1, len(jobs)))()
    T = slot_mapping.shape[0]
    for i, (src, codes, scales) in enumerate(jobs):
        arr[i] = _store_job(src, T, codes, scales)
    for t in (cu_q, seq_len):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise TypeError("cu_q and seq_len must be contiguous int32 tensors")
    dev = cu_q.device
    if row_req is None:
        row_req = torch.empty(R, dtype=torch.int32, device=dev)
    if row_len is None:
        row_len = torch.empty(R, dtype=torch.int32, device=dev)
    rc = load().m3s_nvfp4_store_batch_rows(arr, len(jobs), T, _ptr(slot_mapping), _ptr(cu_q), _ptr(seq_len),
                                           seq_len.shape[0], R, _ptr(row_req), _ptr(row_len), _ptr(err),
                                           _stream(stream))
    _check(rc, "m3s_nvfp4_store_batch_rows")
    return row_req, row_len


def m3s_qk_norm_rope_store(jobs, slot_mapping, rope_cos=None, rope_sin=None, rotary_dim: int = 0,
                           eps: float = 1e-6, err=None, stream=None) -> None:
    """Quantise-at-write. jobs: sequence of (src bf16 [T, H, 128], norm_weight fp32 [128] or
    None, rope: bool, destination) with the destination either a (codes, scales) plane pair
    or a bf16 tensor [T, H, 128] for the normalised rows."""
    arr = (WriteJob * max(1, len(jobs)))()
    T = None
    for i, (src, weight, rope, dst) in enumerate(jobs):
        if src.dtype != torch.bfloat16 or src.dim() != 3 or src.stride(2) != 1:
            raise TypeError("src must be bfloat16 [T, H, 128] with unit element stride")
        if weight is not None and (weight.dtype != torch.float32 or not weight.is_contiguous()):
            raise TypeError("norm_weight must be a contiguous float32 [128] tensor")
        T = src.shape[0] if T is None else T
        if src.shape[0] != T or (src.shape[1] != 1 and src.stride(1) != HEAD_DIM):
            raise TypeError("every job has T rows of [H, 128] with unit head stride")
        if isinstance(dst, torch.Tensor):
            if dst.dtype is not torch.bfloat16 or dst.shape != src.shape or dst.stride(2) != 1:
                raise TypeError("a BF16 destination has the source's shape and unit element stride")
            arr[i] = WriteJob(src.data_ptr(), src.stride(0), src.shape[1], _ptr(weight), int(rope),
                              Plane(), dst.data_ptr(), dst.stride(0))
        else:
            arr[i] = WriteJob(src.data_ptr(), src.stride(0), src.shape[1], _ptr(weight), int(rope),
                              plane(*dst), None, 0)
    for t in (rope_cos, rope_sin):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise TypeError("rope_cos / rope_sin must be contiguous float32 [T, rotary_dim / 2]")
    if slot_mapping is not None and slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    rc = load().m3s_qk_norm_rope_store(arr, len(jobs), 0 if T is None else T, _ptr(slot_mapping),
                                       _ptr(rope_cos), _ptr(rope_sin), rotary_dim, float(eps),
                                       _ptr(err), _stream(stream))
    _check(rc, "m3s_qk_norm_rope_store")


def m3s_decode_rows(cu_q: torch.Tensor, seq_len: torch.Tensor, R: int,
                    row_req: torch.Tensor | None = None, row_len: torch.Tensor | None = None,
                    stream=None):
    B = seq_len.shape[0]
    dev = cu_q.device
    if row_req is None:
        row_req = torch.empty(R, dtype=torch.int32, device=dev)
    if row_len is None:
        row_len = torch.empty(R, dtype=torch.int32, device=dev)
    rc = load().m3s_decode_rows(_ptr(cu_q), _ptr(seq_len), B, R, _ptr(row_req), _ptr(row_len),
                                _stream(stream))
    _check(rc, "m3s_decode_rows")
    return row_req, row_len


def _index_inputs(q_idx, w, block_table, *int32s):
    """The dtypes the C calls assume for the index-scoring tensors (they pass raw
    pointers: a float64 weight tensor would be read as fp32 pairs)."""
    if q_idx.dtype != torch.bfloat16 or not q_idx.is_contiguous():
        raise TypeError("q_idx must be a contiguous bfloat16 tensor [R, Hi, 128]")
    if w.dtype != torch.float32 or not w.is_contiguous() or tuple(w.shape) != tuple(q_idx.shape[:2]):
        raise TypeError("w must be a contiguous float32 tensor [R, Hi]")
    for t in (block_table,) + int32s:
        if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
            raise TypeError("block tables, row maps and cu_q must be contiguous int32 tensors")


def m3s_index_score_topk(q_idx, w, codes, scales, block_table, row_req, row_len, topk: int,
                         topk_ids=None, block_scores=None, ws=None, err=None, stream=None,
                         init_blocks: int = 0, local_blocks: int = 0):
    _index_inputs(q_idx, w, block_table, row_req, row_len)
    R, Hi = q_idx.shape[0], q_idx.shape[1]
    B, bt_stride = block_table.shape
    if topk_ids is None:
        topk_ids = torch.empty((R, topk), dtype=torch.int32, device=q_idx.device)
    if ws is None:   # zeroed once, as the call requires (each call leaves it so)
        nb = m3s_workspace_bytes(OP_INDEX_SCORE_TOPK, R, B, bt_stride, 0, 0, Hi, topk)
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=q_idx.device)
    rc = load().m3s_index_score_topk(
        _ptr(q_idx), _ptr(w), Hi, plane(codes, scales), _ptr(block_table), bt_stride,
        _ptr(row_req), _ptr(row_len), R, B, topk, init_blocks, local_blocks, _ptr(topk_ids),
        _ptr(block_scores), _ptr(ws), ws.numel() * ws.element_size(),
        _ptr(err), _stream(stream))
    _check(rc, "m3s_index_score_topk")
    return topk_ids


def m3s_index_score_topk_static(q_idx, w, codes, scales, block_table, row_req, row_len, topk: int,
                                topk_ids=None, err=None, stream=None):
    _index_inputs(q_idx, w, block_table, row_req, row_len)
    R, Hi = q_idx.shape[0], q_idx.shape[1]
    B, bt_stride = block_table.shape
    if topk_ids is None:
        topk_ids = torch.empty((R, topk), dtype=torch.int32, device=q_idx.device)
    rc = load().m3s_index_score_topk_static(
        _ptr(q_idx), _ptr(w), Hi, plane(codes, scales), _ptr(block_table), bt_stride,
        _ptr(row_req), _ptr(row_len), R, B, topk, _ptr(topk_ids), _ptr(err), _stream(stream))
    _check(rc, "m3s_index_score_topk_static")
    return topk_ids


def m3s_index_block_scores(q_idx, w, codes, scales, block_table, row_req, row_len, block_scores,
                           err=None, stream=None):
    _index_inputs(q_idx, w, block_table, row_req, row_len)
    if block_scores.dtype != torch.float32:
        raise TypeError("block_scores must be float32")
    R, Hi = q_idx.shape[0], q_idx.shape[1]
    B, bt_stride = block_table.shape
    rc = load().m3s_index_block_scores(
        _ptr(q_idx), _ptr(w), Hi, plane(codes, scales), _ptr(block_table), bt_stride,
        _ptr(row_req), _ptr(row_len), R, B, _ptr(block_scores), block_scores.shape[1], _ptr(err),
        _stream(stream))
    _check(rc, "m3s_index_block_scores")
    return block_scores


def m3s_block_topk(block_scores, row_req, row_len, B: int, bt_stride: int, topk: int,
                   topk_ids=None, stream=None, init_blocks: int = 0, local_blocks: int = 0):
    R = row_len.shape[0]
    if topk_ids is None:
        topk_ids = torch.empty((R, topk), dtype=torch.int32, device=row_len.device)
    rc = load().m3s_block_topk(_ptr(block_scores), block_scores.shape[1], _ptr(row_req),
                               _ptr(row_len), R, B, bt_stride, topk, init_blocks, local_blocks,
                               _ptr(topk_ids), _stream(stream))
    _check(rc, "m3s_block_topk")
    return topk_ids


def m3s_verify_score_topk(q_idx, w, codes, scales, block_table, cu_q, row_len, max_q: int,
                          topk: int, topk_ids=None, ws=None, err=None, stream=None,
                          init_blocks: int = 0, local_blocks: int = 0):
    _index_inputs(q_idx, w, block_table, cu_q, row_len)
    R, Hi = q_idx.shape[0], q_idx.shape[1]
    B, bt_stride = block_table.shape
    if topk_ids is None:
        topk_ids = torch.empty((R, topk), dtype=torch.int32, device=q_idx.device)
    if ws is None:   # zeroed once, as the call requires (each call leaves it so)
        nb = m3s_workspace_bytes(OP_VERIFY_SCORE_TOPK, R, B, bt_stride, 0, 0, Hi, topk, max_q)
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=q_idx.device)
    rc = load().m3s_verify_score_topk(
        _ptr(q_idx), _ptr(w), Hi, plane(codes, scales), _ptr(block_table), bt_stride, _ptr(cu_q),
        _ptr(row_len), B, R, max_q, topk, init_blocks, local_blocks, _ptr(topk_ids), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(err), _stream(stream))
    _check(rc, "m3s_verify_score_topk")
    return topk_ids


def m3s_sparse_attention(q, hkv: int, k_codes, k_scales, v_codes, v_scales, block_table, row_req,
                         row_len, topk_ids, sm_scale: float | None = None, out=None, lse=None,
                         ws=None, err=None, stream=None):
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise TypeError("q must be a contiguous bfloat16 tensor [R, Hq, 128]")
    for t in (block_table, row_req, row_len, topk_ids):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise TypeError("block tables, row maps and top-k ids must be contiguous int32 tensors")
    R, Hq = q.shape[0], q.shape[1]
    B, bt_stride = block_table.shape
    topk = topk_ids.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        nb = m3s_workspace_bytes(OP_SPARSE_ATTENTION, R, B, bt_stride, Hq, hkv, 0, topk)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=q.device)
    rc = load().m3s_sparse_attention(
        _ptr(q), Hq, hkv, plane(k_codes, k_scales), plane(v_codes, v_scales), _ptr(block_table),
        bt_stride, B, _ptr(row_req), _ptr(row_len), _ptr(topk_ids), topk, R, float(sm_scale),
        _ptr(out), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(), _ptr(err),
        _stream(stream))
    _check(rc, "m3s_sparse_attention")
    return out


def m3s_index_score_candidates(q_idx, w, codes, scales, block_table, blk_begin, blk_count, row_req,
                               row_len, topk: int, cand_keys=None, ws=None, err=None, stream=None,
                               init_blocks: int = 0, local_blocks: int = 0):
    """A slice's candidate keys, int64 [R, topk] (the uint64 keys' bits)."""
    _index_inputs(q_idx, w, block_table, row_req, row_len, blk_begin, blk_count)
    R, Hi = q_idx.shape[0], q_idx.shape[1]
    B, bt_stride = block_table.shape
    if cand_keys is None:
        cand_keys = torch.empty((R, topk), dtype=torch.int64, device=q_idx.device)
    if cand_keys.dtype != torch.int64 or not cand_keys.is_contiguous():
        raise TypeError("cand_keys must be a contiguous int64 tensor [R, topk]")
    if ws is None:   # zeroed once, as the call requires (each call leaves it so)
        nb = m3s_workspace_bytes(OP_INDEX_CANDIDATES, R, B, bt_stride, 0, 0, Hi, topk)
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=q_idx.device)
    rc = load().m3s_index_score_candidates(
        _ptr(q_idx), _ptr(w), Hi, plane(codes, scales), _ptr(block_table), bt_stride, _ptr(blk_begin),
        _ptr(blk_count), _ptr(row_req), _ptr(row_len), R, B, topk, init_blocks, local_blocks,
        _ptr(cand_keys), _ptr(ws), ws.numel() * ws.element_size(), _ptr(err), _stream(stream))
    _check(rc, "m3s_index_score_candidates")
    return cand_keys


def m3s_merge_candidates(cand_keys, topk_ids=None, stream=None):
    """cand_keys int64 [n_lists, R, topk] -> topk_ids int32 [R, topk]."""
    if cand_keys.dtype != torch.int64 or cand_keys.dim() != 3 or not cand_keys.is_contiguous():
        raise TypeError("cand_keys must be a contiguous int64 tensor [n_lists, R, topk]")
    n, R, topk = cand_keys.shape
    if topk_ids is None:
        topk_ids = torch.empty((R, topk), dtype=torch.int32, device=cand_keys.device)
    rc = load().m3s_merge_candidates(_ptr(cand_keys), n, R, topk, _ptr(topk_ids), _stream(stream))
    _check(rc, "m3s_merge_candidates")
    return topk_ids


def m3s_index_attention(q_idx, w, idx_codes, idx_scales, q, hkv: int, k_codes, k_scales, v_codes,
                        v_scales, block_table, row_req, row_len, topk: int, sm_scale: float,
                        topk_ids=None, out=None, lse=None, ws=None, err=None, stream=None,
                        init_blocks: int = 0, local_blocks: int = 0):
    """Index scoring, top-k and attention of decode rows (two launches);
    returns (topk_ids int32 [R, topk], out bf16 [R, Hq, 128])."""
    _index_inputs(q_idx, w, block_table, row_req, row_len)
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise TypeError("q must be a contiguous bfloat16 tensor [R, Hq, 128]")
    R, Hi = q_idx.shape[0], q_idx.shape[1]
    Hq = q.shape[1]
    B, bt_stride = block_table.shape
    if topk_ids is None:
        topk_ids = torch.empty((R, topk), dtype=torch.int32, device=q.device)
    if out is None:
        out = torch.empty((R, Hq, 128), dtype=torch.bfloat16, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise TypeError("lse must be a contiguous float32 tensor [R, Hq]")
    if ws is None:
        nb = m3s_workspace_bytes(OP_INDEX_ATTENTION, R, B, bt_stride, Hq, hkv, Hi, topk)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=q.device)
    rc = load().m3s_index_attention(
        _ptr(q_idx), _ptr(w), Hi, plane(idx_codes, idx_scales), _ptr(q), Hq, hkv, plane(k_codes, k_scales),
        plane(v_codes, v_scales), _ptr(block_table), bt_stride, B, _ptr(row_req), _ptr(row_len), R, topk,
        init_blocks, local_blocks, sm_scale, _ptr(topk_ids), _ptr(out), _ptr(lse), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(err), _stream(stream))
    _check(rc, "m3s_index_attention")
    return topk_ids, out


def m3s_verify_index_attention(q_idx, w, idx_codes, idx_scales, q, hkv: int, k_codes, k_scales, v_codes,
                               v_scales, block_table, cu_q, row_req, row_len, max_q: int, topk: int,
                               sm_scale: float, topk_ids=None, out=None, lse=None, ws=None, err=None,
                               stream=None, init_blocks: int = 0, local_blocks: int = 0):
    """Verify scoring, top-k and attention of verify rows (two launches);
    returns (topk_ids int32 [R, topk], out bf16 [R, Hq, 128])."""
    _index_inputs(q_idx, w, block_table, cu_q, row_req, row_len)
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise TypeError("q must be a contiguous bfloat16 tensor [R, Hq, 128]")
    R, Hi = q_idx.shape[0], q_idx.shape[1]
    Hq = q.shape[1]
    B, bt_stride = block_table.shape
    if topk_ids is None:
        topk_ids = torch.empty((R, topk), dtype=torch.int32, device=q.device)
    if out is None:
        out = torch.empty((R, Hq, 128), dtype=torch.bfloat16, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise TypeError("lse must be a contiguous float32 tensor [R, Hq]")
    if ws is None:
        nb = m3s_workspace_bytes(OP_VERIFY_INDEX_ATTENTION, R, B, bt_stride, Hq, hkv, Hi, topk, max_q)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=q.device)
    rc = load().m3s_verify_index_attention(
        _ptr(q_idx), _ptr(w), Hi, plane(idx_codes, idx_scales), _ptr(q), Hq, hkv, plane(k_codes, k_scales),
        plane(v_codes, v_scales), _ptr(block_table), bt_stride, B, _ptr(cu_q), _ptr(row_req), _ptr(row_len), R,
        max_q, topk, init_blocks, local_blocks, sm_scale, _ptr(topk_ids), _ptr(out), _ptr(lse), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(err), _stream(stream))
    _check(rc, "m3s_verify_index_attention")
    return topk_ids, out
