"""Seeded synthetic inputs for the NVFP4 block-sparse decode/verify step.

This module only *draws* inputs: BF16 bit patterns, fp32 index weights, the
paged layout (block tables, slots) and the row grouping. It holds none of the
method's arithmetic (no quantisation, no scoring, no attention), so both the
CUDA path and the fp64 oracle consume exactly the same bits from it.

Random numbers come from a counter-based generator: SplitMix64 (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014)
evaluated at ``key + (i + 1) * GAMMA`` for element ``i`` of a named stream, so
any slice of any stream can be drawn independently and in parallel. Normal
variates use the Box-Muller transform (Box and Muller, 1958) on pairs of
53-bit uniforms; each pair yields two variates.

The workload shapes follow the five configurations of the NVFP4 sparse KV
work (MiniMax-M3.1 sparse layers): head_dim 128, 128-token pages, one KV head,
and the page/block tables of a paged KV pool. Where the pages name contexts
in "K" tokens, 1K = 1024 tokens (450K = 460,800 and 150K = 153,600, both whole
pages).
"""

from __future__ import annotations

import dataclasses
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HEAD_DIM = 128
PAGE = 128

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (in place on a uint64 array)."""
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, name: str) -> np.uint64:
    """Key of the named stream under a workload seed."""
    with np.errstate(over="ignore"):
        z = np.array([np.uint64(seed) * _GAMMA + np.uint64(zlib.crc32(name.encode()))],
                     dtype=np.uint64)
        return _mix(z)[0]


def u64(seed: int, name: str, start: int, count: int) -> np.ndarray:
    """Elements [start, start+count) of the named uint64 stream."""
    key = stream_key(seed, name)
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        i *= _GAMMA
        i += key
        return _mix(i)


def uniform(seed: int, name: str, start: int, count: int) -> np.ndarray:
    """Float64 uniforms in the open interval (0, 1), 53 random bits each."""
    b = u64(seed, name, start, count) >> np.uint64(11)
    return (b.astype(np.float64) + 0.5) * (2.0 ** -53)


def normal_slice(seed: int, name: str, start: int, count: int) -> np.ndarray:
    """Elements [start, start+count) of the named standard-normal stream (start, count even).

    Variates 2i and 2i+1 are the cosine and sine outputs of the Box-Muller
    transform of uniforms 2i and 2i+1 of the stream.
    """
    assert start % 2 == 0 and count % 2 == 0
    u = uniform(seed, name, start, count)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    th = (2.0 * np.pi) * u[1::2]
    out = np.empty(count, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal(seed: int, name: str, count: int) -> np.ndarray:
    """``count`` standard normal float64 variates of the named stream."""
    return normal_slice(seed, name, 0, count + (count & 1))[:count]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (round to nearest, ties to even) -> uint16 bits.

    Inputs here are finite. This is how the *inputs* are made BF16; both sides
    then read the same bits.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def permutation(seed: int, name: str, n: int) -> np.ndarray:
    """A uniform random permutation of range(n) (sort by 64-bit random keys)."""
    return np.argsort(u64(seed, name, 0, n), kind="stable").astype(np.int64)


def outlier_channels(seed: int, name: str, n_out: int) -> np.ndarray:
    return np.sort(permutation(seed, name + ".outliers", HEAD_DIM)[:n_out])


def bf16_tensor(seed: int, name: str, shape: tuple, n_out: int = 0, factor: float = 1.0,
                rows: tuple | None = None) -> np.ndarray:
    """BF16 bits of N(0,1) values; ``n_out`` channels of the last axis scaled by ``factor``.

    ``rows=(r0, r1)`` draws only rows r0..r1-1 of the first axis; they are
    bit-identical to the same rows of the full draw. Large draws run in threads.
    """
    per_row = int(np.prod(shape[1:]))
    r0, r1 = rows if rows is not None else (0, shape[0])
    out = np.empty((r1 - r0,) + tuple(shape[1:]), dtype=np.uint16)
    ch = outlier_channels(seed, name, n_out) if n_out else None
    pad = per_row & 1            # keep every row on a Box-Muller pair boundary

    def work(a: int, b: int) -> None:
        x = normal_slice(seed, name, a * (per_row + pad), (b - a) * (per_row + pad))
        x = x.reshape(b - a, per_row + pad)[:, :per_row].reshape((b - a,) + tuple(shape[1:]))
        if ch is not None:
            x[..., ch] *= factor
        out[a - r0: b - r0] = f32_to_bf16_bits(x.astype(np.float32))

    step = max(1, (1 << 20) // max(per_row, 1))
    spans = [(a, min(r1, a + step)) for a in range(r0, r1, step)]
    if len(spans) <= 1:
        for a, b in spans:
            work(a, b)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(lambda ab: work(*ab), spans))
    return out


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape of one synthetic workload."""

    name: str
    seed: int
    ctx: tuple            # total tokens per request after this step (seq_len)
    q_rows: tuple         # query rows per request in this step
    hq: int               # q heads (all on one KV head group per KV head)
    hkv: int
    hi: int               # index heads
    topk: int
    n_out: int            # outlier channels per tensor
    out_factor: float
    store_all: bool       # the step stores every cache row (the tiny case)
    description: str

    @property
    def batch(self) -> int:
        return len(self.ctx)

    @property
    def rows(self) -> int:
        return int(sum(self.q_rows))


def _w3_ctx() -> tuple:
    # 16 contexts drawn uniformly from [64K, 192K] tokens (1K = 1024).
    lo, hi = 64 * 1024, 192 * 1024
    u = u64(2, "ctx", 0, 16)
    return tuple(int(lo + int(v % np.uint64(hi - lo + 1))) for v in u)


SPECS = {
    "tiny": Spec("tiny", 0, (4096,), (1,), 4, 1, 4, 8, 4, 20.0, True,
                 "tiny decode: 1 request, ctx 4096, 4 q heads, 4 index heads, top-k 8"),
    "decode": Spec("decode", 1, (32768,) * 8, (1,) * 8, 16, 1, 16, 16, 3, 10.0, False,
                   "decode bs8 x 32768 ctx, 16 q heads, 16 index heads, top-k 16"),
    "verify": Spec("verify", 2, _w3_ctx(), (8,) * 16, 16, 1, 16, 16, 3, 10.0, False,
                   "speculative verify 16 requests x 8 rows, ctx U[64K,192K]"),
    "skewed": Spec("skewed", 3, (460800,) + (153600,) * 7, (1,) * 8, 16, 1, 16, 16, 3, 10.0,
                   False, "skewed decode bs8: 1 x 450K + 7 x 150K ctx, top-k 16"),
    "prefill": Spec("prefill", 4, (262144 + 8192,), (8192,), 16, 1, 16, 16, 0, 1.0, False,
                    "prefill chunk: 8192 new rows on a 256K cached context, top-k 16"),
}


@dataclasses.dataclass
class Workload:
    """All host arrays of one synthetic workload (numpy, C-contiguous)."""

    spec: Spec
    seq_len: np.ndarray      # int32 [B]
    cu_q: np.ndarray         # int32 [B+1]
    block_table: np.ndarray  # int32 [B, bt_stride]; unused entries -1
    num_pages: int
    tok_off: np.ndarray      # int64 [B+1] first global token index of each request
    slot_all: np.ndarray     # int64 [Ntok] slot of every cache token
    new_tok: np.ndarray      # int64 [T] global token indices stored by this step
    k_src: np.ndarray        # uint16 bf16 bits [Ntok, Hkv, 128]
    v_src: np.ndarray        # uint16 bf16 bits [Ntok, Hkv, 128]
    ik_src: np.ndarray       # uint16 bf16 bits [Ntok, 1, 128]
    q: np.ndarray            # uint16 bf16 bits [R, Hq, 128]
    q_idx: np.ndarray        # uint16 bf16 bits [R, Hi, 128]
    w: np.ndarray            # float32 [R, Hi]

    @property
    def bt_stride(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def ntok(self) -> int:
        return int(self.slot_all.shape[0])

    @property
    def new_slots(self) -> np.ndarray:
        return self.slot_all[self.new_tok]


def layout(seed: int, ctx: tuple) -> tuple:
    """Block tables: request b owns a seeded random set of whole pages of the pool.

    The pool holds exactly sum(ceil(L/128)) pages, shuffled by a seeded random
    permutation, so a request's pages are scattered over the pool.
    Returns (block_table [B, max_blocks] int32, num_pages, tok_off, slot_all).
    """
    nblk = [(L + PAGE - 1) // PAGE for L in ctx]
    num_pages = int(sum(nblk))
    perm = permutation(seed, "pool", num_pages)
    bt = np.full((len(ctx), max(nblk)), -1, dtype=np.int32)
    tok_off = np.zeros(len(ctx) + 1, dtype=np.int64)
    slots = []
    p0 = 0
    for b, L in enumerate(ctx):
        pages = perm[p0: p0 + nblk[b]]
        p0 += nblk[b]
        bt[b, : nblk[b]] = pages
        t = np.arange(L, dtype=np.int64)
        slots.append(pages[t // PAGE] * PAGE + t % PAGE)
        tok_off[b + 1] = tok_off[b] + L
    return bt, num_pages, tok_off, np.concatenate(slots)


def make(spec: Spec | str, ctx: tuple | None = None, q_rows: tuple | None = None,
         with_cache_src: bool = True) -> Workload:
    """Draw a workload. ``ctx``/``q_rows`` override the spec's shape (smaller test cases)."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    if ctx is not None or q_rows is not None:
        spec = dataclasses.replace(spec, ctx=tuple(ctx or spec.ctx),
                                   q_rows=tuple(q_rows or spec.q_rows))
    assert len(spec.ctx) == len(spec.q_rows)
    assert all(0 <= q <= L for q, L in zip(spec.q_rows, spec.ctx))
    s = spec.seed
    bt, num_pages, tok_off, slot_all = layout(s, spec.ctx)
    ntok = int(tok_off[-1])
    cu_q = np.zeros(spec.batch + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(spec.q_rows)
    if spec.store_all:
        new_tok = np.arange(ntok, dtype=np.int64)
    else:
        new_tok = np.concatenate([np.arange(tok_off[b + 1] - q, tok_off[b + 1], dtype=np.int64)
                                  for b, q in enumerate(spec.q_rows)])
    R = spec.rows
    if with_cache_src:
        k_src = bf16_tensor(s, "k", (ntok, spec.hkv, HEAD_DIM), spec.n_out, spec.out_factor)
        v_src = bf16_tensor(s, "v", (ntok, spec.hkv, HEAD_DIM), spec.n_out, spec.out_factor)
        ik_src = bf16_tensor(s, "ik", (ntok, 1, HEAD_DIM), spec.n_out, spec.out_factor)
    else:
        k_src = v_src = ik_src = np.zeros((0, 1, HEAD_DIM), dtype=np.uint16)
    q = bf16_tensor(s, "q", (R, spec.hq, HEAD_DIM), spec.n_out, spec.out_factor)
    q_idx = bf16_tensor(s, "q_idx", (R, spec.hi, HEAD_DIM), spec.n_out, spec.out_factor)
    w = uniform(s, "w", 0, R * spec.hi).astype(np.float32).reshape(R, spec.hi)
    return Workload(spec, np.asarray(spec.ctx, dtype=np.int32), cu_q, bt, num_pages, tok_off,
                    slot_all, new_tok, k_src, v_src, ik_src, q, q_idx, w)
