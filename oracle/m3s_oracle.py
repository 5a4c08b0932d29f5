"""Oracle for the NVFP4 block-sparse decode / verify step (plain CPU, fp64).

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
this module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
arm of ``bench.py`` use it. It shares no code with the CUDA library.

What it computes, and where each definition comes from (the pages are the
three pull requests on the MiniMax-M3.1 NVFP4 caches):

* NVFP4 record -- "NVFP4 sparse KV" (ROCm/ATOM #2746), Summary, and
  "[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (ROCm/ATOM
  #2744), opening paragraph: per token and head, a 64 B e2m1 payload plus
  8 B of E4M3 scales (one scale per 16 of the 128 elements).
* Quantisation -- #2744, Design / Write path: per 16 elements
  scale = e4m3(amax / 6); codes rounded half-to-even, saturating at 6.
* Paged planes -- #2746, Summary (pool): uint8 code planes and scale planes;
  the order inside a page follows "MXFP4 KV cache for MiniMax-M3.1 on gfx950"
  (vllm #64198), Claims: a page is [128 x payload][128 x scales].
* Row map -- #2744, Design / Attention and the row-map commit message: each
  row gets (request, causal length); rows of request b are its last Q_b
  positions.
* Index scoring -- the lightning indexer of #2744, Design / Index and Decode
  score grid: token score = sum_h w_h * ReLU(q_h . k_t) over FP4 keys, block
  score = max over the block's causal tokens, top-k blocks by score.
* Fused verify top-k -- #2744, Fused verify top-k: the same selection as
  score + top-k, ids only.
* MXFP4 record -- #2744, Follow-up: MXFP4 caches, and vllm #64198, Overview /
  Claims: e2m1 data with one E8M0 scale per 32 elements, 68 B per token and
  head, a page [128 x 64 B e2m1][128 x 4 B e8m0]. The pages name the format
  and not its rounding; the shared exponent is the OCP MX one,
  floor(log2(amax)) - 2 (2 = the exponent of e2m1's largest value, 6),
  clamped to E8M0's range, and each element is rounded half-to-even on the
  e2m1 grid after division by 2^exponent, saturating at 6.
* Sparse attention -- #2746 Summary / Attention and #2744 Design / Attention:
  softmax attention over the tokens of the selected blocks, addressed through
  the block table, against the dequantised cache.

Readings where the pages are silent (each is listed with its reason in the
design notes of this repository):
  - E4M3 is OCP e4m3fn; amax/6 above 448 saturates to 448 (0x7E);
  - the e2m1 code of x is the nearest grid value to the exact quotient
    |x|/s (not x*(1/s)), ties to the even code, sign = IEEE sign bit of x;
  - a block whose scale rounds to 0 stores all-zero code bytes;
  - byte i of the payload holds element 2i in its low nibble, 2i+1 high;
  - forced blocks (init / local) rank above every scored block, init
    above local; init blocks lower id first, local blocks most recent first;
  - top-k ties break to the lower block id; the ids are returned sorted
    ascending and padded with -1;
  - sm_scale is an argument (the workloads pass 1/sqrt(128)).

All rounding decisions are taken by exact comparisons in float64 (every
product compared is exactly representable), so this module reproduces the
mathematical definition, not a float approximation of it.
"""

from __future__ import annotations

import math

import numpy as np

HEAD_DIM = 128
PAGE = 128
GROUP = 16
PAYLOAD_BYTES = HEAD_DIM // 2       # 64 B of e2m1 codes per token and head
SCALE_BYTES = HEAD_DIM // GROUP     # 8 B of E4M3 scales per token and head
MX_GROUP = 32
MX_SCALE_BYTES = HEAD_DIM // MX_GROUP   # 4 B of E8M0 scales per token and head (MXFP4)

# error bits reported by the store / scorer / attention (same meaning as the
# CUDA library's device error word)
ERR_SLOT = 1
ERR_BLOCK_ID = 2
ERR_PAGE = 4
ERR_ROW = 8

# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

#: e2m1 magnitudes, indexed by the 3-bit magnitude code (OCP FP4 E2M1).
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_value(code: int) -> float:
    """Value of an OCP E4M3 (e4m3fn) byte: bias 7, subnormals m*2^-9, 0x7F/0xFF NaN."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


#: the 127 finite non-negative E4M3 values, indexed by code 0x00..0x7E (increasing)
E4M3_POS = np.array([e4m3_value(c) for c in range(0x7F)])
#: value of every E4M3 byte (NaN for 0x7F / 0xFF)
E4M3_ALL = np.array([e4m3_value(c) for c in range(256)])


def _nearest_even(x: np.ndarray, values: np.ndarray, scale=None) -> np.ndarray:
    """Index of the entry of the increasing table ``values * scale`` nearest to x.

    Ties go to the even index; x beyond the last entry gives the last index
    (saturation). The comparisons are against ``scale * midpoint``, which the
    callers guarantee to be exact in float64.
    """
    mids = (values[:-1] + values[1:]) / 2.0          # exact: few significant bits
    x = np.asarray(x, dtype=np.float64)
    if scale is None or np.ndim(scale) == 0:
        thr = mids * (1.0 if scale is None else float(scale))
        below = np.searchsorted(thr, x, side="left")  # midpoints strictly below x
        at = np.searchsorted(thr, x, side="right") > below   # x sits on a midpoint
    else:
        thr = np.asarray(scale, dtype=np.float64)[..., None] * mids   # [..., n-1]
        below = (thr < x[..., None]).sum(axis=-1)
        at = (thr == x[..., None]).any(axis=-1)
    # on a tie between index `below` and `below + 1`, keep the even one
    return np.where(at & (below % 2 == 1), below + 1, below)


def e8m0_value(code: int) -> float:
    """Value of an OCP E8M0 byte: 2^(code - 127); 0xFF is NaN."""
    code = int(code) & 0xFF
    return math.nan if code == 0xFF else math.ldexp(1.0, code - 127)


#: value of every E8M0 byte (NaN for 0xFF)
E8M0_ALL = np.array([e8m0_value(c) for c in range(256)])


def e4m3_encode_nonneg(v: np.ndarray) -> np.ndarray:
    """Round non-negative reals to E4M3 (nearest, ties to even code, saturate at 448)."""
    return _nearest_even(v, E4M3_POS).astype(np.uint8)


# --------------------------------------------------------------------------
# Quantisation of BF16 rows into NVFP4 records
# --------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def quantize(bits: np.ndarray, mx: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4- (or, with ``mx``, MXFP4-) quantise BF16 rows (see ``_quantize`` and
    ``_quantize_mx``), in slices to bound memory."""
    bits = np.asarray(bits, dtype=np.uint16)
    flat = bits.reshape(-1, HEAD_DIM)
    n = flat.shape[0]
    nsb = MX_SCALE_BYTES if mx else SCALE_BYTES
    codes = np.empty((n, PAYLOAD_BYTES), dtype=np.uint8)
    scales = np.empty((n, nsb), dtype=np.uint8)
    step = 1 << 15
    fn = _quantize_mx if mx else _quantize
    for i in range(0, n, step):
        codes[i:i + step], scales[i:i + step] = fn(flat[i:i + step])
    lead = bits.shape[:-1]
    return codes.reshape(lead + (PAYLOAD_BYTES,)), scales.reshape(lead + (nsb,))


def _quantize(bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4-quantise BF16 rows.

    ``bits``: uint16 BF16 bit patterns, shape [..., 128].
    Returns (codes uint8 [..., 64], scales uint8 [..., 8]).

    Per group of 16 elements: amax = max |x|; the scale byte is E4M3(amax/6)
    (nearest, ties to even, saturating at 448); each element's magnitude code
    is the e2m1 grid value nearest to |x|/s (ties to the even code, values
    beyond 6 saturate to 6) and its sign bit is the sign bit of x. A group
    whose scale is 0 stores code 0 for every element.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    lead = bits.shape[:-1]
    assert bits.shape[-1] == HEAD_DIM
    x = bf16_to_f64(bits).reshape(lead + (SCALE_BYTES, GROUP))
    sign = ((bits >> np.uint16(15)) & np.uint16(1)).astype(np.uint8).reshape(x.shape)
    amax = np.abs(x).max(axis=-1)                             # [..., 8]
    # nearest E4M3 to amax/6  <=>  compare amax with 6 x (E4M3 midpoints), exact
    scode = _nearest_even(amax, E4M3_POS, 6.0).astype(np.uint8)
    s = E4M3_POS[scode]                                       # [..., 8]
    # nearest grid value to |x|/s  <=>  compare |x| with s x (grid midpoints), exact
    mag = _nearest_even(np.abs(x), E2M1_GRID, s[..., None]).astype(np.uint8)
    code = (sign << np.uint8(3)) | mag
    code = np.where((s == 0.0)[..., None], np.uint8(0), code).astype(np.uint8)
    code = code.reshape(lead + (HEAD_DIM,))
    packed = (code[..., 0::2] | (code[..., 1::2] << np.uint8(4))).astype(np.uint8)
    return packed, scode


def _quantize_mx(bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """MXFP4-quantise BF16 rows.

    ``bits``: uint16 BF16 bit patterns, shape [..., 128].
    Returns (codes uint8 [..., 64], scales uint8 [..., 4]).

    Per group of 32 elements: amax = max |x|; the shared exponent is
    E = floor(log2(amax)) - 2, clamped to [-127, 127] (amax = 0 gives -127);
    the scale byte is E + 127 (E8M0). Each element's magnitude code is the
    e2m1 grid value nearest to |x| / 2^E (ties to the even code, beyond 6
    saturating to 6) and its sign bit is the sign bit of x.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    lead = bits.shape[:-1]
    assert bits.shape[-1] == HEAD_DIM
    x = bf16_to_f64(bits).reshape(lead + (MX_SCALE_BYTES, MX_GROUP))
    sign = ((bits >> np.uint16(15)) & np.uint16(1)).astype(np.uint8).reshape(x.shape)
    amax = np.abs(x).max(axis=-1)                             # [..., 4]
    _, e = np.frexp(amax)                                     # amax = m 2^e, m in [0.5, 1)
    E = np.where(amax > 0.0, e.astype(np.int64) - 1 - 2, -127)
    E = np.clip(E, -127, 127)
    scode = (E + 127).astype(np.uint8)
    s = np.ldexp(1.0, E)                                      # exact powers of two
    # nearest grid value to |x| / 2^E  <=>  compare |x| with 2^E x (grid midpoints), exact
    mag = _nearest_even(np.abs(x), E2M1_GRID, s[..., None]).astype(np.uint8)
    code = ((sign << np.uint8(3)) | mag).reshape(lead + (HEAD_DIM,))
    packed = (code[..., 0::2] | (code[..., 1::2] << np.uint8(4))).astype(np.uint8)
    return packed, scode


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """x_hat = e2m1(code) * scale, float64, shape [..., 128].

    The format follows the scale array: 8 bytes per record are E4M3 scales of
    16 elements each (NVFP4), 4 bytes are E8M0 scales of 32 elements (MXFP4).
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    lo = codes & np.uint8(0xF)
    hi = codes >> np.uint8(4)
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (HEAD_DIM,))
    val = E2M1_GRID[c & 7] * np.where(c & 8, -1.0, 1.0)
    if scales.shape[-1] == MX_SCALE_BYTES:
        return val * np.repeat(E8M0_ALL[scales], MX_GROUP, axis=-1)
    assert scales.shape[-1] == SCALE_BYTES
    return val * np.repeat(E4M3_ALL[scales], GROUP, axis=-1)


def new_planes(num_pages: int, heads: int, mx: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Zeroed planes: codes [P, H, 128, 64] and scales [P, H, 128, 8] (NVFP4) or
    [P, H, 128, 4] (MXFP4), uint8."""
    return (np.zeros((num_pages, heads, PAGE, PAYLOAD_BYTES), dtype=np.uint8),
            np.zeros((num_pages, heads, PAGE, MX_SCALE_BYTES if mx else SCALE_BYTES),
                     dtype=np.uint8))


def nvfp4_store(src: np.ndarray, slot_mapping: np.ndarray, codes: np.ndarray,
                scales: np.ndarray) -> int:
    """Quantise rows ``src`` [T, H, 128] (BF16 bits) into the planes at their slots.

    The planes' format follows the scale plane (8 bytes per record: NVFP4, 4:
    MXFP4). slot = page * 128 + offset. A negative slot is a pad row and is
    skipped, leaving the planes untouched; a slot beyond the planes sets
    ERR_SLOT and is skipped. Returns the error bits.
    """
    src = np.asarray(src, dtype=np.uint16)
    slot_mapping = np.asarray(slot_mapping, dtype=np.int64)
    P, H = codes.shape[0], codes.shape[1]
    assert src.shape[1] == H
    err = 0
    c, s = quantize(src, mx=scales.shape[-1] == MX_SCALE_BYTES)
    for r, slot in enumerate(slot_mapping):
        if slot < 0:
            continue
        if slot >= P * PAGE:
            err |= ERR_SLOT
            continue
        codes[slot // PAGE, :, slot % PAGE] = c[r]
        scales[slot // PAGE, :, slot % PAGE] = s[r]
    return err


# --------------------------------------------------------------------------
# Row map
# --------------------------------------------------------------------------

def decode_rows(cu_q: np.ndarray, seq_len: np.ndarray, R: int) -> tuple[np.ndarray, np.ndarray]:
    """(row_req, row_len) for R query rows.

    Row r = cu_q[b] + j of request b (which has Q_b = cu_q[b+1] - cu_q[b] rows
    and seq_len[b] tokens including them) is the token at position
    seq_len[b] - Q_b + j, so it attends causally to seq_len[b] - Q_b + j + 1
    tokens. Rows at or past cu_q[B] are padding: (-1, 0).
    """
    row_req = np.full(R, -1, dtype=np.int32)
    row_len = np.zeros(R, dtype=np.int32)
    B = len(seq_len)
    for b in range(B):
        qb = int(cu_q[b + 1]) - int(cu_q[b])
        for j in range(qb):
            r = int(cu_q[b]) + j
            if r < R:
                row_req[r] = b
                row_len[r] = int(seq_len[b]) - qb + j + 1
    return row_req, row_len


# --------------------------------------------------------------------------
# Index scoring and block top-k
# --------------------------------------------------------------------------

def _request_pages(block_table: np.ndarray, b: int, nblk: int, num_pages: int
                   ) -> tuple[np.ndarray, int]:
    pages = np.asarray(block_table[b, :nblk], dtype=np.int64)
    err = 0
    if nblk > block_table.shape[1]:
        err |= ERR_ROW
    if np.any((pages < 0) | (pages >= num_pages)):
        err |= ERR_PAGE
    return pages, err


def dequant_tokens(codes: np.ndarray, scales: np.ndarray, pages: np.ndarray, head: int,
                   L: int) -> np.ndarray:
    """Dequantised tokens 0..L-1 of a request whose blocks live on ``pages``; [L, 128]."""
    if L <= 0:
        return np.zeros((0, HEAD_DIM))
    nb = (L + PAGE - 1) // PAGE
    x = dequantize(codes[pages[:nb], head], scales[pages[:nb], head])   # [nb, 128, 128]
    return x.reshape(nb * PAGE, HEAD_DIM)[:L]


def token_scores(q_idx_row: np.ndarray, w_row: np.ndarray, k_hat: np.ndarray) -> np.ndarray:
    """score[t] = sum_h w[h] * ReLU(q[h] . k_hat[t]) in float64."""
    q = bf16_to_f64(q_idx_row)                        # [Hi, 128]
    s = k_hat @ q.T                                    # [L, Hi] (library matmul, fp64)
    return np.maximum(s, 0.0) @ np.asarray(w_row, dtype=np.float64)


def block_max(score: np.ndarray, L: int) -> np.ndarray:
    """Block score = max of the token scores of its causal tokens (t < L)."""
    nb = (L + PAGE - 1) // PAGE
    out = np.empty(nb)
    for b in range(nb):
        out[b] = score[b * PAGE: min((b + 1) * PAGE, L)].max()
    return out


def topk_ids(bscore: np.ndarray, k: int, init_blocks: int = 0, local_blocks: int = 0) -> np.ndarray:
    """The k best blocks (higher score first, the lower id on equal scores).

    Forced blocks -- #2744's review of the fused verify top-k and vllm #64198,
    Design (the init / local sentinels 1e30 and 1e29 written before the
    top-k): the first ``init_blocks`` blocks and the last ``local_blocks``
    blocks of the row rank above every scored block, init above local. Init
    blocks rank lower id first; local blocks rank most recent (higher id)
    first, so that when init + local exceeds k the row's newest blocks -- its
    current token's block among them -- are the ones kept (the review's
    correction of the fused path). A block that is both counts as init.

    Returned sorted by ascending id, padded with -1 when there are fewer than k blocks.
    """
    nb = len(bscore)
    ids = np.arange(nb)
    init = ids < init_blocks
    local = (ids >= nb - local_blocks) & ~init
    cls = np.where(init, 2, np.where(local, 1, 0))
    within = np.where(init, ids.astype(np.float64),
                      np.where(local, -ids.astype(np.float64), -np.asarray(bscore, dtype=np.float64)))
    order = np.lexsort((ids, within, -cls))     # class, then the in-class order, then lower id
    sel = np.sort(order[: min(k, nb)])
    out = np.full(k, -1, dtype=np.int32)
    out[: len(sel)] = sel
    return out


def rank_records(bscore: np.ndarray, ids, nb: int, init_blocks: int = 0, local_blocks: int = 0) -> list:
    """The order topk_ids selects by, as sortable records (class, in-class value, id):
    a record ranks higher with a larger class, then a larger in-class value, then a
    lower id. Init blocks (class 2) by lower id, local blocks (class 1) by higher id,
    scored blocks (class 0) by score; ``nb`` is the row's block count (the forced
    blocks are the row's first and last ones)."""
    out = []
    for i in ids:
        i = int(i)
        if i < init_blocks:
            out.append((2, -float(i), i))
        elif i >= nb - local_blocks:
            out.append((1, float(i), i))
        else:
            out.append((0, float(bscore[i]), i))
    return out


def _best_first(records):
    return sorted(records, key=lambda rec: (-rec[0], -rec[1], rec[2]))


def slice_candidates(bscore: np.ndarray, lo: int, hi: int, k: int, init_blocks: int = 0,
                     local_blocks: int = 0) -> list:
    """Indexer context parallelism ("[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV
    cache" (#2744), review thread on the unused page-16 tables: the indexer-CP decode path
    merges per-rank candidate keys): the candidates of the rank that holds blocks
    [lo, hi) of a row whose block scores are ``bscore`` -- the k best of its blocks in
    the order topk_ids uses (forced blocks by the row's own block count), best first,
    as rank_records."""
    nb = len(bscore)
    recs = rank_records(bscore, range(max(0, lo), min(hi, nb)), nb, init_blocks, local_blocks)
    return _best_first(recs)[:k]


def merge_candidates(lists, k: int) -> np.ndarray:
    """The k best of the union of the ranks' candidate lists (rank_records), as
    topk_ids returns them: ids ascending, padded with -1. Because every block of
    the row's top k is among its own rank's k best, this equals the top k of the
    whole row."""
    union = _best_first([rec for lst in lists for rec in lst])[:k]
    out = np.full(k, -1, dtype=np.int32)
    out[: len(union)] = np.sort([rec[2] for rec in union]).astype(np.int32)
    return out


def index_score_topk(q_idx: np.ndarray, w: np.ndarray, idx_codes: np.ndarray,
                     idx_scales: np.ndarray, block_table: np.ndarray, row_req: np.ndarray,
                     row_len: np.ndarray, topk: int, rows=None, init_blocks: int = 0,
                     local_blocks: int = 0):
    """Per query row: index scores over its causal keys, block maxima, top-k block ids.

    Returns (topk_ids int32 [R, topk], block_scores list of float64 arrays
    (one per row, length ceil(row_len/128)), err bits). ``rows`` restricts the
    work to a subset of rows (others get -1 ids and empty scores).
    """
    R = len(row_req)
    out = np.full((R, topk), -1, dtype=np.int32)
    bscores = [np.zeros(0) for _ in range(R)]
    err = 0
    num_pages = idx_codes.shape[0]
    cache = {}
    for r in (range(R) if rows is None else rows):
        b, L = int(row_req[r]), int(row_len[r])
        if b < 0 or L <= 0:
            continue
        nb = (L + PAGE - 1) // PAGE
        pages, e = _request_pages(block_table, b, nb, num_pages)
        err |= e
        if e:
            continue
        key = (b, nb)
        if key not in cache:
            cache.clear()
            cache[key] = dequant_tokens(idx_codes, idx_scales, pages, 0, nb * PAGE)
        k_hat = cache[key][:L]
        sc = token_scores(q_idx[r], w[r], k_hat)
        bscores[r] = block_max(sc, L)
        out[r] = topk_ids(bscores[r], topk, init_blocks, local_blocks)
    return out, bscores, err


def verify_score_topk(q_idx, w, idx_codes, idx_scales, block_table, cu_q, seq_len, R, topk,
                      rows=None, init_blocks: int = 0, local_blocks: int = 0):
    """Fused verify score + top-k: the same selection as the row map followed by
    score + top-k (the fused kernel only changes how the work is grouped)."""
    row_req, row_len = decode_rows(cu_q, seq_len, R)
    ids, _, err = index_score_topk(q_idx, w, idx_codes, idx_scales, block_table, row_req,
                                   row_len, topk, rows, init_blocks, local_blocks)
    return ids, err


# --------------------------------------------------------------------------
# Block-sparse attention
# --------------------------------------------------------------------------

def sparse_attention(q: np.ndarray, hkv: int, k_codes, k_scales, v_codes, v_scales,
                     block_table, row_req, row_len, ids, sm_scale: float, rows=None):
    """o[r, h] = sum_t softmax_t(sm_scale * q[r,h] . k_hat[t]) v_hat[t].

    t runs over the tokens of the listed blocks (logical ids within the
    request; -1 entries skipped) that lie before the row's causal length. q head
    h reads KV head h // (Hq / Hkv). A row with no such token outputs zeros and
    lse = -inf. An id at or beyond the row's block count sets ERR_BLOCK_ID and
    is skipped. Returns (out float64 [R, Hq, 128], lse float64 [R, Hq], err).
    """
    R, Hq, _ = q.shape
    G = Hq // hkv
    out = np.zeros((R, Hq, HEAD_DIM))
    lse = np.full((R, Hq), -np.inf)
    err = 0
    num_pages = k_codes.shape[0]
    for r in (range(R) if rows is None else rows):
        b, L = int(row_req[r]), int(row_len[r])
        if b < 0 or L <= 0:
            continue
        nb = (L + PAGE - 1) // PAGE
        toks = []
        for i in np.asarray(ids[r]):
            i = int(i)
            if i < 0:
                continue
            if i >= nb or i >= block_table.shape[1]:
                err |= ERR_BLOCK_ID
                continue
            toks.append((i, min(PAGE, L - i * PAGE)))
        if not toks:
            continue
        pages = np.array([block_table[b, i] for i, _ in toks], dtype=np.int64)
        if np.any((pages < 0) | (pages >= num_pages)):
            err |= ERR_PAGE
            continue
        q_r = bf16_to_f64(q[r])
        for kvh in range(hkv):
            kh = np.concatenate([dequantize(k_codes[p, kvh, :n], k_scales[p, kvh, :n])
                                 for p, (_, n) in zip(pages, toks)])
            vh = np.concatenate([dequantize(v_codes[p, kvh, :n], v_scales[p, kvh, :n])
                                 for p, (_, n) in zip(pages, toks)])
            for h in range(kvh * G, (kvh + 1) * G):
                logits = sm_scale * (kh @ q_r[h])
                m = logits.max()
                p = np.exp(logits - m)
                l = p.sum()
                out[r, h] = (p @ vh) / l
                lse[r, h] = m + math.log(l)
    return out, lse, err


# --------------------------------------------------------------------------
# Quantise-at-write: the normalise / rotate / cache-write step with the
# quantisation inside it ("[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV
# cache" (#2744), Follow-up: MXFP4 caches -- "the quantization happens inside
# the fused qk-norm/RoPE/cache kernel, so there is no staging buffer and no
# store launch"; the unfused path of the same page, Summary / Write, writes
# the normalised rows BF16 to a staging buffer and quantises them after).
# --------------------------------------------------------------------------

def _f32(x):
    return np.asarray(x, dtype=np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16, nearest, ties to even (NaN kept quiet)."""
    u = _f32(x).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7F800000) == 0x7F800000
    nan &= (u & 0x007FFFFF) != 0
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = np.where(nan, (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def head_sum_sq_f32(x: np.ndarray) -> np.ndarray:
    """sum of x^2 over the last axis (128) in float32, in the order the write
    kernel's warp takes it: lane l owns elements 4l .. 4l+3 and adds their
    squares left to right; the 32 lane sums are then combined by an xor
    butterfly (offsets 16, 8, 4, 2, 1) and lane 0's value is the result.
    Float addition is commutative, so only this tree of additions matters."""
    sq = _f32(x) * _f32(x)                                   # rounded products
    sq = sq.reshape(sq.shape[:-1] + (32, 4))
    p = ((sq[..., 0] + sq[..., 1]) + sq[..., 2]) + sq[..., 3]
    lanes = np.arange(32)
    for off in (16, 8, 4, 2, 1):
        p = p + p[..., lanes ^ off]
    return p[..., 0]


def norm_rope_rows(bits: np.ndarray, weight, cos, sin, rotary_dim: int, eps: float) -> np.ndarray:
    """The normalised, rotated BF16 rows [T, H, 128] of BF16 rows ``bits``.

    Per (row, head), in float32 with every operation rounded (no fused
    multiply-add), as the write kernel computes it:
      - RMSNorm (``weight`` [128] given): r = 1 / sqrt(sum(x^2) / 128 + eps),
        y_i = (x_i * r) * weight_i; else y = x;
      - RoPE (``cos``/``sin`` [T, rotary_dim / 2] given): for i < rotary_dim / 2,
        with j = i + rotary_dim / 2, c = cos[t, i], s = sin[t, i]:
        o_i = y_i * c - y_j * s,  o_j = y_j * c + y_i * s;  dims >= rotary_dim
        pass unchanged;
      - the result rounded to BF16 (nearest, ties to even), as the staging
        buffer of the unfused path holds it.
    """
    x = bf16_to_f64(bits).astype(np.float32)                 # exact
    T, H, D = x.shape
    assert D == HEAD_DIM
    if weight is not None:
        ss = head_sum_sq_f32(x)                              # [T, H]
        v = ss * np.float32(1.0 / 128) + np.float32(eps)
        r = np.float32(1.0) / np.sqrt(v)
        y = (x * r[..., None]) * _f32(weight)
    else:
        y = x
    if cos is not None:
        h = rotary_dim // 2
        c = _f32(cos)[:, None, :h]
        s = _f32(sin)[:, None, :h]
        y1, y2 = y[..., :h], y[..., h:rotary_dim]
        o1 = y1 * c - y2 * s
        o2 = y2 * c + y1 * s
        y = np.concatenate([o1, o2, y[..., rotary_dim:]], axis=-1)
    return f32_to_bf16_bits(y)


def norm_rope_rows_f64(bits: np.ndarray, weight, cos, sin, rotary_dim: int, eps: float) -> np.ndarray:
    """The normalised, rotated rows [T, H, 128] of BF16 rows ``bits`` in float64,
    unrounded: the definition itself, with no float32 step and no order of
    summation (the sum of squares is math.fsum's, exact then rounded once).

      - RMSNorm (``weight`` [128] given): y = x / sqrt(mean(x^2) + eps) * weight;
      - RoPE (``cos``/``sin`` [T, rotary_dim / 2] given), rotate-half on the first
        rotary_dim dims: o_i = y_i c - y_j s, o_j = y_j c + y_i s (j = i + rd/2).
    """
    x = bf16_to_f64(bits)
    T, H, D = x.shape
    assert D == HEAD_DIM
    if weight is not None:
        ss = np.array([[math.fsum(v * v for v in x[t, h]) for h in range(H)] for t in range(T)])
        y = x / np.sqrt(ss / HEAD_DIM + float(eps))[..., None] * np.asarray(weight, np.float64)
    else:
        y = x.copy()
    if cos is not None:
        h = rotary_dim // 2
        c = np.asarray(cos, np.float64)[:, None, :h]
        s = np.asarray(sin, np.float64)[:, None, :h]
        y1, y2 = y[..., :h].copy(), y[..., h:rotary_dim].copy()
        y[..., :h] = y1 * c - y2 * s
        y[..., h:rotary_dim] = y2 * c + y1 * s
    return y


def qk_norm_rope_store(jobs, slot_mapping, cos, sin, rotary_dim: int, eps: float) -> int:
    """The fused write: each job is (src bits [T, H, 128], weight [128] or None,
    rope: bool, destination), the destination either a (codes, scales) plane
    pair, filled as ``nvfp4_store`` would fill it from the normalised rows, or
    a BF16 array [T, H, 128] that receives them. Returns the store's error bits."""
    err = 0
    for src, weight, rope, dst in jobs:
        rows = norm_rope_rows(src, weight, cos if rope else None, sin if rope else None,
                              rotary_dim, eps)
        if isinstance(dst, tuple):
            err |= nvfp4_store(rows, slot_mapping, dst[0], dst[1])
        else:
            dst[...] = rows
    return err
