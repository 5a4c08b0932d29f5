"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: hand-worked
values (tests/golden), a library routine (torch's float8_e4m3fn conversion,
torch's scaled_dot_product_attention), exact rational arithmetic, brute force
over every subset on tiny inputs, closed forms and invariants.
"""

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from nvfp4_block_sparse_m3s_gb300 import workloads as W
from oracle import m3s_oracle as O

GOLDEN = __file__.rsplit("/", 1)[0] + "/golden/nvfp4_quant_blocks.txt"


def _golden_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("case "):
            cur = {"name": line[5:]}
            cases.append(cur)
        else:
            k, v = line.split(":", 1)
            cur[k] = v.split()
    return cases


def _block(values):
    """16 decimal values -> a 128-element BF16 row (group 0 = values, rest zero)."""
    x = np.zeros(128, dtype=np.float32)
    x[:16] = [float(v) for v in values]
    bits = W.f32_to_bf16_bits(x)
    # the golden inputs are BF16-exact: the rounding must not have moved them
    assert np.array_equal(W.bf16_bits_to_f32(bits)[:16], x[:16])
    return bits


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_quantiser_hand_worked(case):
    codes, scales = O.quantize(_block(case["x"]))
    assert scales[0] == int(case["scale"][0], 16)
    got = [(codes[i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
    assert got == [int(c, 16) for c in case["codes"]]
    # the other 7 groups are zero
    assert not codes[8:].any() and not scales[1:].any()


def test_e4m3_table_matches_torch():
    """Every E4M3 byte decodes as torch's float8_e4m3fn does (library routine)."""
    allb = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()
    ours = O.E4M3_ALL
    nan = np.isnan(allb)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(allb[~nan], ours[~nan])
    assert O.E4M3_POS[-1] == 448.0 and O.E4M3_POS[1] == 2.0 ** -9


def test_e4m3_encoder_matches_torch_rne():
    """Nearest / ties-to-even E4M3 rounding agrees with torch's float32 -> e4m3fn cast
    on every in-range float32 value tried (all midpoints, neighbours of every
    value, and random reals)."""
    v = O.E4M3_POS
    mids = (v[:-1] + v[1:]) / 2
    rng = np.random.default_rng(0)
    cand = np.concatenate([v, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
                           rng.uniform(0, 448, 20000), rng.uniform(0, 2 ** -6, 20000)])
    cand = cand.astype(np.float32).astype(np.float64)      # exactly float32
    cand = cand[cand <= 448.0]
    t = torch.from_numpy(cand.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(O.e4m3_encode_nonneg(cand), t.numpy())


def _exact_quantise_group(xs):
    """Independent restatement in exact rationals (Fraction) of one 16-group."""
    fr = [Fraction(float(x)) for x in xs]
    amax = max(abs(x) for x in fr)
    target = amax / 6
    vals = [Fraction(float(O.e4m3_value(c))) for c in range(0x7F)]
    best = min(range(0x7F), key=lambda c: (abs(vals[c] - target), c % 2))
    s = vals[best]
    grid = [Fraction(g) for g in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    codes = []
    for x, xf in zip(xs, fr):
        if s == 0:
            codes.append(0)
            continue
        q = abs(xf) / s
        m = min(range(8), key=lambda i: (abs(grid[i] - q), i % 2))
        codes.append(m | (8 if math.copysign(1.0, float(x)) < 0 else 0))
    return best, codes


def test_quantiser_equals_exact_rational_definition():
    """Vectorised oracle == exact-rational brute force on random groups spanning the
    whole E4M3 scale range, with ties planted."""
    rng = np.random.default_rng(1)
    rows = []
    for i in range(48):
        e = rng.integers(-14, 12)
        x = rng.standard_normal(128) * 2.0 ** e
        if i % 3 == 0:        # plant exact ties: grid midpoints x a power-of-two scale
            x[:7] = np.array([.25, .75, 1.25, 1.75, 2.5, 3.5, 5]) * 2.0 ** e
            x[7] = 6 * 2.0 ** e
        rows.append(x)
    bits = W.f32_to_bf16_bits(np.array(rows, dtype=np.float32))
    xs = W.bf16_bits_to_f32(bits).astype(np.float64)
    codes, scales = O.quantize(bits)
    for r in range(len(rows)):
        for g in range(8):
            s, c = _exact_quantise_group(xs[r, 16 * g: 16 * g + 16])
            assert scales[r, g] == s
            got = [(codes[r, 8 * g + i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
            assert got == c, (r, g)


def test_round_trip_error_bound_and_idempotence():
    """|x - x_hat| <= half the local e2m1 step x s for unsaturated elements, and
    quantising the dequantised values again gives the same bytes when the group's
    largest code is 7."""
    bits = W.bf16_tensor(7, "rt", (512, 128), 4, 20.0)
    x = W.bf16_bits_to_f32(bits).astype(np.float64)
    c, s = O.quantize(bits)
    xh = O.dequantize(c, s)
    sv = np.repeat(O.E4M3_ALL[s], 16, axis=-1)
    q = np.abs(x) / np.where(sv > 0, sv, 1)
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    unsat = q <= 6
    assert np.all(np.abs(x - xh)[unsat] <= (0.5 * step * sv)[unsat] + 0.0)
    cmax = np.stack([(c >> 4) & 7, c & 7], -1).reshape(512, 8, 16).max(-1)
    again_c, again_s = O.quantize(W.f32_to_bf16_bits(xh.astype(np.float32)))
    full = cmax == 7
    assert np.array_equal(again_s[full], s[full])
    cg = c.reshape(512, 8, 8)
    assert np.array_equal(again_c.reshape(512, 8, 8)[full], cg[full])


def test_store_head_split_and_pad_rows():
    """An H-head store equals H single-head stores ("NVFP4 sparse KV", Tests:
    kv_nvfp4_store over H heads equals the per-head index store); pad rows
    (slot < 0) leave the planes untouched; an out-of-range slot is reported."""
    H, T, P = 3, 40, 4
    src = W.bf16_tensor(3, "st", (T, H, 128), 2, 10.0)
    slots = W.permutation(3, "slots", P * 128)[:T].astype(np.int64)
    slots[5] = -1
    slots[17] = -7
    c, s = O.new_planes(P, H)
    c[:] = 0xA5
    s[:] = 0x5A
    assert O.nvfp4_store(src, slots, c, s) == 0
    for h in range(H):
        ch, sh = O.new_planes(P, 1)
        ch[:] = 0xA5
        sh[:] = 0x5A
        O.nvfp4_store(src[:, h: h + 1], slots, ch, sh)
        assert np.array_equal(ch[:, 0], c[:, h]) and np.array_equal(sh[:, 0], s[:, h])
    written = set(int(v) for v in slots if v >= 0)
    for slot in range(P * 128):
        if slot not in written:
            assert (c[slot // 128, :, slot % 128] == 0xA5).all()
            assert (s[slot // 128, :, slot % 128] == 0x5A).all()
    bad = slots.copy()
    bad[3] = P * 128
    c2, s2 = O.new_planes(P, H)
    assert O.nvfp4_store(src, bad, c2, s2) == O.ERR_SLOT


def test_record_size_reproduces_pages_block_bytes():
    """72 B per token and head reproduces the pages' KV block bytes: the drop from
    3,179,520 to 1,827,840 B per 128-token block over 60 sparse layers is exactly
    2 x (132 - 72) + (128 - 72) bytes per token per layer ("NVFP4 sparse KV",
    Results / KV capacity; FP8 record 128 + 4 B, FP8 index key 128 B)."""
    c, s = O.quantize(np.zeros((1, 128), dtype=np.uint16))
    rec = c.shape[-1] + s.shape[-1]
    assert rec == 72
    per_token = (3_179_520 - 1_827_840) // 128
    assert per_token * 128 == 3_179_520 - 1_827_840
    assert per_token == 60 * (2 * (132 - rec) + (128 - rec))


def test_row_map_closed_form_vs_searchsorted():
    """decode_rows against a brute-force mapping built the way the pages' prefill
    row map is (searchsorted over the row offsets)."""
    rng = np.random.default_rng(2)
    for trial in range(50):
        B = int(rng.integers(1, 12))
        qb = rng.integers(0, 9, B)
        seq = (qb + rng.integers(0, 500, B)).astype(np.int32)
        cu = np.concatenate([[0], np.cumsum(qb)]).astype(np.int32)
        R = int(cu[-1] + rng.integers(0, 4))
        rr, rl = O.decode_rows(cu, seq, R)
        r = np.arange(R)
        b = np.searchsorted(cu, r, side="right") - 1
        valid = r < cu[-1]
        exp_req = np.where(valid, b, -1)
        bb = np.clip(b, 0, B - 1)
        exp_len = np.where(valid, seq[bb] - (cu[bb + 1] - cu[bb]) + (r - cu[bb]) + 1, 0)
        assert np.array_equal(rr, exp_req) and np.array_equal(rl, exp_len)


def _tiny_index_case(seed, L, hi=2, nb_pages=None):
    """A tiny request of L tokens on shuffled pages, quantised by the oracle."""
    nb = (L + 127) // 128
    P = nb_pages or nb + 2
    pages = W.permutation(seed, "tp", P)[:nb]
    bt = pages[None, :].astype(np.int32)
    src = W.bf16_tensor(seed, "tk", (nb * 128, 1, 128), 2, 10.0)
    c, s = O.new_planes(P, 1)
    slots = (pages[np.arange(nb * 128) // 128] * 128 + np.arange(nb * 128) % 128)
    O.nvfp4_store(src, slots, c, s)
    q = W.bf16_tensor(seed, "tq", (1, hi, 128))
    w = W.uniform(seed, "tw", 0, hi).astype(np.float32).reshape(1, hi)
    return bt, c, s, q, w, src


def test_scores_brute_force_and_topk_all_subsets():
    """Token scores by explicit Python loops; the top-k set is the best of every
    k-subset under (higher block score, then lower id). The last two cases give
    the second head a negative weight: the formula puts no sign on w_h, so a
    head can only lower a token's score (block scores may then be negative)."""
    for seed, L, k, neg in [(11, 300, 2, False), (12, 512, 3, False), (13, 129, 1, False),
                            (14, 385, 2, False), (15, 300, 2, True), (16, 640, 3, True)]:
        bt, c, s, q, w, _ = _tiny_index_case(seed, L)
        if neg:
            w[0, 1] = -2.0 * w[0, 1]
        rr, rl = np.array([0], np.int32), np.array([L], np.int32)
        ids, bsc, err = O.index_score_topk(q, w, c, s, bt, rr, rl, k)
        assert err == 0
        qf = W.bf16_bits_to_f32(q[0]).astype(np.float64)
        nb = (L + 127) // 128
        brute = []
        for b in range(nb):
            best = -math.inf
            for t in range(b * 128, min(b * 128 + 128, L)):
                page = bt[0, t // 128]
                kh = O.dequantize(c[page, 0, t % 128], s[page, 0, t % 128])
                tot = 0.0
                for h in range(q.shape[1]):
                    dot = sum(float(qf[h, d]) * float(kh[d]) for d in range(128))
                    tot += float(w[0, h]) * max(dot, 0.0)
                best = max(best, tot)
            brute.append(best)
        np.testing.assert_allclose(bsc[0], brute, rtol=1e-12, atol=1e-12)
        kk = min(k, nb)

        def rank_key(sub):
            return sorted(((brute[i], -i) for i in sub), reverse=True)

        best_sub = max(itertools.combinations(range(nb), kk), key=rank_key)
        assert list(ids[0][:kk]) == sorted(best_sub)
        assert (ids[0][kk:] == -1).all()


def test_block_max_closed_form():
    """A block's score is the largest score of its causal tokens: with token
    scores increasing in t that is the block's last causal token, with scores
    decreasing its first token, for lengths with a ragged last block."""
    for L in (1, 127, 128, 129, 300, 512):
        t = np.arange(L, dtype=np.float64)
        nb = (L + 127) // 128
        assert O.block_max(t, L).tolist() == [float(min(128 * (b + 1), L) - 1) for b in range(nb)]
        assert O.block_max(-t, L).tolist() == [-float(128 * b) for b in range(nb)]


def test_rows_of_a_request_score_alone_or_together():
    """Scoring a request's rows in one call gives each row what scoring it alone
    gives, for rows whose causal lengths cross block boundaries (253..260
    tokens: 2 and 3 blocks), in increasing and in decreasing row order."""
    bt, c, s, _, _, _ = _tiny_index_case(41, 260)
    R = 8
    q = W.bf16_tensor(41, "rq", (R, 2, 128))
    w = W.uniform(41, "rw", 0, 2 * R).astype(np.float32).reshape(R, 2)
    for lens in (np.arange(253, 261), np.arange(260, 252, -1)):
        rl = lens.astype(np.int32)
        ids, bs, err = O.index_score_topk(q, w, c, s, bt, np.zeros(R, np.int32), rl, 2)
        assert err == 0
        for r in range(R):
            ids1, bs1, _ = O.index_score_topk(q[r:r + 1], w[r:r + 1], c, s, bt, np.zeros(1, np.int32),
                                              rl[r:r + 1], 2)
            assert len(bs[r]) == (int(rl[r]) + 127) // 128
            assert np.array_equal(bs[r], bs1[0]) and np.array_equal(ids[r], ids1[0])


def test_bad_pages_rows_and_ids_are_reported():
    """Error bits and skipped rows: in scoring, a block-table entry outside the
    pool (PAGE) and a row longer than its block table (ROW); in attention, a
    page outside the pool (PAGE). A reported row gets no ids, or zero output and
    lse -inf."""
    bt, c, s, q, w, _ = _tiny_index_case(42, 300)
    P = c.shape[0]
    bad = bt.copy()
    bad[0, 1] = P
    ids, _, err = O.index_score_topk(q, w, c, s, bad, np.zeros(1, np.int32), np.array([300], np.int32), 2)
    assert err == O.ERR_PAGE and (ids == -1).all()
    bad[0, 1] = -3
    _, _, err = O.index_score_topk(q, w, c, s, bad, np.zeros(1, np.int32), np.array([300], np.int32), 2)
    assert err == O.ERR_PAGE
    long = np.array([bt.shape[1] * 128 + 1], np.int32)
    ids, _, err = O.index_score_topk(q, w, c, s, bt, np.zeros(1, np.int32), long, 2)
    assert err & O.ERR_ROW and (ids == -1).all()
    bt, kc, ks, vc, vs, qa = _attn_case(43, 300)
    bad = bt.copy()
    bad[0, 2] = kc.shape[0]
    out, lse, err = O.sparse_attention(qa, 1, kc, ks, vc, vs, bad, np.zeros(1, np.int32),
                                       np.array([300], np.int32), np.array([[0, 2]]), 0.1)
    assert err == O.ERR_PAGE and not out.any() and np.isneginf(lse).all()


def test_zero_queries_select_lowest_ids():
    """All-zero queries give every block the score 0; ties go to the lower block id
    (the pages' fused top-k tie test uses zero queries)."""
    bt, c, s, q, w, _ = _tiny_index_case(21, 1000)
    q[:] = 0
    ids, bsc, _ = O.index_score_topk(q, w, c, s, bt, np.array([0], np.int32),
                                     np.array([1000], np.int32), 3)
    assert (bsc[0] == 0).all() and list(ids[0]) == [0, 1, 2]


def test_hot_token_is_selected():
    """A key aligned with the query planted in block b* wins the top-1."""
    for bstar in range(4):
        bt, c, s, q, w, src = _tiny_index_case(30 + bstar, 512)
        t = bstar * 128 + 77
        hot = W.bf16_bits_to_f32(q[0, 0]).astype(np.float32) * 8
        row = W.f32_to_bf16_bits(hot)[None, None, :]
        page = int(bt[0, t // 128])
        O.nvfp4_store(row, np.array([page * 128 + t % 128]), c, s)
        w[:] = [[1.0, 0.0]]
        ids, _, _ = O.index_score_topk(q, w, c, s, bt, np.array([0], np.int32),
                                       np.array([512], np.int32), 1)
        assert ids[0, 0] == bstar


def _attn_case(seed, L, hq=4, hkv=1):
    nb = (L + 127) // 128
    P = nb + 1
    pages = W.permutation(seed, "ap", P)[:nb]
    bt = pages[None, :].astype(np.int32)
    kc, ks = O.new_planes(P, hkv)
    vc, vs = O.new_planes(P, hkv)
    t = np.arange(nb * 128)
    slots = pages[t // 128] * 128 + t % 128
    O.nvfp4_store(W.bf16_tensor(seed, "ak", (nb * 128, hkv, 128), 2, 10.0), slots, kc, ks)
    O.nvfp4_store(W.bf16_tensor(seed, "av", (nb * 128, hkv, 128), 2, 10.0), slots, vc, vs)
    q = W.bf16_tensor(seed, "aq", (1, hq, 128))
    return bt, kc, ks, vc, vs, q


def test_attention_full_cover_equals_dense_sdpa():
    """Top-k covering every causal block == dense causal softmax attention over the
    whole dequantised cache (torch scaled_dot_product_attention, float64)."""
    for L, hq, hkv in [(300, 4, 1), (640, 8, 2), (128, 2, 1)]:
        bt, kc, ks, vc, vs, q = _attn_case(L, L, hq, hkv)
        nb = (L + 127) // 128
        ids = np.arange(nb, dtype=np.int32)[None, :]
        sm = 1 / math.sqrt(128)
        out, lse, err = O.sparse_attention(q, hkv, kc, ks, vc, vs, bt, np.array([0]),
                                           np.array([L]), ids, sm)
        assert err == 0
        pages = bt[0]
        K = O.dequantize(kc[pages], ks[pages]).transpose(1, 0, 2, 3).reshape(hkv, -1, 128)[:, :L]
        V = O.dequantize(vc[pages], vs[pages]).transpose(1, 0, 2, 3).reshape(hkv, -1, 128)[:, :L]
        G = hq // hkv
        Kt = torch.from_numpy(np.repeat(K, G, axis=0))[None]
        Vt = torch.from_numpy(np.repeat(V, G, axis=0))[None]
        Qt = torch.from_numpy(W.bf16_bits_to_f32(q[0]).astype(np.float64))[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(Qt, Kt, Vt, scale=sm)
        np.testing.assert_allclose(out[0], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)
        logits = torch.einsum("hd,htd->ht", Qt[0, :, 0], Kt[0]) * sm
        np.testing.assert_allclose(lse[0], torch.logsumexp(logits, -1).numpy(), rtol=1e-13)


def test_attention_special_cases():
    bt, kc, ks, vc, vs, q = _attn_case(41, 256)
    p0 = bt[0, 0]
    v0 = O.dequantize(vc[p0, 0, 0], vs[p0, 0, 0])
    # row_len = 1: the output is exactly the first value row
    out, lse, _ = O.sparse_attention(q, 1, kc, ks, vc, vs, bt, np.array([0]), np.array([1]),
                                     np.array([[0, -1]]), 0.088)
    assert np.array_equal(out[0, 0], v0)
    # all keys equal: the output is the plain mean of V; lse = logit + log(n)
    kc2, ks2 = kc.copy(), ks.copy()
    kc2[:] = kc[p0, 0, 3]
    ks2[:] = ks[p0, 0, 3]
    L = 200
    out, lse, _ = O.sparse_attention(q, 1, kc2, ks2, vc, vs, bt, np.array([0]), np.array([L]),
                                     np.array([[0, 1]]), 0.088)
    V = np.concatenate([O.dequantize(vc[bt[0, 0], 0], vs[bt[0, 0], 0]),
                        O.dequantize(vc[bt[0, 1], 0], vs[bt[0, 1], 0])])[:L]
    np.testing.assert_allclose(out[0, 0], V.mean(0), rtol=1e-12, atol=1e-14)
    k0 = O.dequantize(kc[p0, 0, 3], ks[p0, 0, 3])
    qf = W.bf16_bits_to_f32(q[0, 0]).astype(np.float64)
    assert math.isclose(lse[0, 0], 0.088 * float(qf @ k0) + math.log(L), rel_tol=1e-12)
    # pad rows and empty id lists give zeros and -inf
    out, lse, err = O.sparse_attention(q, 1, kc, ks, vc, vs, bt, np.array([-1]), np.array([0]),
                                       np.array([[0, 1]]), 0.088)
    assert not out.any() and np.isneginf(lse).all() and err == 0
    # an id beyond the causal blocks is an error and is skipped
    _, _, err = O.sparse_attention(q, 1, kc, ks, vc, vs, bt, np.array([0]), np.array([100]),
                                   np.array([[0, 1]]), 0.088)
    assert err == O.ERR_BLOCK_ID


def test_verify_equals_rowmap_plus_score_topk():
    """The fused verify selection equals row map + score + top-k ("[MiniMax-M3.1]
    FP4 index cache ...", Tests: the fused top-k selects what score + top-k selects)."""
    wl = W.make("verify", ctx=(700, 1500, 333), q_rows=(3, 8, 1))
    P = wl.num_pages
    c, s = O.new_planes(P, 1)
    O.nvfp4_store(wl.ik_src, wl.slot_all, c, s)
    R = wl.spec.rows
    ids_v, err = O.verify_score_topk(wl.q_idx, wl.w, c, s, wl.block_table, wl.cu_q,
                                     wl.seq_len, R, 4)
    rr, rl = O.decode_rows(wl.cu_q, wl.seq_len, R)
    ids_u, _, _ = O.index_score_topk(wl.q_idx, wl.w, c, s, wl.block_table, rr, rl, 4)
    assert err == 0 and np.array_equal(ids_v, ids_u)
    # row j of a request sees one more token than row j-1
    assert list(rl[3:11]) == [1500 - 8 + j + 1 for j in range(8)]


# ---------------------------------------------------------------------------
# Forced init / local blocks in the top-k
# ---------------------------------------------------------------------------

def _forced_rank_restatement(scores, k, init, local):
    """Independent restatement: every block gets a tuple whose maximum ranks first."""
    nb = len(scores)
    ranked = []
    for b in range(nb):
        if b < init:
            ranked.append(((2, -b, 0.0, 0), b))
        elif b >= nb - local:
            ranked.append(((1, b, 0.0, 0), b))
        else:
            ranked.append(((0, 0, float(scores[b]), -b), b))
    ranked.sort(reverse=True)
    return sorted(b for _, b in ranked[: min(k, nb)])


def test_forced_blocks_reviews_worked_example():
    """#2744 review: topk 16, init 4, local 16 on a long row. The ids kept are the
    four init blocks and the twelve newest blocks, the current token's block
    (the last) among them; not the four init blocks plus local n-16 .. n-5."""
    nb = 100
    scores = np.linspace(5.0, -5.0, nb)              # scores alone would pick blocks 0 .. 15
    got = O.topk_ids(scores, 16, init_blocks=4, local_blocks=16)
    assert got.tolist() == [0, 1, 2, 3] + list(range(88, 100))


def test_forced_blocks_special_cases():
    rng = np.random.default_rng(5)
    sc = rng.standard_normal(40)
    # no forced blocks: the plain top-k
    assert np.array_equal(O.topk_ids(sc, 8, 0, 0), O.topk_ids(sc, 8))
    # forced blocks that fit are all kept; the rest are the best scored blocks
    got = set(O.topk_ids(sc, 8, 2, 3).tolist())
    assert {0, 1, 37, 38, 39} <= got
    rest = sorted(range(2, 37), key=lambda b: (-sc[b], b))[:3]
    assert got == {0, 1, 37, 38, 39} | set(rest)
    # init blocks alone filling k: exactly the first k blocks
    assert O.topk_ids(sc, 8, 10, 5).tolist() == list(range(8))
    # a row no longer than k: every block, whatever is forced
    assert O.topk_ids(sc[:5], 8, 2, 2).tolist() == [0, 1, 2, 3, 4, -1, -1, -1]
    # init and local overlapping on a short row: the block counts once, as init
    assert O.topk_ids(sc[:12], 4, 3, 10).tolist() == [0, 1, 2, 11]


def test_forced_blocks_against_restatement():
    rng = np.random.default_rng(6)
    for _ in range(300):
        nb = int(rng.integers(1, 60))
        k = int(rng.integers(1, 20))
        init, local = int(rng.integers(0, 8)), int(rng.integers(0, 24))
        sc = np.round(rng.standard_normal(nb), 1)   # ties
        got = O.topk_ids(sc, k, init, local)
        exp = _forced_rank_restatement(sc, k, init, local)
        cnt = min(k, nb)
        assert got[:cnt].tolist() == exp and (got[cnt:] == -1).all()


# --------------------------------------------------------------------------
# MXFP4 (e2m1 + E8M0 per 32): "[MiniMax-M3.1] FP4 index cache and NVFP4
# sparse KV cache" (#2744), Follow-up: MXFP4 caches; vllm #64198, Overview
# --------------------------------------------------------------------------

MX_GOLDEN = __file__.rsplit("/", 1)[0] + "/golden/mxfp4_quant_groups.txt"


def _mx_golden_cases():
    cases, cur = [], None
    for line in open(MX_GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("case "):
            cur = {"name": line[5:]}
            cases.append(cur)
        else:
            k, v = line.split(":", 1)
            cur[k] = v.split()
    return cases


def _mx_value(tok):
    return float.fromhex(tok) if tok.lstrip("-").startswith("0x") else float(tok)


def _mx_row(case):
    g = int(case["group"][0])
    x = np.zeros(128, dtype=np.float32)
    vals = [_mx_value(t) for t in case["x"]]
    x[32 * g: 32 * g + len(vals)] = vals
    bits = W.f32_to_bf16_bits(x)
    assert np.array_equal(W.bf16_bits_to_f32(bits), x)   # BF16-exact inputs
    return bits, g, len(vals)


@pytest.mark.parametrize("case", _mx_golden_cases(), ids=lambda c: c["name"])
def test_mx_quantiser_hand_worked(case):
    bits, g, n = _mx_row(case)
    codes, scales = O.quantize(bits, mx=True)
    assert scales.shape == (4,) and codes.shape == (64,)
    for j in range(4):
        assert scales[j] == (int(case["scale"][0], 16) if j == g else 0), j
    got = [(codes[(32 * g + i) // 2] >> (4 * (i % 2))) & 0xF for i in range(32)]
    assert got[:n] == [int(c, 16) for c in case["codes"]]
    assert not any(got[n:])
    other = np.delete(codes.reshape(4, 16), g, axis=0)
    assert not other.any()


def test_e8m0_table_matches_torch():
    """Every E8M0 byte decodes as torch's float8_e8m0fnu does (library routine)."""
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    allb = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).float().double().numpy()
    nan = np.isnan(allb)
    assert nan.sum() == 1 and nan[255]
    assert np.array_equal(allb[~nan], O.E8M0_ALL[~nan])


def _exact_quantise_mx_group(xs):
    """Independent restatement in exact rationals of one 32-group: the shared
    exponent is the largest k with 2^(k+2) <= amax (found by stepping), clamped."""
    fr = [Fraction(float(x)) for x in xs]
    amax = max(abs(x) for x in fr)
    if amax == 0:
        k = -127
    else:
        k = 0
        while Fraction(2) ** (k + 2) > amax:
            k -= 1
        while Fraction(2) ** (k + 3) <= amax:
            k += 1
        k = max(-127, min(127, k))
    s = Fraction(2) ** k
    grid = [Fraction(g) for g in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    codes = []
    for x, xf in zip(xs, fr):
        q = abs(xf) / s
        m = min(range(8), key=lambda i: (abs(grid[i] - q), i % 2))
        codes.append(m | (8 if math.copysign(1.0, float(x)) < 0 else 0))
    return k + 127, codes


def test_mx_quantiser_equals_exact_rational_definition():
    """Vectorised MX quantiser == exact-rational brute force on random groups over
    a wide exponent range (BF16 subnormals included), with ties planted."""
    rng = np.random.default_rng(11)
    rows = []
    for i in range(40):
        e = int(rng.integers(-135, 120))
        x = rng.standard_normal(128) * 2.0 ** e
        if i % 3 == 0:        # exact ties at a power-of-two scale
            x[:7] = np.array([.25, .75, 1.25, 1.75, 2.5, 3.5, 5]) * 2.0 ** (e - 3)
            x[7] = 7 * 2.0 ** (e - 3)
        rows.append(x)
    bits = W.f32_to_bf16_bits(np.array(rows, dtype=np.float32))
    bits[(bits & 0x7F80) == 0x7F80] &= 0x807F     # no inf / NaN from the float32 range
    xs = W.bf16_bits_to_f32(bits).astype(np.float64)
    codes, scales = O.quantize(bits, mx=True)
    for r in range(len(rows)):
        for g in range(4):
            s, c = _exact_quantise_mx_group(xs[r, 32 * g: 32 * g + 32])
            assert scales[r, g] == s, (r, g)
            got = [(codes[r, 16 * g + i // 2] >> (4 * (i % 2))) & 0xF for i in range(32)]
            assert got == c, (r, g)


def test_mx_round_trip_error_bound():
    """|x - x_hat| <= half the local e2m1 step x 2^E below 6 x 2^E, and <= 2 x 2^E
    in the saturating band (6, 8) x 2^E; every group uses its top code range
    (amax / 2^E lies in [4, 8))."""
    bits = W.bf16_tensor(7, "mxrt", (512, 128), 4, 20.0)
    x = W.bf16_bits_to_f32(bits).astype(np.float64)
    c, s = O.quantize(bits, mx=True)
    xh = O.dequantize(c, s)
    sv = np.repeat(O.E8M0_ALL[s], 32, axis=-1)
    q = np.abs(x) / sv
    step = np.where(q < 2, 0.5, np.where(q < 4, 1.0, 2.0))
    unsat = q <= 6
    assert np.all(np.abs(x - xh)[unsat] <= (0.5 * step * sv)[unsat])
    assert np.all(np.abs(x - xh)[~unsat] <= (2.0 * sv)[~unsat])
    amax_q = q.reshape(512, 4, 32).max(-1)
    assert np.all((amax_q >= 4) & (amax_q < 8))


def test_mx_record_and_page_size_reproduce_pages():
    """68 B per token and head, and a 128-token page per head of
    [128 x 64 B e2m1][128 x 4 B e8m0] = 8704 B (vllm #64198, Claims)."""
    c, s = O.new_planes(1, 1, mx=True)
    assert c.shape[-1] + s.shape[-1] == 68
    assert c[0, 0].nbytes + s[0, 0].nbytes == 8704


def test_mx_and_nvfp4_dequantise_alike_where_both_represent_the_values():
    """Records whose every group has scale 1 in both formats (E8M0 0x7f, E4M3
    0x38) dequantise to the same values, and the oracle's scorer and attention
    give the same results over them."""
    rng = np.random.default_rng(5)
    P, L = 3, 300
    codes = rng.integers(0, 256, size=(P, 1, 128, 64), dtype=np.uint8)
    s_nv = np.full((P, 1, 128, 8), 0x38, dtype=np.uint8)
    s_mx = np.full((P, 1, 128, 4), 0x7F, dtype=np.uint8)
    assert np.array_equal(O.dequantize(codes, s_nv), O.dequantize(codes, s_mx))
    bt = np.array([[2, 0, 1]], dtype=np.int32)
    rr, rl = np.array([0], dtype=np.int32), np.array([L], dtype=np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((1, 2, 128)).astype(np.float32))
    w = rng.random((1, 2))
    ids_nv, bs_nv, _ = O.index_score_topk(q, w, codes, s_nv, bt, rr, rl, 2)
    ids_mx, bs_mx, _ = O.index_score_topk(q, w, codes, s_mx, bt, rr, rl, 2)
    assert np.array_equal(ids_nv, ids_mx) and np.array_equal(bs_nv, bs_mx)
    qa = W.f32_to_bf16_bits(rng.standard_normal((1, 4, 128)).astype(np.float32))
    ids = np.array([[0, 2]], dtype=np.int32)
    o_nv, l_nv, _ = O.sparse_attention(qa, 1, codes, s_nv, codes, s_nv, bt, rr, rl, ids, 0.1)
    o_mx, l_mx, _ = O.sparse_attention(qa, 1, codes, s_mx, codes, s_mx, bt, rr, rl, ids, 0.1)
    assert np.array_equal(o_nv, o_mx) and np.array_equal(l_nv, l_mx)


def test_mx_store_into_mx_planes():
    """The store picks the MXFP4 quantiser from the planes' 4-byte scale records and
    leaves pad rows untouched."""
    H, T, P = 2, 30, 3
    src = W.bf16_tensor(4, "mxst", (T, H, 128), 2, 10.0)
    slots = W.permutation(4, "mxslots", P * 128)[:T].astype(np.int64)
    slots[4] = -1
    c, s = O.new_planes(P, H, mx=True)
    c[:] = 0xA5
    s[:] = 0x5A
    assert O.nvfp4_store(src, slots, c, s) == 0
    qc, qs = O.quantize(src, mx=True)
    for r, slot in enumerate(slots):
        if slot < 0:
            continue
        assert np.array_equal(c[slot // 128, :, slot % 128], qc[r])
        assert np.array_equal(s[slot // 128, :, slot % 128], qs[r])
    written = set(int(v) for v in slots if v >= 0)
    for slot in range(P * 128):
        if slot not in written:
            assert (c[slot // 128, :, slot % 128] == 0xA5).all()
            assert (s[slot // 128, :, slot % 128] == 0x5A).all()


# --------------------------------------------------------------------------
# Quantise-at-write (normalise / rotate / write, the quantisation inside):
# #2744, Follow-up: MXFP4 caches ("the quantization happens inside the fused
# qk-norm/RoPE/cache kernel, so there is no staging buffer and no store launch")
# --------------------------------------------------------------------------

def _rope_tables(T, half, base=10000.0, pos0=3):
    t = (pos0 + np.arange(T))[:, None] * (base ** (-np.arange(half) / half))[None, :]
    return np.cos(t).astype(np.float32), np.sin(t).astype(np.float32)


def test_bf16_rounding_matches_torch():
    """f32 -> BF16 (nearest, ties to even) equals torch's conversion, ties included."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal(4096).astype(np.float32) * np.float32(2.0) ** rng.integers(-60, 60, 4096)
    hi = rng.integers(0, 1 << 16, 512).astype(np.uint32)
    hi = hi[(hi & 0x7F80) != 0x7F80]                      # finite patterns only
    ties = ((hi << np.uint32(16)) | np.uint32(0x8000)).astype(np.uint32)
    x = np.concatenate([x, ties.view(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_bits(x), want)


def test_head_sum_of_squares_within_f32_rounding_of_exact():
    """The kernel-order float32 sum of squares lies within the rounding bound of
    the exact sum (math.fsum over the exact squares)."""
    rng = np.random.default_rng(4)
    x = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((64, 128)).astype(np.float32) * 3))
    got = O.head_sum_sq_f32(x)
    for r in range(64):
        exact = math.fsum(float(v) * float(v) for v in x[r].astype(np.float64))
        assert abs(float(got[r]) - exact) <= 140 * 2.0 ** -24 * exact


def test_norm_rope_against_torch_rms_norm_and_complex_rotation():
    """RMSNorm (torch.nn.functional.rms_norm, fp64) followed by rotate-half RoPE
    written as complex multiplication: the oracle's BF16 rows agree within BF16
    rounding plus float32 arithmetic."""
    rng = np.random.default_rng(6)
    T, H, r = 6, 3, 64
    x = W.f32_to_bf16_bits((rng.standard_normal((T, H, 128)) * 4).astype(np.float32))
    w = (rng.random(128) + 0.5).astype(np.float32)
    cos, sin = _rope_tables(T, r // 2)
    got = O.bf16_to_f64(O.norm_rope_rows(x, w, cos, sin, r, 1e-6))
    xt = torch.from_numpy(O.bf16_to_f64(x))
    nt = torch.nn.functional.rms_norm(xt, (128,), torch.from_numpy(w.astype(np.float64)), eps=1e-6)
    rot = torch.complex(nt[..., : r // 2], nt[..., r // 2: r]) * torch.complex(
        torch.from_numpy(cos.astype(np.float64))[:, None, :], torch.from_numpy(sin.astype(np.float64))[:, None, :])
    ref = torch.cat([rot.real, rot.imag, nt[..., r:]], -1).numpy()
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)


def test_norm_rope_f64_against_torch_rms_norm_and_complex_rotation():
    """The unrounded float64 rows equal torch's rms_norm (fp64) followed by the
    rotation written as a complex product, to fp64 rounding; with neither step
    the rows come back exactly."""
    rng = np.random.default_rng(16)
    T, H, r = 5, 2, 48
    x = W.f32_to_bf16_bits((rng.standard_normal((T, H, 128)) * 2.0 ** rng.integers(-30, 30, (T, H, 1)))
                           .astype(np.float32))
    w = (rng.random(128) + 0.5).astype(np.float32)
    cos, sin = _rope_tables(T, r // 2)
    got = O.norm_rope_rows_f64(x, w, cos, sin, r, 1e-6)
    xt = torch.from_numpy(O.bf16_to_f64(x))
    nt = torch.nn.functional.rms_norm(xt, (128,), torch.from_numpy(w.astype(np.float64)), eps=1e-6)
    rot = torch.complex(nt[..., : r // 2], nt[..., r // 2: r]) * torch.complex(
        torch.from_numpy(cos.astype(np.float64))[:, None, :], torch.from_numpy(sin.astype(np.float64))[:, None, :])
    ref = torch.cat([rot.real, rot.imag, nt[..., r:]], -1).numpy()
    mag = np.abs(nt.numpy()).max(axis=-1, keepdims=True)
    assert np.all(np.abs(got - ref) <= 1e-13 * mag)
    assert np.array_equal(O.norm_rope_rows_f64(x, None, None, None, 0, 1e-6), O.bf16_to_f64(x))


def test_norm_rope_special_cases():
    """No norm and no rotation give the rows back bit for bit; angle 0 is the
    identity; a zero row stays zero; a constant row of c with unit weights
    normalises to c / sqrt(c^2 + eps); the rotation keeps each pair's norm."""
    rng = np.random.default_rng(8)
    x = W.f32_to_bf16_bits(rng.standard_normal((4, 2, 128)).astype(np.float32))
    assert np.array_equal(O.norm_rope_rows(x, None, None, None, 0, 1e-6), x)
    c1, s0 = np.ones((4, 64), np.float32), np.zeros((4, 64), np.float32)
    assert np.array_equal(O.norm_rope_rows(x, None, c1, s0, 128, 1e-6), x)
    z = np.zeros((1, 1, 128), dtype=np.uint16)
    assert not O.norm_rope_rows(z, np.ones(128, np.float32), None, None, 0, 1e-6).any()
    c = np.full((1, 1, 128), W.f32_to_bf16_bits(np.float32([-0.75]))[0], dtype=np.uint16)
    y = O.bf16_to_f64(O.norm_rope_rows(c, np.ones(128, np.float32), None, None, 0, 1e-6))
    assert np.allclose(y, -0.75 / math.sqrt(0.5625 + 1e-6), rtol=2.0 ** -8)
    # eps equal to the mean square: a constant row of a = 2^-10 with eps = 2^-20
    # normalises to a / sqrt(a^2 + eps) = 1 / sqrt(2)
    a = np.full((1, 1, 128), W.f32_to_bf16_bits(np.float32([2.0 ** -10]))[0], dtype=np.uint16)
    y = O.bf16_to_f64(O.norm_rope_rows(a, np.ones(128, np.float32), None, None, 0, 2.0 ** -20))
    assert np.allclose(y, 1 / math.sqrt(2), rtol=2.0 ** -8)
    y64 = O.norm_rope_rows_f64(a, np.ones(128), None, None, 0, 2.0 ** -20)
    assert np.allclose(y64, 1 / math.sqrt(2), rtol=1e-14)
    cos, sin = _rope_tables(4, 64)
    xr = O.bf16_to_f64(x)
    yr = O.bf16_to_f64(O.norm_rope_rows(x, None, cos, sin, 128, 1e-6))
    n0 = np.hypot(xr[..., :64], xr[..., 64:])
    n1 = np.hypot(yr[..., :64], yr[..., 64:])
    assert np.all(np.abs(n1 - n0) <= n0 * 2.0 ** -7 + 1e-30)


def test_fused_write_job_without_norm_or_rope_is_the_plain_store():
    """A job with no weight and no RoPE stores its rows as the plain store does,
    byte for byte, while another job of the same call is rotated."""
    T, P = 200, 3
    src = W.bf16_tensor(44, "fw", (T, 1, 128), 2, 10.0)
    slots = W.permutation(44, "fs", P * 128)[:T].astype(np.int64)
    cos, sin = _rope_tables(T, 32)
    plain = O.new_planes(P, 1)
    assert O.nvfp4_store(src, slots, *plain) == 0
    fused, rotated = O.new_planes(P, 1), O.new_planes(P, 1)
    O.qk_norm_rope_store([(src, None, False, fused), (src, None, True, rotated)], slots, cos, sin, 64, 1e-6)
    assert np.array_equal(fused[0], plain[0]) and np.array_equal(fused[1], plain[1])
    assert not np.array_equal(rotated[0], plain[0])


def test_quantise_at_write_equals_staging_then_store():
    """The fused write fills the planes exactly as the unfused path does: the
    normalised rows to a BF16 staging buffer, then the store (#2744, Summary /
    Write), for both record formats; BF16 destinations receive the rows."""
    rng = np.random.default_rng(9)
    T, P = 20, 2
    cos, sin = _rope_tables(T, 32)
    slots = rng.permutation(P * 128)[:T].astype(np.int64)
    slots[3] = -1
    k = W.f32_to_bf16_bits(rng.standard_normal((T, 2, 128)).astype(np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((T, 4, 128)).astype(np.float32))
    wk = (rng.random(128) + 0.5).astype(np.float32)
    for mx in (False, True):
        kc, ks = O.new_planes(P, 2, mx=mx)
        qo = np.zeros_like(q)
        assert O.qk_norm_rope_store([(k, wk, True, (kc, ks)), (q, None, True, qo)], slots,
                                    cos, sin, 64, 1e-6) == 0
        staged = O.norm_rope_rows(k, wk, cos, sin, 64, 1e-6)
        rc, rs = O.new_planes(P, 2, mx=mx)
        O.nvfp4_store(staged, slots, rc, rs)
        assert np.array_equal(kc, rc) and np.array_equal(ks, rs)
        assert np.array_equal(qo, O.norm_rope_rows(q, None, cos, sin, 64, 1e-6))


# --------------------------------------------------------------------------
# Indexer context parallelism: per-rank candidates, then a merge (#2744, review
# thread on the unused page-16 tables: merge_candidate_keys)
# --------------------------------------------------------------------------

def test_split_candidates_merge_to_the_unsplit_top_k():
    """For any cut of a row's blocks into contiguous slices, merging each slice's k
    best equals the row's top k (topk_ids, itself pinned by brute force): ties to
    the lower id and forced init / local blocks included."""
    rng = np.random.default_rng(40)
    for trial in range(400):
        nb = int(rng.integers(1, 90))
        k = int(rng.integers(1, 20))
        sc = rng.integers(0, 6, nb).astype(np.float64) if trial % 3 == 0 else rng.standard_normal(nb)
        init = int(rng.integers(0, 4)) if trial % 2 else 0
        local = int(rng.integers(0, 5)) if trial % 2 else 0
        n = int(rng.integers(1, 6))
        cuts = np.sort(rng.integers(0, nb + 1, n - 1))
        bounds = [0, *cuts.tolist(), nb]
        lists = [O.slice_candidates(sc, bounds[i], bounds[i + 1], k, init, local) for i in range(n)]
        assert all(len(lst) <= k for lst in lists)
        assert np.array_equal(O.merge_candidates(lists, k), O.topk_ids(sc, k, init, local)), trial


def test_slice_candidates_special_cases():
    """An empty slice has no candidates; a slice of at most k blocks keeps them all;
    the whole row as one slice gives topk_ids' set, best first."""
    sc = np.array([3.0, 1.0, 4.0, 1.0, 5.0])
    assert O.slice_candidates(sc, 2, 2, 3) == []
    assert sorted(r[2] for r in O.slice_candidates(sc, 1, 3, 5)) == [1, 2]
    best = O.slice_candidates(sc, 0, 5, 3)
    assert [r[2] for r in best] == [4, 2, 0]
    assert np.array_equal(O.merge_candidates([best], 3), O.topk_ids(sc, 3))
    # equal scores: the lower id first; forced: init (lower id first) above local
    assert [r[2] for r in O.slice_candidates(np.zeros(6), 0, 6, 6, 1, 2)] == [0, 5, 4, 1, 2, 3]
