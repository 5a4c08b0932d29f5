"""The GPU parity tests' acceptance checks, run on the CPU against planted wrong
answers: each check must reject a result that breaks its rule and accept one
that the rule allows (exact results, and differences inside the top-k tie
band). Without this, a check that accepted everything would make every GPU
parity test pass."""

import numpy as np
import pytest

from oracle import m3s_oracle as O
from step_helpers import (ATTN_RTOL, SCORE_RTOL, TIE_BAND, attention_rel_err, check_block_scores, check_topk,
                          check_topk_forced)


def _scores():
    rng = np.random.default_rng(5)
    return [rng.standard_normal(40) * 3.0, rng.standard_normal(9), np.abs(rng.standard_normal(130)) + 1.0]


def _gpu_matrix(scores, width=140):
    m = np.full((len(scores), width), np.nan, dtype=np.float32)
    for r, s in enumerate(scores):
        m[r, : len(s)] = s
    return m


def test_block_scores_rule():
    ref = _scores()
    check_block_scores(_gpu_matrix(ref), ref, range(3))
    ok = [s * (1 + 0.5 * SCORE_RTOL) for s in ref]
    check_block_scores(_gpu_matrix(ok), ref, range(3))
    bad = [s.copy() for s in ref]
    bad[2][77] *= 1 + 3 * SCORE_RTOL
    with pytest.raises(AssertionError):
        check_block_scores(_gpu_matrix(bad), ref, range(3))


def _ids(scores, k):
    return np.stack([O.topk_ids(s, k) for s in scores])


def test_top_k_rule_rejects_wrong_selections():
    ref = _scores()
    k = 16
    good = _ids(ref, k)
    assert check_topk(good, ref, k, range(3), _gpu_matrix(ref)) == 0
    # a block well above the band swapped for one well below it
    r = 0
    order = np.argsort(-ref[r], kind="stable")
    wrong = good.copy()
    sel = set(good[r][good[r] >= 0].tolist())
    sel.discard(int(order[0]))
    sel.add(int(order[-1]))
    wrong[r, :k] = sorted(sel)
    with pytest.raises(AssertionError):
        check_topk(wrong, ref, k, range(3))
    # unsorted ids, a missing pad, an id past the row's blocks
    unsorted = good.copy()
    unsorted[0, [0, 1]] = unsorted[0, [1, 0]]
    with pytest.raises(AssertionError):
        check_topk(unsorted, ref, k, range(3))
    nopad = good.copy()
    nopad[1, -1] = 3            # row 1 has 9 blocks: places 9.. must be -1
    with pytest.raises(AssertionError):
        check_topk(nopad, ref, k, range(3))
    past = good.copy()
    past[1, 8] = 9
    with pytest.raises(AssertionError):
        check_topk(past, ref, k, range(3))


def test_top_k_rule_allows_the_tie_band_only():
    k = 4
    base = np.array([9.0, 8.0, 7.0, 5.0, 5.0 * (1 - 0.5 * TIE_BAND), 1.0, 0.5])
    ids_ref = O.topk_ids(base, k)                      # 0, 1, 2, 3
    swapped = np.array([[0, 1, 2, 4]], dtype=np.int32)  # block 4 sits inside the band around block 3
    assert list(ids_ref) == [0, 1, 2, 3]
    assert check_topk(swapped, [base], k, [0]) == 1
    far = base.copy()
    far[4] = 5.0 * (1 - 10 * TIE_BAND)                  # now outside the band
    with pytest.raises(AssertionError):
        check_topk(swapped, [far], k, [0])
    # with the GPU's own scores given, the ids must be exactly their top-k (ties to the lower id)
    own = np.array([[9.0, 8.0, 7.0, 5.0, 5.0, 1.0, 0.5]], dtype=np.float32)
    with pytest.raises(AssertionError):
        check_topk(swapped, [base], k, [0], own)


def test_forced_top_k_rule():
    rng = np.random.default_rng(6)
    sc = rng.standard_normal(30)
    k, init, local = 8, 2, 3
    good = O.topk_ids(sc, k, init, local)[None, :]
    check_topk_forced(good, [sc], k, [0], init, local)
    dropped = good.copy()                     # forced block 0 replaced by the best unforced block not chosen
    free = [b for b in np.argsort(-sc) if init <= b < 30 - local and b not in good[0]]
    row = sorted((set(good[0].tolist()) - {0}) | {int(free[0])})
    dropped[0, :] = row
    with pytest.raises(AssertionError):
        check_topk_forced(dropped, [sc], k, [0], init, local)


def test_attention_error_measure():
    ref = np.zeros((2, 3, 128))
    ref[0, :, 0] = [1.0, -2.0, 4.0]
    ref[1, :, 5] = 10.0
    out = ref.copy()
    out[0, 1, 0] += 2.0 * 0.5 * ATTN_RTOL      # head 1's max magnitude is 2
    assert attention_rel_err(out, ref, range(2)) == pytest.approx(0.5 * ATTN_RTOL)
    out[1, 2, 7] = 10.0 * 2 * ATTN_RTOL
    assert attention_rel_err(out, ref, range(2)) > ATTN_RTOL
    zero = np.zeros((1, 1, 128))
    nonzero = zero.copy()
    nonzero[0, 0, 3] = 1e-3
    with pytest.raises(AssertionError):          # a row the oracle leaves empty must stay zero
        attention_rel_err(nonzero, zero, range(1))
