"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in a copy of the oracle's source: a
dropped term, a wrong sign, constant or index, swapped operands, an off-by-one,
or a wrong tie or priority rule. The case requires that at least one pin in
test_oracle_pins fails on the mutated copy. The mutated copy exists only in
this process; the oracle's file is never modified. A control case runs the
pins on an unmutated copy built the same way, so a failure here means a pin
is blind to that mistake and not that the harness is broken.
"""

import inspect
import types

import pytest

import test_oracle_pins as P
from oracle import m3s_oracle as O

SRC = open(O.__file__).read()

# name -> [(text in the oracle's source, its replacement)]; each text occurs once
MUTANTS = {
    # number formats
    "e4m3 subnormal exponent": [("return sign * m * 2.0 ** -9", "return sign * m * 2.0 ** -10")],
    "e4m3 bias": [("return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)",
                   "return sign * (1.0 + m / 8.0) * 2.0 ** (e - 8)")],
    "ties round up, not to even": [("return np.where(at & (below % 2 == 1), below + 1, below)",
                                    "return np.where(at, below + 1, below)")],
    "ties round down": [("return np.where(at & (below % 2 == 1), below + 1, below)",
                         "return below")],
    "e8m0 bias": [("math.ldexp(1.0, code - 127)", "math.ldexp(1.0, code - 128)")],
    # quantisation
    "nvfp4 scale = e4m3(amax / 4)": [("_nearest_even(amax, E4M3_POS, 6.0)", "_nearest_even(amax, E4M3_POS, 4.0)")],
    "nvfp4 sign bit dropped": [("    code = (sign << np.uint8(3)) | mag\n", "    code = mag + 0 * sign\n")],
    "zero-scale group keeps its codes": [
        ("code = np.where((s == 0.0)[..., None], np.uint8(0), code).astype(np.uint8)", "code = code.astype(np.uint8)")],
    "mx exponent floor(log2 amax) - 1": [("e.astype(np.int64) - 1 - 2", "e.astype(np.int64) - 1 - 1")],
    # (the upper clamp never binds for BF16 input: the largest BF16 gives E = 125)
    "mx exponent clamped at -126": [("E = np.clip(E, -127, 127)", "E = np.clip(E, -126, 127)")],
    "dequantise nibbles swapped": [("c = np.stack([lo, hi], axis=-1)", "c = np.stack([hi, lo], axis=-1)")],
    "dequantise scale of the wrong group": [("return val * np.repeat(E4M3_ALL[scales], GROUP, axis=-1)",
                                             "return val * np.tile(E4M3_ALL[scales], GROUP)")],
    "dequantise mx sign dropped": [("val = E2M1_GRID[c & 7] * np.where(c & 8, -1.0, 1.0)",
                                    "val = E2M1_GRID[c & 7] * np.where(c & 8, 1.0, 1.0)")],
    # store
    "store: page and offset swapped": [("codes[slot // PAGE, :, slot % PAGE] = c[r]",
                                        "codes[slot % PAGE, :, slot // PAGE] = c[r]")],
    "store: slot -1 not a pad row": [("        if slot < 0:\n            continue", "        if slot < -1:\n            continue")],
    "store: out-of-range slot not reported": [("            err |= ERR_SLOT\n", "            err |= 0\n")],
    # row map
    "row map: causal length one short": [("row_len[r] = int(seq_len[b]) - qb + j + 1",
                                          "row_len[r] = int(seq_len[b]) - qb + j")],
    "row map: rows are the first positions": [("row_len[r] = int(seq_len[b]) - qb + j + 1", "row_len[r] = j + 1")],
    # index scoring
    "scores: ReLU dropped": [("return np.maximum(s, 0.0) @ np.asarray(w_row, dtype=np.float64)",
                              "return s @ np.asarray(w_row, dtype=np.float64)")],
    "scores: weights of the reversed heads": [("return np.maximum(s, 0.0) @ np.asarray(w_row, dtype=np.float64)",
                                               "return np.maximum(s, 0.0) @ np.asarray(w_row, dtype=np.float64)[::-1]")],
    "scores: weight inside the ReLU with its sign lost": [
        ("return np.maximum(s, 0.0) @ np.asarray(w_row, dtype=np.float64)",
         "return np.maximum(s * np.abs(np.asarray(w_row, dtype=np.float64)), 0.0).sum(axis=-1)")],
    "block max: one token of the next block": [("out[b] = score[b * PAGE: min((b + 1) * PAGE, L)].max()",
                                                "out[b] = score[b * PAGE: min((b + 1) * PAGE + 1, L)].max()")],
    "block max: first token left out": [("out[b] = score[b * PAGE: min((b + 1) * PAGE, L)].max()",
                                         "out[b] = score[b * PAGE + 1: min((b + 1) * PAGE, L)].max(initial=-np.inf)")],
    "scores past the causal length": [("k_hat = cache[key][:L]", "k_hat = cache[key]"),
                                      ("out[b] = score[b * PAGE: min((b + 1) * PAGE, L)].max()",
                                       "out[b] = score[b * PAGE: (b + 1) * PAGE].max()")],
    # top-k and forced blocks
    "top-k: ties to the higher id": [("order = np.lexsort((ids, within, -cls))", "order = np.lexsort((-ids, within, -cls))")],
    "top-k: lowest scores": [("np.where(local, -ids.astype(np.float64), -np.asarray(bscore, dtype=np.float64))",
                              "np.where(local, -ids.astype(np.float64), np.asarray(bscore, dtype=np.float64))")],
    "top-k: k - 1 kept": [("sel = np.sort(order[: min(k, nb)])", "sel = np.sort(order[: min(k - 1, nb)])")],
    "top-k: ids not sorted": [("sel = np.sort(order[: min(k, nb)])", "sel = order[: min(k, nb)]")],
    "forced: local above init": [("cls = np.where(init, 2, np.where(local, 1, 0))",
                                  "cls = np.where(init, 1, np.where(local, 2, 0))")],
    "forced: local oldest first": [("np.where(local, -ids.astype(np.float64), -np.asarray(",
                                    "np.where(local, ids.astype(np.float64), -np.asarray(")],
    "forced: init highest id first": [("within = np.where(init, ids.astype(np.float64),",
                                       "within = np.where(init, -ids.astype(np.float64),")],
    "forced: local blocks one too many": [("local = (ids >= nb - local_blocks) & ~init",
                                           "local = (ids >= nb - local_blocks - 1) & ~init")],
    # context-parallel candidates
    "cp: local records oldest first": [("out.append((1, float(i), i))", "out.append((1, -float(i), i))")],
    "cp: init records highest id first": [("out.append((2, -float(i), i))", "out.append((2, float(i), i))")],
    "cp: merge keeps k - 1": [("union = _best_first([rec for lst in lists for rec in lst])[:k]",
                               "union = _best_first([rec for lst in lists for rec in lst])[:k - 1]")],
    "cp: ties to the higher id": [("key=lambda rec: (-rec[0], -rec[1], rec[2])", "key=lambda rec: (-rec[0], -rec[1], -rec[2])")],
    "cp: forced blocks by the slice's own count": [
        ("recs = rank_records(bscore, range(max(0, lo), min(hi, nb)), nb, init_blocks, local_blocks)",
         "recs = rank_records(bscore, range(max(0, lo), min(hi, nb)), min(hi, nb), init_blocks, local_blocks)")],
    # attention
    "attention: sm_scale dropped": [("logits = sm_scale * (kh @ q_r[h])", "logits = kh @ q_r[h]")],
    "attention: K and V swapped": [("out[r, h] = (p @ vh) / l", "out[r, h] = (p @ kh) / l")],
    "attention: not normalised": [("out[r, h] = (p @ vh) / l", "out[r, h] = p @ vh")],
    "attention: lse without the maximum": [("lse[r, h] = m + math.log(l)", "lse[r, h] = math.log(l)")],
    "attention: last block past the causal length": [("toks.append((i, min(PAGE, L - i * PAGE)))",
                                                      "toks.append((i, PAGE))")],
    "attention: q heads interleaved over KV heads": [("for h in range(kvh * G, (kvh + 1) * G):",
                                                      "for h in range(kvh, Hq, hkv):")],
    "attention: out-of-range id not reported": [("                err |= ERR_BLOCK_ID\n", "                err |= 0\n")],
    # quantise-at-write
    "rope: sign of the first half": [("o1 = y1 * c - y2 * s", "o1 = y1 * c + y2 * s")],
    "rope: interleaved pairs, not rotate-half": [
        ("y1, y2 = y[..., :h], y[..., h:rotary_dim]", "y1, y2 = y[..., 0:rotary_dim:2], y[..., 1:rotary_dim:2]")],
    "rope f64: sign of the second half": [("y[..., h:rotary_dim] = y2 * c + y1 * s", "y[..., h:rotary_dim] = y2 * c - y1 * s")],
    "rmsnorm: sum, not mean": [("v = ss * np.float32(1.0 / 128) + np.float32(eps)", "v = ss + np.float32(eps)")],
    "rmsnorm: eps outside the root": [("r = np.float32(1.0) / np.sqrt(v)",
                                       "r = np.float32(1.0) / (np.sqrt(v - np.float32(eps)) + np.float32(eps))")],
    "rmsnorm: weight dropped": [("y = (x * r[..., None]) * _f32(weight)", "y = x * r[..., None]")],
    "rmsnorm f64: sum, not mean": [("np.sqrt(ss / HEAD_DIM + float(eps))", "np.sqrt(ss + float(eps))")],
    "rmsnorm f64: eps outside the root": [("np.sqrt(ss / HEAD_DIM + float(eps))", "(np.sqrt(ss / HEAD_DIM) + float(eps))")],
    "bf16 rounding: ties away from zero": [("r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "r = (u + 0x8000) >> 16")],
    "bf16 rounding: truncation": [("r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16", "r = u >> 16")],
    "f32 sum of squares: butterfly one level short": [("for off in (16, 8, 4, 2, 1):", "for off in (16, 8, 4, 2):")],
    "fused write: RoPE on every job": [("cos if rope else None, sin if rope else None", "cos, sin")],
    "fused write: RMSNorm weight ignored": [("rows = norm_rope_rows(src, weight,", "rows = norm_rope_rows(src, None,")],
    # more of the scoring and attention paths
    "mx quantiser: sign dropped": [("code = ((sign << np.uint8(3)) | mag).reshape(lead + (HEAD_DIM,))",
                                    "code = (mag + 0 * sign).reshape(lead + (HEAD_DIM,))")],
    "nvfp4 groups strided, not contiguous": [
        ("x = bf16_to_f64(bits).reshape(lead + (SCALE_BYTES, GROUP))",
         "x = bf16_to_f64(bits).reshape(lead + (GROUP, SCALE_BYTES)).swapaxes(-1, -2)")],
    "request's pages in reverse order": [
        ("x = dequantize(codes[pages[:nb], head], scales[pages[:nb], head])",
         "x = dequantize(codes[pages[:nb][::-1], head], scales[pages[:nb][::-1], head])")],
    "scoring: bad page not reported": [("        err |= ERR_PAGE\n    return pages, err",
                                        "        err |= 0\n    return pages, err")],
    "scoring: row past the block table not reported": [("        err |= ERR_ROW\n", "        err |= 0\n")],
    "scoring: token cache keyed by request only": [("key = (b, nb)", "key = b")],
    "forced: init blocks counted from the end": [("init = ids < init_blocks", "init = ids >= nb - init_blocks")],
    "attention: softmax without the maximum": [("p = np.exp(logits - m)", "p = np.exp(logits)")],
    "attention: lse in base 2": [("lse[r, h] = m + math.log(l)", "lse[r, h] = m + math.log2(l)")],
    "attention: ids past the causal length attended": [("if i >= nb or i >= block_table.shape[1]:",
                                                        "if i >= block_table.shape[1]:")],
    "attention: bad page not reported": [("            err |= ERR_PAGE\n            continue",
                                          "            continue")],
    "attention: K of the next KV head": [("kh = np.concatenate([dequantize(k_codes[p, kvh, :n], k_scales[p, kvh, :n])",
                                           "kh = np.concatenate([dequantize(k_codes[p, (kvh + 1) % hkv, :n], "
                                           "k_scales[p, (kvh + 1) % hkv, :n])")],
    "row map: padding rows take the last request": [("row_req = np.full(R, -1, dtype=np.int32)",
                                                     "row_req = np.full(R, len(seq_len) - 1, dtype=np.int32)")],
}


def _mutant(edits):
    src = SRC
    for old, new in edits:
        assert src.count(old) == 1, f"mutation site not found exactly once: {old!r}"
        src = src.replace(old, new)
    mod = types.ModuleType("m3s_oracle_mutant")
    mod.__file__ = O.__file__
    exec(compile(src, O.__file__ + " (mutated copy)", "exec"), mod.__dict__)
    return mod


def _pins():
    out = []
    for name, fn in inspect.getmembers(P, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != P.__name__:
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if marks:
            argname, values = marks[0].args[0], marks[0].args[1]
            out.extend((f"{name}[{i}]", fn, {argname: v}) for i, v in enumerate(values))
        else:
            out.append((name, fn, {}))
    return out


PINS = _pins()


def _first_failing_pin(mod, monkeypatch):
    monkeypatch.setattr(P, "O", mod)
    for name, fn, kw in PINS:
        try:
            fn(**kw)
        except (Exception, pytest.fail.Exception):   # an assertion, or an error the mistake causes
            return name
    return None


def test_unmutated_copy_passes_every_pin(monkeypatch):
    assert len(PINS) > 30
    assert _first_failing_pin(_mutant([]), monkeypatch) is None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    caught = _first_failing_pin(_mutant(MUTANTS[name]), monkeypatch)
    assert caught is not None, f"no pin fails when the oracle has this mistake: {name}"
