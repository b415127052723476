"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (on the CPU, by replacing one of
its functions for the duration of the test) and runs every pin of
``test_oracle_pins``; at least one pin must fail.  The mistakes are the kind
a restatement of the pages could make: a dropped term, a wrong constant, an
off-by-one window, a transposed operand, a wrong tie rule, a rounding mode,
a byte layout.  The untouched oracle passes every pin (the pins' own run).
"""
import inspect
import math
import os

import numpy as np
import pytest

from oracle import kvc_oracle as O
from tests import test_oracle_pins as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pin_cases():
    """(name, kwargs, function) for every pin, parametrisations expanded."""
    cases = []
    for name, f in sorted(vars(P).items()):
        if not (name.startswith("test_") and callable(f)):
            continue
        params = list(inspect.signature(f).parameters)
        grid = [{}]
        for m in getattr(f, "pytestmark", []):
            if m.name != "parametrize":
                continue
            names = [s.strip() for s in m.args[0].split(",")]
            grid = [dict(g, **dict(zip(names, v if len(names) > 1 else (v,)))) for g in grid for v in m.args[1]]
        for g in grid:
            kw = dict(g)
            if "golden_dir" in params:
                kw["golden_dir"] = GOLDEN
            cases.append((name, kw, f))
    return cases


PINS = _pin_cases()


# --------------------------------------------------------------------------
# mutant builders
# --------------------------------------------------------------------------

def _quantize(round_fn=np.rint, eps=0.0):
    def quantize_rows(x, bits):
        x = np.asarray(x, dtype=np.float32)
        qmax = np.float32(O.qmax_for_bits(bits))
        amax = np.max(np.abs(x), axis=-1)
        scale = (amax / qmax + np.float32(eps)).astype(np.float32)
        safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = (x / safe[..., None]).astype(np.float32)
        lo, hi = O.code_range(bits)
        codes = np.clip(round_fn(ratio), lo, hi)
        return np.where(scale[..., None] > 0, codes, 0).astype(np.int8), scale
    return quantize_rows


def _half_away(r):
    return np.sign(r) * np.floor(np.abs(r) + 0.5)


def _quantize_e4m3(fmax):
    def quantize_rows_e4m3(x):
        x = np.asarray(x, dtype=np.float32)
        amax = np.max(np.abs(x), axis=-1)
        scale = (amax / np.float32(fmax)).astype(np.float32)
        safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
        codes = O.e4m3_encode((x / safe[..., None]).astype(np.float32))
        return np.where(scale[..., None] > 0, codes, 0).astype(np.uint8), scale
    return quantize_rows_e4m3


def _attention(scale_one=False, values_are_keys=False, wrong_axis=False):
    def attention(q, keys, values, sm_scale=None):
        q = np.asarray(q, np.float64)
        k = np.asarray(keys, np.float64)
        v = np.asarray(k if values_are_keys else values, np.float64)
        s = 1.0 if scale_one else (1.0 / math.sqrt(q.shape[-1]) if sm_scale is None else sm_scale)
        logits = (q @ k.T) * s
        ax = 0 if wrong_axis else -1
        e = np.exp(logits - logits.max(axis=ax, keepdims=True))
        probs = e / e.sum(axis=ax, keepdims=True)
        return probs @ v, probs
    return attention


def _select_h2o(ties_high=False, recent_strict=False, sinks_free=False):
    def select_h2o(pos, score, pos_total, budget, recent, n_sink_present=O.NUM_SINK):
        pos = np.asarray(pos, np.int64)
        score = np.asarray(score, np.float64)
        n = pos.shape[0]
        if (n if sinks_free else n_sink_present + n) <= budget:
            return np.ones(n, dtype=bool)
        heavy = budget - (0 if sinks_free else O.NUM_SINK) - recent
        if heavy < 0:
            raise ValueError("budget")
        keep = pos > pos_total - recent if recent_strict else pos >= pos_total - recent
        cand = np.nonzero(~keep)[0]
        order = np.lexsort(((-pos if ties_high else pos)[cand], -score[cand]))
        keep[cand[order[:heavy]]] = True
        return keep
    return select_h2o


def _select_streaming_strict():
    def select_streaming(pos, pos_total, window, n_sink_present=O.NUM_SINK):
        pos = np.asarray(pos, np.int64)
        if pos.shape[0] <= window:
            return np.ones(pos.shape[0], dtype=bool)
        return pos > pos_total - window
    return select_streaming


def _select_blocks(evict_retained=False, ties_late=False, first_head_only=False):
    def select_blocks(scores, n_slots, recent, retention):
        n_cand = max(0, n_slots - recent) // O.PAGE
        n_evict = int(n_cand * (retention if evict_retained else 1.0 - retention))
        heads = scores[:1] if first_head_only else scores
        sums = [sum(float(sc[t]) for sc in heads for t in range(p * O.PAGE, (p + 1) * O.PAGE))
                for p in range(n_cand)]
        order = sorted(range(n_cand), key=lambda p: (sums[p], -p if ties_late else p))
        keep = np.ones(n_slots, dtype=bool)
        for p in order[:n_evict]:
            keep[p * O.PAGE:(p + 1) * O.PAGE] = False
        return keep
    return select_blocks


def _prefill_not_causal():
    def prefill_attention(q, k, v, sm_scale=None):
        q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
        hq, n, d = q.shape
        g = hq // k.shape[0]
        s = 1.0 / math.sqrt(d) if sm_scale is None else sm_scale
        out = np.zeros((hq, n, d))
        scores = np.zeros((k.shape[0], n))
        for j in range(hq):
            logits = (q[j] @ k[j // g].T) * s
            e = np.exp(logits - logits.max(axis=-1, keepdims=True))
            probs = e / e.sum(axis=-1, keepdims=True)
            out[j] = probs @ v[j // g]
            scores[j // g] += probs.sum(axis=0)
        return out, scores
    return prefill_attention


def _prefill_variant(first_head_scores_only=False, mask_offset=1):
    def prefill_attention(q, k, v, sm_scale=None):
        q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
        hq, n, d = q.shape
        g = hq // k.shape[0]
        s = 1.0 / math.sqrt(d) if sm_scale is None else sm_scale
        future = np.triu(np.ones((n, n), dtype=bool), mask_offset)
        out = np.zeros((hq, n, d))
        scores = np.zeros((k.shape[0], n))
        for j in range(hq):
            logits = (q[j] @ k[j // g].T) * s
            logits[future] = -np.inf
            e = np.exp(logits - logits.max(axis=-1, keepdims=True))
            probs = e / e.sum(axis=-1, keepdims=True)
            out[j] = probs @ v[j // g]
            if not first_head_scores_only or j % g == 0:
                scores[j // g] += probs.sum(axis=0)
        return out, scores
    return prefill_attention


def _pack_swapped(codes):
    c = np.asarray(codes, dtype=np.int8).astype(np.uint8) & np.uint8(0x0F)
    return (c[..., 1::2] | (c[..., 0::2] << np.uint8(4))).astype(np.uint8)


def _unpack_swapped(packed):
    p = np.asarray(packed, dtype=np.uint8)
    hi = (p & np.uint8(0x0F)).astype(np.int16)
    lo = (p >> np.uint8(4)).astype(np.int16)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int8)
    out[..., 0::2] = np.where(lo >= 8, lo - 16, lo)
    out[..., 1::2] = np.where(hi >= 8, hi - 16, hi)
    return out


def _attend_without_window(orig):
    def attend(self, b, q, sm_scale=None, accumulate=True):
        w = self.bf16_window
        self.bf16_window = 0
        try:
            return orig(self, b, q, sm_scale, accumulate)
        finally:
            self.bf16_window = w
    return attend


def _evict_complement(orig):
    def evict(self, b, masks):
        return orig(self, b, [~np.asarray(m, dtype=bool) for m in masks])
    return evict


def _attend_modulo_heads(orig):
    """Query head j reads KV head j % Hkv instead of j // G."""
    def attend(self, b, q, sm_scale=None, accumulate=True):
        g, hkv = self.group, self.hkv
        perm = np.array([gi * hkv + h for h in range(hkv) for gi in range(g)])
        out = np.empty((self.hq, self.d))
        out[perm] = orig(self, b, np.asarray(q)[perm], sm_scale, accumulate)
        return out
    return attend


def _dequantize_as_int(orig):
    def dequantize(self, codes, scale):
        return O.dequantize(codes, scale)
    return dequantize


def _prefill_without_scores(orig):
    def prefill(self, b, q, k, v, sm_scale=None):
        out = orig(self, b, q, k, v, sm_scale)
        s = self.seqs[b]
        for h in range(self.hkv):
            s.sink_score[h] = np.zeros_like(s.sink_score[h])
            s.heads[h].score = np.zeros_like(s.heads[h].score)
        return out
    return prefill


def _keep_masks_without_recent(orig):
    def keep_masks(self, b, mode, budget=0, recent=0, window=0, retention=1.0):
        return orig(self, b, mode, budget, 0 if mode == "h2o" else recent, window, retention)
    return keep_masks


def _chunk_without_scores(orig):
    def prefill_chunk(self, b, q, k, v, sm_scale=None, accumulate=True):
        return orig(self, b, q, k, v, sm_scale, False)
    return prefill_chunk


def _attend_window_one_long(orig):
    def attend(self, b, q, sm_scale=None, accumulate=True):
        w = self.bf16_window
        if w > 0:
            self.bf16_window = w + 1
        try:
            return orig(self, b, q, sm_scale, accumulate)
        finally:
            self.bf16_window = w
    return attend


def _block_masks_without_recent(orig):
    def keep_masks(self, b, mode, budget=0, recent=0, window=0, retention=1.0):
        return orig(self, b, mode, budget, 0 if mode == "block" else recent, window, retention)
    return keep_masks


# name -> list of (object, attribute, factory(original) -> replacement)
MUTANTS = {
    "INT8 scale divides by 128": [(O, "qmax_for_bits", lambda f: lambda bits: 128 if bits == 8 else f(bits))],
    "codes rounded half away from zero": [(O, "quantize_rows", lambda f: _quantize(round_fn=_half_away))],
    "scale with an epsilon term": [(O, "quantize_rows", lambda f: _quantize(eps=1e-8))],
    "codes truncated instead of rounded": [(O, "quantize_rows", lambda f: _quantize(round_fn=np.trunc))],
    "dequantisation drops the scale": [(O, "dequantize", lambda f: lambda c, s: np.asarray(c, np.float64))],
    "attention ignores sm_scale": [(O, "attention", lambda f: _attention(scale_one=True))],
    "attention reads K as V": [(O, "attention", lambda f: _attention(values_are_keys=True))],
    "softmax over the query axis": [(O, "attention", lambda f: _attention(wrong_axis=True))],
    "H2O increment averaged over the group": [(O, "h2o_increments",
                                               lambda f: lambda p: np.asarray(p, np.float64).mean(axis=0))],
    "H2O ties to the higher position": [(O, "select_h2o", lambda f: _select_h2o(ties_high=True))],
    "recent window one short": [(O, "select_h2o", lambda f: _select_h2o(recent_strict=True))],
    "sinks outside the budget": [(O, "select_h2o", lambda f: _select_h2o(sinks_free=True))],
    "StreamingLLM window one short": [(O, "select_streaming", lambda f: _select_streaming_strict())],
    "block eviction count uses the retention": [(O, "select_blocks", lambda f: _select_blocks(evict_retained=True))],
    "block ties to the later page": [(O, "select_blocks", lambda f: _select_blocks(ties_late=True))],
    "block key from the first head only": [(O, "select_blocks", lambda f: _select_blocks(first_head_only=True))],
    "prefill without the causal mask": [(O, "prefill_attention", lambda f: _prefill_not_causal())],
    "INT4 nibbles swapped": [(O, "pack_int4", lambda f: _pack_swapped), (O, "unpack_int4", lambda f: _unpack_swapped)],
    "E4M3 decoded with bias 8": [(O, "e4m3_decode", lambda f: lambda c: f(c) * 0.5)],
    "FP8 scale from the E4M3-FNUZ maximum 240": [(O, "quantize_rows_e4m3", lambda f: _quantize_e4m3(240.0))],
    "KV size counts K only": [(O, "kv_cache_bytes", lambda f: lambda *a, **k: f(*a, **k) // 2)],
    "bf16 window ignored by the decode attention": [(O.OracleCache, "attend", _attend_without_window)],
    "eviction keeps the complement of the mask": [(O.OracleCache, "evict", _evict_complement)],
    "three sink tokens": [(O, "NUM_SINK", lambda f: 3)],
    "query head j reads KV head j mod Hkv": [(O.OracleCache, "attend", _attend_modulo_heads)],
    "FP8 codes dequantised as integers": [(O.OracleCache, "dequantize", _dequantize_as_int)],
    "prefill leaves the scores at zero": [(O.OracleCache, "prefill", _prefill_without_scores)],
    "H2O keep masks drop the recent window": [(O.OracleCache, "keep_masks", _keep_masks_without_recent)],
    "prompt over context adds no scores": [(O.OracleCache, "prefill_chunk", _chunk_without_scores)],
    "bf16 window one position too long": [(O.OracleCache, "attend", _attend_window_one_long)],
    "block keep masks drop the recent pages": [(O.OracleCache, "keep_masks", _block_masks_without_recent)],
    "prefill scores from one query head of the group": [(O, "prefill_attention",
                                                         lambda f: _prefill_variant(first_head_scores_only=True))],
    "prefill mask lets a query see the next key": [(O, "prefill_attention", lambda f: _prefill_variant(mask_offset=2))],
    "E4M3 saturates at 240": [(O, "e4m3_encode", lambda f: lambda y: f(np.clip(np.asarray(y, np.float32), -240, 240)))],
    "H2O increment from the first query head only": [(O, "h2o_increments",
                                                      lambda f: lambda p: np.asarray(p, np.float64)[0])],
    "StreamingLLM keeps the oldest window": [(O, "select_streaming", lambda f: lambda pos, pt, w, ns=O.NUM_SINK:
                                             np.argsort(np.argsort(np.asarray(pos))) < w
                                             if np.asarray(pos).shape[0] > w else np.ones(len(pos), bool))],
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_a_pin_catches_the_planted_mistake(name, monkeypatch):
    for obj, attr, make in MUTANTS[name]:
        monkeypatch.setattr(obj, attr, make(getattr(obj, attr)))
    for pin, kw, f in PINS:
        try:
            f(**kw)
        except pytest.skip.Exception:
            continue
        except Exception:
            return  # caught
    pytest.fail(f"no pin fails with the planted mistake: {name}")
