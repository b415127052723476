"""Reference oracle for the compressed-KV decode step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product path
(the CUDA library and its Python binding) never calls it, and this module never
imports the product package: the two share no code.

What it computes, step by step, each citing the page passage it restates:

* ``kv_cache_bytes`` -- the KV-memory closed form of "KV Cache optimization
  techniques" (metaphor-xennon), section "KV Cache的挑战" (kv_cache_memory_analysis).
* ``quantize_rows`` -- per-token symmetric quantisation, "KV Cache optimization
  techniques" section 1.2 (PerTokenKVQuantizer) and "Technical Report: KV Cache
  Compression for Text-Only LLMs" section 3.2 (quantize_kv): one scale per
  (token, head) = amax over head_dim / (2^(bits-1) - 1), code = round-half-even
  of x / scale, clamped.  Computed in IEEE fp32 exactly as the pages' fp32
  tensors would be (division, not reciprocal multiplication).
* ``quantize_rows_e4m3`` -- FP8 codes (the techniques page lists FP8 among
  its quantisation strategies, section 1.1; the Technical Report's section 2
  lists INT8/FP8/INT4): the same per-token symmetric scale with the E4M3
  range (amax / 448), and each x / scale rounded to E4M3, ties to even,
  saturating at 448 (``e4m3_encode``, written from the OCP 8-bit floating
  point format: 4 exponent bits with bias 7, 3 fraction bits, subnormals).
* ``attention`` -- the dense definition softmax(Q K^T / sqrt(d)) V of the
  Technical Report section 1.1, evaluated in fp64 on the dequantised keys and
  values (code * scale, section 3.2) and on the bf16 sink tokens (section 3.2:
  sinks are not quantised).
* ``h2o_increments`` -- the H2O heavy-hitter score: column sums of the softmax
  probabilities (Technical Report section 3.4, ``attention_scores.sum(dim=0)``;
  the survey page's section 3.3 calls it the cumulative attention a token
  receives from all later tokens).  With grouped-query attention the G query
  heads that read one KV head all add to that head's score.
* ``select_h2o`` / ``select_streaming`` -- the kept set: the attention sinks,
  the recent window, and the top-k of the remaining tokens by accumulated
  score, ties to the lower position (Technical Report sections 3.3-3.4,
  "KV Cache optimization techniques" sections 2.2 and 2.4).
* ``select_blocks`` -- block-granular eviction (the eviction-and-reuse survey
  page, section 4, the block manager's eviction by attention): blocks sorted
  by their mean attention score, the lowest int(n * (1 - ratio)) evicted.
* ``prefill_attention`` -- the prompt's causal attention over itself and the
  H2O scores it gives (Technical Report section 3.4: the score is the sum of
  the attention matrix over its query rows; the survey page's section 3.3:
  a token's cumulative attention from all later tokens), in fp64 on the exact
  bf16 inputs.
* ``OracleCache.prefill_chunk`` -- a prompt appended to a sequence that may
  already hold context, each query attending causally to the compressed
  cache as the decode step does.
* ``OracleCache(bf16_window=W)`` -- hybrid precision ("KV Cache optimization
  techniques" section 1.3, HybridPrecisionKVCache: recent tokens at 16 bits,
  older ones at INT4/INT8): the tokens at the last W positions attend with
  their unquantised bf16 values, older ones with their codes.

Where the pages are silent or disagree, the reading taken is restated beside
the function whose arithmetic it affects.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, worked examples with exact scales, library witnesses, invariants,
brute force).  None is "parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 128
NUM_SINK = 4
PAGE = 16  # tokens per block of the paged pool


# ---------------------------------------------------------------------------
# Closed form for KV bytes
# ---------------------------------------------------------------------------

def kv_cache_bytes(batch: int, seq_len: int, num_layers: int, num_heads: int,
                   head_dim: int, bytes_per_element: int) -> int:
    """Bytes held by an uncompressed KV cache.

    "KV Cache optimization techniques", section "KV Cache的挑战": per token the
    cache holds a key and a value vector for every layer and head, i.e.
    2 * layers * heads * head_dim * bytes_per_element bytes; the whole cache is
    that times batch * seq_len.
    """
    per_token = 2 * num_layers * num_heads * head_dim * bytes_per_element
    return per_token * batch * seq_len


def kv_cache_gib(batch, seq_len, num_layers, num_heads, head_dim, bytes_per_element) -> float:
    """The same closed form in GiB (the page divides by 1024**3)."""
    return kv_cache_bytes(batch, seq_len, num_layers, num_heads, head_dim,
                          bytes_per_element) / float(1024 ** 3)


def stored_bytes_per_token_head(bits: int, head_dim: int = HEAD_DIM,
                                with_scales: bool = True) -> int:
    """Bytes one (token, KV head) occupies in the compressed cache: K and V codes
    (bits/8 bytes per element) plus, optionally, one fp32 scale each for K and V
    (per-token scales, "KV Cache optimization techniques" section 1.2)."""
    code_bytes = 2 * (head_dim * bits // 8)
    return code_bytes + (2 * 4 if with_scales else 0)


# ---------------------------------------------------------------------------
# bf16 helpers (input decoding only: bf16 -> fp32 is exact)
# ---------------------------------------------------------------------------

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bit patterns (uint16) to fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


# ---------------------------------------------------------------------------
# Per-token quantisation
# ---------------------------------------------------------------------------

def qmax_for_bits(bits: int) -> int:
    """2^(bits-1) - 1: 127 for INT8, 7 for INT4 ("KV Cache optimization
    techniques" section 1.2, ``max_val``)."""
    if bits not in (4, 8):
        # The quantiser of section 1.1 raises on unsupported widths.
        raise ValueError(f"unsupported bits: {bits}")
    return (1 << (bits - 1)) - 1


def code_range(bits: int) -> tuple[int, int]:
    """Clamp range of the codes.

    INT8: [-127, 127] (Technical Report section 3.2 clamps symmetric; the
    techniques page clamps to [-128, 127] -- the bound never binds because
    |x / scale| <= 127 * (1 + 2^-24) rounds to at most 127).
    INT4: [-8, 7] (techniques page section 1.1); again only [-7, 7] is reached.
    """
    return (-127, 127) if bits == 8 else (-8, 7)


def quantize_rows(x: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """Quantise each row (last axis = head_dim) of an fp32 array.

    Returns (codes as int8 with the same shape as ``x``, scales fp32 of shape
    ``x.shape[:-1]``).

    Steps, in the order of "KV Cache optimization techniques" section 1.2:
      1. amax = max |x| over the row (exact in fp32);
      2. scale = amax / qmax, one IEEE fp32 division (no epsilon: the
         Technical Report's quantize_kv adds none, and the techniques page's
         +1e-8 would change the codes of tiny rows);
      3. code = round-half-to-even(x / scale) with an IEEE fp32 division,
         then clamp to ``code_range(bits)``.
    A row whose amax is 0 has scale 0 and all codes 0 (0/0 is avoided).
    """
    x = np.asarray(x, dtype=np.float32)
    qmax = np.float32(qmax_for_bits(bits))
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / qmax).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (x / safe[..., None]).astype(np.float32)
    codes = np.rint(ratio)  # numpy rint: round half to even
    lo, hi = code_range(bits)
    codes = np.clip(codes, lo, hi)
    codes = np.where(scale[..., None] > 0, codes, 0).astype(np.int8)
    return codes, scale


E4M3_MAX = 448.0  # largest finite FP8 E4M3 value: 1.75 * 2^8


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """FP8 E4M3 codes (uint8) of fp32 values: round to nearest, ties to even,
    saturating to +-448 (no infinities in E4M3).

    Format (OCP 8-bit floating point, E4M3): sign bit, 4 exponent bits with
    bias 7, 3 fraction bits; exponent field 0 holds the subnormals m * 2^-9
    (m = 0..7); the largest finite value is 1.75 * 2^8 = 448.  Rounding:
    the representable values near |y| are spaced 2^(e-3) apart, e =
    max(floor(log2 |y|), -6); |y| / 2^(e-3) rounded half to even, times
    2^(e-3), is the nearest value (exact in fp64: power-of-two scaling)."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    sign = np.signbit(y).astype(np.uint8)
    a = np.minimum(np.abs(y), E4M3_MAX)  # saturation (values above 448 round to 448 or beyond)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))  # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    e = np.maximum(ex - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    v = np.rint(a / quantum) * quantum  # rounded magnitude, <= 448
    sub = v < 2.0 ** -6
    fm, fe = np.frexp(np.where(v > 0, v, 1.0))  # v = (2 fm) * 2^(fe - 1)
    exp_field = np.where(sub, 0, fe - 1 + 7)
    frac = np.where(sub, v / 2.0 ** -9, (2.0 * fm - 1.0) * 8.0)
    code = (exp_field.astype(np.int64) << 3) | np.rint(frac).astype(np.int64)
    return ((sign.astype(np.int64) << 7) | code).astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Exact fp64 values of FP8 E4M3 codes (the NaN codes 0x7F / 0xFF are
    never produced by ``e4m3_encode``)."""
    c = np.asarray(codes).astype(np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(ef == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, ef - 7))
    return sign * mag


def quantize_rows_e4m3(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """FP8 (E4M3) per-token quantisation of each row (last axis): amax over
    the row, scale = amax / 448 (one IEEE fp32 division), code =
    e4m3_encode(x / scale) with an IEEE fp32 division; a zero row has scale 0
    and codes 0.  Returns (uint8 codes, fp32 scales)."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    ratio = (x / safe[..., None]).astype(np.float32)
    codes = e4m3_encode(ratio)
    codes = np.where(scale[..., None] > 0, codes, 0).astype(np.uint8)
    return codes, scale


def pack_int4(codes: np.ndarray) -> np.ndarray:
    """Two INT4 codes per byte: element 2i in the low nibble, 2i+1 in the high
    nibble, two's complement (the page's ``.to(torch.int4)`` is not a real
    dtype; this packing is our stated reading)."""
    c = np.asarray(codes, dtype=np.int8).astype(np.uint8) & np.uint8(0x0F)
    return (c[..., 0::2] | (c[..., 1::2] << np.uint8(4))).astype(np.uint8)


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    """Inverse of ``pack_int4`` (sign-extends each nibble)."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & np.uint8(0x0F)).astype(np.int16)
    hi = (p >> np.uint8(4)).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def dequantize(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """code * scale in fp64 ("KV Cache optimization techniques" section 1.2,
    dequantize; Technical Report section 3.2, K_q * scale_k)."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[..., None]


# ---------------------------------------------------------------------------
# Attention (fp64 definition)
# ---------------------------------------------------------------------------

def attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray,
              sm_scale: float | None = None) -> tuple[np.ndarray, np.ndarray]:
    """softmax(q K^T * sm_scale) V for a set of query rows, in fp64.

    q: [G, D]; keys, values: [N, D].  Returns (out [G, D], probs [G, N]).
    sm_scale defaults to 1/sqrt(D) (Technical Report section 1.1).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(keys, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    d = q.shape[-1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    logits = (q @ k.T) * sm_scale
    m = logits.max(axis=-1, keepdims=True)
    e = np.exp(logits - m)
    probs = e / e.sum(axis=-1, keepdims=True)
    return probs @ v, probs


def h2o_increments(probs: np.ndarray) -> np.ndarray:
    """H2O score added this step to each attended token: the column sum of the
    softmax probabilities over the query rows that read this KV head
    (Technical Report section 3.4, ``attention_scores.sum(dim=0)``)."""
    return np.asarray(probs, dtype=np.float64).sum(axis=0)


# ---------------------------------------------------------------------------
# Selection
# ---------------------------------------------------------------------------

def prefill_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                      sm_scale: float | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Causal attention of a prompt over itself, and the H2O scores it gives.

    q: [Hq, n, D]; k, v: [Hkv, n, D] (exact bf16 values, fp32).  Query head j
    reads KV head j // G; query i attends keys 0..i.  Returns, in fp64,
    (out [Hq, n, D], scores [Hkv, n]) where scores[h, t] is the sum, over the
    G query heads of KV head h and over every query, of the probability that
    query gives key t: the column sums of the attention matrix (Technical
    Report section 3.4, ``attention_scores.sum(dim=0)``).  Reading: the prompt
    attends with its exact values; the compressed cache is what the decode
    steps read."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    hq, n, d = q.shape
    hkv = k.shape[0]
    g = hq // hkv
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    future = np.triu(np.ones((n, n), dtype=bool), 1)  # key index > query index
    out = np.zeros((hq, n, d), np.float64)
    scores = np.zeros((hkv, n), np.float64)
    for j in range(hq):
        h = j // g
        logits = (q[j] @ k[h].T) * sm_scale
        logits[future] = -np.inf
        e = np.exp(logits - logits.max(axis=-1, keepdims=True))
        probs = e / e.sum(axis=-1, keepdims=True)
        out[j] = probs @ v[h]
        scores[h] += probs.sum(axis=0)
    return out, scores


def select_h2o(pos: np.ndarray, score: np.ndarray, pos_total: int, budget: int,
               recent: int, n_sink_present: int = NUM_SINK) -> np.ndarray:
    """Keep-mask over the non-sink tokens of one (sequence, KV head).

    The attention sinks (always kept, not in ``pos``) take ``n_sink_present``
    places of the budget.  If every token fits, nothing is evicted.  Otherwise
    the recent window (positions >= pos_total - recent) is kept, and of the
    other tokens the ``budget - NUM_SINK - recent`` with the largest scores,
    ties to the lower position (Technical Report section 3.4: keep heavy
    hitters and recent tokens; "KV Cache optimization techniques" section 2.2:
    evict once the cache exceeds its limit, keep by top-k of the score).
    """
    pos = np.asarray(pos, dtype=np.int64)
    score = np.asarray(score, dtype=np.float64)
    n = pos.shape[0]
    if n_sink_present + n <= budget:
        return np.ones(n, dtype=bool)
    heavy = budget - NUM_SINK - recent
    if heavy < 0:
        raise ValueError("budget must cover the sinks and the recent window")
    keep = pos >= pos_total - recent
    cand = np.nonzero(~keep)[0]
    # order: score descending, then position ascending
    order = np.lexsort((pos[cand], -score[cand]))
    keep[cand[order[:heavy]]] = True
    return keep


def select_streaming(pos: np.ndarray, pos_total: int, window: int,
                     n_sink_present: int = NUM_SINK) -> np.ndarray:
    """StreamingLLM keep-mask: the sinks (kept outside this mask) plus the last
    ``window`` positions (Technical Report section 3.3 SlidingWindow: sink
    tokens then a deque of the most recent ``window_size`` tokens)."""
    pos = np.asarray(pos, dtype=np.int64)
    if pos.shape[0] <= window:
        return np.ones(pos.shape[0], dtype=bool)
    return pos >= pos_total - window


def select_blocks(scores: list, n_slots: int, recent: int, retention: float) -> np.ndarray:
    """Block-granular eviction (the eviction-and-reuse survey page, section 4:
    the block manager's eviction by attention sorts the blocks by the mean
    attention score of their tokens and evicts the first int(len * (1 -
    ratio)) of them).

    The pool of one sequence, in slot order, is cut into blocks of PAGE slots;
    all KV heads share a block, so a block's score covers its PAGE slots of
    every head.  Readings: the candidates are the full blocks that lie before
    the last ``recent`` slots (the recent window and the unfilled last block
    always stay; the sinks are not in the pool); a block is ordered by the
    sum of its PAGE x Hkv scores, accumulated in fp64 head by head and slot by
    slot (the sum orders blocks exactly as the mean does); ties go to the
    earlier block, as a stable sort leaves them.  ``scores`` holds one score
    array per KV head, in slot order.  Returns the keep mask over the
    ``n_slots`` slots, the same for every head."""
    n_cand = max(0, n_slots - recent) // PAGE
    n_evict = int(n_cand * (1.0 - retention))
    sums = []
    for p in range(n_cand):
        acc = 0.0
        for sc in scores:
            for t in range(p * PAGE, (p + 1) * PAGE):
                acc += float(sc[t])
        sums.append(acc)
    order = sorted(range(n_cand), key=lambda p: (sums[p], p))
    keep = np.ones(n_slots, dtype=bool)
    for p in order[:n_evict]:
        keep[p * PAGE:(p + 1) * PAGE] = False
    return keep


# ---------------------------------------------------------------------------
# Dense per-(sequence, KV head) cache that runs the decode step
# ---------------------------------------------------------------------------

@dataclass
class HeadState:
    """Non-sink tokens of one (sequence, KV head), in insertion order."""
    pos: np.ndarray            # int64 [N]
    kcodes: np.ndarray         # int8  [N, D]  (unpacked codes)
    kscale: np.ndarray         # fp32  [N]
    vcodes: np.ndarray         # int8  [N, D]
    vscale: np.ndarray         # fp32  [N]
    score: np.ndarray          # fp64  [N]


@dataclass
class SeqState:
    pos_total: int = 0
    raw_k: list = field(default_factory=list)    # per head: fp32 [pos_total, D], every token's bf16 values
    raw_v: list = field(default_factory=list)
    sink_k: list = field(default_factory=list)   # per head: fp32 [ns, D]
    sink_v: list = field(default_factory=list)
    sink_score: list = field(default_factory=list)  # per head: fp64 [ns]
    heads: list = field(default_factory=list)   # per head: HeadState


def _empty_head(d: int) -> HeadState:
    return HeadState(np.zeros(0, np.int64), np.zeros((0, d), np.int8), np.zeros(0, np.float32),
                     np.zeros((0, d), np.int8), np.zeros(0, np.float32), np.zeros(0, np.float64))


class OracleCache:
    """One layer of the compressed cache for a batch of sequences, dense (no
    paging), evaluated token by token.

    Per decode step the order is append -> attention (the new token attends to
    itself) -> score accumulation -> select -> evict ("KV Cache optimization
    techniques" section 2.2: append, then evict once over the limit).
    """

    def __init__(self, batch: int, num_q_heads: int, num_kv_heads: int, bits: int,
                 head_dim: int = HEAD_DIM, bf16_window: int = 0, codes: str = "int"):
        if num_q_heads % num_kv_heads:
            raise ValueError("num_q_heads must be a multiple of num_kv_heads")
        if bf16_window < 0:
            raise ValueError("bf16_window must be >= 0")
        qmax_for_bits(bits)
        if codes not in ("int", "e4m3") or (codes == "e4m3" and bits != 8):
            raise ValueError("codes: 'int', or 'e4m3' with bits = 8")
        self.batch, self.hq, self.hkv, self.bits, self.d = batch, num_q_heads, num_kv_heads, bits, head_dim
        self.bf16_window = bf16_window
        self.codes = codes
        self.group = num_q_heads // num_kv_heads
        self.seqs = []
        for _ in range(batch):
            s = SeqState()
            for _ in range(num_kv_heads):
                s.sink_k.append(np.zeros((0, head_dim), np.float32))
                s.sink_v.append(np.zeros((0, head_dim), np.float32))
                s.sink_score.append(np.zeros(0, np.float64))
                s.heads.append(_empty_head(head_dim))
                s.raw_k.append(np.zeros((0, head_dim), np.float32))
                s.raw_v.append(np.zeros((0, head_dim), np.float32))
            self.seqs.append(s)

    # -- write path ---------------------------------------------------------
    def append(self, b: int, k: np.ndarray, v: np.ndarray) -> None:
        """Append n tokens to sequence b.  k, v: fp32 [Hkv, n, D] (exact bf16
        values).  Positions < NUM_SINK are stored unquantised (Technical Report
        section 3.2: sink KV stay in half precision); the others are quantised
        once, at write time."""
        s = self.seqs[b]
        n = k.shape[1]
        for h in range(self.hkv):
            s.raw_k[h] = np.concatenate([s.raw_k[h], k[h].astype(np.float32)])
            s.raw_v[h] = np.concatenate([s.raw_v[h], v[h].astype(np.float32)])
        for i in range(n):
            p = s.pos_total + i
            for h in range(self.hkv):
                if p < NUM_SINK:
                    s.sink_k[h] = np.vstack([s.sink_k[h], k[h, i][None]])
                    s.sink_v[h] = np.vstack([s.sink_v[h], v[h, i][None]])
                    s.sink_score[h] = np.append(s.sink_score[h], 0.0)
        first_q = max(0, NUM_SINK - s.pos_total)
        if first_q < n:
            if self.codes == "e4m3":  # byte codes kept in the int8 arrays
                kc, ks = quantize_rows_e4m3(k[:, first_q:])
                vc, vs = quantize_rows_e4m3(v[:, first_q:])
                kc, vc = kc.view(np.int8), vc.view(np.int8)
            else:
                kc, ks = quantize_rows(k[:, first_q:], self.bits)
                vc, vs = quantize_rows(v[:, first_q:], self.bits)
            newpos = np.arange(s.pos_total + first_q, s.pos_total + n, dtype=np.int64)
            for h in range(self.hkv):
                hs = s.heads[h]
                hs.pos = np.concatenate([hs.pos, newpos])
                hs.kcodes = np.concatenate([hs.kcodes, kc[h]])
                hs.kscale = np.concatenate([hs.kscale, ks[h]])
                hs.vcodes = np.concatenate([hs.vcodes, vc[h]])
                hs.vscale = np.concatenate([hs.vscale, vs[h]])
                hs.score = np.concatenate([hs.score, np.zeros(n - first_q)])
        s.pos_total += n

    def prefill(self, b: int, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                sm_scale: float | None = None) -> np.ndarray:
        """The prompt of a fresh sequence b: append its n tokens (k, v: fp32
        [Hkv, n, D]), run ``prefill_attention`` with q (fp32 [Hq, n, D]) and
        set every prompt token's H2O score (sinks included) to its column
        sum.  Returns the attention output fp64 [Hq, n, D]."""
        s = self.seqs[b]
        if s.pos_total != 0:
            raise ValueError("prefill needs a fresh sequence")
        self.append(b, k, v)
        out, sc = prefill_attention(q, k, v, sm_scale)
        for h in range(self.hkv):
            ns = s.sink_k[h].shape[0]
            s.sink_score[h] = sc[h, :ns].copy()
            s.heads[h].score = sc[h, s.heads[h].pos].copy()
        return out

    def dequantize(self, codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
        """code value * scale in fp64 (INT codes, or E4M3 codes decoded)."""
        if self.codes == "e4m3":
            return e4m3_decode(np.asarray(codes).view(np.uint8)) * np.asarray(scale, np.float64)[..., None]
        return dequantize(codes, scale)

    def prefill_chunk(self, b: int, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                      sm_scale: float | None = None, accumulate: bool = True) -> np.ndarray:
        """A prompt of n tokens appended to sequence b, which may already
        hold context (a later turn; the survey's prefill over the compressed
        pool): append the tokens (quantised as on every append), then query
        i (position P_old + i) attends, as the decode step does, to every
        held token at a position <= P_old + i in its stored form (sinks and
        bf16-window tokens exact, pool tokens dequantised).  With
        ``accumulate`` every held token's score grows by the probabilities all
        n queries (and the G query heads of its KV head) give it.  q: fp32
        [Hq, n, D]; k, v: fp32 [Hkv, n, D].  Returns fp64 [Hq, n, D]."""
        s = self.seqs[b]
        p_old = s.pos_total
        n = q.shape[1]
        self.append(b, k, v)
        d = self.d
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(d)
        out = np.zeros((self.hq, n, d), np.float64)
        for h in range(self.hkv):
            hs = s.heads[h]
            ns = s.sink_k[h].shape[0]
            kq = self.dequantize(hs.kcodes, hs.kscale)
            vq = self.dequantize(hs.vcodes, hs.vscale)
            if self.bf16_window > 0:
                recent = hs.pos >= s.pos_total - self.bf16_window
                kq[recent] = s.raw_k[h][hs.pos[recent]].astype(np.float64)
                vq[recent] = s.raw_v[h][hs.pos[recent]].astype(np.float64)
            keys = np.vstack([s.sink_k[h].astype(np.float64), kq])
            vals = np.vstack([s.sink_v[h].astype(np.float64), vq])
            kpos = np.concatenate([np.arange(ns), hs.pos])
            inc = np.zeros(keys.shape[0], np.float64)
            for i in range(n):
                seen = kpos <= p_old + i
                o, pr = attention(q[h * self.group:(h + 1) * self.group, i], keys[seen], vals[seen], sm_scale)
                out[h * self.group:(h + 1) * self.group, i] = o
                inc[seen] += h2o_increments(pr)
            if accumulate:
                s.sink_score[h] = s.sink_score[h] + inc[:ns]
                hs.score = hs.score + inc[ns:]
        return out

    # -- read path ----------------------------------------------------------
    def attend(self, b: int, q: np.ndarray, sm_scale: float | None = None,
               accumulate: bool = True) -> np.ndarray:
        """Decode attention of sequence b.  q: fp32 [Hq, D].  Returns fp64
        [Hq, D].  Query head j reads KV head j // G (consecutive query heads
        share a KV head).  With ``accumulate`` the H2O scores of every attended
        token (sinks included) grow by the column sums of this step's
        probabilities.

        Hybrid precision (bf16_window = W > 0; "KV Cache optimization
        techniques" section 1.3): a held token whose position is one of the
        last W (>= pos_total - W) attends with its unquantised bf16 values,
        every older one with its codes.  Reading: the page's "recent" slice
        is the most recent tokens (its code slices the oldest, a bug), over a
        window of fixed length that slides with the sequence."""
        s = self.seqs[b]
        out = np.zeros((self.hq, self.d), np.float64)
        for h in range(self.hkv):
            hs = s.heads[h]
            kq = self.dequantize(hs.kcodes, hs.kscale)
            vq = self.dequantize(hs.vcodes, hs.vscale)
            if self.bf16_window > 0:
                recent = hs.pos >= s.pos_total - self.bf16_window
                kq[recent] = s.raw_k[h][hs.pos[recent]].astype(np.float64)
                vq[recent] = s.raw_v[h][hs.pos[recent]].astype(np.float64)
            keys = np.vstack([s.sink_k[h].astype(np.float64), kq])
            vals = np.vstack([s.sink_v[h].astype(np.float64), vq])
            qg = q[h * self.group:(h + 1) * self.group]
            o, p = attention(qg, keys, vals, sm_scale)
            out[h * self.group:(h + 1) * self.group] = o
            if accumulate:
                inc = h2o_increments(p)
                ns = s.sink_k[h].shape[0]
                s.sink_score[h] = s.sink_score[h] + inc[:ns]
                hs.score = hs.score + inc[ns:]
        return out

    # -- eviction -----------------------------------------------------------
    def keep_masks(self, b: int, mode: str, budget: int = 0, recent: int = 0,
                   window: int = 0, retention: float = 1.0) -> list:
        s = self.seqs[b]
        if mode == "block":
            # slot order is insertion order while only whole blocks are evicted
            keep = select_blocks([hs.score for hs in s.heads], s.heads[0].pos.shape[0], recent, retention)
            return [keep.copy() for _ in range(self.hkv)]
        masks = []
        for h in range(self.hkv):
            hs = s.heads[h]
            ns = s.sink_k[h].shape[0]
            if mode == "h2o":
                masks.append(select_h2o(hs.pos, hs.score, s.pos_total, budget, recent, ns))
            elif mode == "streaming":
                masks.append(select_streaming(hs.pos, s.pos_total, window, ns))
            else:
                raise ValueError(mode)
        return masks

    def evict(self, b: int, masks: list) -> None:
        """Drop the tokens whose mask entry is False (order of the rest kept)."""
        s = self.seqs[b]
        for h, m in enumerate(masks):
            hs = s.heads[h]
            s.heads[h] = HeadState(hs.pos[m], hs.kcodes[m], hs.kscale[m],
                                   hs.vcodes[m], hs.vscale[m], hs.score[m])

    def kept_positions(self, b: int, h: int) -> np.ndarray:
        """Sorted positions of the non-sink tokens held for (b, h)."""
        return np.sort(self.seqs[b].heads[h].pos)

    def load_head(self, b: int, h: int, pos, kcodes, kscale, vcodes, vscale, score) -> None:
        """Replace the state of (b, h) (lock-step re-synchronisation)."""
        self.seqs[b].heads[h] = HeadState(np.asarray(pos, np.int64), np.asarray(kcodes, np.int8),
                                          np.asarray(kscale, np.float32), np.asarray(vcodes, np.int8),
                                          np.asarray(vscale, np.float32), np.asarray(score, np.float64))
