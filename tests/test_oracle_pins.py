"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test ties one oracle function to something other than itself: values the
pages print, closed forms, worked examples whose scale is exact, library
witnesses, invariants and brute force on tiny inputs.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O


def _read_table(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


# --------------------------------------------------------------------------
# closed form and ratios
# --------------------------------------------------------------------------

def test_closed_form_matches_printed_and_report(golden_dir):
    rows = _read_table(os.path.join(golden_dir, "kv_closed_form.txt"))
    assert len(rows) == 6
    for src, seq, bpe, gib in rows:
        got = O.kv_cache_gib(1, int(seq), 32, 32, 128, int(bpe))
        assert got == pytest.approx(float(gib), abs=0.005), (src, seq)
    # the report's per-token figure: 0.5 MB for fp16
    assert O.kv_cache_bytes(1, 1, 32, 32, 128, 2) == 512 * 1024


def test_closed_form_scales_linearly():
    a = O.kv_cache_bytes(3, 100, 2, 5, 128, 2)
    assert a == 2 * 2 * 5 * 128 * 2 * 3 * 100
    assert O.kv_cache_bytes(3, 200, 2, 5, 128, 2) == 2 * a


def test_compression_ratios_match_checklist(golden_dir):
    rows = _read_table(os.path.join(golden_dir, "compression_ratios.txt"))
    x = np.random.default_rng(0).standard_normal((64, 128)).astype(np.float32)
    bf16_bytes = x.size * 2
    for name, bits, ratio in rows:
        bits = int(bits)
        if bits == 16:
            stored = bf16_bytes
        else:
            codes, _ = O.quantize_rows(x, bits)
            stored = (O.pack_int4(codes) if bits == 4 else codes).nbytes
            assert O.stored_bytes_per_token_head(bits, with_scales=False) / (2 * 128 * 2) == float(ratio)
        assert stored / bf16_bytes == float(ratio), name
    # with the two fp32 scales per token-head
    assert O.stored_bytes_per_token_head(8) == 264
    assert O.stored_bytes_per_token_head(4) == 136


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------

def test_quant_worked_int8_exact_scale():
    # amax = 127 makes the scale exactly 1.0, so the codes are the
    # round-half-to-even of the inputs (torch.round on the page is half-even).
    row = np.zeros(128, np.float32)
    vals = [127.0, 2.5, 3.5, -2.5, 0.5, -0.5, 1.5, -126.5, 0.49999997, 100.25]
    row[:len(vals)] = vals
    codes, scale = O.quantize_rows(row[None], 8)
    assert scale[0] == np.float32(1.0)
    assert codes[0, :len(vals)].tolist() == [127, 2, 4, -2, 0, 0, 2, -126, 0, 100]


def test_quant_worked_int4_exact_scale():
    row = np.zeros(128, np.float32)
    vals = [7.0, 1.5, 2.5, -3.5, -6.5, 0.5, -7.0]
    row[:len(vals)] = vals
    codes, scale = O.quantize_rows(row[None], 4)
    assert scale[0] == np.float32(1.0)
    assert codes[0, :len(vals)].tolist() == [7, 2, 2, -4, -6, 0, -7]


def test_quant_power_of_two_scale():
    # amax = 254 -> scale 2.0 exactly; x = 5 -> 2.5 -> 2; x = 7 -> 3.5 -> 4.
    row = np.zeros(128, np.float32)
    row[:3] = [254.0, 5.0, 7.0]
    codes, scale = O.quantize_rows(row[None], 8)
    assert scale[0] == np.float32(2.0)
    assert codes[0, :3].tolist() == [127, 2, 4]


@pytest.mark.parametrize("bits", [8, 4])
def test_quant_invariants(bits):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((500, 128)) * rng.uniform(0.01, 50, (500, 1))).astype(np.float32)
    codes, scale = O.quantize_rows(x, bits)
    qmax = 127 if bits == 8 else 7
    # the amax element maps to +-qmax
    i = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(500), i].astype(int)
    assert np.all(np.abs(top) == qmax)
    assert np.all(np.sign(top) == np.sign(x[np.arange(500), i]))
    # codes stay in range
    assert codes.min() >= -qmax and codes.max() <= qmax
    # per-element dequantisation error <= scale/2 (+ fp32 division rounding)
    err = np.abs(x.astype(np.float64) - O.dequantize(codes, scale))
    bound = scale.astype(np.float64)[:, None] / 2 + np.abs(x.astype(np.float64)) * 2.0 ** -23
    assert np.all(err <= bound)
    # scale is amax / qmax in fp32
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(scale, (amax / np.float32(qmax)).astype(np.float32))


def test_quant_zero_row():
    codes, scale = O.quantize_rows(np.zeros((2, 128), np.float32), 8)
    assert np.all(codes == 0) and np.all(scale == 0)


@pytest.mark.parametrize("bits", [8, 4])
def test_quant_torch_witness(bits):
    # Library witness: the page's per-token quantiser written with torch ops in
    # fp32, without the techniques page's 1e-8 epsilon (the Technical Report's
    # quantize_kv has none).
    rng = np.random.default_rng(2)
    x = rng.standard_normal((300, 128)).astype(np.float32)
    x[:, 7] *= 10
    t = torch.from_numpy(x)
    qmax = (1 << (bits - 1)) - 1
    s = t.abs().amax(dim=-1, keepdim=True) / qmax
    want = torch.round(t / s).clamp(-qmax - 1, qmax).to(torch.int8).numpy()
    codes, scale = O.quantize_rows(x, bits)
    assert np.array_equal(codes, want)
    assert np.array_equal(scale, s[:, 0].numpy())


def test_int4_packing_layout_and_roundtrip():
    codes = np.zeros(128, np.int8)
    codes[:4] = [1, -1, -8, 7]
    p = O.pack_int4(codes[None])[0]
    assert p[0] == 0xF1 and p[1] == 0x78
    rng = np.random.default_rng(3)
    c = rng.integers(-8, 8, (10, 128)).astype(np.int8)
    assert np.array_equal(O.unpack_int4(O.pack_int4(c)), c)


def test_quant_rejects_bits():
    with pytest.raises(ValueError):
        O.quantize_rows(np.ones((1, 128), np.float32), 2)


def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x4049], np.uint16)
    assert O.bf16_bits_to_f32(bits).tolist() == [1.0, -2.0, 0.0, 3.140625]


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def test_attention_sdpa_witness():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((5, 128))
    k = rng.standard_normal((37, 128)) * 2
    v = rng.standard_normal((37, 128))
    out, probs = O.attention(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None])[0]
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(probs.sum(axis=1), 1.0)


def test_attention_bruteforce_loops():
    rng = np.random.default_rng(5)
    d = 8
    q = rng.standard_normal((2, d))
    k = rng.standard_normal((5, d))
    v = rng.standard_normal((5, d))
    out, _ = O.attention(q, k, v)
    for g in range(2):
        w = [math.exp(sum(q[g, i] * k[t, i] for i in range(d)) / math.sqrt(d)) for t in range(5)]
        z = sum(w)
        for j in range(d):
            assert out[g, j] == pytest.approx(sum(w[t] * v[t, j] for t in range(5)) / z, rel=1e-12)


def test_attention_equal_keys_gives_mean_values():
    rng = np.random.default_rng(6)
    k = np.tile(rng.standard_normal(128), (20, 1))
    v = rng.standard_normal((20, 128))
    out, _ = O.attention(rng.standard_normal((3, 128)), k, v)
    assert np.allclose(out, v.mean(axis=0)[None], atol=1e-12)


def test_attention_planted_token_dominates():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((50, 128)) * 0.1
    k[17] = q[0] * (30 * math.sqrt(128) / float(q[0] @ q[0]))  # logit +30
    v = rng.standard_normal((50, 128))
    out, probs = O.attention(q, k, v)
    assert probs[0, 17] > 1 - 1e-10
    assert np.allclose(out[0], v[17], atol=1e-9)


def test_attention_permutation_invariant():
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal((4, 128)), rng.standard_normal((33, 128)), rng.standard_normal((33, 128))
    perm = rng.permutation(33)
    a, pa = O.attention(q, k, v)
    b, pb = O.attention(q, k[perm], v[perm])
    assert np.allclose(a, b, atol=1e-13)
    assert np.allclose(pa[:, perm], pb, atol=1e-15)


def _fill_cache(bits, B, Hq, Hkv, T, seed):
    rng = np.random.default_rng(seed)
    c = O.OracleCache(B, Hq, Hkv, bits)
    k = rng.standard_normal((B, Hkv, T, 128)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, T, 128)).astype(np.float32)
    for b in range(B):
        c.append(b, k[b], v[b])
    return c, k, v, rng


def test_gqa_grouping_matches_repeat_interleave():
    # Query head j reads KV head j // G: the layout transformers and vLLM use
    # (repeat_interleave of the KV heads), checked through torch sdpa.
    B, Hq, Hkv, T = 1, 6, 2, 23
    c, k, v, rng = _fill_cache(8, B, Hq, Hkv, T, 9)
    q = rng.standard_normal((Hq, 128)).astype(np.float32)
    out = c.attend(0, q, accumulate=False)
    hs = c.seqs[0]
    keys, vals = [], []
    for h in range(Hkv):
        keys.append(np.vstack([hs.sink_k[h], O.dequantize(hs.heads[h].kcodes, hs.heads[h].kscale)]))
        vals.append(np.vstack([hs.sink_v[h], O.dequantize(hs.heads[h].vcodes, hs.heads[h].vscale)]))
    K = torch.from_numpy(np.stack(keys)).double().repeat_interleave(Hq // Hkv, dim=0)
    V = torch.from_numpy(np.stack(vals)).double().repeat_interleave(Hq // Hkv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).double()[:, None, :], K, V)[:, 0, :]
    assert np.allclose(out, ref.numpy(), atol=1e-12)


def test_sinks_stored_exactly_and_rest_quantised():
    c, k, v, _ = _fill_cache(8, 1, 2, 2, 9, 10)
    s = c.seqs[0]
    for h in range(2):
        assert np.array_equal(s.sink_k[h], k[0, h, :4])
        assert np.array_equal(s.sink_v[h], v[0, h, :4])
        assert s.heads[h].pos.tolist() == list(range(4, 9))
        codes, scale = O.quantize_rows(k[0, h, 4:], 8)
        assert np.array_equal(s.heads[h].kcodes, codes)
        assert np.array_equal(s.heads[h].kscale, scale)


def test_short_context_all_sinks():
    c, k, v, rng = _fill_cache(8, 1, 1, 1, 3, 11)
    assert c.seqs[0].heads[0].pos.size == 0
    q = rng.standard_normal((1, 128)).astype(np.float32)
    out = c.attend(0, q)
    ref, _ = O.attention(q, k[0, 0], v[0, 0])
    assert np.allclose(out, ref, atol=1e-12)


# --------------------------------------------------------------------------
# scores and selection
# --------------------------------------------------------------------------

def test_score_increments_sum_to_group_size():
    B, Hq, Hkv, T = 2, 8, 2, 40
    c, _, _, rng = _fill_cache(8, B, Hq, Hkv, T, 12)
    for step in range(3):
        before = [[c.seqs[b].heads[h].score.sum() + c.seqs[b].sink_score[h].sum() for h in range(Hkv)]
                  for b in range(B)]
        for b in range(B):
            c.attend(b, rng.standard_normal((Hq, 128)).astype(np.float32))
        for b in range(B):
            for h in range(Hkv):
                tot = c.seqs[b].heads[h].score.sum() + c.seqs[b].sink_score[h].sum()
                assert tot - before[b][h] == pytest.approx(Hq // Hkv, abs=1e-12)


def _brute_select(pos, score, pos_total, budget, recent):
    n = len(pos)
    if 4 + n <= budget:
        return set(pos)
    keep = {p for p in pos if p >= pos_total - recent}
    cand = sorted(((-s, p) for p, s in zip(pos, score) if p < pos_total - recent))
    keep |= {p for _, p in cand[:budget - 4 - recent]}
    return keep


def test_select_h2o_bruteforce():
    rng = np.random.default_rng(13)
    for trial in range(200):
        n = int(rng.integers(0, 30))
        pos_total = 4 + n + int(rng.integers(0, 5))
        pos = rng.choice(np.arange(4, pos_total), size=n, replace=False)
        # make the recent window fully present, as it always is in the cache
        recent = int(rng.integers(0, 6))
        pos = np.unique(np.concatenate([pos, np.arange(max(4, pos_total - recent), pos_total)]))
        rng.shuffle(pos)
        score = rng.integers(0, 4, size=pos.size).astype(np.float64)  # many ties
        budget = 4 + recent + int(rng.integers(0, 10))
        keep = O.select_h2o(pos, score, pos_total, budget, recent)
        assert set(pos[keep].tolist()) == _brute_select(pos.tolist(), score.tolist(), pos_total, budget, recent)
        if 4 + pos.size > budget:
            assert keep.sum() == budget - 4


def test_select_ties_go_to_lower_position():
    pos = np.array([10, 5, 7, 20, 21])
    score = np.array([1.0, 1.0, 1.0, 0.0, 0.0])
    keep = O.select_h2o(pos, score, pos_total=22, budget=4 + 2 + 2, recent=2)
    assert sorted(pos[keep].tolist()) == [5, 7, 20, 21]


def test_streaming_rule_exact():
    for n_total, window in [(5000, 2048), (2053, 2048), (2052, 2048), (100, 2048), (40, 8)]:
        pos = np.arange(4, n_total)
        keep = O.select_streaming(pos, n_total, window)
        kept = pos[keep].tolist()
        if n_total - 4 <= window:
            assert kept == list(range(4, n_total))
        else:
            assert kept == list(range(n_total - window, n_total))
            assert len(kept) == window


def test_identity_budget_covers_context():
    # Evicting nothing must equal full attention by brute force.
    B, Hq, Hkv, T = 1, 4, 2, 30
    c, k, v, rng = _fill_cache(8, B, Hq, Hkv, T, 14)
    q = rng.standard_normal((Hq, 128)).astype(np.float32)
    out = c.attend(0, q)
    masks = c.keep_masks(0, "h2o", budget=4 + T, recent=8)
    assert all(m.all() for m in masks)
    c.evict(0, masks)
    out2 = c.attend(0, q, accumulate=False)
    assert np.array_equal(out, out2)
    s = c.seqs[0]
    for h in range(Hkv):
        keys = np.vstack([k[0, h, :4], O.dequantize(*O.quantize_rows(k[0, h, 4:], 8))])
        vals = np.vstack([v[0, h, :4], O.dequantize(*O.quantize_rows(v[0, h, 4:], 8))])
        for g in range(2):
            qq = q[h * 2 + g].astype(np.float64)
            w = np.exp(keys @ qq / math.sqrt(128) - (keys @ qq / math.sqrt(128)).max())
            assert np.allclose(out[h * 2 + g], (w[:, None] * vals).sum(0) / w.sum(), atol=1e-12)


def test_planted_heavy_hitters_kept_tiny_workload():
    # Tiny single-layer workload: every planted token outside the sinks and the
    # recent window survives the first eviction (10 planted <= 92 heavy places).
    from compressed_kv_cache_kvc_gb300 import workloads as W
    w = W.WORKLOADS["tiny_b1_h8_t512_int8_h2o"]
    d = W.gen_layer(w, 0)
    c = O.OracleCache(w.batch, w.num_q_heads, w.num_kv_heads, w.bits)
    f = O.bf16_bits_to_f32
    c.append(0, f(d["k"][0]), f(d["v"][0]))
    c.append(0, f(d["k_new"][0]), f(d["v_new"][0]))
    c.attend(0, f(d["q"][0]))
    masks = c.keep_masks(0, "h2o", budget=w.budget, recent=w.recent)
    c.evict(0, masks)
    p_total = w.context + 1
    for h in range(w.num_kv_heads):
        kept = set(c.kept_positions(0, h).tolist())
        assert len(kept) == w.budget - 4
        planted = set(np.nonzero(d["planted"][0, h])[0].tolist())
        assert planted and planted <= kept | set(range(p_total - w.recent, p_total))


def test_cache_keep_masks_brute_force():
    """keep_masks("h2o") of a cache after a few decode steps keeps what the
    plain-Python rule keeps on that cache's positions and scores."""
    B, Hq, Hkv, T = 1, 4, 2, 60
    c, _, _, rng = _fill_cache(8, B, Hq, Hkv, T, 15)
    for _ in range(3):
        c.attend(0, rng.standard_normal((Hq, 128)).astype(np.float32))
    s = c.seqs[0]
    for budget, recent in [(30, 8), (20, 0), (14, 10), (4 + T, 8)]:
        masks = c.keep_masks(0, "h2o", budget=budget, recent=recent)
        for h in range(Hkv):
            hs = s.heads[h]
            want = _brute_select(hs.pos.tolist(), hs.score.tolist(), s.pos_total, budget, recent)
            assert set(hs.pos[masks[h]].tolist()) == want, (budget, recent, h)


# ---------------------------------------------------------------------------
# block-granular eviction (the survey page's block manager)
# ---------------------------------------------------------------------------

def _block_scores(block_sums, hkv=2, extra=0):
    """Per-head score arrays whose block sums (over heads and slots) are the
    given values: the whole sum sits on slot 0 of head 0."""
    n = len(block_sums) * 16 + extra
    sc = [np.zeros(n) for _ in range(hkv)]
    for p, v in enumerate(block_sums):
        sc[0][16 * p] = v
    return sc


def test_blocks_worked_example_with_a_tie():
    # 100 slots, recent 20: candidates are the 5 full blocks before slot 80;
    # retention 0.4 evicts int(5 * 0.6) = 3 of them: sums 5, 1, 4, 1, 9 ->
    # blocks 1 and 3 (tie at 1, earlier first), then block 2
    sc = _block_scores([5.0, 1.0, 4.0, 1.0, 9.0], extra=20)
    keep = O.select_blocks(sc, 100, recent=20, retention=0.4)
    want = np.ones(100, dtype=bool)
    want[16:64] = False
    assert np.array_equal(keep, want)


def test_blocks_tie_at_the_eviction_boundary():
    # sums 5, 1, 4, 1, 9 with retention 0.7: int(5 * 0.3) = 1 block goes, and
    # blocks 1 and 3 tie for it: the earlier one goes (a stable sort, as the
    # survey page's sorted() leaves equal keys)
    sc = _block_scores([5.0, 1.0, 4.0, 1.0, 9.0], extra=20)
    keep = O.select_blocks(sc, 100, recent=20, retention=0.7)
    assert np.array_equal(np.nonzero(~keep)[0], np.arange(16, 32))


def test_blocks_edges():
    sc = _block_scores([3.0, 2.0, 1.0], extra=7)  # 55 slots
    assert O.select_blocks(sc, 55, recent=7, retention=1.0).all()          # keep everything
    assert O.select_blocks(sc, 55, recent=60, retention=0.1).all()         # no candidate
    keep = O.select_blocks(sc, 55, recent=7, retention=1e-9)                # int(3 * (1 - 1e-9)) = 2
    assert np.array_equal(np.nonzero(~keep)[0], np.arange(16, 48))         # blocks 2 and 1 go
    keep = O.select_blocks(sc, 55, recent=8, retention=0.5)                 # 47 slots -> 2 candidates, evict 1
    assert np.array_equal(np.nonzero(~keep)[0], np.arange(16, 32))


def test_blocks_against_numpy_means():
    rng = np.random.default_rng(8)
    for trial in range(20):
        hkv = int(rng.integers(1, 5))
        n_slots = int(rng.integers(1, 300))
        recent = int(rng.integers(0, 80))
        retention = float(rng.uniform(0.05, 1.0))
        sc = [rng.random(n_slots) for _ in range(hkv)]
        keep = O.select_blocks(sc, n_slots, recent, retention)
        n_cand = max(0, n_slots - recent) // 16
        n_evict = int(n_cand * (1.0 - retention))
        means = np.array([np.mean([s[16 * p:16 * p + 16] for s in sc]) for p in range(n_cand)])
        lowest = np.argsort(means, kind="stable")[:n_evict]
        want = np.ones(n_slots, dtype=bool)
        for p in lowest:
            want[16 * p:16 * p + 16] = False
        assert np.array_equal(keep, want), trial
        # whole blocks only, never the recent window or the unfilled last block
        assert (~keep).sum() == 16 * n_evict
        assert keep[16 * n_cand:].all()


def test_cache_block_masks_against_numpy_means():
    """keep_masks("block") of a cache after a few decode steps: whole pages
    of the pool (slot order), the lowest mean scores over all heads go, the
    last `recent` slots and the unfilled page stay; the same mask for every
    head."""
    B, Hq, Hkv, T = 1, 4, 2, 150
    c, _, _, rng = _fill_cache(8, B, Hq, Hkv, T, 16)
    for _ in range(3):
        c.attend(0, rng.standard_normal((Hq, 128)).astype(np.float32))
    s = c.seqs[0]
    n_slots = T - 4
    for recent, retention in [(20, 0.5), (0, 0.25), (40, 0.9)]:
        masks = c.keep_masks(0, "block", recent=recent, retention=retention)
        n_cand = (n_slots - recent) // 16
        means = np.array([np.mean([s.heads[h].score[16 * p:16 * p + 16] for h in range(Hkv)])
                          for p in range(n_cand)])
        want = np.ones(n_slots, dtype=bool)
        for p in np.argsort(means, kind="stable")[:int(n_cand * (1.0 - retention))]:
            want[16 * p:16 * p + 16] = False
        for h in range(Hkv):
            assert np.array_equal(masks[h], want), (recent, retention, h)


# ---------------------------------------------------------------------------
# Hybrid precision (the last W positions attend in bf16)
# ---------------------------------------------------------------------------

def _bf16_round(x):
    b = np.asarray(x, np.float32).view(np.uint32)
    b = ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    return O.bf16_bits_to_f32(b)


def test_hybrid_window_covering_the_context_is_bf16_attention():
    """A window longer than the sequence keeps every token unquantised: the
    output is plain fp64 attention over the bf16 inputs (torch SDPA witness
    with the KV heads repeated for GQA)."""
    rng = np.random.default_rng(40)
    Hq, Hkv, n = 8, 2, 45
    k = _bf16_round(rng.standard_normal((Hkv, n, 128)) * 2.0)
    v = _bf16_round(rng.standard_normal((Hkv, n, 128)))
    q = _bf16_round(rng.standard_normal((Hq, 128)))
    c = O.OracleCache(1, Hq, Hkv, 4, bf16_window=1000)
    c.append(0, k, v)
    out = c.attend(0, q)
    K = torch.from_numpy(k).double().repeat_interleave(Hq // Hkv, dim=0)
    V = torch.from_numpy(v).double().repeat_interleave(Hq // Hkv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q).double()[:, None, :], K, V)[:, 0, :]
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)
    # and it differs from the INT4 cache: the window matters
    plain = O.OracleCache(1, Hq, Hkv, 4)
    plain.append(0, k, v)
    assert np.abs(plain.attend(0, q) - out).max() > 1e-3


def test_hybrid_window_zero_is_the_quantised_cache():
    rng = np.random.default_rng(41)
    k = _bf16_round(rng.standard_normal((2, 30, 128)))
    v = _bf16_round(rng.standard_normal((2, 30, 128)))
    q = _bf16_round(rng.standard_normal((4, 128)))
    a, b = O.OracleCache(1, 4, 2, 8), O.OracleCache(1, 4, 2, 8, bf16_window=0)
    a.append(0, k, v)
    b.append(0, k, v)
    assert np.array_equal(a.attend(0, q), b.attend(0, q))
    for h in range(2):
        assert np.array_equal(a.seqs[0].heads[h].score, b.seqs[0].heads[h].score)


def test_hybrid_window_boundary_brute_force():
    """One KV head, one query, INT4, window 3: every key row has one large
    outlier, so INT4 rounds its other entries to 0 and the choice of
    precision per token is visible.  Brute force in plain Python: positions
    0-3 are sinks (bf16), positions >= P - 3 use the bf16 values, the rest
    code * scale; checked before and after one more token moves position
    P - 3 out of the window."""
    rng = np.random.default_rng(42)
    n = 10
    base = rng.uniform(0.2, 0.6, (1, n + 1, 128))
    base[..., 0] = 60.0
    k = _bf16_round(base)
    v = _bf16_round(rng.uniform(-1.0, 1.0, (1, n + 1, 128)))
    q = _bf16_round(rng.uniform(-1.0, 1.0, (1, 128)))
    q[0, 0] = 0.0  # the outlier column does not decide the logits

    def brute(ntok, window):
        kc, ks = O.quantize_rows(k[0, :ntok], 4)
        vc, vs = O.quantize_rows(v[0, :ntok], 4)
        logits, rows = [], []
        for p in range(ntok):
            exact = p < 4 or p >= ntok - window
            kr = [float(x) for x in k[0, p]] if exact else [float(kc[p, d]) * float(ks[p]) for d in range(128)]
            vr = [float(x) for x in v[0, p]] if exact else [float(vc[p, d]) * float(vs[p]) for d in range(128)]
            logits.append(sum(float(q[0, d]) * kr[d] for d in range(128)) / math.sqrt(128))
            rows.append(vr)
        m = max(logits)
        e = [math.exp(x - m) for x in logits]
        z = sum(e)
        return np.array([sum(e[p] / z * rows[p][d] for p in range(ntok)) for d in range(128)])

    c = O.OracleCache(1, 1, 1, 4, bf16_window=3)
    c.append(0, k[:, :n], v[:, :n])
    got = c.attend(0, q, accumulate=False)[0]
    np.testing.assert_allclose(got, brute(n, 3), rtol=0, atol=1e-12)
    assert np.abs(got - brute(n, 0)).max() > 1e-4 and np.abs(got - brute(n, n)).max() > 1e-4
    c.append(0, k[:, n:n + 1], v[:, n:n + 1])
    np.testing.assert_allclose(c.attend(0, q, accumulate=False)[0], brute(n + 1, 3), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Prefill: causal attention of the prompt and the H2O scores it gives
# ---------------------------------------------------------------------------

def test_prefill_attention_against_causal_sdpa():
    rng = np.random.default_rng(50)
    Hq, Hkv, n = 8, 2, 37
    q = _bf16_round(rng.standard_normal((Hq, n, 128)))
    k = _bf16_round(rng.standard_normal((Hkv, n, 128)))
    v = _bf16_round(rng.standard_normal((Hkv, n, 128)))
    out, sc = O.prefill_attention(q, k, v)
    K = torch.from_numpy(k).double().repeat_interleave(Hq // Hkv, dim=0)
    V = torch.from_numpy(v).double().repeat_interleave(Hq // Hkv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q).double(), K, V, is_causal=True)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)
    # every query's probabilities sum to 1: a KV head's scores sum to G * n
    np.testing.assert_allclose(sc.sum(axis=1), [Hq // Hkv * n] * Hkv, rtol=1e-12)


def test_prefill_scores_brute_force():
    """Column sums written out in plain Python on a tiny prompt (head dim 8):
    key t collects, from every query i >= t of the two query heads, that
    query's softmax probability on t."""
    rng = np.random.default_rng(51)
    Hq, Hkv, n, d = 2, 1, 6, 8
    q = rng.standard_normal((Hq, n, d))
    k = rng.standard_normal((Hkv, n, d))
    v = rng.standard_normal((Hkv, n, d))
    out, sc = O.prefill_attention(q, k, v)
    want = [0.0] * n
    for j in range(Hq):
        for i in range(n):
            lg = [sum(q[j, i, e] * k[0, t, e] for e in range(d)) / math.sqrt(d) for t in range(i + 1)]
            m = max(lg)
            ex = [math.exp(x - m) for x in lg]
            z = sum(ex)
            for t in range(i + 1):
                want[t] += ex[t] / z
            o = [sum(ex[t] / z * v[0, t, e] for t in range(i + 1)) for e in range(d)]
            np.testing.assert_allclose(out[j, i], o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(sc[0], want, rtol=0, atol=1e-12)
    # the last key is seen by the last query only
    assert sc[0, -1] < Hq and sc[0, 0] > sc[0, -1]


def test_oracle_cache_prefill_sets_the_scores():
    rng = np.random.default_rng(52)
    Hq, Hkv, n = 4, 2, 30
    q = _bf16_round(rng.standard_normal((Hq, n, 128)))
    k = _bf16_round(rng.standard_normal((Hkv, n, 128)))
    v = _bf16_round(rng.standard_normal((Hkv, n, 128)))
    c = O.OracleCache(1, Hq, Hkv, 8)
    out = c.prefill(0, q, k, v)
    _, sc = O.prefill_attention(q, k, v)
    np.testing.assert_array_equal(out, O.prefill_attention(q, k, v)[0])
    for h in range(Hkv):
        assert np.array_equal(c.seqs[0].sink_score[h], sc[h, :4])
        assert np.array_equal(c.seqs[0].heads[h].score, sc[h, 4:])
    with pytest.raises(ValueError):
        c.prefill(0, q, k, v)


# ---------------------------------------------------------------------------
# FP8 E4M3 codes
# ---------------------------------------------------------------------------

def test_e4m3_against_torch_float8():
    """Library witness: torch's float8_e4m3fn conversion (round to nearest
    even) on values within the finite range, and its decoding of every
    finite code."""
    rng = np.random.default_rng(70)
    y = (rng.standard_normal(100000) * np.exp(rng.uniform(-12, 7, 100000))).astype(np.float32)
    y = np.clip(y, -448, 448).astype(np.float32)
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(y), want)
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]  # the NaN codes
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(O.e4m3_decode(codes), ref)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes).astype(np.float32)), codes)


@pytest.mark.parametrize("y,code", [
    (1.0, 0x38), (448.0, 0x7E), (-2.5, 0xC2),
    (2.0 ** -9, 0x01),                  # smallest subnormal
    (2.0 ** -10, 0x00),                 # half of it: tie to the even code 0
    (0.75 * 2.0 ** -9, 0x01),
    (2.0 ** -6, 0x08),                  # smallest normal
    (17.0, 0x58), (19.0, 0x5A),         # ties between 16/18 and 18/20 go to the even fraction
    (460.0, 0x7E),                      # nearest is 448
    (1.0e6, 0x7E), (-1.0e6, 0xFE),      # saturation to the largest finite value
])
def test_e4m3_worked_values(y, code):
    assert int(O.e4m3_encode(np.array([y], np.float32))[0]) == code


def test_e4m3_row_quantiser_invariants():
    rng = np.random.default_rng(71)
    x = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-4, 4, (64, 1)))).astype(np.float32)
    x[3] = 0.0
    codes, scale = O.quantize_rows_e4m3(x)
    amax = np.abs(x).max(axis=1)
    np.testing.assert_array_equal(scale, (amax / np.float32(448.0)).astype(np.float32))
    assert scale[3] == 0 and not codes[3].any()
    rows = np.arange(64) != 3
    # the amax element maps to +-448 (code 0x7E / 0xFE)
    j = np.abs(x).argmax(axis=1)
    assert np.all((codes[rows, j[rows]] & 0x7F) == 0x7E)
    # within half a quantum: 2^-4 relative for normals, 2^-10 * scale for subnormals
    dec = O.e4m3_decode(codes) * scale[:, None].astype(np.float64)
    err = np.abs(dec - x.astype(np.float64))
    bound = np.abs(x) * 2.0 ** -4 * (1 + 1e-6) + scale[:, None] * 2.0 ** -10 * (1 + 1e-6)
    assert np.all(err <= bound)


def test_fp8_cache_attends_with_torch_float8_values():
    """Library witness: an E4M3 cache's decode attention is torch SDPA over
    the bf16 sinks and torch's float8_e4m3fn reading of the stored codes
    times their scales; the codes are torch's conversion of x / scale."""
    rng = np.random.default_rng(72)
    Hq, Hkv, T = 4, 2, 50
    k = _bf16_round(rng.standard_normal((Hkv, T, 128)) * 3)
    v = _bf16_round(rng.standard_normal((Hkv, T, 128)))
    q = _bf16_round(rng.standard_normal((Hq, 128)))
    c = O.OracleCache(1, Hq, Hkv, 8, codes="e4m3")
    c.append(0, k, v)
    out = c.attend(0, q, accumulate=False)
    s = c.seqs[0]

    def f8(codes, scale):
        t = torch.from_numpy(np.ascontiguousarray(codes).view(np.uint8)).view(torch.float8_e4m3fn).double()
        return t * torch.from_numpy(np.asarray(scale, np.float64))[:, None]

    keys, vals = [], []
    for h in range(Hkv):
        hs = s.heads[h]
        keys.append(torch.cat([torch.from_numpy(s.sink_k[h]).double(), f8(hs.kcodes, hs.kscale)]))
        vals.append(torch.cat([torch.from_numpy(s.sink_v[h]).double(), f8(hs.vcodes, hs.vscale)]))
        x = torch.from_numpy(k[h, 4:])
        sc = x.abs().amax(dim=-1, keepdim=True) / 448.0
        want = (x / sc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(hs.kcodes.view(np.uint8), want)
    K = torch.stack(keys).repeat_interleave(Hq // Hkv, dim=0)
    V = torch.stack(vals).repeat_interleave(Hq // Hkv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q).double()[:, None, :], K, V)[:, 0]
    assert np.allclose(out, ref.numpy(), atol=1e-12)


# ---------------------------------------------------------------------------
# Prefill over the compressed cache (a prompt on a sequence with context)
# ---------------------------------------------------------------------------

def test_prefill_chunk_of_one_token_is_the_decode_step():
    rng = np.random.default_rng(53)
    Hq, Hkv, n = 8, 2, 60
    k = _bf16_round(rng.standard_normal((Hkv, n + 1, 128)))
    v = _bf16_round(rng.standard_normal((Hkv, n + 1, 128)))
    q = _bf16_round(rng.standard_normal((Hq, 128)))
    a, c = O.OracleCache(1, Hq, Hkv, 4), O.OracleCache(1, Hq, Hkv, 4)
    for o in (a, c):
        o.append(0, k[:, :n], v[:, :n])
    a.append(0, k[:, n:], v[:, n:])
    want = a.attend(0, q)
    got = c.prefill_chunk(0, q[:, None, :], k[:, n:], v[:, n:])[:, 0]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)
    for h in range(Hkv):
        np.testing.assert_allclose(c.seqs[0].heads[h].score, a.seqs[0].heads[h].score, rtol=0, atol=1e-13)


def test_prefill_chunk_with_an_all_covering_window_is_the_exact_prefill():
    """On a fresh sequence whose bf16 window covers every token, the chunk's
    attention is the exact causal prefill, scores included."""
    rng = np.random.default_rng(54)
    Hq, Hkv, n = 4, 2, 40
    q = _bf16_round(rng.standard_normal((Hq, n, 128)))
    k = _bf16_round(rng.standard_normal((Hkv, n, 128)))
    v = _bf16_round(rng.standard_normal((Hkv, n, 128)))
    c = O.OracleCache(1, Hq, Hkv, 8, bf16_window=1000)
    got = c.prefill_chunk(0, q, k, v)
    want, sc = O.prefill_attention(q, k, v)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    for h in range(Hkv):
        np.testing.assert_allclose(c.seqs[0].sink_score[h], sc[h, :4], rtol=0, atol=1e-12)
        np.testing.assert_allclose(c.seqs[0].heads[h].score, sc[h, 4:], rtol=0, atol=1e-12)


def test_prefill_chunk_brute_force_after_eviction():
    """A context with evicted tokens, then a 3-token chunk: plain-Python
    causal attention over the held tokens in their stored form."""
    rng = np.random.default_rng(55)
    Hq, Hkv, n0, n, d = 2, 1, 12, 3, 128
    k = _bf16_round(rng.standard_normal((Hkv, n0 + n, d)))
    v = _bf16_round(rng.standard_normal((Hkv, n0 + n, d)))
    q = _bf16_round(rng.standard_normal((Hq, n, d)))
    c = O.OracleCache(1, Hq, Hkv, 4)
    c.append(0, k[:, :n0], v[:, :n0])
    c.evict(0, [np.array([True, False, True, True, False, True, False, True])])  # pool positions 4..11
    got = c.prefill_chunk(0, q, k[:, n0:], v[:, n0:], accumulate=False)
    hs = c.seqs[0].heads[0]
    kept_pos = [0, 1, 2, 3] + hs.pos.tolist()
    rows_k = {p: (k[0, p].astype(np.float64) if p < 4 else None) for p in kept_pos}
    rows_v = {p: (v[0, p].astype(np.float64) if p < 4 else None) for p in kept_pos}
    kq = O.dequantize(hs.kcodes, hs.kscale)
    vq = O.dequantize(hs.vcodes, hs.vscale)
    for j, p in enumerate(hs.pos.tolist()):
        rows_k[p], rows_v[p] = kq[j], vq[j]
    for g in range(Hq):
        for i in range(n):
            lim = n0 + i
            ps = [p for p in kept_pos if p <= lim]
            lg = [sum(float(q[g, i, e]) * float(rows_k[p][e]) for e in range(d)) / math.sqrt(d) for p in ps]
            m = max(lg)
            ex = [math.exp(x - m) for x in lg]
            z = sum(ex)
            want = [sum(ex[t] / z * float(rows_v[p][e]) for t, p in enumerate(ps)) for e in range(d)]
            np.testing.assert_allclose(got[g, i], want, rtol=0, atol=1e-12)
