"""Hybrid precision: the last W positions of each sequence in a bf16 ring,
older tokens quantised in the pool (bf16_window = W).  Checked against the
oracle with the same window: the pool holds exactly the tokens older than the
window, with the codes the oracle gives; the ring holds the window's bf16
values; the outputs are within the attention tolerance; the kept sets agree;
and the one-call step leaves the same state as the separate calls."""
import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O
from tests import kvc_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()


def _bits(rng, shape):
    from compressed_kv_cache_kvc_gb300.workloads import bf16_bits
    return bf16_bits(rng.standard_normal(shape).astype(np.float32))


def _check_state(cache, ora, B):
    W = cache.bf16_window
    st = T.StateView(cache)
    for b in range(B):
        s = ora.seqs[b]
        P = s.pos_total
        assert int(st.seen[b]) == P
        for h in range(cache.num_kv_heads):
            hs = s.heads[h]
            old = hs.pos < P - W
            pos, kc, ks, vc, vs, sc = st.head(b, h)
            o, oo = np.argsort(pos), np.argsort(hs.pos[old])
            assert np.array_equal(pos[o], hs.pos[old][oo]), (b, h)
            assert np.array_equal(kc[o], hs.kcodes[old][oo]) and np.array_equal(vc[o], hs.vcodes[old][oo]), (b, h)
            assert np.array_equal(ks[o].view(np.uint32), hs.kscale[old][oo].view(np.uint32)), (b, h)
            assert np.array_equal(vs[o].view(np.uint32), hs.vscale[old][oo].view(np.uint32)), (b, h)
            np.testing.assert_allclose(sc[o], hs.score[old][oo], rtol=1e-3, atol=1e-6)
            rpos, rk, rv, rsc = st.ring_head(b, h)
            assert np.array_equal(rpos, np.sort(hs.pos[~old])), (b, h)
            assert np.array_equal(O.bf16_bits_to_f32(rk), s.raw_k[h][rpos])
            assert np.array_equal(O.bf16_bits_to_f32(rv), s.raw_v[h][rpos])
            by_pos = dict(zip(hs.pos.tolist(), hs.score.tolist()))
            np.testing.assert_allclose(rsc, [by_pos[p] for p in rpos.tolist()], rtol=1e-3, atol=1e-6)


ATTN_CASES = [
    # bits, hq, hkv, lengths, W, steps, codes
    (8, 8, 2, [300, 41, 130], 64, 4, "int"),
    (4, 40, 8, [500, 90], 50, 3, "int"),
    (8, 16, 4, [20, 70], 100, 3, "int"),     # the first sequence stays inside the window: empty pool
    (4, 8, 8, [1000], 16, 2, "int"),
    (8, 32, 8, [260], 200, 2, "int"),        # more than one window chunk
    (8, 16, 4, [300, 77], 48, 3, "e4m3"),    # FP8 codes for the tokens that leave the window
]


@pytest.mark.parametrize("bits,hq,hkv,lengths,W,steps,codes", ATTN_CASES)
def test_hybrid_attention_and_state_against_oracle(bits, hq, hkv, lengths, W, steps, codes):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits + hq + W)
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + steps + 15) // 16 + 2
    cache = KVCache(hq, hkv, bits, B * mbps, B, mbps, bf16_window=W, codes=codes)
    ora = O.OracleCache(B, hq, hkv, bits, bf16_window=W, codes=codes)
    f = O.bf16_bits_to_f32
    k = _bits(rng, (B, hkv, T_, 128))
    v = _bits(rng, (B, hkv, T_, 128))
    for b, n in enumerate(lengths):
        # the prefill in three chunks: appends that push window tokens into the pool
        cuts = [0, n // 3, n // 3 + max(1, n // 7), n]
        for a, e in zip(cuts[:-1], cuts[1:]):
            if e > a:
                cache.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, a:e])),
                                      T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, a:e])), seq_begin=b)
                ora.append(b, f(k[b, :, a:e]), f(v[b, :, a:e]))
    _check_state(cache, ora, B)
    for _ in range(steps):
        kn = _bits(rng, (B, hkv, 1, 128))
        vn = _bits(rng, (B, hkv, 1, 128))
        q = _bits(rng, (B, hq, 128))
        cache.quantize_append(T.to_dev_bf16(kn), T.to_dev_bf16(vn))
        out = T.bf16_tensor_to_f32(cache.decode_attention(T.to_dev_bf16(q), accumulate_h2o=True))
        for b in range(B):
            ora.append(b, f(kn[b]), f(vn[b]))
            ref = ora.attend(b, f(q[b]), T.sm_scale())
            T.assert_attention_close(out[b], ref, f"hybrid W={W} b={b}")
        _check_state(cache, ora, B)
    assert cache.read_status() == 0


def _same_hybrid_state(a, b):
    sa, sb = T.StateView(a), T.StateView(b)
    assert np.array_equal(sa.slots, sb.slots) and np.array_equal(sa.seen, sb.seen)
    for seq in range(a.max_batch):
        for h in range(a.num_kv_heads):
            for x, y in zip(sa.head(seq, h), sb.head(seq, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (seq, h)
            for x, y in zip(sa.ring_head(seq, h), sb.ring_head(seq, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (seq, h)
    assert np.array_equal(sa.sink_score.view(np.uint32), sb.sink_score.view(np.uint32))
    assert np.array_equal(sa.counters[:3], sb.counters[:3])


STEP_CASES = [
    # bits, hq, hkv, lengths, W, mode, budget, recent, window, steps
    (8, 16, 4, [600, 333, 50], 64, "h2o", 200, 64, 0, 3),
    (4, 40, 8, [700, 129], 48, "h2o", 300, 100, 0, 3),
    (8, 8, 2, [400, 90], 32, "streaming", 0, 0, 128, 3),
    (8, 8, 2, [30, 45], 64, "h2o", 100, 64, 0, 2),  # the window holds everything: empty pools
]


@pytest.mark.parametrize("bits,hq,hkv,lengths,W,mode,budget,recent,window,steps", STEP_CASES)
def test_hybrid_step_equals_separate_calls(bits, hq, hkv, lengths, W, mode, budget, recent, window, steps):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits * 11 + W + len(lengths))
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + steps + 15) // 16 + 2
    order = np.random.default_rng(4).permutation(B * mbps).astype(np.int32)
    ca = KVCache(hq, hkv, bits, B * mbps, B, mbps, block_order=order, bf16_window=W)
    cb = KVCache(hq, hkv, bits, B * mbps, B, mbps, block_order=order, bf16_window=W)
    k = _bits(rng, (B, hkv, T_, 128))
    v = _bits(rng, (B, hkv, T_, 128))
    for c in (ca, cb):
        for b, n in enumerate(lengths):
            c.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :n])), seq_begin=b)
    for _ in range(steps):
        q = T.to_dev_bf16(_bits(rng, (B, hq, 128)))
        kn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
        vn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
        oa = ca.step(q, kn, vn, mode=mode, budget=budget, recent=recent, window=window)
        ob = cb.decode_step(q, kn, vn, mode=mode, budget=budget, recent=recent, window=window)
        assert cb.last_launch_count() in (4, 5)  # append, split, window, post (+ moves when > 32 rows)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
        _same_hybrid_state(ca, cb)
    assert ca.read_status() == 0 and cb.read_status() == 0


@pytest.mark.parametrize("bits,W,recent", [(8, 64, 64), (4, 32, 80)])
def test_hybrid_h2o_selection_against_oracle(bits, W, recent):
    """One-call step with H2O: the window is kept; the pool keeps the rest of
    the recent window and the heavy hitters the oracle's rule gives."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits + W)
    B, hq, hkv, n, budget = 2, 16, 4, 700, 260
    mbps = (n + 1 + 15) // 16 + 2
    cache = KVCache(hq, hkv, bits, B * mbps, B, mbps, bf16_window=W)
    f = O.bf16_bits_to_f32
    k = _bits(rng, (B, hkv, n, 128))
    v = _bits(rng, (B, hkv, n, 128))
    q = _bits(rng, (B, hq, 128))
    kn = _bits(rng, (B, hkv, 1, 128))
    vn = _bits(rng, (B, hkv, 1, 128))
    cache.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(v))
    out = T.bf16_tensor_to_f32(cache.decode_step(T.to_dev_bf16(q), T.to_dev_bf16(kn), T.to_dev_bf16(vn),
                                                 mode="h2o", budget=budget, recent=recent))
    st = T.StateView(cache)
    for b in range(B):
        ora = O.OracleCache(1, hq, hkv, bits, bf16_window=W)
        ora.append(0, f(k[b]), f(v[b]))
        ora.append(0, f(kn[b]), f(vn[b]))
        T.assert_attention_close(out[b], ora.attend(0, f(q[b]), T.sm_scale()), f"b={b}")
        masks = ora.keep_masks(0, "h2o", budget=budget, recent=recent)
        P = n + 1
        for h in range(hkv):
            hs = ora.seqs[0].heads[h]
            kept_gpu = set(st.head(b, h)[0].tolist()) | set(st.ring_head(b, h)[0].tolist())
            assert len(kept_gpu) == budget - 4
            assert T.kept_sets_agree(kept_gpu, set(hs.pos[masks[h]].tolist()), hs.pos, hs.score,
                                     budget - 4 - recent, P - recent), (b, h)
        assert cache.lengths(b) == (budget - 4 - W, P)
    assert cache.read_status() == 0


@pytest.mark.parametrize("bits,W,recent,budget", [(8, 48, 64, 200), (4, 32, 32, 150)])
def test_hybrid_h2o_steps_lock_step(bits, W, recent, budget):
    """Twelve one-call steps with a bf16 window and H2O eviction, in lock-step
    with the oracle: each step's attention within tolerance, the window the
    last W positions, the kept set (pool and window) the oracle's rule on its
    scores up to near-ties, the kept tokens' scores close to the oracle's;
    then the oracle takes the GPU's state (pool and window)."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits * 13 + W)
    hq, hkv, lengths, steps = 16, 4, [400, 211, 60], 12
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + steps + 15) // 16 + 2
    cache = KVCache(hq, hkv, bits, B * mbps, B, mbps, bf16_window=W)
    ora = O.OracleCache(B, hq, hkv, bits, bf16_window=W)
    f = O.bf16_bits_to_f32
    k = _bits(rng, (B, hkv, T_, 128))
    v = _bits(rng, (B, hkv, T_, 128))
    for b, n in enumerate(lengths):
        cache.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :n])), seq_begin=b)
        ora.append(b, f(k[b, :, :n]), f(v[b, :, :n]))
    for step in range(steps):
        kn = _bits(rng, (B, hkv, 1, 128))
        vn = _bits(rng, (B, hkv, 1, 128))
        q = _bits(rng, (B, hq, 128))
        out = T.bf16_tensor_to_f32(cache.decode_step(T.to_dev_bf16(q), T.to_dev_bf16(kn), T.to_dev_bf16(vn),
                                                     mode="h2o", budget=budget, recent=recent))
        st = T.StateView(cache)
        for b in range(B):
            ora.append(b, f(kn[b]), f(vn[b]))
            T.assert_attention_close(out[b], ora.attend(b, f(q[b]), T.sm_scale()), f"step {step} b={b}")
            s = ora.seqs[b]
            P = s.pos_total
            ns = min(P, 4)
            for h in range(hkv):
                hs = s.heads[h]
                pos, kc, ks, vc, vs, sc = st.head(b, h)
                rpos, _, _, rsc = st.ring_head(b, h)
                assert np.array_equal(rpos, np.arange(max(4, P - W), P))
                kept = set(pos.tolist()) | set(rpos.tolist())
                by_pos = dict(zip(hs.pos.tolist(), hs.score.tolist()))
                exact = O.select_h2o(hs.pos, hs.score, P, budget, recent, ns)
                ora_kept = set(hs.pos[exact].tolist())
                if kept != ora_kept:
                    assert T.kept_sets_agree(kept, ora_kept, hs.pos, hs.score, budget - 4 - recent, P - recent), \
                        (step, b, h)
                assert len(kept) == min(len(hs.pos), budget - 4)
                np.testing.assert_allclose(sc, [by_pos[p] for p in pos.tolist()], rtol=2e-3, atol=1e-5)
                np.testing.assert_allclose(rsc, [by_pos[p] for p in rpos.tolist()], rtol=2e-3, atol=1e-5)
                # lock-step: the oracle takes the GPU's kept tokens; the window
                # tokens' codes are the oracle's own (the ageing reproduces them)
                idx = {p: i for i, p in enumerate(hs.pos.tolist())}
                ri = np.array([idx[p] for p in rpos.tolist()], dtype=np.int64)
                ora.load_head(b, h, np.concatenate([pos, rpos]),
                              np.concatenate([kc, hs.kcodes[ri]]), np.concatenate([ks, hs.kscale[ri]]),
                              np.concatenate([vc, hs.vcodes[ri]]), np.concatenate([vs, hs.vscale[ri]]),
                              np.concatenate([sc, rsc]).astype(np.float64))
                s.sink_score[h] = st.sink_score[b, h, :ns].astype(np.float64)
        used = np.concatenate([st.used_blocks(b) for b in range(B)])
        free = st.free_stack[:int(st.counters[0])]
        assert np.unique(np.concatenate([used, free])).size == B * mbps == used.size + free.size
    assert cache.read_status() == 0
