"""A prompt on sequences that already hold context (a later turn): every
prompt query attends causally to the compressed cache (sinks bf16, pool
tokens dequantised, earlier prompt tokens included) and adds its
probabilities to the H2O scores, against the oracle's prefill_chunk; the
context is empty, a few sink tokens, a fresh prefill, or a prefill followed
by a StreamingLLM eviction (pool slots no longer follow positions)."""
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


CASES = [
    # bits, codes, hq, hkv, batch, context, n1, streaming window (0: no eviction)
    (8, "int", 8, 2, 2, 0, 20, 0),        # an empty sequence: the first queries see only sinks
    (4, "int", 16, 4, 2, 2, 30, 0),       # two sink tokens of context, appended one call earlier
    (4, "int", 32, 8, 2, 100, 17, 0),     # a prefill's context, a prompt ending mid-page
    (8, "int", 40, 8, 1, 200, 40, 64),    # G = 5, after a StreamingLLM eviction
    (8, "e4m3", 16, 4, 1, 50, 25, 0),     # FP8 codes
    (4, "int", 40, 8, 2, 300, 64, 0),     # G = 5: 320 attention rows per KV head, 5 CTAs each
    (8, "int", 8, 8, 2, 130, 70, 0),      # G = 1 (MHA), rows in 5 tiles of 16
    (8, "int", 16, 2, 1, 40, 520, 0),     # 4160 rows per KV head: 64 CTAs, two rounds of row tiles each
    (4, "int", 8, 2, 1, 33100, 9, 0),     # more pages than the kernel stages block ids for (2048)
]


@pytest.mark.parametrize("bits,codes,hq,hkv,batch,ctx,n1,window", CASES)
def test_prefill_context_against_oracle(bits, codes, hq, hkv, batch, ctx, n1, window):
    """Outputs, codes, lengths and every held token's score against the
    oracle; the kernel runs as three launches (the append, the two passes of
    the multi-query attention)."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits + hq + ctx + n1)
    mbps = (ctx + n1 + 15) // 16 + 2
    cache = KVCache(hq, hkv, bits, batch * mbps, batch, mbps, codes=codes)
    f = O.bf16_bits_to_f32
    ora = O.OracleCache(batch, hq, hkv, bits, codes=codes)
    if ctx:
        k0 = _bits(rng, (batch, hkv, ctx, 128))
        v0 = _bits(rng, (batch, hkv, ctx, 128))
        if ctx < 4 or ctx > 4096:  # a long context by appends (the oracle's prefill would take minutes)
            cache.quantize_append(T.to_dev_bf16(k0), T.to_dev_bf16(v0))
            for b in range(batch):
                ora.append(b, f(k0[b]), f(v0[b]))
        else:
            q0 = _bits(rng, (batch, hq, ctx, 128))
            cache.prefill(T.to_dev_bf16(q0), T.to_dev_bf16(k0), T.to_dev_bf16(v0))
            for b in range(batch):
                ora.prefill(b, f(q0[b]), f(k0[b]), f(v0[b]), T.sm_scale())
    if window:
        mask = cache.h2o_select_evict(batch, mode="streaming", window=window)
        cache.compact_blocks(mask, batch)
        for b in range(batch):
            ora.evict(b, ora.keep_masks(b, "streaming", window=window))
    q1 = _bits(rng, (batch, hq, n1, 128))
    k1 = _bits(rng, (batch, hkv, n1, 128))
    v1 = _bits(rng, (batch, hkv, n1, 128))
    out = T.bf16_tensor_to_f32(cache.prefill_context(T.to_dev_bf16(q1), T.to_dev_bf16(k1), T.to_dev_bf16(v1)))
    append_launches = 2 if n1 >= 64 else 1
    assert cache.last_launch_count() == append_launches + 2
    st = T.StateView(cache)
    for b in range(batch):
        ref = ora.prefill_chunk(b, f(q1[b]), f(k1[b]), f(v1[b]), T.sm_scale())
        T.assert_attention_close(out[b].reshape(hq * n1, 128), ref.reshape(hq * n1, 128), f"b={b}")
        s = ora.seqs[b]
        assert cache.lengths(b) == (s.heads[0].pos.shape[0], s.pos_total)
        assert int(st.slots[b]) == s.heads[0].pos.shape[0] and int(st.seen[b]) == s.pos_total
        for h in range(hkv):
            T.check_codes(st, ora, b, h)
            ns = s.sink_k[h].shape[0]
            np.testing.assert_allclose(st.sink_score[b, h, :ns], s.sink_score[h], rtol=1e-3, atol=1e-5)
            pos, *_, score = st.head(b, h)
            hs = s.heads[h]
            np.testing.assert_allclose(score[np.argsort(pos)], hs.score[np.argsort(hs.pos)], rtol=1e-3, atol=1e-5)
    assert cache.read_status() == 0


def test_prefill_context_then_decode_step():
    """A decode step after the second turn's prompt evicts by the scores of
    both turns and its own: the kept sets are the oracle's."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(62)
    hq, hkv, batch, n0, n1, budget, recent = 16, 4, 2, 150, 30, 100, 24
    mbps = (n0 + n1 + 1 + 15) // 16 + 2
    cache = KVCache(hq, hkv, 8, batch * mbps, batch, mbps)
    f = O.bf16_bits_to_f32
    q0, k0, v0 = (_bits(rng, (batch, x, n0, 128)) for x in (hq, hkv, hkv))
    q1, k1, v1 = (_bits(rng, (batch, x, n1, 128)) for x in (hq, hkv, hkv))
    qn = _bits(rng, (batch, hq, 128))
    kn, vn = (_bits(rng, (batch, hkv, 1, 128)) for _ in range(2))
    cache.prefill(T.to_dev_bf16(q0), T.to_dev_bf16(k0), T.to_dev_bf16(v0))
    cache.prefill_context(T.to_dev_bf16(q1), T.to_dev_bf16(k1), T.to_dev_bf16(v1))
    out = T.bf16_tensor_to_f32(cache.decode_step(T.to_dev_bf16(qn), T.to_dev_bf16(kn), T.to_dev_bf16(vn),
                                                 mode="h2o", budget=budget, recent=recent))
    st = T.StateView(cache)
    for b in range(batch):
        ora = O.OracleCache(1, hq, hkv, 8)
        ora.prefill(0, f(q0[b]), f(k0[b]), f(v0[b]), T.sm_scale())
        ora.prefill_chunk(0, f(q1[b]), f(k1[b]), f(v1[b]), T.sm_scale())
        ora.append(0, f(kn[b]), f(vn[b]))
        T.assert_attention_close(out[b], ora.attend(0, f(qn[b]), T.sm_scale()), f"b={b}")
        masks = ora.keep_masks(0, "h2o", budget=budget, recent=recent)
        for h in range(hkv):
            hs = ora.seqs[0].heads[h]
            kept = set(st.head(b, h)[0].tolist())
            assert T.kept_sets_agree(kept, set(hs.pos[masks[h]].tolist()), hs.pos, hs.score,
                                     budget - 4 - recent, n0 + n1 + 1 - recent), (b, h)
    assert cache.read_status() == 0


WINDOW_CASES = [
    # bits, codes, hq, hkv, batch, context, n1, bf16 window W
    (8, "int", 16, 4, 2, 100, 30, 32),    # a prompt shorter than the window: older window tokens age into the pool
    (4, "int", 40, 8, 1, 200, 80, 48),    # a prompt longer than the window: its own first tokens age out too
    (8, "e4m3", 8, 2, 1, 10, 40, 64),     # the window holds the whole context and prompt: an empty pool
    (4, "int", 8, 2, 2, 0, 50, 16),       # an empty sequence
    (8, "int", 16, 2, 1, 300, 200, 96),   # several window tiles, 400 attention rows per KV head
]


@pytest.mark.parametrize("bits,codes,hq,hkv,batch,ctx,n1,W", WINDOW_CASES)
def test_prefill_context_with_bf16_window(bits, codes, hq, hkv, batch, ctx, n1, W):
    """Hybrid precision: the last W positions stay bf16 (exact), older tokens
    are quantised; each prompt query attends to the sinks, the pool and the
    window tokens at positions up to its own.  Outputs, the pool and window
    contents and every held token's score against the oracle."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits + hq + ctx + n1 + W)
    mbps = (ctx + n1 + 15) // 16 + 2
    cache = KVCache(hq, hkv, bits, batch * mbps, batch, mbps, bf16_window=W, codes=codes)
    f = O.bf16_bits_to_f32
    ora = O.OracleCache(batch, hq, hkv, bits, bf16_window=W, codes=codes)
    if ctx:
        q0 = _bits(rng, (batch, hq, ctx, 128))
        k0 = _bits(rng, (batch, hkv, ctx, 128))
        v0 = _bits(rng, (batch, hkv, ctx, 128))
        cache.prefill(T.to_dev_bf16(q0), T.to_dev_bf16(k0), T.to_dev_bf16(v0))
        for b in range(batch):
            ora.prefill(b, f(q0[b]), f(k0[b]), f(v0[b]), T.sm_scale())
    q1 = _bits(rng, (batch, hq, n1, 128))
    k1 = _bits(rng, (batch, hkv, n1, 128))
    v1 = _bits(rng, (batch, hkv, n1, 128))
    out = T.bf16_tensor_to_f32(cache.prefill_context(T.to_dev_bf16(q1), T.to_dev_bf16(k1), T.to_dev_bf16(v1)))
    st = T.StateView(cache)
    for b in range(batch):
        ref = ora.prefill_chunk(b, f(q1[b]), f(k1[b]), f(v1[b]), T.sm_scale())
        T.assert_attention_close(out[b].reshape(hq * n1, 128), ref.reshape(hq * n1, 128), f"b={b}")
        s = ora.seqs[b]
        P = s.pos_total
        assert int(st.seen[b]) == P
        for h in range(hkv):
            hs = s.heads[h]
            old = hs.pos < P - W
            pos, kc, ks, vc, vs, sc = st.head(b, h)
            o, oo = np.argsort(pos), np.argsort(hs.pos[old])
            assert np.array_equal(pos[o], hs.pos[old][oo]), (b, h)
            assert np.array_equal(kc[o], hs.kcodes[old][oo]) and np.array_equal(vc[o], hs.vcodes[old][oo]), (b, h)
            np.testing.assert_allclose(sc[o], hs.score[old][oo], rtol=1e-3, atol=1e-5)
            rpos, rk, rv, rsc = st.ring_head(b, h)
            assert np.array_equal(rpos, np.sort(hs.pos[~old])), (b, h)
            assert np.array_equal(f(rk), s.raw_k[h][rpos]) and np.array_equal(f(rv), s.raw_v[h][rpos])
            by_pos = dict(zip(hs.pos.tolist(), hs.score.tolist()))
            np.testing.assert_allclose(rsc, [by_pos[p] for p in rpos.tolist()], rtol=1e-3, atol=1e-5)
            ns = s.sink_k[h].shape[0]
            np.testing.assert_allclose(st.sink_score[b, h, :ns], s.sink_score[h], rtol=1e-3, atol=1e-5)
    assert cache.read_status() == 0
