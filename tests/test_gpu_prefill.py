"""Prefill of fresh sequences: the causal attention of the prompt over its
bf16 K/V and the H2O scores it gives every prompt token (column sums of the
attention matrix over all queries and the query heads of the KV head),
against the oracle's prefill_attention; then a decode step whose H2O
selection uses those scores, against the oracle's rule."""
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
    # bits, hq, hkv, batch, n, W
    (8, 8, 2, 2, 100, 0),
    (4, 40, 8, 1, 300, 0),     # G = 5, several query and key tiles, a ragged last tile
    (8, 16, 4, 3, 64, 0),      # exactly one tile
    (8, 8, 8, 2, 3, 0),        # sinks only
    (8, 32, 8, 1, 257, 0),
    (4, 16, 4, 2, 150, 50),    # with a bf16 window: the last 50 tokens in the ring
    (8, 64, 8, 1, 130, 0),     # the largest query group (G = 8)
    (4, 8, 1, 2, 1, 0),        # a one-token prompt, one KV head
    # long prompts: dozens of key tiles per query block, the K/V ring wrapping
    # many times, blocks of every length, the lazy maximum over many tiles
    (4, 10, 2, 1, 4100, 0),    # GQA 5, a ragged last block and tile
    (8, 4, 4, 1, 4096, 0),     # G = 1, whole blocks
    (8, 8, 2, 1, 2050, 300),   # with a bf16 window
]


@pytest.mark.parametrize("bits,hq,hkv,batch,n,W", CASES)
def test_prefill_against_oracle(bits, hq, hkv, batch, n, W):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits + hq + n + W)
    mbps = (n + 15) // 16 + 1
    cache = KVCache(hq, hkv, bits, batch * mbps, batch, mbps, bf16_window=W)
    q = _bits(rng, (batch, hq, n, 128))
    k = _bits(rng, (batch, hkv, n, 128))
    v = _bits(rng, (batch, hkv, n, 128))
    out = cache.prefill(T.to_dev_bf16(q), T.to_dev_bf16(k), T.to_dev_bf16(v))
    assert cache.last_launch_count() == (4 if n >= 64 else 3)  # append (1 or 2), attention, scores
    gpu = T.bf16_tensor_to_f32(out)
    st = T.StateView(cache)
    f = O.bf16_bits_to_f32
    for b in range(batch):
        ref, sc = O.prefill_attention(f(q[b]), f(k[b]), f(v[b]), T.sm_scale())
        T.assert_attention_close(gpu[b].reshape(hq * n, 128), ref.reshape(hq * n, 128), f"prefill b={b}")
        assert cache.lengths(b) == (max(0, n - 4 - W) if W else max(0, n - 4), n)
        for h in range(hkv):
            ns = min(n, 4)
            np.testing.assert_allclose(st.sink_score[b, h, :ns], sc[h, :ns], rtol=1e-3, atol=1e-5)
            pos, *_, score = st.head(b, h)
            np.testing.assert_allclose(score, sc[h, pos], rtol=1e-3, atol=1e-5)
            if W:
                rpos, _, _, rsc = st.ring_head(b, h)
                np.testing.assert_allclose(rsc, sc[h, rpos], rtol=1e-3, atol=1e-5)
            # a KV head's scores add up to G * n
            tot = st.sink_score[b, h, :ns].sum() + score.sum() + (st.ring_head(b, h)[3].sum() if W else 0.0)
            np.testing.assert_allclose(tot, hq // hkv * n, rtol=1e-4)
    assert cache.read_status() == 0


def test_prefill_then_h2o_step_against_oracle():
    """The first decode step after the prompt evicts by the prompt's scores
    plus its own: the kept set is the oracle's."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(60)
    hq, hkv, batch, n, budget, recent = 16, 4, 2, 400, 120, 32
    mbps = (n + 1 + 15) // 16 + 1
    cache = KVCache(hq, hkv, 8, batch * mbps, batch, mbps)
    q = _bits(rng, (batch, hq, n, 128))
    k = _bits(rng, (batch, hkv, n, 128))
    v = _bits(rng, (batch, hkv, n, 128))
    qn = _bits(rng, (batch, hq, 128))
    kn = _bits(rng, (batch, hkv, 1, 128))
    vn = _bits(rng, (batch, hkv, 1, 128))
    cache.prefill(T.to_dev_bf16(q), T.to_dev_bf16(k), T.to_dev_bf16(v))
    out = T.bf16_tensor_to_f32(cache.decode_step(T.to_dev_bf16(qn), T.to_dev_bf16(kn), T.to_dev_bf16(vn),
                                                 mode="h2o", budget=budget, recent=recent))
    st = T.StateView(cache)
    f = O.bf16_bits_to_f32
    for b in range(batch):
        ora = O.OracleCache(1, hq, hkv, 8)
        ora.prefill(0, f(q[b]), f(k[b]), f(v[b]), T.sm_scale())
        ora.append(0, f(kn[b]), f(vn[b]))
        T.assert_attention_close(out[b], ora.attend(0, f(qn[b]), T.sm_scale()), f"b={b}")
        masks = ora.keep_masks(0, "h2o", budget=budget, recent=recent)
        for h in range(hkv):
            hs = ora.seqs[0].heads[h]
            kept = set(st.head(b, h)[0].tolist())
            assert T.kept_sets_agree(kept, set(hs.pos[masks[h]].tolist()), hs.pos, hs.score,
                                     budget - 4 - recent, n + 1 - recent), (b, h)
    assert cache.read_status() == 0


def test_prefill_errors():
    from compressed_kv_cache_kvc_gb300 import _lib as L
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(61)
    cache = KVCache(8, 2, 8, 16, 2, 8)
    q = T.to_dev_bf16(_bits(rng, (1, 8, 20, 128)))
    k = T.to_dev_bf16(_bits(rng, (1, 2, 20, 128)))
    cache.prefill(q, k, k)
    with pytest.raises(L.KvcError) as e:
        cache.prefill(q, k, k)  # the sequence is no longer empty
    assert e.value.status == L.KVC_ERR_STATE
    cache.prefill(q, k, k, seq_begin=1, accumulate_h2o=False)
    assert cache.last_launch_count() == 2
    assert cache.read_status() == 0


PREFILL_RANGE = 0x80


def test_prefill_value_range():
    """The prompt's P.V product takes V in fp16.  V up to 65280 in magnitude
    (the largest bf16 below fp16's overflow) converts without saturation: no
    status bit, and the error stays within fp16 rounding of P and V (2^-11
    each) on the sum of p |v|, plus the bf16 output's own rounding.  One
    entry of 70000 saturates to 65504: the prompt's status bit is set and
    every output stays finite."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    from compressed_kv_cache_kvc_gb300.workloads import bf16_bits
    rng = np.random.default_rng(62)
    hq, hkv, n = 8, 2, 200
    f = O.bf16_bits_to_f32
    q = _bits(rng, (1, hq, n, 128))
    k = _bits(rng, (1, hkv, n, 128))
    vf = rng.standard_normal((1, hkv, n, 128)).astype(np.float32) * 1000.0
    vf[0, 0, rng.integers(0, n, 40), rng.integers(0, 128, 40)] = 65280.0
    vf[0, 1, rng.integers(0, n, 40), rng.integers(0, 128, 40)] = -65280.0
    v = bf16_bits(vf)
    assert np.abs(f(v)).max() == 65280.0
    cache = KVCache(hq, hkv, 8, 2 * 15, 2, 15)
    out = T.bf16_tensor_to_f32(cache.prefill(T.to_dev_bf16(q), T.to_dev_bf16(k), T.to_dev_bf16(v)))
    assert cache.read_status() == 0
    ref, _ = O.prefill_attention(f(q[0]), f(k[0]), f(v[0]), T.sm_scale())
    mag, _ = O.prefill_attention(f(q[0]), f(k[0]), np.abs(f(v[0])), T.sm_scale())
    err = np.abs(out[0].astype(np.float64) - ref)
    bound = 2e-3 + 2.0 ** -8 * np.abs(ref) + 2.0 * 2.0 ** -11 * mag
    assert (err <= bound).all(), float((err / bound).max())

    vf[0, 1, 7, 3] = 70000.0
    v2 = bf16_bits(vf)
    out2 = T.bf16_tensor_to_f32(cache.prefill(T.to_dev_bf16(q), T.to_dev_bf16(k), T.to_dev_bf16(v2), seq_begin=1))
    assert cache.read_status() & PREFILL_RANGE
    assert np.isfinite(out2).all()
