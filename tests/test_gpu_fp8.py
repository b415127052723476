"""FP8 E4M3 codes (codes = "e4m3", 8-bit): the quantised pool bit for bit
against the oracle's E4M3 quantiser, the attention and H2O selection against
the oracle, and the one-call step against the separate calls."""
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


def _bits_of(x):
    from compressed_kv_cache_kvc_gb300.workloads import bf16_bits
    return bf16_bits(np.asarray(x, np.float32))


def _bits(rng, shape):
    return _bits_of(rng.standard_normal(shape))


@pytest.mark.parametrize("hq,hkv,lengths,steps", [(8, 2, [300, 41], 3), (40, 8, [500], 2), (32, 8, [77, 200, 16], 2)])
def test_fp8_codes_and_attention_against_oracle(hq, hkv, lengths, steps):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(hq + len(lengths))
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + steps + 15) // 16 + 2
    cache = KVCache(hq, hkv, 8, B * mbps, B, mbps, codes="e4m3")
    ora = O.OracleCache(B, hq, hkv, 8, codes="e4m3")
    f = O.bf16_bits_to_f32
    # rows of very different magnitudes, a zero row, rows with one outlier
    mag = np.exp(rng.uniform(-20, 6, (B, hkv, T_, 1))).astype(np.float32)
    x = (rng.standard_normal((B, hkv, T_, 128)) * mag).astype(np.float32)
    x[:, :, 7] = 0.0
    x[:, :, 9, 5] = 300.0
    k = _bits_of(x)
    v = _bits(rng, (B, hkv, T_, 128))
    for b, n in enumerate(lengths):
        cache.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :n])), seq_begin=b)
        ora.append(b, f(k[b, :, :n]), f(v[b, :, :n]))
    st = T.StateView(cache)
    for b in range(B):
        for h in range(hkv):
            T.check_codes(st, ora, b, h)
    for _ in range(steps):
        kn = _bits(rng, (B, hkv, 1, 128))
        vn = _bits(rng, (B, hkv, 1, 128))
        q = _bits(rng, (B, hq, 128))
        cache.quantize_append(T.to_dev_bf16(kn), T.to_dev_bf16(vn))
        out = T.bf16_tensor_to_f32(cache.decode_attention(T.to_dev_bf16(q)))
        for b in range(B):
            ora.append(b, f(kn[b]), f(vn[b]))
            T.assert_attention_close(out[b], ora.attend(b, f(q[b]), T.sm_scale()), f"fp8 b={b}")
    st = T.StateView(cache)
    for b in range(B):
        for h in range(hkv):
            T.check_codes(st, ora, b, h)
    assert cache.read_status() == 0


def test_fp8_step_equals_separate_calls_and_oracle_selection():
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(80)
    hq, hkv, B, n, budget, recent = 16, 4, 2, 600, 200, 40
    mbps = (n + 3 + 15) // 16 + 2
    order = np.random.default_rng(5).permutation(B * mbps).astype(np.int32)
    ca = KVCache(hq, hkv, 8, B * mbps, B, mbps, block_order=order, codes="e4m3")
    cb = KVCache(hq, hkv, 8, B * mbps, B, mbps, block_order=order, codes="e4m3")
    k = _bits(rng, (B, hkv, n, 128))
    v = _bits(rng, (B, hkv, n, 128))
    for c in (ca, cb):
        c.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(v))
    f = O.bf16_bits_to_f32
    q = _bits(rng, (B, hq, 128))
    kn = _bits(rng, (B, hkv, 1, 128))
    vn = _bits(rng, (B, hkv, 1, 128))
    oa = ca.step(T.to_dev_bf16(q), T.to_dev_bf16(kn), T.to_dev_bf16(vn), mode="h2o", budget=budget, recent=recent)
    ob = cb.decode_step(T.to_dev_bf16(q), T.to_dev_bf16(kn), T.to_dev_bf16(vn), mode="h2o", budget=budget,
                        recent=recent)
    torch.cuda.synchronize()
    assert torch.equal(oa, ob)
    sa, sb = T.StateView(ca), T.StateView(cb)
    for b in range(B):
        for h in range(hkv):
            for x, y in zip(sa.head(b, h), sb.head(b, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (b, h)
        ora = O.OracleCache(1, hq, hkv, 8, codes="e4m3")
        ora.append(0, f(k[b]), f(v[b]))
        ora.append(0, f(kn[b]), f(vn[b]))
        T.assert_attention_close(T.bf16_tensor_to_f32(ob)[b], ora.attend(0, f(q[b]), T.sm_scale()), f"b={b}")
        masks = ora.keep_masks(0, "h2o", budget=budget, recent=recent)
        for h in range(hkv):
            hs = ora.seqs[0].heads[h]
            assert T.kept_sets_agree(set(sb.head(b, h)[0].tolist()), set(hs.pos[masks[h]].tolist()), hs.pos,
                                     hs.score, budget - 4 - recent, n + 1 - recent), (b, h)
    assert ca.read_status() == 0 and cb.read_status() == 0
