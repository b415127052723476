"""Block-granular eviction (KVC_EVICT_BLOCK): whole pages by mean H2O score,
dropped from the block table without moving anything in the pool.  The keep
mask must equal the oracle's rule (select_blocks) applied to the GPU's own
accumulated scores, bit for bit; after the compaction every head holds
exactly its pre-eviction slots minus the evicted pages, in the same order."""
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
    # bits, hq, hkv, lengths, recent, retention, steps
    (8, 16, 4, [600, 333], 40, 0.5, 3),
    (4, 40, 8, [1000, 257, 64], 64, 0.3, 2),
    (8, 32, 8, [700, 1300], 128, 0.05, 2),
    (8, 8, 8, [200], 0, 1.0, 2),      # keep everything
    (8, 8, 2, [300], 400, 0.2, 2),    # the recent window covers the pool: no candidate
    (8, 8, 2, [9000, 4100], 100, 0.4, 2),  # more pages than the selection CTA has threads
]


@pytest.mark.parametrize("bits,hq,hkv,lengths,recent,retention,steps", CASES)
def test_block_eviction(bits, hq, hkv, lengths, recent, retention, steps):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits * 3 + hq + len(lengths))
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + steps + 15) // 16 + 2
    nb = B * mbps
    cache = KVCache(hq, hkv, bits, nb, B, mbps, block_order=np.random.default_rng(2).permutation(nb).astype(np.int32))
    k = _bits(rng, (B, hkv, T_, 128))
    v = _bits(rng, (B, hkv, T_, 128))
    for b, n in enumerate(lengths):
        cache.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :n])), seq_begin=b)
    evicted_any = False
    for step in range(steps):
        cache.quantize_append(T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128))), T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128))))
        cache.decode_attention(T.to_dev_bf16(_bits(rng, (B, hq, 128))), accumulate_h2o=True)
        pre = T.StateView(cache)
        mask = cache.h2o_select_evict(B, mode="block", recent=recent, retention=retention)
        assert cache.last_launch_count() == 2  # page sums, then the selection
        mask_h = mask.cpu().numpy()
        cache.compact_blocks(mask, B)
        assert cache.last_launch_count() == 1
        post = T.StateView(cache)
        for b in range(B):
            S = int(pre.slots[b])
            heads = [pre.head(b, h) for h in range(hkv)]
            want = O.select_blocks([hd[5].astype(np.float64) for hd in heads], S, recent, retention)
            evicted_any |= not want.all()
            for h in range(hkv):
                assert np.array_equal(mask_h[b, h, :S] == 1, want), (step, b, h)
                for x, y in zip(heads[h], post.head(b, h)):
                    assert np.array_equal(np.asarray(x)[want], np.asarray(y)), (step, b, h)
            assert int(post.slots[b]) == int(want.sum())
            assert int(post.seen[b]) == int(pre.seen[b])
        used = np.concatenate([post.used_blocks(b) for b in range(B)])
        free = post.free_stack[:int(post.counters[0])]
        allb = np.concatenate([used, free])
        assert allb.size == nb and np.unique(allb).size == nb
        assert cache.read_status() == 0
    if retention < 1.0 and recent < min(lengths) - 32:
        assert evicted_any


def test_block_eviction_ties_to_the_earlier_page():
    """With no attention run every score is 0, so every page sum ties: the
    earliest candidate pages go."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(11)
    hq, hkv, n, recent, retention = 8, 2, 900, 32, 0.35
    mbps = (n + 15) // 16 + 1
    cache = KVCache(hq, hkv, 8, mbps, 1, mbps)
    cache.quantize_append(T.to_dev_bf16(_bits(rng, (1, hkv, n, 128))), T.to_dev_bf16(_bits(rng, (1, hkv, n, 128))))
    S = cache.lengths(0)[0]
    mask = cache.h2o_select_evict(1, mode="block", recent=recent, retention=retention).cpu().numpy()
    n_cand = (S - recent) // 16
    n_evict = int(n_cand * (1.0 - retention))
    want = np.ones(S, dtype=bool)
    want[:16 * n_evict] = False
    assert np.array_equal(want, O.select_blocks([np.zeros(S)] * hkv, S, recent, retention))
    for h in range(hkv):
        assert np.array_equal(mask[0, h, :S] == 1, want)
    cache.compact_blocks(torch.from_numpy(mask).cuda(), 1)
    assert cache.lengths(0)[0] == S - 16 * n_evict
    assert cache.read_status() == 0


def test_block_sums_exact_on_planted_scores():
    """Scores planted directly in the pool: subnormals, zeros, tiny and huge
    normals side by side, so the fp64 page sums round at many steps.  The
    mask must still be the oracle's (its sums are exact conversions of the
    fp32 scores added in the same order)."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(21)
    hq, hkv, n, recent = 16, 4, 2000, 48
    mbps = (n + 15) // 16 + 1
    cache = KVCache(hq, hkv, 8, mbps, 1, mbps)
    cache.quantize_append(T.to_dev_bf16(_bits(rng, (1, hkv, n, 128))), T.to_dev_bf16(_bits(rng, (1, hkv, n, 128))))
    sc = cache.buffer("SCORE").view(torch.int32)
    kind = rng.integers(0, 5, sc.numel())
    bits = np.where(kind == 0, rng.integers(1, 1 << 23, sc.numel()),                  # subnormal
           np.where(kind == 1, 0,                                                     # zero
           np.where(kind == 2, rng.integers(1 << 23, 20 << 23, sc.numel()),           # tiny normal
           np.where(kind == 3, rng.integers(190 << 23, 230 << 23, sc.numel()),        # huge normal
                    rng.integers(100 << 23, 130 << 23, sc.numel())))))                # ordinary
    planted = bits.astype(np.int64).astype(np.int32)
    sc.copy_(torch.from_numpy(planted).to(sc.device))
    st = T.StateView(cache)
    S = int(st.slots[0])
    heads = [st.head(0, h)[5].astype(np.float64) for h in range(hkv)]
    for retention in (0.7, 0.2):
        mask = cache.h2o_select_evict(1, mode="block", recent=recent, retention=retention).cpu().numpy()
        want = O.select_blocks(heads, S, recent, retention)
        assert not want.all()
        for h in range(hkv):
            assert np.array_equal(mask[0, h, :S] == 1, want), (retention, h)
    assert cache.read_status() == 0
