"""Failure detection without a GPU fault: a corrupted block-table entry
(planted on the host through the state buffer) must be reported in the
device status word (KVC_DEV_BAD_BLOCK_ID) and skipped.  Every kernel checks
a block id before it touches the pool, and the compaction lists carry -1 for
a slot on a bad page, which the row mover rejects, so no access leaves the
pool; the other sequences' results are exactly those of an intact cache."""
import numpy as np
import pytest
import torch

from tests import kvc_testlib as T

pytestmark = pytest.mark.gpu

BAD_BLOCK_ID = 0x2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()


def _bits(rng, shape):
    from compressed_kv_cache_kvc_gb300.workloads import bf16_bits
    return bf16_bits(rng.standard_normal(shape).astype(np.float32))


def _pair(bits=8, hq=16, hkv=4, lengths=(500, 300, 200)):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(7)
    B, n = len(lengths), max(lengths)
    mbps = (n + 4 + 15) // 16 + 2
    caches = [KVCache(hq, hkv, bits, B * mbps, B, mbps) for _ in range(2)]
    k = _bits(rng, (B, hkv, n, 128))
    v = _bits(rng, (B, hkv, n, 128))
    for c in caches:
        for b, nb in enumerate(lengths):
            c.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :nb])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :nb])), seq_begin=b)
    torch.cuda.synchronize()
    q = T.to_dev_bf16(_bits(rng, (B, hq, 128)))
    kn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
    vn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
    return caches, mbps, q, kn, vn


@pytest.mark.parametrize("bad", ["past_the_pool", "negative"])
def test_bad_block_id_in_the_one_call_step(bad):
    (clean, corrupt), mbps, q, kn, vn = _pair()
    bt = corrupt.buffer("BLOCK_TABLE").view(torch.int32)
    bt[2] = corrupt.num_blocks + 7 if bad == "past_the_pool" else -1  # sequence 0, its third page
    torch.cuda.synchronize()
    oa = clean.decode_step(q, kn, vn, mode="h2o", budget=120, recent=16)
    ob = corrupt.decode_step(q, kn, vn, mode="h2o", budget=120, recent=16)
    torch.cuda.synchronize()
    assert clean.read_status() == 0
    assert corrupt.read_status() & BAD_BLOCK_ID
    assert corrupt.read_status() == 0  # read_status cleared the word
    assert torch.equal(oa[1:], ob[1:])  # the other sequences are untouched
    sa, sb = T.StateView(clean), T.StateView(corrupt)
    for b in (1, 2):
        for h in range(clean.num_kv_heads):
            for x, y in zip(sa.head(b, h), sb.head(b, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (b, h)


def test_bad_block_id_in_the_separate_calls():
    (clean, corrupt), mbps, q, kn, vn = _pair(bits=4, hq=40, hkv=8)
    bt = corrupt.buffer("BLOCK_TABLE").view(torch.int32)
    bt[5] = 1 << 30
    torch.cuda.synchronize()
    outs = []
    for c in (clean, corrupt):
        c.quantize_append(kn, vn)
        outs.append(c.decode_attention(q))
        mask = c.h2o_select_evict(q.shape[0], budget=150, recent=32)
        c.compact_blocks(mask, q.shape[0])
    torch.cuda.synchronize()
    assert clean.read_status() == 0
    assert corrupt.read_status() & BAD_BLOCK_ID
    assert torch.equal(outs[0][1:], outs[1][1:])


STALE_HOST = 0x20


def _close(a, b):
    a, b = a.float(), b.float()
    assert bool(((a - b).abs() <= 2e-3 + 1e-2 * a.abs()).all())


def test_state_restored_without_host_resync_is_flagged():
    """The host sizes the selection's shared key buffer from its mirror of the
    lengths.  Device state bytes restored from a snapshot without
    kvc_cache_sync_host leave the device longer than that mirror: the step and
    the separate selection must flag KVC_DEV_STALE_HOST and keep the slots
    (never write past the buffer); the attention itself reads the device
    lengths and is unaffected (up to the summation order: the stream-K grid
    follows the host's page count).  After a resync the step is exact again."""
    (c, _), mbps, q, kn, vn = _pair()
    snap = c.state_view.clone()
    o1 = c.decode_step(q, kn, vn, mode="h2o", budget=120, recent=16)
    torch.cuda.synchronize()
    assert c.read_status() == 0
    after = [c.lengths(b)[0] for b in range(q.shape[0])]
    assert max(after) < 200
    # restore without a resync: the host still plans for the evicted lengths
    c.state_view.copy_(snap)
    o2 = c.decode_step(q, kn, vn, mode="h2o", budget=120, recent=16)
    torch.cuda.synchronize()
    assert c.read_status() & STALE_HOST
    _close(o1, o2)
    # the separate selection call takes the same guard
    c.state_view.copy_(snap)
    c.quantize_append(kn, vn)
    o3 = c.decode_attention(q)
    c.h2o_select_evict(q.shape[0], budget=120, recent=16)
    torch.cuda.synchronize()
    assert c.read_status() & STALE_HOST
    _close(o1, o3)
    # resynchronised, the step is the first one again
    c.state_view.copy_(snap)
    c.sync_host()
    o4 = c.decode_step(q, kn, vn, mode="h2o", budget=120, recent=16)
    torch.cuda.synchronize()
    assert c.read_status() == 0
    assert torch.equal(o1, o4)
    assert [c.lengths(b)[0] for b in range(q.shape[0])] == after
