"""kvc_decode_step (one call per layer: append, split attention, the fused
merge/score/select/list kernel, the move kernel) must
leave exactly the device state and outputs that the four separate calls leave,
step after step; plus one direct check against the oracle."""
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


def _same_state(a, b):
    """Same logical cache: per (sequence, KV head) the slots in slot order
    (positions, codes, scales, scores), the sinks and their scores, the
    lengths and the number of free blocks.  Physical block ids may differ:
    the two paths push released blocks in different orders."""
    sa, sb = T.StateView(a), T.StateView(b)
    assert np.array_equal(sa.slots, sb.slots) and np.array_equal(sa.seen, sb.seen)
    for seq in range(a.max_batch):
        for h in range(a.num_kv_heads):
            for x, y in zip(sa.head(seq, h), sb.head(seq, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (seq, h)
    assert np.array_equal(sa.sink_k, sb.sink_k) and np.array_equal(sa.sink_v, sb.sink_v)
    assert np.array_equal(sa.sink_score.view(np.uint32), sb.sink_score.view(np.uint32))
    assert np.array_equal(sa.counters[:3], sb.counters[:3])  # free-stack top, status, ticket


CASES = [
    # bits, hq, hkv, lengths, mode, budget, recent, window, steps
    (8, 8, 8, [512], "h2o", 128, 32, 0, 4),
    (4, 40, 8, [600, 433, 70], "h2o", 180, 40, 0, 3),
    (8, 32, 8, [700, 100, 257, 260], "streaming", 0, 0, 256, 3),
    (8, 8, 2, [150], "h2o", 4 + 160, 8, 0, 2),        # budget covers the context: nothing evicted
    (4, 4, 2, [90], "h2o", 4, 0, 0, 2),               # only the sinks are kept
    (8, 16, 4, [1000, 1000], "h2o", 300, 64, 0, 2),
    (8, 8, 2, [21000, 300], "h2o", 2100, 256, 0, 2),  # keys in shared memory, positions in the workspace
    (4, 8, 2, [41000], "h2o", 4100, 512, 0, 2),       # keys and positions in the workspace
]


@pytest.mark.parametrize("bits,hq,hkv,lengths,mode,budget,recent,window,steps", CASES)
def test_step_equals_separate_calls(bits, hq, hkv, lengths, mode, budget, recent, window, steps):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits * 7 + hq + len(lengths))
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + steps + 15) // 16 + 2
    order = np.random.default_rng(1).permutation(B * mbps).astype(np.int32)
    ca = KVCache(hq, hkv, bits, B * mbps, B, mbps, block_order=order)
    cb = KVCache(hq, hkv, bits, B * mbps, B, mbps, block_order=order)
    k = _bits(rng, (B, hkv, T_, 128))
    v = _bits(rng, (B, hkv, T_, 128))
    for c in (ca, cb):
        for b, n in enumerate(lengths):
            c.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :n])), seq_begin=b)
    _same_state(ca, cb)
    for _ in range(steps):
        q = T.to_dev_bf16(_bits(rng, (B, hq, 128)))
        kn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
        vn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
        oa = ca.step(q, kn, vn, mode=mode, budget=budget, recent=recent, window=window)
        ob = cb.decode_step(q, kn, vn, mode=mode, budget=budget, recent=recent, window=window)
        assert cb.last_launch_count() in (3, 4)  # the move kernel only when a pair moves > 32 rows
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
        _same_state(ca, cb)
        for b in range(B):
            assert ca.lengths(b) == cb.lengths(b)
    assert ca.read_status() == 0 and cb.read_status() == 0


BLOCK_CASES = [
    # bits, hq, hkv, lengths, recent, retention, steps
    (8, 16, 4, [600, 333], 40, 0.5, 3),
    (4, 40, 8, [1000, 257, 64], 64, 0.3, 3),
    (8, 8, 2, [9000, 70], 100, 0.6, 2),
    (4, 8, 8, [200], 0, 1.0, 2),  # keep everything
]


@pytest.mark.parametrize("bits,hq,hkv,lengths,recent,retention,steps", BLOCK_CASES)
def test_block_step_equals_separate_calls(bits, hq, hkv, lengths, recent, retention, steps):
    """Block-granular eviction through the one-call step (five launches):
    the same outputs and logical state as the separate calls."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits * 5 + hq + len(lengths))
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + steps + 15) // 16 + 2
    order = np.random.default_rng(3).permutation(B * mbps).astype(np.int32)
    ca = KVCache(hq, hkv, bits, B * mbps, B, mbps, block_order=order)
    cb = KVCache(hq, hkv, bits, B * mbps, B, mbps, block_order=order)
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
        oa = ca.step(q, kn, vn, mode="block", recent=recent, retention=retention)
        ob = cb.decode_step(q, kn, vn, mode="block", recent=recent, retention=retention)
        assert cb.last_launch_count() == 5
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
        _same_state(ca, cb)
        for b in range(B):
            assert ca.lengths(b) == cb.lengths(b)
    assert ca.read_status() == 0 and cb.read_status() == 0


def test_step_against_oracle_tiny_workload():
    from compressed_kv_cache_kvc_gb300 import workloads as W
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    w = W.WORKLOADS["tiny_b1_h8_t512_int8_h2o"]
    d = W.gen_layer(w, 0)
    mbps = (w.context + 16) // 16 + 1
    c = KVCache(w.num_q_heads, w.num_kv_heads, w.bits, mbps, 1, mbps)
    c.quantize_append(T.to_dev_bf16(d["k"]), T.to_dev_bf16(d["v"]))
    out = c.decode_step(T.to_dev_bf16(d["q"]), T.to_dev_bf16(d["k_new"]), T.to_dev_bf16(d["v_new"]),
                        mode="h2o", budget=w.budget, recent=w.recent)
    ora = O.OracleCache(1, w.num_q_heads, w.num_kv_heads, w.bits)
    f = O.bf16_bits_to_f32
    ora.append(0, f(d["k"][0]), f(d["v"][0]))
    ora.append(0, f(d["k_new"][0]), f(d["v_new"][0]))
    ref = ora.attend(0, f(d["q"][0]), T.sm_scale())
    T.assert_attention_close(T.bf16_tensor_to_f32(out)[0], ref, "decode_step")
    masks = ora.keep_masks(0, "h2o", budget=w.budget, recent=w.recent)
    st = T.StateView(c)
    for h in range(w.num_kv_heads):
        hs = ora.seqs[0].heads[h]
        kept_ora = set(hs.pos[masks[h]].tolist())
        kept_gpu = set(st.head(0, h)[0].tolist())
        assert T.kept_sets_agree(kept_gpu, kept_ora, hs.pos, hs.score, w.budget - 4 - w.recent,
                                 w.context + 1 - w.recent)
    assert c.lengths(0) == (w.budget - 4, w.context + 1)


@pytest.mark.parametrize("bits,hq,hkv", [(8, 16, 4), (4, 40, 8)])
def test_step_on_batch_slices(bits, hq, hkv):
    """Slices of the batch (seq_begin > 0, batch < max_batch) step exactly as
    the separate calls on the same slices do, and leave the other sequences
    untouched."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits + hq)
    lengths = [300, 530, 47, 1000, 260]
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + 16 + 15) // 16 + 2
    ca = KVCache(hq, hkv, bits, B * mbps, B, mbps)
    cb = KVCache(hq, hkv, bits, B * mbps, B, mbps)
    k = _bits(rng, (B, hkv, T_, 128))
    v = _bits(rng, (B, hkv, T_, 128))
    for c in (ca, cb):
        for b, n in enumerate(lengths):
            c.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :n])), seq_begin=b)
    for seq_begin, batch in [(1, 3), (0, 2), (3, 2)]:
        before = T.StateView(cb)
        q = T.to_dev_bf16(_bits(rng, (batch, hq, 128)))
        kn = T.to_dev_bf16(_bits(rng, (batch, hkv, 1, 128)))
        vn = T.to_dev_bf16(_bits(rng, (batch, hkv, 1, 128)))
        oa = ca.step(q, kn, vn, mode="h2o", budget=200, recent=32, seq_begin=seq_begin)
        ob = cb.decode_step(q, kn, vn, mode="h2o", budget=200, recent=32, seq_begin=seq_begin)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
        _same_state(ca, cb)
        after = T.StateView(cb)
        for b in list(range(seq_begin)) + list(range(seq_begin + batch, B)):
            assert after.slots[b] == before.slots[b] and after.seen[b] == before.seen[b]
            for h in range(hkv):
                for x, y in zip(before.head(b, h), after.head(b, h)):
                    assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (b, h)
    assert ca.read_status() == 0 and cb.read_status() == 0


def test_step_with_pyramid_budgets():
    """Per-layer budgets (the linear PyramidKV schedule) through the one-call
    step: every layer keeps exactly its budget, the kept set the oracle's rule
    gives for that budget."""
    from compressed_kv_cache_kvc_gb300.budgets import pyramid_budgets
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(5)
    L, B, hq, hkv, T_, recent = 4, 2, 16, 4, 600, 32
    budgets = pyramid_budgets(L, "linear", recent=recent, base=300)
    assert budgets == [300, 240, 180, 119]  # 300 * (1 - 0.8 * 3/4) = 119.99999999999997 in floating point
    mbps = (T_ + 1 + 15) // 16 + 2
    f = O.bf16_bits_to_f32
    for budget in budgets:
        c = KVCache(hq, hkv, 8, B * mbps, B, mbps)
        k = _bits(rng, (B, hkv, T_, 128))
        v = _bits(rng, (B, hkv, T_, 128))
        q = _bits(rng, (B, hq, 128))
        kn = _bits(rng, (B, hkv, 1, 128))
        vn = _bits(rng, (B, hkv, 1, 128))
        c.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(v))
        out = c.decode_step(T.to_dev_bf16(q), T.to_dev_bf16(kn), T.to_dev_bf16(vn), mode="h2o", budget=budget,
                            recent=recent)
        gpu = T.bf16_tensor_to_f32(out)
        st = T.StateView(c)
        for b in range(B):
            ora = O.OracleCache(1, hq, hkv, 8)
            ora.append(0, f(k[b]), f(v[b]))
            ora.append(0, f(kn[b]), f(vn[b]))
            ref = ora.attend(0, f(q[b]), T.sm_scale())
            T.assert_attention_close(gpu[b], ref, f"budget {budget} b={b}")
            masks = ora.keep_masks(0, "h2o", budget=budget, recent=recent)
            for h in range(hkv):
                hs = ora.seqs[0].heads[h]
                kept_gpu = set(st.head(b, h)[0].tolist())
                assert len(kept_gpu) == budget - 4
                assert T.kept_sets_agree(kept_gpu, set(hs.pos[masks[h]].tolist()), hs.pos, hs.score,
                                         budget - 4 - recent, T_ + 1 - recent), (budget, b, h)
            assert c.lengths(b) == (budget - 4, T_ + 1)
        assert c.read_status() == 0


@pytest.mark.parametrize("bits,hq,hkv", [(8, 64, 8), (4, 64, 8), (8, 8, 1), (4, 12, 4), (8, 42, 7), (8, 14, 2)])
def test_step_head_layouts_against_oracle(bits, hq, hkv):
    """The one-call step at the largest query group (G = 8: every MMA column
    used), multi-query attention (one KV head) and odd groups (G = 3, 6, 7):
    outputs within tolerance and kept sets the oracle's rule."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits * 100 + hq * 10 + hkv)
    B, n, budget, recent = 2, 300, 100, 24
    lengths = [300, 137]
    mbps = (n + 1 + 15) // 16 + 2
    cache = KVCache(hq, hkv, bits, B * mbps, B, mbps)
    k = _bits(rng, (B, hkv, n, 128))
    v = _bits(rng, (B, hkv, n, 128))
    for b, nb in enumerate(lengths):
        cache.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :nb])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :nb])), seq_begin=b)
    q = _bits(rng, (B, hq, 128))
    kn = _bits(rng, (B, hkv, 1, 128))
    vn = _bits(rng, (B, hkv, 1, 128))
    out = T.bf16_tensor_to_f32(cache.decode_step(T.to_dev_bf16(q), T.to_dev_bf16(kn), T.to_dev_bf16(vn),
                                                 mode="h2o", budget=budget, recent=recent))
    st = T.StateView(cache)
    f = O.bf16_bits_to_f32
    for b, nb in enumerate(lengths):
        ora = O.OracleCache(1, hq, hkv, bits)
        ora.append(0, f(k[b, :, :nb]), f(v[b, :, :nb]))
        ora.append(0, f(kn[b]), f(vn[b]))
        T.assert_attention_close(out[b], ora.attend(0, f(q[b]), T.sm_scale()), f"G={hq // hkv} b={b}")
        masks = ora.keep_masks(0, "h2o", budget=budget, recent=recent)
        for h in range(hkv):
            hs = ora.seqs[0].heads[h]
            assert T.kept_sets_agree(set(st.head(b, h)[0].tolist()), set(hs.pos[masks[h]].tolist()), hs.pos,
                                     hs.score, budget - 4 - recent, nb + 1 - recent), (b, h)
    assert cache.read_status() == 0


def test_checkpoint_to_host_and_resume_in_another_arena():
    """Checkpoint/resume: after a few steps the state arena is copied to host
    memory and restored into a second cache of the same geometry (another
    device allocation), whose host mirror is then reloaded
    (kvc_cache_sync_host).  The state holds block ids, never addresses, so
    the next steps give the same outputs and the same logical state in both
    caches."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(77)
    hq, hkv, bits, lengths, budget, recent = 16, 4, 4, [300, 170], 120, 24
    B = len(lengths)
    mbps = (max(lengths) + 4 + 15) // 16 + 2
    ca = KVCache(hq, hkv, bits, B * mbps, B, mbps)
    k = _bits(rng, (B, hkv, max(lengths), 128))
    v = _bits(rng, (B, hkv, max(lengths), 128))
    for b, n in enumerate(lengths):
        ca.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                           T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :n])), seq_begin=b)

    def inputs():
        return (T.to_dev_bf16(_bits(rng, (B, hq, 128))), T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128))),
                T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128))))

    for _ in range(2):
        ca.decode_step(*inputs(), mode="h2o", budget=budget, recent=recent)
    torch.cuda.synchronize()
    checkpoint = ca.state_view.cpu()
    cb = KVCache(hq, hkv, bits, B * mbps, B, mbps)
    assert cb.state_view.data_ptr() != ca.state_view.data_ptr()
    cb.state_view.copy_(checkpoint.to(cb.device))
    cb.sync_host()
    for b in range(B):
        assert cb.lengths(b) == ca.lengths(b)
    for _ in range(2):
        q, kn, vn = inputs()
        oa = ca.decode_step(q, kn, vn, mode="h2o", budget=budget, recent=recent)
        ob = cb.decode_step(q, kn, vn, mode="h2o", budget=budget, recent=recent)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
        _same_state(ca, cb)
    assert ca.read_status() == 0 and cb.read_status() == 0


@pytest.mark.parametrize("length,budget,first_launches", [(600, 180, 4), (200, 190, 3)])
def test_step_moves_inline_or_in_their_own_kernel(length, budget, first_launches):
    """Pairs that move at most 32 rows have them moved by the post kernel (no
    move kernel: 3 launches), more take the move kernel (4 launches); either
    way the outputs and the cache equal those of the separate calls, step
    after step (the second step evicts one token: inline)."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(length + budget)
    hq, hkv, B = 16, 4, 2
    mbps = (length + 3 + 15) // 16 + 2
    ca = KVCache(hq, hkv, 8, B * mbps, B, mbps)
    cb = KVCache(hq, hkv, 8, B * mbps, B, mbps)
    k = _bits(rng, (B, hkv, length, 128))
    v = _bits(rng, (B, hkv, length, 128))
    for c in (ca, cb):
        c.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(v))
    for step in range(3):
        q = T.to_dev_bf16(_bits(rng, (B, hq, 128)))
        kn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
        vn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
        oa = ca.step(q, kn, vn, mode="h2o", budget=budget, recent=24)
        ob = cb.decode_step(q, kn, vn, mode="h2o", budget=budget, recent=24)
        assert cb.last_launch_count() == (first_launches if step == 0 else 3)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
        _same_state(ca, cb)
    assert ca.read_status() == 0 and cb.read_status() == 0
