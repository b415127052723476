"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars (the output bar is elementwise because a 2e-3 max-abs bar alone is below
half a bf16 ulp for outputs in [1, 2)):
  * INT8/INT4 codes, fp32 scales, positions, bf16 sinks: bit-exact;
  * kept sets: identical when the oracle selects on the GPU's own scores;
    against the oracle's fp64 scores, different only within 1e-5 relative of
    the k-th score;
  * attention outputs (bf16): |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise;
  * H2O scores (fp32 vs fp64): |gpu - ref| <= 1e-6 + 1e-4 |ref|.
"""
import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O
from tests import kvc_testlib as T

pytestmark = pytest.mark.gpu

SCORE_ATOL, SCORE_RTOL = 1e-6, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()


def _cache(hq, hkv, bits, batch, max_ctx, extra_blocks=0, block_order=None):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    mbps = (max_ctx + 15) // 16 + 2
    nb = batch * mbps + extra_blocks
    return KVCache(hq, hkv, bits, nb, batch, mbps, block_order=block_order)


def _rand_bits(rng, shape, scale=1.0, outliers=None):
    from compressed_kv_cache_kvc_gb300.workloads import bf16_bits
    x = rng.standard_normal(shape).astype(np.float32) * np.float32(scale)
    if outliers is not None:
        x[..., outliers] *= 10
    return bf16_bits(x)


def _prefill(cache, k_bits, v_bits, lengths):
    for b, n in enumerate(lengths):
        n = int(n)
        if n == 0:
            continue
        k = T.to_dev_bf16(np.ascontiguousarray(k_bits[b:b + 1, :, :n]))
        v = T.to_dev_bf16(np.ascontiguousarray(v_bits[b:b + 1, :, :n]))
        cache.quantize_append(k, v, seq_begin=b)


def _oracle(hq, bits, k_bits, v_bits, lengths):
    return T.oracle_from_inputs(hq, bits, k_bits, v_bits, lengths)


# ---------------------------------------------------------------------------
# quantise-on-write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [8, 4])
def test_append_codes_bit_exact(bits):
    rng = np.random.default_rng(100 + bits)
    B, hq, hkv, T_ = 4, 8, 2, 300
    lengths = [1, 4, 17, 300]          # sinks only / exactly the sinks / page edge / ragged
    k = _rand_bits(rng, (B, hkv, T_, 128), outliers=[3, 50])
    v = _rand_bits(rng, (B, hkv, T_, 128))
    k[2, 0, 9] = 0                     # an all-zero row: scale 0, codes 0
    cache = _cache(hq, hkv, bits, B, T_ + 8)
    _prefill(cache, k, v, lengths)
    # then one batched decode append
    kn = _rand_bits(rng, (B, hkv, 1, 128))
    vn = _rand_bits(rng, (B, hkv, 1, 128))
    cache.quantize_append(T.to_dev_bf16(kn), T.to_dev_bf16(vn))
    ora = _oracle(hq, bits, k, v, lengths)
    for b in range(B):
        ora.append(b, O.bf16_bits_to_f32(kn[b]), O.bf16_bits_to_f32(vn[b]))
    st = T.StateView(cache)
    for b in range(B):
        assert st.slots[b] == max(0, lengths[b] + 1 - 4)
        assert st.seen[b] == lengths[b] + 1
        assert cache.lengths(b) == (int(st.slots[b]), int(st.seen[b]))
        for h in range(hkv):
            T.check_codes(st, ora, b, h)
    assert cache.read_status() == 0


def test_append_prefill_sink_boundary_split():
    # sinks arrive over several appends: 2 tokens, then 1, then 5
    rng = np.random.default_rng(7)
    hq, hkv = 4, 4
    cache = _cache(hq, hkv, 8, 1, 64)
    ora = O.OracleCache(1, hq, hkv, 8)
    for n in (2, 1, 5, 16, 1):
        k = _rand_bits(rng, (1, hkv, n, 128))
        v = _rand_bits(rng, (1, hkv, n, 128))
        cache.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(v))
        ora.append(0, O.bf16_bits_to_f32(k[0]), O.bf16_bits_to_f32(v[0]))
    st = T.StateView(cache)
    assert st.seen[0] == 25 and st.slots[0] == 21
    for h in range(hkv):
        T.check_codes(st, ora, 0, h)


# ---------------------------------------------------------------------------
# attention (+ H2O score accumulation)
# ---------------------------------------------------------------------------

ATTN_CASES = [
    # bits, hq, hkv, context
    (8, 8, 8, 700),
    (8, 32, 8, 1000),
    (4, 40, 8, 999),
    (8, 8, 1, 333),
    (4, 4, 4, 50),
    (8, 10, 2, 3),      # all sinks
    (4, 8, 2, 5),       # one pool slot
    (8, 16, 4, 20),     # one full page + ragged tail
    (4, 6, 2, 4100),    # many splits
]


@pytest.mark.parametrize("bits,hq,hkv,ctx", ATTN_CASES)
def test_decode_attention_and_scores(bits, hq, hkv, ctx):
    rng = np.random.default_rng(bits * 1000 + hq * 10 + ctx)
    B = 2
    lengths = [ctx, max(1, ctx // 2 + 3)]
    k = _rand_bits(rng, (B, hkv, ctx, 128), outliers=[1, 2, 77, 100])
    v = _rand_bits(rng, (B, hkv, ctx, 128))
    q = _rand_bits(rng, (B, hq, 128))
    cache = _cache(hq, hkv, bits, B, ctx + 4)
    _prefill(cache, k, v, lengths)
    out = cache.decode_attention(T.to_dev_bf16(q), accumulate_h2o=True)
    gpu = T.bf16_tensor_to_f32(out)
    ora = _oracle(hq, bits, k, v, lengths)
    st = T.StateView(cache)
    for b in range(B):
        ref = ora.attend(b, O.bf16_bits_to_f32(q[b]), T.sm_scale(), accumulate=True)
        T.assert_attention_close(gpu[b], ref, f"b={b}")
        s = ora.seqs[b]
        for h in range(hkv):
            pos, *_, sc = st.head(b, h)
            hs = s.heads[h]
            want = dict(zip(hs.pos.tolist(), hs.score.tolist()))
            w = np.array([want[p] for p in pos.tolist()])
            assert np.all(np.abs(sc - w) <= SCORE_ATOL + SCORE_RTOL * np.abs(w)), (b, h)
            ns = s.sink_k[h].shape[0]
            ss = st.sink_score[b, h, :ns]
            assert np.all(np.abs(ss - s.sink_score[h]) <= SCORE_ATOL + SCORE_RTOL * np.abs(s.sink_score[h]))
            # invariant: this step's increments sum to the group size
            assert abs(sc.sum() + ss.sum() - hq // hkv) <= 1e-4 * (hq // hkv)
    assert cache.read_status() == 0


def test_attention_without_h2o_leaves_scores():
    rng = np.random.default_rng(3)
    hq, hkv, ctx = 8, 2, 200
    k = _rand_bits(rng, (1, hkv, ctx, 128))
    v = _rand_bits(rng, (1, hkv, ctx, 128))
    q = _rand_bits(rng, (1, hq, 128))
    cache = _cache(hq, hkv, 8, 1, ctx + 4)
    _prefill(cache, k, v, [ctx])
    cache.decode_attention(T.to_dev_bf16(q), accumulate_h2o=False)
    st = T.StateView(cache)
    assert np.all(st.head(0, 0)[5] == 0) and np.all(st.sink_score == 0)


def test_attention_planted_token_and_scaled_inputs():
    # a token aligned with q dominates; inputs far from unit scale keep parity
    rng = np.random.default_rng(11)
    hq, hkv, ctx = 4, 1, 400
    from compressed_kv_cache_kvc_gb300.workloads import bf16_bits
    qf = rng.standard_normal((1, hq, 128)).astype(np.float32) * 3e-3
    kf = rng.standard_normal((1, hkv, ctx, 128)).astype(np.float32) * 200.0
    vf = rng.standard_normal((1, hkv, ctx, 128)).astype(np.float32) * 1e-3
    kf[0, 0, 123] = qf[0].mean(0) * 5e5
    q, k, v = bf16_bits(qf), bf16_bits(kf), bf16_bits(vf)
    cache = _cache(hq, hkv, 8, 1, ctx + 4)
    _prefill(cache, k, v, [ctx])
    gpu = T.bf16_tensor_to_f32(cache.decode_attention(T.to_dev_bf16(q)))
    ora = _oracle(hq, 8, k, v, [ctx])
    ref = ora.attend(0, O.bf16_bits_to_f32(q[0]), T.sm_scale())
    # relative bound only (outputs are ~1e-3): scale the absolute term
    err = np.abs(gpu[0] - ref)
    assert np.all(err <= 2e-3 * 1e-3 + 1e-2 * np.abs(ref)), err.max()


# ---------------------------------------------------------------------------
# the whole step: append -> attention -> select -> compact, in lock-step
# ---------------------------------------------------------------------------

def _run_steps(hq, hkv, bits, k, v, lengths, steps, mode, budget=0, recent=0, window=0, seed=0,
               block_order=None):
    rng = np.random.default_rng(seed)
    B = k.shape[0]
    G = hq // hkv
    cache = _cache(hq, hkv, bits, B, max(lengths) + steps + 4, block_order=block_order)
    if block_order is not None:
        pass
    _prefill(cache, k, v, lengths)
    ora = _oracle(hq, bits, k, v, lengths)
    h2o = mode == "h2o"
    stats = dict(max_err=0.0, tie_diffs=0)
    for step in range(steps):
        kn = _rand_bits(rng, (B, hkv, 1, 128))
        vn = _rand_bits(rng, (B, hkv, 1, 128))
        q = _rand_bits(rng, (B, hq, 128))
        cache.quantize_append(T.to_dev_bf16(kn), T.to_dev_bf16(vn))
        out = cache.decode_attention(T.to_dev_bf16(q), accumulate_h2o=h2o)
        gpu = T.bf16_tensor_to_f32(out)
        pre = T.StateView(cache)
        mask = cache.h2o_select_evict(B, mode=mode, budget=budget, recent=recent, window=window)
        mask_h = mask.cpu().numpy()
        cache.compact_blocks(mask, B)
        post = T.StateView(cache)
        for b in range(B):
            ora.append(b, O.bf16_bits_to_f32(kn[b]), O.bf16_bits_to_f32(vn[b]))
            ref = ora.attend(b, O.bf16_bits_to_f32(q[b]), T.sm_scale(), accumulate=h2o)
            stats["max_err"] = max(stats["max_err"], T.assert_attention_close(gpu[b], ref, f"step {step} b={b}"))
            P = int(pre.seen[b])
            for h in range(hkv):
                T.check_codes(pre, ora, b, h)
                pos, kc, ks, vc, vs, sc = pre.head(b, h)
                S = pos.size
                kept_gpu = set(pos[mask_h[b, h, :S] == 1].tolist())
                ns = min(P, 4)
                hs = ora.seqs[b].heads[h]
                if h2o:
                    want = dict(zip(hs.pos.tolist(), hs.score.tolist()))
                    w = np.array([want[p] for p in pos.tolist()])
                    assert np.all(np.abs(sc - w) <= SCORE_ATOL + SCORE_RTOL * np.abs(w)), (step, b, h)
                    # exact: the oracle's rule on the GPU's own scores
                    exact = O.select_h2o(pos, sc.astype(np.float64), P, budget, recent, ns)
                    assert set(pos[exact].tolist()) == kept_gpu, (step, b, h)
                    # against the oracle's own scores: near-ties only
                    om = O.select_h2o(hs.pos, hs.score, P, budget, recent, ns)
                    kept_ora = set(hs.pos[om].tolist())
                    heavy = budget - 4 - recent
                    if kept_gpu != kept_ora:
                        stats["tie_diffs"] += 1
                    assert T.kept_sets_agree(kept_gpu, kept_ora, hs.pos, hs.score, heavy, P - recent), (step, b, h)
                else:
                    om = O.select_streaming(hs.pos, P, window, ns)
                    assert set(hs.pos[om].tolist()) == kept_gpu, (step, b, h)
                    if S > window:
                        assert kept_gpu == set(range(P - window, P))
                # compaction: kept multiset moved intact
                keep_idx = np.nonzero(mask_h[b, h, :S] == 1)[0]
                ppos, pkc, pks, pvc, pvs, psc = post.head(b, h)
                assert ppos.size == keep_idx.size
                o1 = np.argsort(pos[keep_idx])
                o2 = np.argsort(ppos)
                assert np.array_equal(pos[keep_idx][o1], ppos[o2])
                assert np.array_equal(kc[keep_idx][o1], pkc[o2]) and np.array_equal(vc[keep_idx][o1], pvc[o2])
                assert np.array_equal(ks[keep_idx][o1].view(np.uint32), pks[o2].view(np.uint32))
                assert np.array_equal(vs[keep_idx][o1].view(np.uint32), pvs[o2].view(np.uint32))
                assert np.array_equal(sc[keep_idx][o1].view(np.uint32), psc[o2].view(np.uint32))
                # kept slots inside the keep window [w, w + n') did not move
                # (they are slots t - w now); only the ones outside it moved
                npr = keep_idx.size
                w = 16 * ((S - npr) // 16) if npr < S else 0
                stay = keep_idx[(keep_idx >= w) & (keep_idx < w + npr)]
                assert np.array_equal(pos[stay], ppos[stay - w])
            T.load_oracle_from_state(ora, post, b)
        # block conservation: used + free = all, no id twice
        used = np.concatenate([post.used_blocks(b) for b in range(B)] + [np.zeros(0, np.int32)])
        top = int(post.counters[0])
        free = post.free_stack[:top]
        allb = np.concatenate([used, free])
        assert allb.size == post.num_blocks and np.unique(allb).size == post.num_blocks
        assert cache.read_status() == 0
    return stats


def test_tiny_workload_h2o_eight_steps():
    from compressed_kv_cache_kvc_gb300 import workloads as W
    w = W.WORKLOADS["tiny_b1_h8_t512_int8_h2o"]
    d = W.gen_layer(w, 0)
    st = _run_steps(w.num_q_heads, w.num_kv_heads, w.bits, d["k"], d["v"], d["lengths"], 8, "h2o",
                    budget=w.budget, recent=w.recent, seed=5)
    assert st["max_err"] < 2e-2


@pytest.mark.parametrize("bits,hq,hkv", [(8, 32, 8), (4, 40, 8), (8, 8, 8)])
def test_h2o_steps_gqa(bits, hq, hkv):
    rng = np.random.default_rng(bits + hq)
    B, ctx = 3, 600
    lengths = [600, 433, 70]
    k = _rand_bits(rng, (B, hkv, ctx, 128), outliers=[5, 9, 60, 61])
    v = _rand_bits(rng, (B, hkv, ctx, 128))
    _run_steps(hq, hkv, bits, k, v, lengths, 4, "h2o", budget=180, recent=40, seed=bits)


def test_h2o_budget_covers_context_is_identity():
    rng = np.random.default_rng(21)
    hq, hkv, ctx = 8, 2, 150
    k = _rand_bits(rng, (1, hkv, ctx, 128))
    v = _rand_bits(rng, (1, hkv, ctx, 128))
    _run_steps(hq, hkv, 8, k, v, [ctx], 2, "h2o", budget=4 + ctx + 10, recent=8, seed=1)


def test_h2o_zero_heavy_and_only_sinks():
    rng = np.random.default_rng(22)
    hq, hkv, ctx = 4, 2, 90
    k = _rand_bits(rng, (1, hkv, ctx, 128))
    v = _rand_bits(rng, (1, hkv, ctx, 128))
    _run_steps(hq, hkv, 8, k, v, [ctx], 2, "h2o", budget=4 + 16, recent=16, seed=2)
    _run_steps(hq, hkv, 4, k, v, [ctx], 2, "h2o", budget=4, recent=0, seed=3)


def test_streaming_ragged_steps():
    rng = np.random.default_rng(23)
    hq, hkv = 32, 8
    lengths = [700, 100, 257, 260, 1000]
    B, ctx = len(lengths), max(lengths)
    k = _rand_bits(rng, (B, hkv, ctx, 128))
    v = _rand_bits(rng, (B, hkv, ctx, 128))
    _run_steps(hq, hkv, 8, k, v, lengths, 4, "streaming", window=256, seed=4)


def test_shuffled_block_order():
    rng = np.random.default_rng(24)
    hq, hkv, ctx, B = 8, 8, 300, 2
    k = _rand_bits(rng, (B, hkv, ctx, 128))
    v = _rand_bits(rng, (B, hkv, ctx, 128))
    mbps = (ctx + 3 + 4 + 15) // 16 + 2
    order = np.random.default_rng(0).permutation(B * mbps).astype(np.int32)
    _run_steps(hq, hkv, 8, k, v, [ctx, 211], 3, "h2o", budget=64, recent=16, seed=6, block_order=order)


def test_capacity_error_leaves_cache_unchanged():
    from compressed_kv_cache_kvc_gb300 import _lib as L
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(25)
    cache = KVCache(4, 2, 8, num_blocks=3, max_batch=1, max_blocks_per_seq=8)
    k = _rand_bits(rng, (1, 2, 40, 128))
    cache.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(k))  # 36 slots -> 3 blocks
    before = cache.state_view.clone()
    k1 = _rand_bits(rng, (1, 2, 13, 128))
    with pytest.raises(L.KvcError) as ei:
        cache.quantize_append(T.to_dev_bf16(k1), T.to_dev_bf16(k1))
    assert ei.value.status == L.KVC_ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.equal(before, cache.state_view)
    assert cache.lengths(0) == (36, 40)


def test_launch_counts():
    rng = np.random.default_rng(26)
    cache = _cache(8, 2, 8, 1, 100)
    k = _rand_bits(rng, (1, 2, 80, 128))
    cache.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(k))
    assert cache.last_launch_count() == 2  # a long append: page allocation, then rows over token chunks
    cache.quantize_append(T.to_dev_bf16(k[:, :, :10]), T.to_dev_bf16(k[:, :, :10]))
    assert cache.last_launch_count() == 1
    q = _rand_bits(rng, (1, 8, 128))
    cache.decode_attention(T.to_dev_bf16(q))
    assert cache.last_launch_count() == 2
    m = cache.h2o_select_evict(1, budget=40, recent=8)
    assert cache.last_launch_count() == 1
    cache.compact_blocks(m, 1)
    assert cache.last_launch_count() == 2  # compaction, page release


@pytest.mark.parametrize("bits,W", [(8, 0), (4, 0), (8, 40)])
def test_bulk_append_equals_token_by_token(bits, W):
    """A long append (page allocation, then rows spread over token chunks)
    leaves the same device state, byte for byte, as the same tokens appended
    one at a time (one CTA per sequence)."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(bits + W)
    lengths = [300, 77, 129]
    B, hkv, n = 3, 4, max(lengths)
    mbps = (n + 15) // 16 + 1
    ca = KVCache(16, hkv, bits, B * mbps, B, mbps, bf16_window=W)
    cb = KVCache(16, hkv, bits, B * mbps, B, mbps, bf16_window=W)
    k = _rand_bits(rng, (B, hkv, n, 128))
    v = _rand_bits(rng, (B, hkv, n, 128))
    for b, nb in enumerate(lengths):
        ca.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :nb])),
                           T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :nb])), seq_begin=b)
        assert ca.last_launch_count() == 2
        for t in range(nb):
            cb.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, t:t + 1])),
                               T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, t:t + 1])), seq_begin=b)
    torch.cuda.synchronize()
    sa, sb = T.StateView(ca), T.StateView(cb)
    for b, nb in enumerate(lengths):
        for h in range(hkv):
            for x, y in zip(sa.head(b, h), sb.head(b, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (b, h)
            if W:
                for x, y in zip(sa.ring_head(b, h), sb.ring_head(b, h)):
                    assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (b, h)
    for name in ["BLOCK_TABLE", "SEQ_SLOTS", "SEQ_POS", "SINK_K", "SINK_V"]:
        assert torch.equal(ca.buffer(name), cb.buffer(name)), name
    assert ca.read_status() == 0 and cb.read_status() == 0


def _edge_rows(bits, rng, n_rows):
    """bf16 bit patterns of 128-value rows at the edges of the rounding:
    exact half-integer quotients, quotients within 2^-12 of a half-integer
    (found by enumerating every bf16 value), subnormal and near-overflow
    scales, zero and negative-zero rows, a lone nonzero value."""
    qmax = 127 if bits == 8 else 7
    allb = np.arange(65536, dtype=np.uint32)
    allf = (allb << 16).view(np.float32)
    rows = []
    # exact ties, scale 1 and 2^-3
    for div in (1.0, 8.0):
        ks = np.arange(-qmax, qmax) + 0.5
        r = np.resize(ks, 128).astype(np.float32) / np.float32(div)
        r[0] = np.float32(qmax / div)
        rows.append(r)
    # near ties for a few non-power-of-two scales
    for amax in (100.0, 3.0, 0.0371, 5.5e-20):
        a = np.float32((np.uint32(np.float32(amax).view(np.uint32)) & 0xFFFF0000).view(np.float32))
        scale = np.float32(a / np.float32(qmax))
        with np.errstate(all="ignore"):
            t = (allf / scale).astype(np.float32)
            d = np.abs(t - np.floor(t) - np.float32(0.5))
        ok = np.isfinite(allf) & (np.abs(allf) <= a)
        near = allf[ok & (d < 2.0 ** -12)]
        assert near.size > 0
        r = np.resize(rng.permutation(near), 128).astype(np.float32)
        r[0] = a
        rows.append(r)
    sub = lambda hi: (rng.integers(0, hi, 128).astype(np.uint32) << 16).view(np.float32)
    rows.append(sub(6) * np.where(rng.random(128) < 0.5, -1, 1).astype(np.float32))  # subnormal amax
    rows.append(rng.uniform(-1, 1, 128).astype(np.float32) * np.float32(2.0 ** -120))  # scale in (2^-128, 2^-126)
    rows.append(rng.uniform(-1, 1, 128).astype(np.float32) * np.float32(3.0e38))  # huge
    rows.append(np.zeros(128, np.float32))
    rows.append(np.full(128, -0.0, np.float32))
    lone = np.zeros(128, np.float32)
    lone[77] = -2.5
    rows.append(lone)
    from compressed_kv_cache_kvc_gb300.workloads import bf16_bits
    out = [bf16_bits(r) for r in rows]
    return [out[i % len(out)] for i in range(n_rows)]


@pytest.mark.parametrize("bits", [8, 4])
def test_bulk_append_rounding_edges(bits):
    """Rows whose quotients x / scale sit on or within 2^-12 of a half-integer,
    subnormal and near-overflow scales, zero rows: the long append (16-byte
    loads, the product with the reciprocal deciding where it can) gives the
    oracle's codes and scales bit for bit."""
    rng = np.random.default_rng(400 + bits)
    B, hq, hkv, n = 2, 4, 2, 96
    k = _rand_bits(rng, (B, hkv, n, 128))
    v = _rand_bits(rng, (B, hkv, n, 128))
    edge = _edge_rows(bits, rng, 2 * B * hkv * 40)
    i = 0
    for b in range(B):
        for h in range(hkv):
            for t in range(4, 44):
                k[b, h, t] = edge[i]
                v[b, h, n - 1 - (t - 4)] = edge[(i + 7) % len(edge)]
                i += 1
    cache = _cache(hq, hkv, bits, B, n + 8)
    _prefill(cache, k, v, [n] * B)
    assert cache.last_launch_count() == 2
    ora = _oracle(hq, bits, k, v, [n] * B)
    st = T.StateView(cache)
    for b in range(B):
        for h in range(hkv):
            T.check_codes(st, ora, b, h)
    assert cache.read_status() == 0


@pytest.mark.parametrize("B,n", [(10, 1000), (5, 1000), (4, 601), (3, 700)])
def test_bulk_append_chunk_sizes(B, n):
    """One batched long append whose grid takes 32, 16, 8 and 4 tokens per
    CTA (on 152 SMs: the chunk halves while fewer than two CTAs per SM would
    run), ragged tails included: codes and scales equal the oracle's bit for
    bit in both code widths."""
    for bits in (8, 4):
        rng = np.random.default_rng(1000 * B + n + bits)
        hq, hkv = 2, 2
        k = _rand_bits(rng, (B, hkv, n, 128), outliers=[5])
        v = _rand_bits(rng, (B, hkv, n, 128))
        cache = _cache(hq, hkv, bits, B, n + 8)
        cache.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(v))
        assert cache.last_launch_count() == 2
        ora = _oracle(hq, bits, k, v, [n] * B)
        st = T.StateView(cache)
        for b in range(B):
            for h in range(hkv):
                T.check_codes(st, ora, b, h)
        assert cache.read_status() == 0


@pytest.mark.parametrize("bits", [8, 4])
def test_long_window_append_equals_token_by_token(bits):
    """A long append that pushes window tokens into the pool runs on the
    one-CTA-per-sequence kernel and writes more pool pages than that kernel
    stages in shared memory (13 here): the state equals the same tokens
    appended one at a time, byte for byte."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(77 + bits)
    hkv, W, n1, n2 = 2, 40, 300, 200
    mbps = (n1 + n2) // 16 + 2
    ca = KVCache(4, hkv, bits, mbps, 1, mbps, bf16_window=W)
    cb = KVCache(4, hkv, bits, mbps, 1, mbps, bf16_window=W)
    k = _rand_bits(rng, (1, hkv, n1 + n2, 128))
    v = _rand_bits(rng, (1, hkv, n1 + n2, 128))
    for a, e in ((0, n1), (n1, n1 + n2)):
        ca.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[:, :, a:e])),
                           T.to_dev_bf16(np.ascontiguousarray(v[:, :, a:e])))
    assert ca.last_launch_count() == 1  # window tokens pushed out: the one-CTA kernel
    for t in range(n1 + n2):
        cb.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[:, :, t:t + 1])),
                           T.to_dev_bf16(np.ascontiguousarray(v[:, :, t:t + 1])))
    torch.cuda.synchronize()
    sa, sb = T.StateView(ca), T.StateView(cb)
    for h in range(hkv):
        for x, y in zip(sa.head(0, h), sb.head(0, h)):
            assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), h
        for x, y in zip(sa.ring_head(0, h), sb.ring_head(0, h)):
            assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), h
    for name in ["BLOCK_TABLE", "SEQ_SLOTS", "SEQ_POS", "SINK_K", "SINK_V"]:
        assert torch.equal(ca.buffer(name), cb.buffer(name)), name
    assert ca.read_status() == 0 and cb.read_status() == 0


def test_append_8_byte_aligned_input():
    """A long append from inputs aligned to 8 bytes but not 16 runs on the
    one-CTA-per-sequence kernel and leaves the same state as the same rows
    appended from aligned inputs."""
    rng = np.random.default_rng(31)
    B, hq, hkv, n = 2, 4, 2, 100
    k = _rand_bits(rng, (B, hkv, n, 128))
    v = _rand_bits(rng, (B, hkv, n, 128))
    ca, cb = _cache(hq, hkv, 8, B, n + 8), _cache(hq, hkv, 8, B, n + 8)

    def shifted(bits):
        flat = T.to_dev_bf16(bits.reshape(-1))
        buf = torch.empty(flat.numel() + 4, dtype=torch.bfloat16, device=flat.device)
        view = buf[4:].view(bits.shape)
        view.copy_(flat.view(bits.shape))
        assert view.data_ptr() % 16 == 8
        return view

    ca.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(v))
    assert ca.last_launch_count() == 2
    cb.quantize_append(shifted(k), shifted(v))
    assert cb.last_launch_count() == 1
    torch.cuda.synchronize()
    sa, sb = T.StateView(ca), T.StateView(cb)
    for b in range(B):
        for h in range(hkv):
            for x, y in zip(sa.head(b, h), sb.head(b, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (b, h)
    # (the block ids differ: the one-CTA kernel's sequences take their pages
    # from the free stack in launch order, not sequence order)
    for name in ["SEQ_SLOTS", "SEQ_POS", "SINK_K", "SINK_V"]:
        assert torch.equal(ca.buffer(name), cb.buffer(name)), name
    assert ca.read_status() == 0 and cb.read_status() == 0


def test_release_sequences():
    """Releasing a sequence returns its pages (no block lost or duplicated),
    empties it, leaves the others alone, is idempotent, and the freed slot
    takes a new prompt that leaves the state a fresh cache would hold."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(90)
    lengths = [300, 170, 90]
    B, hkv, hq = 3, 2, 8
    mbps = 24
    cache = KVCache(hq, hkv, 8, B * mbps, B, mbps)
    k = _rand_bits(rng, (B, hkv, 300, 128))
    for b, n in enumerate(lengths):
        cache.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                              T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])), seq_begin=b)
    q = T.to_dev_bf16(_rand_bits(rng, (B, hq, 128)))
    kn = T.to_dev_bf16(_rand_bits(rng, (B, hkv, 1, 128)))
    cache.decode_step(q, kn, kn, mode="h2o", budget=120, recent=16)
    before = T.StateView(cache)
    cache.release(1, 1)
    assert cache.last_launch_count() == 1
    after = T.StateView(cache)
    assert cache.lengths(1) == (0, 0) and int(after.slots[1]) == 0 and int(after.seen[1]) == 0
    for b in (0, 2):
        assert cache.lengths(b) == (int(before.slots[b]), int(before.seen[b]))
        for h in range(hkv):
            for x, y in zip(before.head(b, h), after.head(b, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))
    used = np.concatenate([after.used_blocks(b) for b in (0, 2)])
    free = after.free_stack[:int(after.counters[0])]
    assert np.unique(np.concatenate([used, free])).size == B * mbps == used.size + free.size
    cache.release(1, 1)  # idempotent
    assert cache.last_launch_count() == 0
    # a new prompt in the freed slot equals the same prompt in a fresh cache
    k2 = _rand_bits(rng, (1, hkv, 200, 128))
    cache.quantize_append(T.to_dev_bf16(k2), T.to_dev_bf16(k2), seq_begin=1)
    fresh = KVCache(hq, hkv, 8, B * mbps, B, mbps)
    fresh.quantize_append(T.to_dev_bf16(k2), T.to_dev_bf16(k2), seq_begin=1)
    sa, sb = T.StateView(cache), T.StateView(fresh)
    for h in range(hkv):
        for x, y in zip(sa.head(1, h), sb.head(1, h)):
            assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))
    assert cache.read_status() == 0


def test_binding_refuses_mis_sized_buffers():
    """The binding refuses, before any launch, an output, keep mask or
    workspace whose shape, dtype or device differs from what the call's sizes
    imply, and inputs that are not on the cache's device; the cache is left
    usable."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    c = KVCache(8, 2, 8, 16, 2, 8)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(2, 8, 128, **bf)
    k = torch.zeros(2, 2, 1, 128, **bf)
    c.quantize_append(k, k)
    bad = [
        lambda: c.decode_attention(q, out=torch.empty(1, 8, 128, **bf)),
        lambda: c.decode_attention(q, workspace=torch.empty(1 << 20, dtype=torch.float32, device="cuda")),
        lambda: c.decode_attention(q.cpu()),
        lambda: c.decode_step(q, k, k, out=torch.empty(2, 8, 64, **bf)),
        lambda: c.h2o_select_evict(2, budget=8, recent=2, keep_mask=torch.empty(2, 2, 8, dtype=torch.uint8,
                                                                                  device="cuda")),
        lambda: c.compact_blocks(torch.zeros(1, 2, c.s_cap, dtype=torch.uint8, device="cuda"), 2),
        lambda: c.prefill_context(torch.zeros(2, 8, 3, 128, **bf), torch.zeros(2, 2, 3, 128, **bf),
                                  torch.zeros(2, 2, 3, 128, **bf), out=torch.empty(2, 8, 2, 128, **bf)),
    ]
    for f in bad:
        with pytest.raises(ValueError):
            f()
    assert c.lengths(0) == (0, 1) and c.lengths(1) == (0, 1)
    out = c.decode_attention(q)
    assert out.shape == q.shape and c.read_status() == 0
