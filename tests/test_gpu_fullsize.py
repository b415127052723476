"""Full-size parity: one layer of each large workload, at the launch
configuration the bench uses (the library picks the grid from the device), on
outputs the oracle can compute one sequence at a time, plus properties checked
on every (sequence, KV head).

Per step: append -> attention (+H2O) -> select -> compact.  For a few sampled
sequences the oracle (re-synchronised to the GPU state after each step) checks
codes, scales, outputs, scores and kept sets with the bars of
test_gpu_parity.py; for all pairs: kept counts, the per-step score increment
sum (= group size), and block conservation.
"""
import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O
from tests import kvc_testlib as T

pytestmark = pytest.mark.gpu

SCORE_ATOL, SCORE_RTOL = 1e-6, 1e-4

FULL = [
    ("llama7b_b16_h32_t4096_int8_h2o", 2),
    ("llama3_8b_b64_gqa_ragged_int8_streaming", 2),
    ("qwen14b_b32_gqa5_t8192_int4_h2o_48l", 2),
    ("longctx_b4_gqa4_t32768_int8_h2o_32l_64s", 3),
]


def _same_logical_state(a, b):
    """Two caches hold the same logical state: per (sequence, KV head) the
    slots in slot order (positions, codes, scales, scores) bit for bit, the
    sinks and their scores, the lengths and the free-block count."""
    sa, sb = T.StateView(a), T.StateView(b)
    assert np.array_equal(sa.slots, sb.slots) and np.array_equal(sa.seen, sb.seen)
    for seq in range(a.max_batch):
        for h in range(a.num_kv_heads):
            for x, y in zip(sa.head(seq, h), sb.head(seq, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (seq, h)
    assert np.array_equal(sa.sink_k, sb.sink_k) and np.array_equal(sa.sink_v, sb.sink_v)
    assert np.array_equal(sa.sink_score.view(np.uint32), sb.sink_score.view(np.uint32))
    assert sa.counters[0] == sb.counters[0]
    return sb


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_cache_kvc_gb300.build import build_library
    build_library()


@pytest.mark.parametrize("name,steps", FULL)
def test_full_size_sampled(name, steps):
    _full_size(name, steps, with_step=False)


# The one-call step at the shapes the bench times: 256 (Qwen-shaped INT4) and
# 512 (LLaMA-shaped INT8) (sequence, KV head) pairs, more than the SMs, so the
# library runs the 512-thread post kernel beside the split and move kernels;
# the 32k-context stack has 32 pairs (the 1024-thread post kernel).
STEP_FULL = [
    ("qwen14b_b32_gqa5_t8192_int4_h2o_48l", 2),
    ("llama7b_b16_h32_t4096_int8_h2o", 2),
    ("longctx_b4_gqa4_t32768_int8_h2o_32l_64s", 3),
]


@pytest.mark.parametrize("name,steps", STEP_FULL)
def test_full_size_decode_step(name, steps):
    """The benchmarked path itself: kvc_decode_step on a full-size layer,
    step after step.  A second cache runs the separate calls on the same
    inputs and gets every check of the sampled test (oracle outputs, codes,
    scores and kept sets on sampled sequences; on every pair the kept set the
    oracle's rule gives on the GPU's own scores, the score-sum invariant,
    block conservation); the one-call step must give the same outputs bit for
    bit and the same logical state after every step, so every check carries
    over to it.  Its own outputs are also checked against the oracle."""
    _full_size(name, steps, with_step=True)


def _full_size(name, steps, with_step):
    from compressed_kv_cache_kvc_gb300 import workloads as W
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    w = W.WORKLOADS[name]
    d = W.gen_layer(w, 0)
    lengths = d["lengths"]
    B, hq, hkv, G = w.batch, w.num_q_heads, w.num_kv_heads, w.group
    mbps = (int(lengths.max()) + steps + 15) // 16 + 1
    nb = B * mbps
    order = W.block_order(w, nb) if w.shuffled_blocks else None
    cache = KVCache(hq, hkv, w.bits, nb, B, mbps, block_order=order)
    caches = [cache]
    if with_step:
        stepper = KVCache(hq, hkv, w.bits, nb, B, mbps, block_order=order)
        caches.append(stepper)
    for c in caches:
        if np.all(lengths == lengths[0]):
            c.quantize_append(T.to_dev_bf16(d["k"]), T.to_dev_bf16(d["v"]))
        else:
            for b in range(B):
                n = int(lengths[b])
                c.quantize_append(T.to_dev_bf16(np.ascontiguousarray(d["k"][b:b + 1, :, :n])),
                                  T.to_dev_bf16(np.ascontiguousarray(d["v"][b:b + 1, :, :n])), seq_begin=b)
    rng = np.random.default_rng(99)
    sample = sorted(rng.choice(B, size=min(2, B), replace=False).tolist())
    oras = {}
    for b in sample:
        o = O.OracleCache(1, hq, hkv, w.bits)
        n = int(lengths[b])
        o.append(0, O.bf16_bits_to_f32(d["k"][b, :, :n]), O.bf16_bits_to_f32(d["v"][b, :, :n]))
        oras[b] = o
    del d["k"], d["v"]
    h2o = w.mode == "h2o"
    prev_sum = np.zeros((B, hkv))
    for step in range(steps):
        s = d if step == 0 else W.gen_step(w, 0, step)
        if with_step:
            sout = stepper.decode_step(T.to_dev_bf16(s["q"]), T.to_dev_bf16(s["k_new"]), T.to_dev_bf16(s["v_new"]),
                                       mode=w.mode, budget=w.budget, recent=w.recent, window=w.window)
            # the first step moves hundreds of rows per pair (a move kernel); later
            # steps move one (inside the post kernel)
            assert stepper.last_launch_count() == (4 if step == 0 else 3)
        cache.quantize_append(T.to_dev_bf16(s["k_new"]), T.to_dev_bf16(s["v_new"]))
        out = cache.decode_attention(T.to_dev_bf16(s["q"]), accumulate_h2o=h2o)
        gpu = T.bf16_tensor_to_f32(out)
        pre = T.StateView(cache)
        mask = cache.h2o_select_evict(B, mode=w.mode, budget=w.budget, recent=w.recent, window=w.window)
        mask_h = mask.cpu().numpy()
        cache.compact_blocks(mask, B)
        post = T.StateView(cache)
        for b in range(B):
            P = int(pre.seen[b])
            for h in range(hkv):
                pos, kc, ks, vc, vs, sc = pre.head(b, h)
                S = pos.size
                kept = mask_h[b, h, :S] == 1
                if h2o:
                    want = S if 4 + S <= w.budget else w.budget - 4
                    tot = float(sc.astype(np.float64).sum() + pre.sink_score[b, h, :min(P, 4)].sum())
                    assert abs(tot - prev_sum[b, h] - G) <= 1e-4 * G * (step + 1), (step, b, h)
                    # kept set = the rule applied to the GPU's own scores
                    exact = O.select_h2o(pos, sc.astype(np.float64), P, w.budget, w.recent, min(P, 4))
                    assert np.array_equal(exact, kept), (step, b, h)
                else:
                    want = S if S <= w.window else w.window
                    if S > w.window:
                        assert set(pos[kept].tolist()) == set(range(P - w.window, P)), (step, b, h)
                assert int(kept.sum()) == want and int(post.slots[b]) == want
                ppos = post.head(b, h)[0]
                assert np.array_equal(np.sort(ppos), np.sort(pos[kept])), (step, b, h)
                prev_sum[b, h] = float(post.head(b, h)[5].astype(np.float64).sum() +
                                       post.sink_score[b, h, :min(P, 4)].sum())
        if with_step:
            torch.cuda.synchronize()
            assert torch.equal(sout, out), f"{name} step {step}: one-call step output differs"
            _same_logical_state(cache, stepper)
            for b in range(B):
                assert stepper.lengths(b) == cache.lengths(b)
        for b in sample:
            ora = oras[b]
            ora.append(0, O.bf16_bits_to_f32(s["k_new"][b]), O.bf16_bits_to_f32(s["v_new"][b]))
            ref = ora.attend(0, O.bf16_bits_to_f32(s["q"][b]), T.sm_scale(), accumulate=h2o)
            T.assert_attention_close(gpu[b], ref, f"{name} step {step} b={b}")
            if with_step:
                T.assert_attention_close(T.bf16_tensor_to_f32(sout)[b], ref, f"{name} one-call step {step} b={b}")
            for h in range(hkv):
                # codes/scales/positions of the sampled sequence, bit for bit
                sv = _single(pre, b)
                T.check_codes(sv, ora, 0, h)
                if h2o:
                    pos, *_, sc = pre.head(b, h)
                    hs = ora.seqs[0].heads[h]
                    wmap = dict(zip(hs.pos.tolist(), hs.score.tolist()))
                    ws = np.array([wmap[p] for p in pos.tolist()])
                    assert np.all(np.abs(sc - ws) <= SCORE_ATOL + SCORE_RTOL * np.abs(ws)), (step, b, h)
                    om = O.select_h2o(hs.pos, hs.score, int(pre.seen[b]), w.budget, w.recent, 4)
                    kept_gpu = set(pos[mask_h[b, h, :pos.size] == 1].tolist())
                    assert T.kept_sets_agree(kept_gpu, set(hs.pos[om].tolist()), hs.pos, hs.score,
                                             w.budget - 4 - w.recent, int(pre.seen[b]) - w.recent), (step, b, h)
            T.load_oracle_from_state(ora, _single(post, b), 0)
        used = np.concatenate([post.used_blocks(b) for b in range(B)])
        free = post.free_stack[:int(post.counters[0])]
        allb = np.concatenate([used, free])
        assert allb.size == nb and np.unique(allb).size == nb
        assert cache.read_status() == 0
    if with_step:
        assert stepper.read_status() == 0


class _single:
    """View of one sequence b of a StateView as sequence 0 (for the oracle helpers)."""

    def __init__(self, sv, b):
        self.sv, self.b = sv, b
        self.hkv = sv.hkv
        self.sink_k = sv.sink_k[b:b + 1]
        self.sink_v = sv.sink_v[b:b + 1]
        self.sink_score = sv.sink_score[b:b + 1]

    def head(self, _b, h):
        return self.sv.head(self.b, h)


FEATURES = [
    ("hybrid", "qwen14b_b32_gqa5_t8192_int4_h2o_48l"),   # bf16 window of the recent 512 positions
    ("fp8", "llama7b_b16_h32_t4096_int8_h2o"),          # FP8 E4M3 codes
    ("block", "qwen14b_b32_gqa5_t8192_int4_h2o_48l"),    # block-granular eviction, 25 % of the pages kept
]


@pytest.mark.parametrize("feature,name", FEATURES)
def test_full_size_features_sampled(feature, name):
    """One full-size layer per feature at the bench's launch configuration:
    two sampled sequences against the oracle (outputs; FP8 codes bit for bit;
    kept sets), and on every (sequence, KV head) the kept counts and block
    conservation; block eviction's mask is the oracle's rule on the GPU's own
    scores for every sequence."""
    from compressed_kv_cache_kvc_gb300 import workloads as W
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    w = W.WORKLOADS[name]
    d = W.gen_layer(w, 0)
    B, hq, hkv, n = w.batch, w.num_q_heads, w.num_kv_heads, w.context
    window = w.recent if feature == "hybrid" else 0
    codes = "e4m3" if feature == "fp8" else "int"
    mbps = (n + 1 + 15) // 16 + 1
    cache = KVCache(hq, hkv, w.bits, B * mbps, B, mbps, bf16_window=window, codes=codes)
    cache.quantize_append(T.to_dev_bf16(d["k"]), T.to_dev_bf16(d["v"]))
    f = O.bf16_bits_to_f32
    sample = sorted(np.random.default_rng(98).choice(B, size=2, replace=False).tolist())
    oras = {}
    for b in sample:
        oras[b] = O.OracleCache(1, hq, hkv, w.bits, bf16_window=window, codes=codes)
        oras[b].append(0, f(d["k"][b]), f(d["v"][b]))
    if feature == "fp8":
        st = T.StateView(cache)
        for b in sample:
            for h in range(hkv):
                T.check_codes(_single(st, b), oras[b], 0, h)
    del d["k"], d["v"]
    q, kn, vn = T.to_dev_bf16(d["q"]), T.to_dev_bf16(d["k_new"]), T.to_dev_bf16(d["v_new"])
    if feature == "block":
        retention = 0.25
        cache.quantize_append(kn, vn)
        out = cache.decode_attention(q)
        pre = T.StateView(cache)
        mask = cache.h2o_select_evict(B, mode="block", recent=w.recent, retention=retention).cpu().numpy()
        cache.compact_blocks(torch.from_numpy(mask).cuda(), B)
        for b in range(B):
            S = int(pre.slots[b])
            want = O.select_blocks([pre.head(b, h)[5].astype(np.float64) for h in range(hkv)], S, w.recent,
                                   retention)
            for h in range(hkv):
                assert np.array_equal(mask[b, h, :S] == 1, want), (b, h)
            assert cache.lengths(b)[0] == int(want.sum())
    else:
        out = cache.decode_step(q, kn, vn, mode="h2o", budget=w.budget, recent=w.recent)
    gpu = T.bf16_tensor_to_f32(out)
    post = T.StateView(cache)
    for b in sample:
        ora = oras[b]
        ora.append(0, f(d["k_new"][b]), f(d["v_new"][b]))
        T.assert_attention_close(gpu[b], ora.attend(0, f(d["q"][b]), T.sm_scale()), f"{feature} b={b}")
        if feature == "block":
            continue
        P = n + 1
        masks = ora.keep_masks(0, "h2o", budget=w.budget, recent=w.recent)
        for h in range(hkv):
            hs = ora.seqs[0].heads[h]
            kept = set(post.head(b, h)[0].tolist())
            if window:
                kept |= set(post.ring_head(b, h)[0].tolist())
            assert T.kept_sets_agree(kept, set(hs.pos[masks[h]].tolist()), hs.pos, hs.score,
                                     w.budget - 4 - w.recent, P - w.recent), (b, h)
    if feature != "block":
        nr = min(window, n + 1 - 4) if window else 0
        for b in range(B):
            assert cache.lengths(b) == (w.budget - 4 - nr, n + 1)
    used = np.concatenate([post.used_blocks(b) for b in range(B)])
    free = post.free_stack[:int(post.counters[0])]
    assert np.unique(np.concatenate([used, free])).size == B * mbps == used.size + free.size
    assert cache.read_status() == 0
