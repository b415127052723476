"""kvc_decode_step_overlap (the merge on the attention's stream, the eviction
on a second stream) must leave exactly the outputs and the logical device
state that kvc_decode_step leaves, step after step.  The steps run back to
back with no synchronisation between them: the library orders each call on a
cache after the eviction the previous call left running.  A multi-layer step
captured into one CUDA graph (the eviction stream forked from the capturing
stream and joined back) and replayed must equal the eager one-call steps."""
import numpy as np
import pytest
import torch

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
    """Same logical cache: per (sequence, KV head) the slots in slot order, the
    sinks and their scores, the bf16 window, the lengths and the free count."""
    sa, sb = T.StateView(a), T.StateView(b)
    assert np.array_equal(sa.slots, sb.slots) and np.array_equal(sa.seen, sb.seen)
    for seq in range(a.max_batch):
        for h in range(a.num_kv_heads):
            for x, y in zip(sa.head(seq, h), sb.head(seq, h)):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8)), (seq, h)
    assert np.array_equal(sa.sink_k, sb.sink_k) and np.array_equal(sa.sink_v, sb.sink_v)
    assert np.array_equal(sa.sink_score.view(np.uint32), sb.sink_score.view(np.uint32))
    for name in ("RING_K", "RING_V", "RING_SCORE"):
        assert torch.equal(a.buffer(name), b.buffer(name)), name
    assert np.array_equal(sa.counters[:2], sb.counters[:2])  # free-stack top, status


def _pair(bits, hq, hkv, lengths, steps, seed, codes="int", bf16_window=0):
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(seed)
    B, T_ = len(lengths), max(lengths)
    mbps = (T_ + steps + 15) // 16 + 2
    order = np.random.default_rng(seed + 1).permutation(B * mbps).astype(np.int32)
    caches = [KVCache(hq, hkv, bits, B * mbps, B, mbps, block_order=order, codes=codes, bf16_window=bf16_window)
              for _ in range(2)]
    k = _bits(rng, (B, hkv, T_, 128))
    v = _bits(rng, (B, hkv, T_, 128))
    for c in caches:
        for b, n in enumerate(lengths):
            c.quantize_append(T.to_dev_bf16(np.ascontiguousarray(k[b:b + 1, :, :n])),
                              T.to_dev_bf16(np.ascontiguousarray(v[b:b + 1, :, :n])), seq_begin=b)
    torch.cuda.synchronize()
    return caches, rng


CASES = [
    # bits, hq, hkv, lengths, mode, budget, recent, window, retention, codes, bf16 window, steps
    (4, 40, 8, [600, 433, 70], "h2o", 180, 40, 0, 1.0, "int", 0, 3),
    (8, 8, 8, [512], "h2o", 128, 32, 0, 1.0, "int", 0, 4),
    (8, 32, 8, [700, 100, 257, 260], "streaming", 0, 0, 256, 1.0, "int", 0, 3),
    (8, 16, 4, [600, 333], "block", 0, 40, 0, 0.5, "int", 0, 3),
    (8, 16, 4, [900, 200], "h2o", 300, 64, 0, 1.0, "e4m3", 0, 3),
    (4, 16, 4, [800, 300, 90], "h2o", 400, 160, 0, 1.0, "int", 128, 3),  # recent >= the window
    (8, 8, 2, [21000, 300], "h2o", 2100, 256, 0, 1.0, "int", 0, 2),
    (4, 8, 2, [41000], "h2o", 4100, 512, 0, 1.0, "int", 0, 2),
]


@pytest.mark.parametrize("bits,hq,hkv,lengths,mode,budget,recent,window,retention,codes,bfw,steps", CASES)
def test_overlap_equals_one_call_step(bits, hq, hkv, lengths, mode, budget, recent, window, retention, codes, bfw,
                                      steps):
    (ca, cb), rng = _pair(bits, hq, hkv, lengths, steps, bits * 11 + hq + len(lengths) + bfw, codes, bfw)
    B = len(lengths)
    s_att, s_ev = torch.cuda.Stream(), torch.cuda.Stream()
    ws_b = cb.workspace(B)
    inputs, outs_a, outs_b = [], [], []
    for _ in range(steps):
        q = T.to_dev_bf16(_bits(rng, (B, hq, 128)))
        kn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
        vn = T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))
        inputs.append((q, kn, vn))  # kept alive: the streams read them later
    s_att.wait_stream(torch.cuda.current_stream())
    for q, kn, vn in inputs:
        outs_a.append(ca.decode_step(q, kn, vn, mode=mode, budget=budget, recent=recent, window=window,
                                     retention=retention))
        n_one = ca.last_launch_count()
        ob = torch.empty_like(q)
        cb.decode_step_overlap(q, kn, vn, s_ev, mode=mode, budget=budget, recent=recent, window=window,
                               retention=retention, out=ob, workspace=ws_b, stream=s_att)
        assert cb.last_launch_count() == n_one + 1  # the merge of its own
        outs_b.append(ob)
    # no synchronisation above: read_status orders itself after the eviction
    assert cb.read_status(stream=s_att) == 0
    torch.cuda.synchronize()
    assert ca.read_status() == 0
    for oa, ob in zip(outs_a, outs_b):
        assert torch.equal(oa, ob)
    _same_state(ca, cb)
    for b in range(B):
        assert ca.lengths(b) == cb.lengths(b)


def test_overlap_graph_over_layers_equals_eager_steps():
    """Three layers captured into one graph on a capturing stream, each
    layer's eviction forked onto a second stream and joined at the end;
    replayed twice from the restored pre-step state.  The first step after
    the prompt (hundreds of rows move per pair) and, captured at the next
    state, a steady step (rows moved inside the post kernel)."""
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    rng = np.random.default_rng(5)
    L, B, hq, hkv, n, budget, recent = 3, 4, 40, 8, 700, 200, 40
    mbps = (n + 4 + 15) // 16 + 2
    ref, cap = [], []
    for _ in range(L):
        k = _bits(rng, (B, hkv, n, 128))
        v = _bits(rng, (B, hkv, n, 128))
        pair = []
        for _ in range(2):
            c = KVCache(hq, hkv, 4, B * mbps, B, mbps)
            c.quantize_append(T.to_dev_bf16(k), T.to_dev_bf16(v))
            pair.append(c)
        ref.append(pair[0])
        cap.append(pair[1])
    steps_in = [[(T.to_dev_bf16(_bits(rng, (B, hq, 128))), T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128))),
                  T.to_dev_bf16(_bits(rng, (B, hkv, 1, 128)))) for _ in range(L)] for _ in range(2)]
    torch.cuda.synchronize()
    s_att, s_ev = torch.cuda.Stream(), torch.cuda.Stream()
    wss = [c.workspace(B) for c in cap]
    outs = [torch.empty(B, hq, 128, dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    for st in range(2):
        ref_out = [ref[l].decode_step(*steps_in[st][l], mode="h2o", budget=budget, recent=recent)
                   for l in range(L)]
        torch.cuda.synchronize()
        snaps = [c.state_view.clone() for c in cap]

        def layers():
            for l in range(L):
                cap[l].decode_step_overlap(*steps_in[st][l], s_ev, mode="h2o", budget=budget, recent=recent,
                                           out=outs[l], workspace=wss[l], stream=s_att)

        # an eager run first (the library creates its events outside any capture)
        s_att.wait_stream(torch.cuda.current_stream())
        layers()
        s_att.wait_stream(s_ev)
        torch.cuda.synchronize()
        for c, s in zip(cap, snaps):
            c.state_view.copy_(s)
        torch.cuda.synchronize()
        for c in cap:
            c.sync_host()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s_att):
            layers()
            s_att.wait_stream(s_ev)  # the join
        torch.cuda.synchronize()
        for rep in range(2):
            for c, s in zip(cap, snaps):
                c.state_view.copy_(s)
            torch.cuda.synchronize()
            with torch.cuda.stream(s_att):
                g.replay()
            torch.cuda.synchronize()
            for l in range(L):
                assert torch.equal(outs[l], ref_out[l]), (st, rep, l)
                _same_state(ref[l], cap[l])
        for c in cap:
            c.sync_host()
            assert c.read_status() == 0
        del g


@pytest.mark.parametrize("name", ["qwen14b_b32_gqa5_t8192_int4_h2o_48l", "llama7b_b16_h32_t4096_int8_h2o"])
def test_overlap_equals_one_call_step_full_size(name):
    """The benchmarked call itself, kvc_decode_step_overlap, on one full-size
    layer of the INT4 Qwen-shaped stack (256 pairs) and of the INT8
    LLaMA-shaped one (512 pairs, shuffled blocks), two steps back to back:
    the same outputs bit for bit and the same logical state as the one-call
    step, which tests/test_gpu_fullsize.py checks against the oracle at these
    sizes.  Inputs from the bench's device-side draw of the same recipe."""
    from compressed_kv_cache_kvc_gb300 import workloads as W
    from compressed_kv_cache_kvc_gb300.cache import KVCache
    w = W.WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, kn, vn = W.gen_layer_torch(w, 0, dev)
    B, hq, hkv, steps = w.batch, w.num_q_heads, w.num_kv_heads, 2
    mbps = (w.context + steps + 15) // 16 + 1
    order = W.block_order(w, B * mbps) if w.shuffled_blocks else None
    ca, cb = [KVCache(hq, hkv, w.bits, B * mbps, B, mbps, block_order=order) for _ in range(2)]
    for c in (ca, cb):
        c.quantize_append(k, v)
    del k, v
    inputs = [(q, kn, vn)] + [W.gen_step_torch(w, 0, st, dev) for st in range(1, steps)]
    s_att, s_ev = torch.cuda.Stream(), torch.cuda.Stream()
    ws_b = cb.workspace(B)
    s_att.wait_stream(torch.cuda.current_stream())
    outs_a, outs_b = [], []
    for qq, kk, vv in inputs:
        outs_a.append(ca.decode_step(qq, kk, vv, mode=w.mode, budget=w.budget, recent=w.recent, window=w.window))
        ob = torch.empty_like(qq)
        cb.decode_step_overlap(qq, kk, vv, s_ev, mode=w.mode, budget=w.budget, recent=w.recent, window=w.window,
                               out=ob, workspace=ws_b, stream=s_att)
        outs_b.append(ob)
    assert cb.read_status(stream=s_att) == 0
    torch.cuda.synchronize()
    assert ca.read_status() == 0
    for oa, ob in zip(outs_a, outs_b):
        assert torch.equal(oa, ob)
    _same_state(ca, cb)
    for b in range(B):
        assert ca.lengths(b) == cb.lengths(b)
