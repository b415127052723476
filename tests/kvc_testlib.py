"""Helpers shared by the GPU parity tests: read the library's device state back
into per-(sequence, KV head) arrays, drive the oracle on the same inputs, and
compare with the tolerances the tests state."""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import kvc_oracle as O

ATOL = 2e-3   # attention outputs: |gpu - ref| <= ATOL + RTOL * |ref|
RTOL = 1e-2
TIE_REL = 1e-5  # selection differences allowed only within this of the k-th score


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_tensor_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


class StateView:
    """Host copy of one cache's device state."""

    def __init__(self, cache):
        torch.cuda.synchronize()
        nb, hkv = cache.num_blocks, cache.num_kv_heads
        rb = 128 * cache.bits // 8

        def get(name, dt):
            return cache.buffer(name).cpu().numpy().view(dt)

        self.bits = cache.bits
        self.hkv = hkv
        self.kc = get("K_CODES", np.uint8).reshape(nb, hkv, 16, rb)
        self.vc = get("V_CODES", np.uint8).reshape(nb, hkv, 16, rb)
        self.ks = get("K_SCALE", np.float32).reshape(nb, hkv, 16)
        self.vs = get("V_SCALE", np.float32).reshape(nb, hkv, 16)
        self.pos = get("SLOT_POS", np.int32).reshape(nb, hkv, 16)
        self.score = get("SCORE", np.float32).reshape(nb, hkv, 16)
        self.sink_k = get("SINK_K", np.uint16).reshape(cache.max_batch, hkv, 4, 128)
        self.sink_v = get("SINK_V", np.uint16).reshape(cache.max_batch, hkv, 4, 128)
        self.sink_score = get("SINK_SCORE", np.float32).reshape(cache.max_batch, hkv, 4)
        self.bt = get("BLOCK_TABLE", np.int32).reshape(cache.max_batch, cache.max_blocks_per_seq)
        self.slots = get("SEQ_SLOTS", np.int32)
        self.seen = get("SEQ_POS", np.int32)
        self.free_stack = get("FREE_STACK", np.int32)
        self.counters = get("COUNTERS", np.int32)
        self.num_blocks = nb
        self.W = getattr(cache, "bf16_window", 0)
        if self.W > 0:
            self.ring_k = get("RING_K", np.uint16).reshape(cache.max_batch, hkv, self.W, 128)
            self.ring_v = get("RING_V", np.uint16).reshape(cache.max_batch, hkv, self.W, 128)
            self.ring_score = get("RING_SCORE", np.float32).reshape(cache.max_batch, hkv, self.W)

    def ring_head(self, b, h):
        """(positions, K bf16 bits, V bf16 bits, scores) of the bf16 window of
        (b, h), in position order: positions P - n .. P - 1 at ring slot
        (position - 4) mod W."""
        P = int(self.seen[b])
        n = min(self.W, max(0, P - 4))
        p = np.arange(P - n, P)
        r = (p - 4) % self.W
        return p, self.ring_k[b, h, r], self.ring_v[b, h, r], self.ring_score[b, h, r]

    def codes(self, raw):
        if self.bits == 8:
            return raw.view(np.int8)
        return O.unpack_int4(raw)

    def head(self, b, h):
        """(pos, kcodes, kscale, vcodes, vscale, score) in slot order."""
        S = int(self.slots[b])
        t = np.arange(S)
        blk = self.bt[b, t // 16]
        off = t % 16
        return (self.pos[blk, h, off].astype(np.int64), self.codes(self.kc[blk, h, off]), self.ks[blk, h, off],
                self.codes(self.vc[blk, h, off]), self.vs[blk, h, off], self.score[blk, h, off])

    def used_blocks(self, b):
        return self.bt[b, :(int(self.slots[b]) + 15) // 16]


def oracle_from_inputs(w_or_shape, bits, k_bits, v_bits, lengths):
    """Oracle cache filled with the prefill of each sequence (k/v bf16 bits
    [B, Hkv, T, D], sequence b uses its first lengths[b] tokens)."""
    B, Hkv = k_bits.shape[0], k_bits.shape[1]
    hq = w_or_shape
    c = O.OracleCache(B, hq, Hkv, bits)
    for b in range(B):
        n = int(lengths[b])
        c.append(b, O.bf16_bits_to_f32(k_bits[b, :, :n]), O.bf16_bits_to_f32(v_bits[b, :, :n]))
    return c


def check_codes(state: StateView, oracle: O.OracleCache, b: int, h: int):
    """Codes, scales and positions of (b, h) equal the oracle's bit for bit."""
    pos, kc, ks, vc, vs, _ = state.head(b, h)
    hs = oracle.seqs[b].heads[h]
    order = np.argsort(pos)
    oorder = np.argsort(hs.pos)
    assert np.array_equal(pos[order], hs.pos[oorder]), f"positions differ at ({b},{h})"
    assert np.array_equal(kc[order], hs.kcodes[oorder]), f"K codes differ at ({b},{h})"
    assert np.array_equal(vc[order], hs.vcodes[oorder]), f"V codes differ at ({b},{h})"
    assert np.array_equal(ks[order].view(np.uint32), hs.kscale[oorder].view(np.uint32)), f"K scales ({b},{h})"
    assert np.array_equal(vs[order].view(np.uint32), hs.vscale[oorder].view(np.uint32)), f"V scales ({b},{h})"
    s = oracle.seqs[b]
    ns = s.sink_k[h].shape[0]
    sk = O.bf16_bits_to_f32(state.sink_k[b, h, :ns])
    sv = O.bf16_bits_to_f32(state.sink_v[b, h, :ns])
    assert np.array_equal(sk, s.sink_k[h]) and np.array_equal(sv, s.sink_v[h]), f"sinks differ at ({b},{h})"


def assert_attention_close(gpu: np.ndarray, ref: np.ndarray, what=""):
    err = np.abs(gpu.astype(np.float64) - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside 2e-3 + 1e-2|ref|; "
                           f"max abs err {err.max():.3e}, max rel {(err / np.maximum(np.abs(ref), 1e-30)).max():.3e}")
    return float(err.max())


def load_oracle_from_state(oracle: O.OracleCache, state: StateView, b: int):
    """Lock-step resync: the oracle's (b, *) state := the GPU's."""
    for h in range(state.hkv):
        pos, kc, ks, vc, vs, sc = state.head(b, h)
        oracle.load_head(b, h, pos, kc, ks, vc, vs, sc.astype(np.float64))
        ns = oracle.seqs[b].sink_k[h].shape[0]
        oracle.seqs[b].sink_score[h] = state.sink_score[b, h, :ns].astype(np.float64)


def kept_sets_agree(gpu_pos: set, ora_pos: set, pos: np.ndarray, score: np.ndarray, n_heavy: int,
                    thr: int) -> bool:
    """Equal, or different only among candidates whose score lies within
    TIE_REL of the k-th candidate score (ties broken by the lower position)."""
    if gpu_pos == ora_pos:
        return True
    if len(gpu_pos) != len(ora_pos):
        return False
    cand = pos < thr
    cs = np.sort(score[cand])[::-1]
    if n_heavy <= 0 or n_heavy > cs.size:
        return False
    kth = cs[n_heavy - 1]
    sd = gpu_pos ^ ora_pos
    by_pos = dict(zip(pos.tolist(), score.tolist()))
    return all(abs(by_pos[p] - kth) <= TIE_REL * max(abs(kth), 1e-30) for p in sd)


def sm_scale():
    return 1.0 / math.sqrt(128)
