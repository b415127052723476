"""Seeded synthetic inputs for the compressed-KV decode step.

This module holds no arithmetic of the method (no quantisation, attention,
scoring or selection): it only draws random bf16 tensors with the shapes and
value structure of the workloads, so that the CUDA path and the oracle can be
fed the same bits.  It imports neither of them.

Recipe (per workload, per layer, per step):
  * K, V, Q ~ N(0, 1), rounded to bf16 (round-to-nearest-even of fp32 bits);
  * K carries 4 outlier channels, drawn once per workload and shared by every
    head and layer, multiplied by 10;
  * planted heavy hitters: round(0.02 * T) positions per (sequence, KV head),
    uniform over 4..T-1, whose whole K row is 3 * qbar + N(0, 1), qbar being
    the mean of the first decode step's queries of that KV head's group;
  * ragged workloads draw each sequence's context uniformly in [lo, hi];
  * the pool's free-block order is a seeded permutation when the workload asks
    for shuffled block tables, else ascending.
Seeds: ``seed + 1009 * layer + 7919 * step`` (step 0 = prefill + first decode
step, whose query is drawn first so that the planted rows can use it).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

HEAD_DIM = 128
PAGE = 16


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    context: int            # fixed context, or the upper end of a ragged range
    bits: int               # 8 or 4
    mode: str               # "h2o" or "streaming"
    budget: int = 0         # kept tokens incl. the 4 sinks (h2o)
    recent: int = 0         # recent window kept by h2o
    window: int = 0         # streaming window
    layers: int = 1
    steps: int = 1
    seed: int = 0
    shuffled_blocks: bool = False
    context_lo: int = 0     # > 0: context ~ U[context_lo, context]
    head_dim: int = HEAD_DIM
    plant_frac: float = 0.02
    n_outlier: int = 4
    outlier_mult: float = 10.0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


# The five synthetic workloads: a tiny single layer; a LLaMA-7B-shaped MHA layer
# with scattered pages; a Llama-3-8B-shaped GQA layer with ragged contexts in
# StreamingLLM mode; a Qwen2.5-14B-shaped 48-layer INT4 stack; a long-context
# GQA stack run for 64 consecutive decode steps.  Budgets that the pages give
# as fractions of the context are floored (int()).
WORKLOADS = {
    "tiny_b1_h8_t512_int8_h2o": Workload(
        "tiny_b1_h8_t512_int8_h2o", batch=1, num_q_heads=8, num_kv_heads=8, context=512,
        bits=8, mode="h2o", budget=128, recent=32, seed=0),
    "llama7b_b16_h32_t4096_int8_h2o": Workload(
        "llama7b_b16_h32_t4096_int8_h2o", batch=16, num_q_heads=32, num_kv_heads=32,
        context=4096, bits=8, mode="h2o", budget=int(0.2 * 4096), recent=256, seed=1,
        shuffled_blocks=True),
    "llama3_8b_b64_gqa_ragged_int8_streaming": Workload(
        "llama3_8b_b64_gqa_ragged_int8_streaming", batch=64, num_q_heads=32, num_kv_heads=8,
        context=8192, context_lo=1024, bits=8, mode="streaming", window=2048, steps=16, seed=2),
    "qwen14b_b32_gqa5_t8192_int4_h2o_48l": Workload(
        "qwen14b_b32_gqa5_t8192_int4_h2o_48l", batch=32, num_q_heads=40, num_kv_heads=8,
        context=8192, bits=4, mode="h2o", budget=int(0.3 * 8192), recent=512, layers=48,
        seed=3),
    "longctx_b4_gqa4_t32768_int8_h2o_32l_64s": Workload(
        "longctx_b4_gqa4_t32768_int8_h2o_32l_64s", batch=4, num_q_heads=32, num_kv_heads=8,
        context=32768, bits=8, mode="h2o", budget=int(0.1 * 32768), recent=1024, layers=32,
        steps=64, seed=4),
}


# ---------------------------------------------------------------------------
# bf16 encoding of the drawn fp32 values (input encoding, not method arithmetic)
# ---------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def rng_for(w: Workload, layer: int, step: int) -> np.random.Generator:
    return np.random.default_rng(w.seed + 1009 * layer + 7919 * step)


def outlier_channels(w: Workload) -> np.ndarray:
    return np.sort(np.random.default_rng(w.seed).choice(w.head_dim, w.n_outlier, replace=False))


def context_lengths(w: Workload) -> np.ndarray:
    """Prefill length per sequence."""
    if w.context_lo > 0:
        r = np.random.default_rng(w.seed + 77)
        return r.integers(w.context_lo, w.context + 1, size=w.batch).astype(np.int64)
    return np.full(w.batch, w.context, dtype=np.int64)


def block_order(w: Workload, num_blocks: int) -> np.ndarray:
    """Order in which the pool hands out blocks (a seeded permutation when the
    workload scatters its pages)."""
    if w.shuffled_blocks:
        return np.random.default_rng(w.seed + 31337).permutation(num_blocks).astype(np.int32)
    return np.arange(num_blocks, dtype=np.int32)


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def gen_layer(w: Workload, layer: int, context: int | None = None,
              batch: int | None = None) -> dict:
    """Prefill K/V and the first decode step (step 0) of one layer.

    Returns bf16 bit arrays: ``q`` [B, Hq, D] (step-0 query), ``k``/``v``
    [B, Hkv, T, D] prefill (T = max context; a sequence with a shorter
    ``lengths[b]`` uses the prefix), ``k_new``/``v_new`` [B, Hkv, 1, D] (the
    token appended at step 0), ``lengths`` [B], and ``planted`` (bool
    [B, Hkv, T]).
    """
    B = w.batch if batch is None else batch
    T = int(w.context if context is None else context)
    D, Hq, Hkv, G = w.head_dim, w.num_q_heads, w.num_kv_heads, w.group
    rng = rng_for(w, layer, 0)
    q = bf16_bits(_normal(rng, (B, Hq, D)))
    qf = bf16_to_f32(q)
    k = _normal(rng, (B, Hkv, T, D))
    k[..., outlier_channels(w)] *= np.float32(w.outlier_mult)
    v = _normal(rng, (B, Hkv, T, D))
    planted = np.zeros((B, Hkv, T), dtype=bool)
    n_plant = int(round(w.plant_frac * T))
    if n_plant > 0 and T > 4:
        qbar = qf.reshape(B, Hkv, G, D).mean(axis=2)
        for b in range(B):
            for h in range(Hkv):
                idx = rng.choice(np.arange(4, T), size=min(n_plant, T - 4), replace=False)
                planted[b, h, idx] = True
                k[b, h, idx] = np.float32(3.0) * qbar[b, h] + _normal(rng, (idx.size, D))
    k_new = _normal(rng, (B, Hkv, 1, D))
    k_new[..., outlier_channels(w)] *= np.float32(w.outlier_mult)
    v_new = _normal(rng, (B, Hkv, 1, D))
    lengths = context_lengths(w)[:B] if context is None else np.full(B, T, np.int64)
    return dict(q=q, k=bf16_bits(k), v=bf16_bits(v), k_new=bf16_bits(k_new),
                v_new=bf16_bits(v_new), lengths=lengths, planted=planted)


def gen_step(w: Workload, layer: int, step: int, batch: int | None = None) -> dict:
    """Fresh query and appended token of decode step ``step`` >= 1."""
    B = w.batch if batch is None else batch
    D, Hq, Hkv = w.head_dim, w.num_q_heads, w.num_kv_heads
    rng = rng_for(w, layer, step)
    q = _normal(rng, (B, Hq, D))
    k_new = _normal(rng, (B, Hkv, 1, D))
    k_new[..., outlier_channels(w)] *= np.float32(w.outlier_mult)
    v_new = _normal(rng, (B, Hkv, 1, D))
    return dict(q=bf16_bits(q), k_new=bf16_bits(k_new), v_new=bf16_bits(v_new))


def gen_layer_torch(w: Workload, layer: int, device, batch: int | None = None):
    """Device-side draw of the same recipe for bench-scale stacks (tens of GB of
    prefill would take minutes through numpy).  Uses torch's seeded device
    generator, so the values differ from ``gen_layer``'s but follow the same
    distribution.  Returns bf16 tensors q, k, v, k_new, v_new."""
    import torch
    B = w.batch if batch is None else batch
    T, D, Hq, Hkv, G = w.context, w.head_dim, w.num_q_heads, w.num_kv_heads, w.group
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 1009 * layer)
    q = torch.randn(B, Hq, D, generator=g, device=device).to(torch.bfloat16)
    k = torch.randn(B, Hkv, T, D, generator=g, device=device)
    oc = torch.as_tensor(outlier_channels(w), device=device)
    k[..., oc] *= w.outlier_mult
    v = torch.randn(B, Hkv, T, D, generator=g, device=device).to(torch.bfloat16)
    n_plant = int(round(w.plant_frac * T))
    if n_plant > 0 and T > 4:
        qbar = q.float().view(B, Hkv, G, D).mean(dim=2)
        scores = torch.rand(B, Hkv, T - 4, generator=g, device=device)
        idx = scores.topk(n_plant, dim=-1).indices + 4
        noise = torch.randn(B, Hkv, n_plant, D, generator=g, device=device)
        rows = 3.0 * qbar[:, :, None, :] + noise
        k.scatter_(2, idx[..., None].expand(B, Hkv, n_plant, D), rows)
    k = k.to(torch.bfloat16)
    k_new = torch.randn(B, Hkv, 1, D, generator=g, device=device)
    k_new[..., oc] *= w.outlier_mult
    v_new = torch.randn(B, Hkv, 1, D, generator=g, device=device)
    return q, k, v, k_new.to(torch.bfloat16), v_new.to(torch.bfloat16)


def gen_step_torch(w: Workload, layer: int, step: int, device, batch: int | None = None):
    import torch
    B = w.batch if batch is None else batch
    D, Hq, Hkv = w.head_dim, w.num_q_heads, w.num_kv_heads
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 1009 * layer + 7919 * step)
    q = torch.randn(B, Hq, D, generator=g, device=device)
    k_new = torch.randn(B, Hkv, 1, D, generator=g, device=device)
    oc = torch.as_tensor(outlier_channels(w), device=device)
    k_new[..., oc] *= w.outlier_mult
    v_new = torch.randn(B, Hkv, 1, D, generator=g, device=device)
    return q.to(torch.bfloat16), k_new.to(torch.bfloat16), v_new.to(torch.bfloat16)
