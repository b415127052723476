"""Per-layer token budgets (PyramidKV-style schedules) for the H2O selection.

The kernels take the budget per call, so a per-layer schedule is host policy:
compute one budget per layer here and pass it to that layer's
`decode_step` / `h2o_select_evict`.

Two schedules appear on the pages, in opposite directions:

* "linear" ("KV Cache optimization techniques", section 1.3, PyramidKV): the
  cache of layer i keeps base * (1 - 0.8 * i / L) tokens, truncated to an
  integer, so shallow layers keep more and the deepest keeps ~0.2 of the base.
* "quadratic" (the eviction-and-reuse survey page, the pyramid ratio of its
  block manager): layer i retains the fraction rho + (1 - rho) * (i / L)^2 of
  the context, so deep layers keep more.  The page fixes L = 80; here L is the
  model's own layer count.

Either way a budget never drops below the 4 sinks plus the recent window,
which the selection always keeps.
"""
from __future__ import annotations

import math

SINKS = 4


def pyramid_budgets(num_layers: int, kind: str, recent: int, base: int | None = None,
                    context: int | None = None, base_ratio: float | None = None) -> list[int]:
    """Token budget (sinks included) of every layer.

    kind="linear":    budget_i = floor(base * (1 - 0.8 * i / num_layers))
    kind="quadratic": budget_i = floor(context * (base_ratio + (1 - base_ratio) * (i / num_layers) ** 2))
    Both are clamped below at 4 + recent.
    """
    if num_layers < 1:
        raise ValueError("num_layers must be >= 1")
    if recent < 0:
        raise ValueError("recent must be >= 0")
    floor_budget = SINKS + recent
    out = []
    for i in range(num_layers):
        if kind == "linear":
            if base is None or base < 1:
                raise ValueError("linear schedule needs base >= 1")
            b = math.floor(base * (1.0 - 0.8 * (i / num_layers)))
        elif kind == "quadratic":
            if context is None or context < 1 or base_ratio is None or not 0.0 < base_ratio <= 1.0:
                raise ValueError("quadratic schedule needs context >= 1 and 0 < base_ratio <= 1")
            b = math.floor(context * (base_ratio + (1.0 - base_ratio) * (i / num_layers) ** 2))
        else:
            raise ValueError(f"unknown schedule {kind!r}")
        out.append(max(floor_budget, b))
    return out
