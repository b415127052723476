"""Per-layer budget schedules ("KV Cache optimization techniques" section 1.3,
PyramidKV linear decay; the eviction-and-reuse survey page's quadratic pyramid
ratio).  Values worked by hand from the pages' formulas at chosen layers, plus
the invariants each schedule fixes."""
import pytest

from compressed_kv_cache_kvc_gb300.budgets import pyramid_budgets


def test_linear_decay_worked_values():
    b = pyramid_budgets(48, "linear", recent=512, base=2457)
    # layer 0 keeps the base; layer 24 keeps 0.6 of it (1474.2 -> 1474);
    # layer 47 keeps 1 - 0.8 * 47/48 = 0.21666.. of it (532.35 -> 532)
    assert (b[0], b[24], b[47]) == (2457, 1474, 532)
    assert all(x >= y for x, y in zip(b, b[1:]))  # shallow layers keep more


def test_quadratic_pyramid_worked_values():
    b = pyramid_budgets(48, "quadratic", recent=512, context=8192, base_ratio=0.3)
    # 0.3 * 8192 = 2457.6; (0.3 + 0.7 * 0.25) * 8192 = 3891.2;
    # (0.3 + 0.7 * (47/48)^2) * 8192 = 7955.55
    assert (b[0], b[24], b[47]) == (2457, 3891, 7955)
    assert all(x <= y for x, y in zip(b, b[1:]))  # deep layers keep more


def test_truncation_follows_the_pages_floating_point():
    # the page computes int(base * (1.0 - 0.8 * i / L)) in double precision:
    # 1 - 0.8 * 0.75 = 0.3999999999999999, so 300 keeps 119 tokens, not 120
    assert pyramid_budgets(4, "linear", recent=32, base=300) == [300, 240, 180, 119]


def test_budgets_never_drop_below_sinks_and_recent():
    b = pyramid_budgets(10, "linear", recent=40, base=100)
    assert b[9] == 44  # 100 * (1 - 0.72) = 28 -> clamped to 4 + 40
    assert min(b) >= 44


def test_single_layer_is_the_base():
    assert pyramid_budgets(1, "linear", recent=8, base=77) == [77]
    assert pyramid_budgets(1, "quadratic", recent=8, context=1000, base_ratio=0.25) == [250]


@pytest.mark.parametrize("kw", [dict(kind="cubic", base=10), dict(kind="linear"), dict(kind="quadratic", context=10)])
def test_bad_arguments(kw):
    with pytest.raises(ValueError):
        pyramid_budgets(4, recent=0, **kw)
