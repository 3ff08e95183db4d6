"""Host side of the recipe cache modes turboquant25 / turboquant35 against the oracle
(oracle/recipe_oracle.py): row bytes, the metadata check and channel order ("vLLM Usage",
Metadata Validation Rules), the energy calibration ("Architecture", vLLM Runtime Mapping)
and the 1-bit codebook the 2-bit groups use.  No GPU work is launched."""

import numpy as np
import pytest

from oracle import recipe_oracle as ro
from oracle import tq_oracle as o

RECIPES = ["turboquant25", "turboquant35"]


@pytest.fixture(scope="module")
def tq():
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


@pytest.mark.parametrize("recipe", RECIPES)
@pytest.mark.parametrize("d", [64, 128])
def test_recipe_row_bytes_match_oracle(tq, recipe, d):
    assert tq.tq_recipe_row_bytes(recipe, d) == ro.recipe_row_bytes(recipe, d)


def test_recipe_row_bytes_worked_values_and_refusals(tq):
    # D 128: high group 64 channels, low group 64 (hand-worked in the oracle's pins)
    assert tq.tq_recipe_row_bytes("turboquant25", 128) == 56
    assert tq.tq_recipe_row_bytes("turboquant35", 128) == 72
    assert tq.lib().tq_recipe_row_bytes(30, 128) == -1  # no such recipe
    assert tq.lib().tq_recipe_row_bytes(25, 256) == -1  # no kernel at head_dim 256
    with pytest.raises(ValueError):
        tq.tq_recipe_row_bytes("turboquant45", 128)


@pytest.mark.parametrize("recipe", RECIPES)
def test_channel_order_matches_oracle(tq, recipe):
    rng = np.random.default_rng(4)
    d, h = 128, 5
    high = np.sort(np.stack([rng.choice(d, d // 2, replace=False) for _ in range(h)]), axis=1)
    got = tq.tq_recipe_channel_order(recipe, d, high).numpy()
    hi = ro.validate_high_groups(high, recipe, d, h)
    want = np.concatenate([hi, ro.low_groups(hi, d)], axis=1)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("case", ["unsorted", "repeated", "too_large", "negative"])
def test_channel_order_rejects_each_broken_rule(tq, case):
    d, h = 64, 2
    high = np.tile(np.arange(0, d, 2), (h, 1))  # valid: even channels
    if case == "unsorted":
        high[1, [3, 4]] = high[1, [4, 3]]
    elif case == "repeated":
        high[0, 5] = high[0, 4]
    elif case == "too_large":
        high[1, -1] = d
    else:
        high[0, 0] = -1
    with pytest.raises(ValueError):
        ro.validate_high_groups(high, "turboquant35", d, h)  # the oracle rejects it too
    with pytest.raises(tq.TQError) as e:
        tq.tq_recipe_channel_order("turboquant35", d, high)
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    msg = str(e.value)
    assert ("sorted and unique" in msg) if case in ("unsorted", "repeated") else ("outside" in msg)


@pytest.mark.parametrize("recipe", RECIPES)
def test_calibration_matches_oracle(tq, recipe):
    rng = np.random.default_rng(21)
    n, h, d = 200, 3, 64
    x = (rng.standard_normal((n, h, d)) * rng.lognormal(0.0, 0.7, (1, h, d))).astype(np.float32)
    got = tq.tq_recipe_calibrate(recipe, x).numpy()
    assert np.array_equal(got, ro.calibrate_high_groups(x.astype(np.float64), recipe))


def test_calibration_ties_go_to_the_lower_channel(tq):
    # integer samples: many channels of equal energy
    rng = np.random.default_rng(3)
    x = rng.integers(-2, 3, size=(6, 2, 32)).astype(np.float32)
    got = tq.tq_recipe_calibrate("turboquant25", x).numpy()
    assert np.array_equal(got, ro.calibrate_high_groups(x.astype(np.float64), "turboquant25"))


@pytest.mark.parametrize("d", [32, 64, 128])
def test_one_bit_codebook_matches_oracle(tq, d):
    c_lib = tq.tq_codebook(d, 1)[0].numpy()
    c_or = o.codebook_f32(d, 1)[0]
    assert np.all(np.abs(c_lib - c_or) <= np.spacing(np.abs(c_or)))
    assert c_lib[0] == -c_lib[1] and c_lib[1] > 0
