"""Pins of the recipe-mode (turboquant25 / turboquant35) oracle against what the names, the
metadata rules and the mathematics fix: the mean bits the names state, the row bytes
worked by hand, each metadata rule, calibration by brute force over channel subsets,
closed forms of a row whose low group is empty, unbiased scores and reconstructions over
sketch draws, and the decode equal to dense attention on the reconstruction."""

import itertools
import math

import numpy as np
import pytest

from oracle import qjl_oracle as qo
from oracle import recipe_oracle as ro
from oracle import tq_oracle as o


@pytest.mark.parametrize("recipe,mean", [("turboquant25", 2.5), ("turboquant35", 3.5)])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_group_bits_average_to_the_recipe_name(recipe, mean, d):
    bh, bl = ro.recipe_bits(recipe)
    n_hi = ro.high_group_count(recipe, d)
    assert (n_hi * bh + (d - n_hi) * bl) / d == mean
    assert bh == bl + 1


def test_unknown_recipe_and_odd_head_dim_raise():
    with pytest.raises(ValueError):
        ro.recipe_bits("turboquant45")
    with pytest.raises(ValueError):
        ro.high_group_count("turboquant25", 7)


def test_row_bytes_worked_by_hand():
    # D = 128, groups of 64 channels.  turboquant25: high 3 bits = 2-bit indices (16 B) + 64
    # sign bits (8 B) + nu, gamma (8 B) = 32 B; low 2 bits = 1-bit indices (8 B) + 8 + 8 = 24 B
    assert ro.recipe_row_bytes("turboquant25", 128) == 32 + 24 == 56
    # turboquant35: high 4 bits = 3-bit indices (24 B) + 16 = 40 B; low 3 bits = 32 B
    assert ro.recipe_row_bytes("turboquant35", 128) == 40 + 32 == 72
    assert ro.recipe_row_bytes("turboquant25", 64) == (8 + 4 + 8) + (4 + 4 + 8)


def test_metadata_rules_each_raise():
    d, h = 16, 2
    good = np.array([[0, 2, 4, 6, 8, 10, 12, 14], [1, 3, 5, 7, 9, 11, 13, 15]])
    assert np.array_equal(ro.validate_high_groups(good, "turboquant35", d, h), good)
    bad = {
        "head count": good[:1],
        "integers": good.astype(np.float64),
        "group count": good[:, :7],
        "range high": np.array([[0, 2, 4, 6, 8, 10, 12, 16], good[1]]),
        "range low": np.array([[-1, 2, 4, 6, 8, 10, 12, 14], good[1]]),
        "sorted": np.array([[2, 0, 4, 6, 8, 10, 12, 14], good[1]]),
        "unique": np.array([[0, 2, 2, 6, 8, 10, 12, 14], good[1]]),
    }
    for name, arr in bad.items():
        with pytest.raises(ValueError):
            ro.validate_high_groups(arr, "turboquant35", d, h)
    low = ro.low_groups(good, d)
    assert np.array_equal(low, good[::-1])
    for k in range(h):
        assert sorted(set(good[k]) | set(low[k])) == list(range(d))


def test_calibration_is_the_max_energy_subset():
    # brute force over every 4-channel subset of 8 channels, per kv head
    rng = np.random.default_rng(21)
    x = rng.standard_normal((50, 3, 8)) * rng.lognormal(0.0, 1.0, (1, 3, 8))
    got = ro.calibrate_high_groups(x, "turboquant25")
    energy = np.sum(x * x, axis=0)
    for k in range(3):
        best = max(itertools.combinations(range(8), 4), key=lambda s: sum(energy[k, list(s)]))
        assert tuple(got[k]) == best
    # equal energies: the lower channels win
    flat = np.ones((5, 1, 8))
    assert list(ro.calibrate_high_groups(flat, "turboquant35")[0]) == [0, 1, 2, 3]


def test_row_with_an_empty_low_group_has_closed_forms():
    # x lives on the high channels only: the low group has nu = 0, every index at the lower
    # middle centroid c_m, residual r = -c_m (1, ..., 1), gamma = |c_m| sqrt(d), and sign bit
    # i = [sum_j S[i][j] |c_m| >= 0] = [row sum i of S >= 0]
    recipe, d = "turboquant25", 32
    codec = ro.RecipeCodec(recipe, d)
    rng = np.random.default_rng(22)
    high = np.sort(rng.permutation(d)[:d // 2])
    low = ro.low_groups(high[None], d)[0]
    x = np.zeros((3, d))
    x[:, high] = rng.standard_normal((3, d // 2)) * 2.0
    rows = ro.encode_recipe_rows(x, high, low, codec)
    nh, _ = codec.group_bytes()
    idx_h, _, nu_h, _ = qo.unpack_prod_rows(rows[:, :nh], codec.d, codec.bits[0])
    idx_l, z_l, nu_l, g_l = qo.unpack_prod_rows(rows[:, nh:], codec.d, codec.bits[1])
    assert np.array_equal(nu_h, np.linalg.norm(x, axis=1).astype(np.float32))
    assert np.all(nu_l == 0.0)
    c_lo = codec.mse[1].astype(np.float64)
    mid = len(c_lo) // 2 - 1
    assert np.all(idx_l == mid)
    assert np.allclose(g_l, abs(c_lo[mid]) * math.sqrt(codec.d), rtol=1e-7)
    assert np.array_equal(z_l, np.broadcast_to((codec.smat.sum(axis=1) >= 0).astype(np.int64), z_l.shape))
    # the high group's indices are the MSE indices of the gathered channels at bits - 1
    want, _, _ = o.encode_rows(x[:, high], codec.rot, codec.mse[0])
    assert np.array_equal(idx_h, want)


def _draws(recipe, d, x, q, high, low, draws):
    est = np.empty(draws)
    rec = np.empty((draws, d))
    for k in range(draws):
        codec = ro.RecipeCodec(recipe, d, smat=qo.normal_matrix(d // 2, d // 2, 5000 + k))
        rows = ro.encode_recipe_rows(x[None], high, low, codec)
        est[k] = ro.recipe_scores(q[None], rows, high, low, codec)[0, 0]
        rec[k] = ro.recipe_dequant(rows, high, low, codec)[0]
    return est, rec


@pytest.mark.parametrize("recipe", ["turboquant25", "turboquant35"])
def test_scores_and_reconstruction_are_unbiased_over_sketch_draws(recipe):
    d, draws = 32, 1500
    rng = np.random.default_rng(23)
    x = rng.standard_normal(d) * rng.lognormal(0.0, 0.7, d)
    q = rng.standard_normal(d)
    high = ro.calibrate_high_groups(x[None, None, :], recipe)[0]
    low = ro.low_groups(high[None], d)[0]
    est, rec = _draws(recipe, d, x, q, high, low, draws)
    truth = float(q @ x)  # the stored norms are fp32: their rounding sits inside the 1e-6 term
    assert abs(est.mean() - truth) < 5.0 * est.std() / math.sqrt(draws) + 1e-6 * abs(truth)
    sd = rec.std(axis=0) / math.sqrt(draws)
    assert np.all(np.abs(rec.mean(axis=0) - x) < 5.0 * sd + 1e-6 * np.abs(x) + 1e-12)


def test_scores_equal_inner_products_with_the_reconstruction():
    d = 64
    rng = np.random.default_rng(24)
    for recipe in ro.RECIPES:
        codec = ro.RecipeCodec(recipe, d)
        high = np.sort(rng.permutation(d)[:d // 2])
        low = ro.low_groups(high[None], d)[0]
        x = rng.standard_normal((9, d))
        q = rng.standard_normal((4, d))
        rows = ro.encode_recipe_rows(x, high, low, codec)
        s = ro.recipe_scores(q, rows, high, low, codec)
        assert np.max(np.abs(s - q @ ro.recipe_dequant(rows, high, low, codec).T)) < 1e-10


def test_more_bits_and_calibrated_groups_lower_the_error():
    # half the channels carry 4x the scale.  With those in the high group (as calibration
    # puts them) the error is lower than with the groups swapped, and turboquant35 beats
    # turboquant25
    d, n = 64, 400
    rng = np.random.default_rng(25)
    loud = np.sort(rng.permutation(d)[:d // 2])
    scale = np.ones(d)
    scale[loud] = 4.0
    x = rng.standard_normal((n, d)) * scale
    err = {}
    for recipe in ro.RECIPES:
        codec = ro.RecipeCodec(recipe, d)
        high = ro.calibrate_high_groups(x[:, None, :], recipe)[0]
        assert np.array_equal(high, loud)
        for name, hi in (("calibrated", high), ("swapped", ro.low_groups(high[None], d)[0])):
            lo = ro.low_groups(hi[None], d)[0]
            xh = ro.recipe_dequant(ro.encode_recipe_rows(x, hi, lo, codec), hi, lo, codec)
            err[recipe, name] = float(np.mean(np.sum((xh - x) ** 2, axis=1) / np.sum(x * x, axis=1)))
    for recipe in ro.RECIPES:
        assert err[recipe, "calibrated"] < 0.8 * err[recipe, "swapped"]
    assert err["turboquant35", "calibrated"] < 0.6 * err["turboquant25", "calibrated"]


def test_write_skips_negative_slots_and_refuses_out_of_range():
    recipe, d, h, bs, nb = "turboquant35", 32, 2, 4, 3
    codec = ro.RecipeCodec(recipe, d)
    rng = np.random.default_rng(26)
    high = np.stack([np.sort(rng.permutation(d)[:d // 2]) for _ in range(h)])
    raw = rng.standard_normal((5, h, d))
    pages = np.full((nb, bs, h, ro.recipe_row_bytes(recipe, d)), 0x5A, dtype=np.uint8)
    slots = np.array([3, -1, 0, 11, -1])
    out = ro.write_recipe_kv(raw, pages, slots, high, codec)
    flat = out.reshape(nb * bs, h, -1)
    for t, s in enumerate(slots):
        if s >= 0:
            for k in range(h):
                lo = ro.low_groups(high[k:k + 1], d)[0]
                assert np.array_equal(flat[s, k], ro.encode_recipe_rows(raw[t:t + 1, k], high[k], lo, codec)[0])
    untouched = np.setdiff1d(np.arange(nb * bs), slots[slots >= 0])
    assert np.all(flat[untouched] == 0x5A)
    with pytest.raises(IndexError):
        ro.write_recipe_kv(raw, pages, np.array([3, -1, 0, 12, -1]), high, codec)


def test_decode_is_dense_attention_on_the_reconstruction():
    recipe, d, h, hq, bs = "turboquant25", 32, 2, 4, 4
    codec = ro.RecipeCodec(recipe, d)
    rng = np.random.default_rng(27)
    lens = np.array([7, 5, 0])
    bt = np.array([[3, 0], [1, 4], [2, 2]], dtype=np.int32)
    nb = 5
    kraw = rng.standard_normal((nb * bs, h, d)) * rng.lognormal(0.0, 0.5, d)
    vraw = rng.standard_normal((nb * bs, h, d))
    high = ro.calibrate_high_groups(kraw, recipe)
    rb = ro.recipe_row_bytes(recipe, d)
    empty = np.zeros((nb, bs, h, rb), dtype=np.uint8)
    kp = ro.write_recipe_kv(kraw, empty, np.arange(nb * bs), high, codec)
    vp = ro.write_recipe_kv(vraw, empty, np.arange(nb * bs), high, codec)
    q = rng.standard_normal((3, hq, d))
    got = ro.paged_decode_recipe(q, kp, vp, bt, lens, high, codec)
    for b in range(3):
        for j in range(hq):
            k = j // (hq // h)
            n = int(lens[b])
            if n == 0:
                assert np.all(got[b, j] == 0.0)
                continue
            slot = bt[b, np.arange(n) // bs] * bs + np.arange(n) % bs
            lo = ro.low_groups(high[k:k + 1], d)[0]
            kh = ro.recipe_dequant(kp.reshape(nb * bs, h, rb)[slot, k], high[k], lo, codec)
            vh = ro.recipe_dequant(vp.reshape(nb * bs, h, rb)[slot, k], high[k], lo, codec)
            sc = (q[b, j] @ kh.T) / math.sqrt(d)
            p = np.exp(sc - sc.max())
            p /= p.sum()
            assert np.max(np.abs(got[b, j] - p @ vh)) < 1e-12
    # a block id past the pages: its tokens are left out
    bad = bt.copy()
    bad[0, 1] = nb + 2
    got_bad = ro.paged_decode_recipe(q, kp, vp, bad, lens, high, codec)
    trimmed = ro.paged_decode_recipe(q, kp, vp, bt, np.array([4, 5, 0]), high, codec)
    assert np.max(np.abs(got_bad - trimmed)) < 1e-12
