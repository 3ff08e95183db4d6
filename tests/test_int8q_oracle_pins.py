"""Pins of the INT8-query oracle (oracle/int8q_oracle.py) against what the arithmetic fixes:
a hand-worked row with ties, the half-step rounding bound, the full code range, the zero
row, fp32 decisions, and the reduction of the int8 prefill to the float prefill on the
dequantised query.  Planted mistakes (round half away from zero, a 128 divisor, a scale per
row instead of per (row, head)) each fail one of them."""

import numpy as np
import pytest

from oracle import int8q_oracle as iq
from oracle import tq_oracle as o


def test_hand_worked_row_with_ties():
    # amax 127 -> s = 1 exactly; -63.5, 0.5, 1.5, -0.5 are ties, which go to the even code
    q = np.array([[127.0, -63.5, 0.5, 1.5, -0.5, 2.5, 0.0, 3.25]], dtype=np.float32)
    codes, s = iq.quantize_queries_int8(q)
    assert s.tolist() == [1.0]
    assert codes.tolist() == [[127, -64, 0, 2, 0, 2, 0, 3]]


def test_rounding_bound_and_full_range():
    rng = np.random.default_rng(0)
    q = (rng.standard_normal((50, 8, 128)) * rng.lognormal(0, 2, (50, 8, 1))).astype(np.float32)
    codes, s = iq.quantize_queries_int8(q)
    assert codes.dtype == np.int8 and s.shape == (50, 8)
    assert np.all(np.abs(codes) <= 127)
    assert np.all(np.max(np.abs(codes.astype(np.int32)), axis=-1) == 127)  # the largest entry maps to +-127
    err = np.abs(q.astype(np.float64) - iq.dequantize_queries(codes, s))
    assert np.all(err <= 0.5 * s.astype(np.float64)[..., None] * (1 + 1e-6))
    # the scale is per (row, head): rescaling one head leaves the other heads' codes alone
    q2 = q.copy()
    q2[:, 3] *= 1000.0
    c2, _ = iq.quantize_queries_int8(q2)
    assert np.array_equal(np.delete(c2, 3, axis=1), np.delete(codes, 3, axis=1))


def test_zero_row_and_fp32_decisions():
    q = np.zeros((2, 3, 16), dtype=np.float32)
    q[1, 2, 5] = -3.0
    codes, s = iq.quantize_queries_int8(q)
    assert np.all(codes[0] == 0) and np.all(s[0] == 0)
    assert codes[1, 2, 5] == -127 and s[1, 2] == np.float32(3.0) / np.float32(127)
    # a ratio that rounds differently in fp32 and fp64: the fp32 quotient decides
    q = np.array([[1.0, 0.0]], dtype=np.float32)
    amax = np.float32(1.0)
    s32 = amax / np.float32(127)
    x = np.float32(s32 * np.float32(2.5))  # about 2.5 codes
    q[0, 1] = x
    codes, _ = iq.quantize_queries_int8(q)
    assert codes[0, 1] == np.rint(np.float32(x / s32))


def test_int8_prefill_is_the_float_prefill_of_the_dequantised_query():
    rng = np.random.default_rng(3)
    d, h, hq, bs = 64, 2, 4, 16
    lens = [20, 7]
    nblk = 4
    bt = np.array([[0, 1], [2, 3]], dtype=np.int32)
    signs = o.splitmix64_signs(d, 42)
    kc, vc = o.codebook_f32(d, 4)[0], o.codebook_f32(d, 2)[0]
    kp = np.zeros((nblk, bs, h, o.row_bytes(d, 4)), np.uint8)
    vp = np.zeros((nblk, bs, h, o.row_bytes(d, 2)), np.uint8)
    for b, n in enumerate(lens):
        slots = np.array([bt[b, t // bs] * bs + t % bs for t in range(n)], dtype=np.int64)
        kp = o.write_kv(rng.standard_normal((n, h, d)), kp, slots, signs, kc, 4)
        vp = o.write_kv(rng.standard_normal((n, h, d)), vp, slots, signs, vc, 2)
    q = rng.standard_normal((5, hq, d)).astype(np.float32)
    q_seq = np.array([0, 0, 0, 1, 1], dtype=np.int32)
    q_len = np.array([18, 19, 20, 6, 7], dtype=np.int32)
    codes, s = iq.quantize_queries_int8(q)
    got = iq.paged_prefill_int8q(codes, s, q_seq, q_len, kp, vp, 4, 2, bt, signs, kc, vc)
    want = o.paged_prefill(codes.astype(np.float64) * s[..., None], q_seq, q_len, kp, vp, 4, 2, bt, signs, kc, vc)
    assert np.array_equal(got, want)
    # and it stays close to the float query's attention (quantisation error only)
    flt = o.paged_prefill(q, q_seq, q_len, kp, vp, 4, 2, bt, signs, kc, vc)
    assert np.max(np.abs(got - flt)) < 0.05 * np.max(np.abs(flt))


def _pins_hold(quantize) -> bool:
    """The hand-worked row and the per-(row, head) scale, as checks of a quantiser."""
    q = np.array([[127.0, -63.5, 0.5, 1.5, -0.5, 2.5, 0.0, 3.25]], dtype=np.float32)
    codes, s = quantize(q)
    if s.tolist() != [1.0] or codes.tolist() != [[127, -64, 0, 2, 0, 2, 0, 3]]:
        return False
    rng = np.random.default_rng(1)
    x = rng.standard_normal((4, 3, 32)).astype(np.float32)
    c1, _ = quantize(x)
    x[:, 1] *= 50.0
    c2, _ = quantize(x)
    return np.array_equal(np.delete(c1, 1, axis=1), np.delete(c2, 1, axis=1))


@pytest.mark.parametrize("mistake", ["half_away", "divisor_128", "per_row_scale"])
def test_planted_mistakes_are_caught(mistake):
    def wrong(x):
        x32 = np.asarray(x, dtype=np.float32)
        amax = np.max(np.abs(x32), axis=-1)
        if mistake == "per_row_scale" and x32.ndim == 3:
            amax = np.broadcast_to(np.max(amax, axis=-1, keepdims=True), amax.shape)
        s = (amax / np.float32(128 if mistake == "divisor_128" else 127)).astype(np.float32)
        r = x32 / np.where(s > 0, s, 1)[..., None]
        c = np.sign(r) * np.floor(np.abs(r) + 0.5) if mistake == "half_away" else np.rint(r)
        return np.clip(c, -127, 127).astype(np.int8), s

    assert _pins_hold(iq.quantize_queries_int8)
    assert not _pins_hold(wrong)
