"""Pins of the product-quantised ("QJL residual") key-row oracle against what the
mathematics fixes: the published generator vector, the Box-Muller definition and the
normal law, the row layout, the exact residual, the unbiasedness of the inner-product
estimate and its closed-form variance, and the reduction to the MSE decode when the
sketch term is dropped."""

import math

import numpy as np
import pytest
from scipy import stats

from conftest import read_golden_rows
from oracle import qjl_oracle as qo
from oracle import tq_oracle as o


def test_stream_is_the_published_splitmix64():
    want = [int(v) for v in read_golden_rows("splitmix64_seed1234567.txt")]
    assert qo.splitmix64_stream(1234567, 5) == want


def test_normal_pair_is_box_muller_of_the_first_two_outputs():
    z1, z2 = [int(v) for v in read_golden_rows("splitmix64_seed1234567.txt")][:2]
    u1 = ((z1 >> 11) + 1) / 2.0 ** 53
    u2 = (z2 >> 11) / 2.0 ** 53
    r = math.sqrt(-2.0 * math.log(u1))
    got = qo.normal_matrix(1, 2, 1234567)[0]
    assert got[0] == pytest.approx(r * math.cos(2 * math.pi * u2), rel=0, abs=1e-15)
    assert got[1] == pytest.approx(r * math.sin(2 * math.pi * u2), rel=0, abs=1e-15)
    # odd count: the last pair is cut after its first number, same stream
    assert np.array_equal(qo.normal_matrix(1, 3, 5)[0], qo.normal_matrix(1, 4, 5)[0, :3])


def test_normal_matrix_follows_the_standard_normal_law():
    s = qo.normal_matrix(128, 128, 43).ravel()
    n = s.size
    assert abs(s.mean()) < 4.0 / math.sqrt(n)
    assert abs(s.var() - 1.0) < 4.0 * math.sqrt(2.0 / n)
    assert stats.kstest(s, "norm").pvalue > 1e-3
    assert np.array_equal(qo.normal_matrix(16, 16, 43), qo.normal_matrix(16, 16, 43))
    assert not np.array_equal(qo.normal_matrix(16, 16, 43), qo.normal_matrix(16, 16, 44))


@pytest.mark.parametrize("bits,rb", [(2, 40), (3, 56), (4, 72), (5, 88)])
def test_prod_row_bytes_at_d128(bits, rb):
    # (bits - 1)-bit indices + one sign bit per coordinate + two fp32 norms
    assert qo.prod_row_bytes(128, bits) == rb


def test_pack_layout_hand_worked_and_round_trip():
    # D = 16, 3 bits: 2-bit indices (4 bytes), 16 sign bits (2 bytes), nu, gamma
    idx = np.array([[3, 0, 1, 2] * 4])
    z = np.array([[1, 0, 0, 0, 0, 0, 0, 0, 1, 1, 1, 1, 0, 0, 0, 1]])
    row = qo.pack_prod_rows(idx, z, np.array([1.0]), np.array([0.5]), 3)[0]
    assert row.size == qo.prod_row_bytes(16, 3) == 14
    # indices 3,0,1,2 LSB-first at 2 bits: 0b10_01_00_11 = 0x93
    assert list(row[:4]) == [0x93] * 4
    assert list(row[4:6]) == [0x01, 0x8F]
    assert list(row[6:10]) == [0x00, 0x00, 0x80, 0x3F]  # fp32 1.0
    assert list(row[10:14]) == [0x00, 0x00, 0x00, 0x3F]  # fp32 0.5
    rng = np.random.default_rng(3)
    for bits in (2, 3, 4, 5):
        d = 64
        idx = rng.integers(0, 1 << (bits - 1), size=(9, d))
        z = rng.integers(0, 2, size=(9, d))
        nu = rng.random(9).astype(np.float32)
        g = rng.random(9).astype(np.float32)
        back = qo.unpack_prod_rows(qo.pack_prod_rows(idx, z, nu, g, bits), d, bits)
        assert np.array_equal(back[0], idx) and np.array_equal(back[1], z)
        assert np.array_equal(back[2], nu) and np.array_equal(back[3], g)


def _setup(d, bits, seed=42, sseed=43):
    signs = o.splitmix64_signs(d, seed)
    rot = o.rotation_matrix(signs)
    c, _ = o.codebook_f32(d, bits - 1)
    return signs, rot, c, qo.normal_matrix(d, d, sseed)


def test_residual_reconstructs_the_row_exactly():
    d, bits = 64, 4
    _, rot, c, smat = _setup(d, bits)
    x = np.random.default_rng(5).standard_normal((7, d)) * 3.0
    enc = qo.encode_prod(x, rot, c, smat)
    nu = np.linalg.norm(x, axis=1)
    rebuilt = (c.astype(np.float64)[enc["idx"]] + enc["residual"]) @ rot * nu[:, None]
    assert np.max(np.abs(rebuilt - x)) < 1e-12
    assert np.allclose(enc["gamma"], np.linalg.norm(enc["residual"], axis=1), rtol=1e-7)
    # the residual is what the MSE codebook misses: no other centroid is closer per coordinate
    y = enc["residual"] + c.astype(np.float64)[enc["idx"]]
    assert np.all(np.abs(enc["residual"]) <= np.min(np.abs(y[..., None] - c[None, None, :]), axis=2) + 1e-15)


def _estimates_over_sketches(d, bits, x, q, draws):
    _, rot, c, _ = _setup(d, bits)
    est = np.empty(draws)
    for k in range(draws):
        smat = qo.normal_matrix(d, d, 1000 + k)
        enc = qo.encode_prod(x[None], rot, c, smat)
        rows = qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], enc["gamma"], bits)
        est[k] = qo.prod_scores(q[None], rows, d, bits, rot, c, smat)[0, 0]
    return est, enc, rot, c


def test_inner_product_estimate_is_unbiased_with_the_closed_form_variance():
    # over draws of S: mean -> <q, x>; variance -> (pi/2)/D (nu gamma)^2 (|qt|^2 - (2/pi) <qt, r/|r|>^2)
    d, bits, draws = 32, 3, 2500
    rng = np.random.default_rng(11)
    x = rng.standard_normal(d) * 2.0
    q = rng.standard_normal(d)
    est, enc, rot, c = _estimates_over_sketches(d, bits, x, q, draws)
    nu = float(enc["nu"][0])
    r = enc["residual"][0]
    gamma = float(np.linalg.norm(r))
    qt = rot @ q
    var = (math.pi / 2) / d * (nu * gamma) ** 2 * (qt @ qt - (2 / math.pi) * (qt @ (r / gamma)) ** 2)
    truth = float(q @ x)  # the stored norms are fp32: their rounding is inside the 1e-6 term
    assert abs(est.mean() - truth) < 5.0 * math.sqrt(var / draws) + 1e-6 * abs(truth)
    assert est.var() == pytest.approx(var, rel=0.15)


def test_mse_part_alone_is_biased_and_the_sketch_removes_it():
    # the MSE reconstruction shrinks inner products (E[ratio] < 1); the product estimate
    # averaged over sketch draws does not
    d, bits = 32, 2
    rng = np.random.default_rng(12)
    x = rng.standard_normal(d)
    q = x + 0.3 * rng.standard_normal(d)
    est, enc, rot, c = _estimates_over_sketches(d, bits, x, q, 1500)
    mse_only = float(enc["nu"][0]) * float((rot @ q) @ c.astype(np.float64)[enc["idx"][0]])
    truth = float(q @ x)
    assert mse_only / truth < 0.97
    assert abs(est.mean() / truth - 1.0) < 0.02


def test_scores_equal_the_inner_products_of_the_reconstruction():
    d, bits = 64, 4
    _, rot, c, smat = _setup(d, bits)
    rng = np.random.default_rng(13)
    x = rng.standard_normal((10, d))
    q = rng.standard_normal((3, d))
    enc = qo.encode_prod(x, rot, c, smat)
    rows = qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], enc["gamma"], bits)
    s = qo.prod_scores(q, rows, d, bits, rot, c, smat)
    xhat = qo.prod_dequant(rows, d, bits, rot, c, smat)
    assert np.max(np.abs(s - q @ xhat.T)) < 1e-10


def test_decode_without_the_sketch_term_is_the_mse_decode():
    # gamma forced to 0 in every key row: the product-key decode is the plain decode over
    # (bits - 1)-bit MSE key rows of the same indices and norms
    d, h, hq, bs, bits, vb = 64, 2, 4, 4, 3, 2
    rng = np.random.default_rng(14)
    signs, rot, c, smat = _setup(d, bits)
    vc, _ = o.codebook_f32(d, vb)
    lens = np.array([7, 5])
    nblk = 4
    bt = np.array([[0, 1], [2, 3]], dtype=np.int32)
    x = rng.standard_normal((nblk * bs * h, d))
    enc = qo.encode_prod(x, rot, c, smat)
    kprod = qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], np.zeros(len(x), np.float32), bits)
    kprod = kprod.reshape(nblk, bs, h, -1)
    kmse = o.make_rows(enc["idx"], enc["nu"], bits - 1).reshape(nblk, bs, h, -1)
    vrows = o.make_rows(rng.integers(0, 1 << vb, size=(nblk * bs * h, d)), rng.random(nblk * bs * h).astype(np.float32),
                        vb).reshape(nblk, bs, h, -1)
    q = rng.standard_normal((2, hq, d))
    got = qo.paged_decode_prod_keys(q, kprod, vrows, bits, vb, bt, lens, signs, c, vc, smat)
    want = o.paged_decode(q, kmse, vrows, bits - 1, vb, bt, lens, signs, c, vc)
    assert np.max(np.abs(got - want)) < 1e-12


def test_decode_with_product_keys_is_dense_attention_on_the_reconstruction():
    d, h, hq, bs, bits, vb = 64, 1, 2, 4, 4, 4
    rng = np.random.default_rng(15)
    signs, rot, c, smat = _setup(d, bits)
    vc, _ = o.codebook_f32(d, vb)
    x = rng.standard_normal((8, d)) * rng.lognormal(0, 0.5, d)
    enc = qo.encode_prod(x, rot, c, smat)
    kprod = qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], enc["gamma"], bits).reshape(2, bs, h, -1)
    vraw = rng.standard_normal((8, d))
    vpages = o.write_kv(vraw[:, None, :].astype(np.float32), np.zeros((2, bs, h, o.row_bytes(d, vb)), np.uint8),
                        np.arange(8), signs, vc, vb)
    q = rng.standard_normal((1, hq, d))
    got = qo.paged_decode_prod_keys(q, kprod, vpages, bits, vb, np.array([[0, 1]]), np.array([8]), signs, c, vc,
                                    smat)
    khat = qo.prod_dequant(kprod.reshape(8, -1), d, bits, rot, c, smat)
    vhat = o.dequant_rows(vpages.reshape(8, -1), d, vb, rot, vc)
    for j in range(hq):
        sc = (q[0, j] @ khat.T) / math.sqrt(d)
        p = np.exp(sc - sc.max())
        p /= p.sum()
        assert np.max(np.abs(got[0, j] - p @ vhat)) < 1e-12
