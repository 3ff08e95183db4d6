"""Pins for the CPU oracle: each check ties the oracle to something other than itself
(values printed on the TurboQuant pages, published tables and test vectors, closed
forms, invariants, independent quadrature, brute force on tiny inputs).

Page citations: "vLLM Usage" (TQ Byte Layout, Slot Mapping, TQ Packed Page Contract),
"vLLM Reference Audit" (Feature Checklist), "Architecture" (PackedPageCache,
Diagnostic vs Serving Paths).
"""

import math

import numpy as np
import pytest
from scipy import integrate
from scipy.special import gammaln

from conftest import read_golden_rows
from oracle import tq_oracle as o


# ---------------------------------------------------------------- row geometry

def test_row_bytes_table_from_pages():
    # "vLLM Usage", TQ Byte Layout table (head_dim 128).
    for line in read_golden_rows("row_bytes_d128.txt"):
        d, b, ib, rb = map(int, line.split())
        assert o.index_bytes(d, b) == ib
        assert o.row_bytes(d, b) == rb


def test_k4_v2_pair_is_104_bytes():
    # "vLLM Usage", TQ Byte Layout: 68 + 36 = 104 bytes per K4/V2 token-head.
    assert o.row_bytes(128, 4) + o.row_bytes(128, 2) == 104


def test_contract_example_page_shape():
    # "vLLM Usage", TQ Packed Page Contract: pages = zeros(32, 16, 2, row_bytes) at dim 128, 4 bits.
    assert (32, 16, 2, o.row_bytes(128, 4)) == (32, 16, 2, 68)


# ---------------------------------------------------------------- rotation

def test_splitmix64_published_vector():
    want = [int(v) for v in read_golden_rows("splitmix64_seed1234567.txt")]
    signs = o.splitmix64_signs(5, 1234567)
    assert list(signs) == [-1.0 if (v >> 63) else 1.0 for v in want]


def test_signs_are_pm1_and_reproducible():
    s1 = o.splitmix64_signs(256, 42)
    s2 = o.splitmix64_signs(256, 42)
    s3 = o.splitmix64_signs(256, 43)
    assert set(np.unique(s1)) <= {-1.0, 1.0}
    assert np.array_equal(s1, s2)
    assert not np.array_equal(s1, s3)
    assert 80 < np.sum(s1 > 0) < 176  # balanced to ~5 sigma


@pytest.mark.parametrize("d", [1, 2, 4, 16, 64, 128])
def test_hadamard_matches_sylvester_recursion(d):
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.kron(np.array([[1.0, 1.0], [1.0, -1.0]]), h)
    assert np.array_equal(o.hadamard(d), h)


@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_rotation_orthogonal(d):
    r = o.rotation_matrix(o.splitmix64_signs(d, 42))
    assert np.max(np.abs(r @ r.T - np.eye(d))) < 1e-12


def _fwht_butterfly(v):
    """Independent in-place natural-order fast Walsh-Hadamard transform (unnormalised)."""
    v = np.array(v, dtype=np.float64)
    h = 1
    while h < v.shape[-1]:
        for i in range(0, v.shape[-1], 2 * h):
            a = v[..., i:i + h].copy()
            b = v[..., i + h:i + 2 * h].copy()
            v[..., i:i + h] = a + b
            v[..., i + h:i + 2 * h] = a - b
        h *= 2
    return v


@pytest.mark.parametrize("d", [32, 128])
def test_rotation_equals_sign_flip_then_fwht(d):
    s = o.splitmix64_signs(d, 7)
    r = o.rotation_matrix(s)
    x = np.random.default_rng(0).standard_normal((5, d))
    want = _fwht_butterfly(x * s) / math.sqrt(d)
    assert np.max(np.abs(x @ r.T - want)) < 1e-12
    # FWHT of a unit vector e_i is column i of H
    e = np.eye(d)
    assert np.array_equal(_fwht_butterfly(e), o.hadamard(d).T)


# ---------------------------------------------------------------- codebook

@pytest.mark.parametrize("d", [32, 128, 256])
def test_density_normalised_and_variance_1_over_d(d):
    mass, _ = integrate.quad(lambda x: o.coord_density(x, d), -1, 1, epsabs=1e-13, epsrel=1e-13, limit=200)
    var, _ = integrate.quad(lambda x: x * x * o.coord_density(x, d), -1, 1, epsabs=1e-14, epsrel=1e-13, limit=200)
    assert abs(mass - 1) < 1e-11
    assert abs(var - 1.0 / d) < 1e-12


@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_one_bit_closed_form(d):
    # b = 1: the two cells are the half-lines, centroid = +-E|X| = Gamma(D/2) / (sqrt(pi) Gamma((D+1)/2)).
    c, b = o.lloyd_max(d, 1)
    want = math.exp(gammaln(d / 2) - 0.5 * math.log(math.pi) - gammaln((d + 1) / 2))
    assert abs(c[1] - want) < 1e-14 and abs(c[0] + want) < 1e-14
    assert b[0] == 0.0


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_lloyd_max_conditions_by_independent_quadrature(d, bits):
    c, b = o.lloyd_max(d, bits)
    n = 1 << bits
    assert c.shape == (n,) and b.shape == (n - 1,)
    assert np.all(np.diff(c) > 0) and c[0] > -1 and c[-1] < 1
    assert np.array_equal(c, -c[::-1]) and b[n // 2 - 1] == 0.0
    assert np.max(np.abs(b - 0.5 * (c[:-1] + c[1:]))) == 0
    edges = np.concatenate([[-1.0], b, [1.0]])
    f = lambda x: o.coord_density(x, d)
    for k in range(n):
        lo, hi = edges[k], edges[k + 1]
        m0, _ = integrate.quad(f, lo, hi, epsabs=1e-15, epsrel=1e-13, limit=200)
        m1, _ = integrate.quad(lambda x: x * f(x), lo, hi, epsabs=1e-16, epsrel=1e-13, limit=200)
        assert abs(m1 / m0 - c[k]) < 1e-10, (k, m1 / m0, c[k])


def test_gaussian_limit_matches_max_1960_table():
    d = 1 << 14
    for line in read_golden_rows("gaussian_lloyd_max_levels.txt"):
        vals = line.split()
        bits = int(vals[0])
        want = np.array([float(v) for v in vals[1:]])
        c, _ = o.lloyd_max(d, bits)
        got = c[len(c) // 2:] * math.sqrt(d)
        assert np.max(np.abs(got - want)) < 1.5e-3, (bits, got, want)


def test_codebook_f32_is_rounded_fp64():
    c, b = o.lloyd_max(128, 4)
    c32, b32 = o.codebook_f32(128, 4)
    assert c32.dtype == np.float32 and np.array_equal(c32, c.astype(np.float32))
    assert np.array_equal(b32, b.astype(np.float32))


# ---------------------------------------------------------------- encode and pack

def test_pack_golden_examples():
    for line in read_golden_rows("pack_examples.txt"):
        bits, idx, hexes = [p.strip() for p in line.split("|")]
        bits = int(bits)
        idx = np.array([[int(v) for v in idx.split()]])
        want = bytes(int(h, 16) for h in hexes.split())
        got = o.pack_indices(idx, bits)[0].tobytes()
        assert got == want, (bits, got.hex(), want.hex())


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("d", [16, 64, 128, 256])
def test_pack_roundtrip(bits, d):
    rng = np.random.default_rng(bits * 1000 + d)
    idx = rng.integers(0, 1 << bits, size=(17, d))
    packed = o.pack_indices(idx, bits)
    assert packed.shape == (17, o.index_bytes(d, bits))
    assert np.array_equal(o.unpack_indices(packed, d, bits), idx)
    # bit-by-bit reading of the stream, independent of numpy's packbits
    row = packed[3]
    for j in range(0, d, 7):
        v = 0
        for i in range(bits):
            k = j * bits + i
            v |= ((int(row[k // 8]) >> (k % 8)) & 1) << i
        assert v == idx[3, j]


def test_norm_bytes_little_endian_fp32():
    rows = o.make_rows(np.zeros((1, 128), dtype=np.int64), np.array([1.0], dtype=np.float32), 4)
    assert rows.shape == (1, 68)
    assert rows[0, -4:].tobytes() == bytes([0x00, 0x00, 0x80, 0x3F])


def test_encode_argmin_equals_boundary_search_away_from_ties():
    d, bits = 128, 4
    c32, _ = o.codebook_f32(d, bits)
    rot = o.rotation_matrix(o.splitmix64_signs(d, 42))
    x = np.random.default_rng(1).standard_normal((300, d))
    idx, norms, margin = o.encode_rows(x, rot, c32)
    u = (x / np.linalg.norm(x, axis=1, keepdims=True)) @ rot.T
    mids = 0.5 * (c32[:-1].astype(np.float64) + c32[1:])
    alt = np.searchsorted(mids, u, side="left")  # #{k : mid_k < u}: ties to the lower index
    away = margin > 1e-12
    assert np.array_equal(idx[away], alt[away])
    assert np.allclose(norms, np.linalg.norm(x, axis=1).astype(np.float32), rtol=0, atol=0)


def test_encode_worked_example_rotated_basis_vector():
    # x = nu * R^T e_0 rotates to nu e_0: coordinate 0 is 1 -> the top centroid; every
    # other coordinate is exactly 0, a tie between the two middle centroids -> lower one.
    d, bits = 64, 3
    c32, _ = o.codebook_f32(d, bits)
    rot = o.rotation_matrix(o.splitmix64_signs(d, 42))
    x = 2.5 * rot.T[:, 0][None, :]
    idx, norms, _ = o.encode_rows(x, rot, c32)
    assert idx[0, 0] == 7
    # R^T e_0 has entries +-1/sqrt(D): rounding leaves |y_j| ~ 1e-17, far inside the middle cells
    assert np.all((idx[0, 1:] == 3) | (idx[0, 1:] == 4))
    assert abs(norms[0] - 2.5) < 1e-6
    # the exact zero row: u = 0, all indices the lower middle one, norm 0
    idx0, n0, _ = o.encode_rows(np.zeros((1, d)), rot, c32)
    assert np.all(idx0 == 3) and n0[0] == 0.0


# ---------------------------------------------------------------- slot scatter

def _tiny_setup(d=32, h=2, bits=4, nblk=3, bs=4, t=6, seed=0):
    rng = np.random.default_rng(seed)
    raw = rng.standard_normal((t, h, d)).astype(np.float32)
    pages = np.zeros((nblk, bs, h, o.row_bytes(d, bits)), dtype=np.uint8)
    signs = o.splitmix64_signs(d, 42)
    c32, _ = o.codebook_f32(d, bits)
    return raw, pages, signs, c32


def test_negative_slots_leave_rows_untouched():
    raw, pages, signs, c32 = _tiny_setup()
    pages[:] = 0xAB
    slots = np.array([0, -1, 5, -7, 11, 2])
    out = o.write_kv(raw, pages, slots, signs, c32, 4)
    written = {0, 5, 11, 2}
    for s in range(12):
        blk, off = divmod(s, 4)
        if s in written:
            assert not np.all(out[blk, off] == 0xAB)
        else:
            assert np.all(out[blk, off] == 0xAB)
    rot = o.rotation_matrix(signs)
    rows, _ = o.encode_to_rows(raw[2], rot, c32, 4)
    assert np.array_equal(out[1, 1], rows)  # slot 5 -> block 1, offset 1, both heads


def test_out_of_range_slot_raises_and_writes_nothing():
    raw, pages, signs, c32 = _tiny_setup()
    before = pages.copy()
    with pytest.raises(o.SlotOutOfRange):
        o.write_kv(raw, pages, np.array([0, 1, 2, 12, 3, 4]), signs, c32, 4)
    assert np.array_equal(pages, before)
    # the last valid slot is fine
    o.write_kv(raw, pages, np.array([0, 1, 2, 11, 3, 4]), signs, c32, 4)


# ---------------------------------------------------------------- decode

def _decode_case(d=64, h=2, hq=4, kb=4, vb=2, bs=4, lens=(7, 1, 0, 9), seed=3):
    rng = np.random.default_rng(seed)
    bsz = len(lens)
    nblk = sum(-(-n // bs) for n in lens) + 2
    perm = rng.permutation(nblk)
    maxb = max(-(-n // bs) for n in lens) or 1
    bt = np.zeros((bsz, maxb), dtype=np.int32)
    pos = 0
    for b, n in enumerate(lens):
        nb = -(-n // bs)
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
    signs = o.splitmix64_signs(d, 42)
    ck, _ = o.codebook_f32(d, kb)
    cv, _ = o.codebook_f32(d, vb)
    kp = np.zeros((nblk, bs, h, o.row_bytes(d, kb)), dtype=np.uint8)
    vp = np.zeros((nblk, bs, h, o.row_bytes(d, vb)), dtype=np.uint8)
    for b, n in enumerate(lens):
        t = np.arange(n)
        slots = bt[b, t // bs].astype(np.int64) * bs + t % bs
        kraw = rng.standard_normal((n, h, d))
        vraw = rng.standard_normal((n, h, d))
        kp = o.write_kv(kraw, kp, slots, signs, ck, kb)
        vp = o.write_kv(vraw, vp, slots, signs, cv, vb)
    q = rng.standard_normal((bsz, hq, d))
    return dict(q=q, k_pages=kp, v_pages=vp, k_bits=kb, v_bits=vb, block_table=bt,
                seq_lens=np.array(lens), signs=signs, k_centroids32=ck, v_centroids32=cv)


def test_decode_dense_form_equals_rotated_form():
    case = _decode_case()
    a = o.paged_decode(**case)
    b = o.paged_decode_rotated(**case)
    assert np.max(np.abs(a - b)) < 1e-12
    assert np.all(a[2] == 0)  # seq_len 0 -> zeros


def test_decode_single_token_returns_its_value_row():
    case = _decode_case(lens=(1,))
    out = o.paged_decode(**case)
    rot = o.rotation_matrix(case["signs"])
    blk = case["block_table"][0, 0]
    for j in range(4):
        vrow = case["v_pages"][blk, 0, j // 2][None]
        want = o.dequant_rows(vrow, 64, 2, rot, case["v_centroids32"])[0]
        assert np.max(np.abs(out[0, j] - want)) < 1e-12


def test_decode_zero_query_is_mean_of_values():
    case = _decode_case(lens=(9,))
    case["q"] = np.zeros_like(case["q"])
    out = o.paged_decode(**case)
    rot = o.rotation_matrix(case["signs"])
    bt = case["block_table"][0]
    rows = np.stack([case["v_pages"][bt[t // 4], t % 4, 1] for t in range(9)])
    want = o.dequant_rows(rows, 64, 2, rot, case["v_centroids32"]).mean(0)
    assert np.max(np.abs(out[0, 3] - want)) < 1e-12


def test_decode_brute_force_tiny():
    # D = 16, a handful of tokens: explicit loops with an independent unpack (bit by bit),
    # an independent Hadamard (Kronecker recursion) and an explicit softmax.
    d, h, hq, kb, vb, bs = 16, 1, 2, 3, 5, 2
    case = _decode_case(d=d, h=h, hq=hq, kb=kb, vb=vb, bs=bs, lens=(3, 4), seed=11)
    out = o.paged_decode(**case)
    hm = np.array([[1.0]])
    while hm.shape[0] < d:
        hm = np.kron(np.array([[1.0, 1.0], [1.0, -1.0]]), hm)
    s = case["signs"]

    def recon(row, bits, cents):
        nb = -(-d * bits // 8)
        idx = []
        for j in range(d):
            v = 0
            for i in range(bits):
                k = j * bits + i
                v |= ((int(row[k // 8]) >> (k % 8)) & 1) << i
            idx.append(v)
        norm = float(np.frombuffer(bytes(row[nb:nb + 4]), dtype="<f4")[0])
        y = np.array([float(cents[i]) for i in idx])
        # x = R^T y with R = H diag(s)/sqrt(d): x_i = s_i sum_j H[j, i] y_j / sqrt(d)
        return norm * np.array([s[i] * sum(hm[j, i] * y[j] for j in range(d)) for i in range(d)]) / math.sqrt(d)

    for b, n in enumerate(case["seq_lens"]):
        for j in range(hq):
            ks, vs = [], []
            for t in range(n):
                blk = case["block_table"][b, t // bs]
                ks.append(recon(case["k_pages"][blk, t % bs, 0], kb, case["k_centroids32"]))
                vs.append(recon(case["v_pages"][blk, t % bs, 0], vb, case["v_centroids32"]))
            sc = [sum(case["q"][b, j, i] * k[i] for i in range(d)) / math.sqrt(d) for k in ks]
            m = max(sc)
            w = [math.exp(v - m) for v in sc]
            tot = sum(w)
            want = [sum(w[t] * vs[t][i] for t in range(n)) / tot for i in range(d)]
            assert np.max(np.abs(out[b, j] - np.array(want))) < 1e-12


def test_decode_skips_out_of_range_block():
    case = _decode_case(lens=(8,))
    good = o.paged_decode(**case)
    nblk = case["k_pages"].shape[0]
    # point the second block at an id past the end: its 4 tokens are left out
    case["block_table"] = case["block_table"].copy()
    case["block_table"][0, 1] = nblk + 5
    bad, flag = o.paged_decode(**case, return_flags=True)
    assert flag
    case2 = dict(case)
    case2["seq_lens"] = np.array([4])
    first_only = o.paged_decode(**case2)
    assert np.max(np.abs(bad - first_only)) < 1e-12
    assert np.max(np.abs(bad - good)) > 1e-6


# ---------------------------------------------------------------- dense readback (tq4_decompress)

def _fwht_butterfly(x):
    """Unnormalised Walsh-Hadamard transform of the last axis by in-place butterflies."""
    y = np.array(x, dtype=np.float64)
    n = y.shape[-1]
    hlen = 1
    while hlen < n:
        for i in range(0, n, 2 * hlen):
            a = y[..., i:i + hlen].copy()
            b = y[..., i + hlen:i + 2 * hlen].copy()
            y[..., i:i + hlen] = a + b
            y[..., i + hlen:i + 2 * hlen] = a - b
        hlen *= 2
    return y


def test_readback_rotates_forward_to_the_centroids():
    # Applying the encoder's forward rotation R x = H_D (s * x) / sqrt(D) (here by butterfly,
    # not the oracle's matrix) to the readback of a row must give nu * c[idx].  A transposed
    # R, a lost sign flip or a wrong bit order in the readback breaks this.
    rng = np.random.default_rng(11)
    for d, bits in ((64, 2), (64, 3), (128, 4), (128, 5), (256, 4)):
        signs = o.splitmix64_signs(d, 42)
        c32, _ = o.codebook_f32(d, bits)
        idx = rng.integers(0, 1 << bits, size=(6, d))
        nu = rng.uniform(0.1, 50.0, size=6).astype(np.float32)
        pages = o.make_rows(idx, nu, bits).reshape(3, 2, 1, -1)  # 3 blocks x 2 slots x 1 head
        back = o.dequant_slots(pages, np.arange(6), signs, c32, bits)[:, 0]
        fwd = _fwht_butterfly(back * signs) / math.sqrt(d)
        want = nu.astype(np.float64)[:, None] * c32.astype(np.float64)[idx]
        assert np.max(np.abs(fwd - want)) <= 1e-12 * float(nu.max())


def test_readback_norm_and_addressing():
    rng = np.random.default_rng(12)
    d, bits, bs, nblk, h = 64, 4, 4, 3, 2
    signs = o.splitmix64_signs(d, 42)
    c32, _ = o.codebook_f32(d, bits)
    idx = rng.integers(0, 16, size=(nblk * bs * h, d))
    nu = rng.uniform(0.5, 4.0, size=nblk * bs * h).astype(np.float32)
    pages = o.make_rows(idx, nu, bits).reshape(nblk, bs, h, -1)
    slots = np.array([7, -1, 0, 11, -3])
    back = o.dequant_slots(pages, slots, signs, c32, bits)
    assert back.shape == (5, h, d)
    assert np.all(back[1] == 0) and np.all(back[4] == 0)  # negative slots: zero rows
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for hh in range(h):
            k = (s // bs * bs + s % bs) * h + hh  # slot s, head hh
            # R is orthogonal: ||nu R^T c[idx]|| = nu ||c[idx]||
            want = float(nu[k]) * np.linalg.norm(c32.astype(np.float64)[idx[k]])
            assert np.linalg.norm(back[t, hh]) == pytest.approx(want, rel=1e-12)
    with pytest.raises(o.SlotOutOfRange):
        o.dequant_slots(pages, np.array([0, nblk * bs]), signs, c32, bits)


# ---------------------------------------------------------------- mixed prefill / decode

def _prefill_case(seed=21):
    rng = np.random.default_rng(seed)
    d, h, hq, kb, vb, bs = 64, 2, 4, 4, 2, 4
    lens = np.array([9, 6, 1])
    nblk = int(sum(-(-n // bs) for n in lens))
    bt = np.zeros((len(lens), 4), dtype=np.int32)
    perm = rng.permutation(nblk)
    pos = 0
    for b, n in enumerate(lens):
        nb = -(-int(n) // bs)
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
    signs = o.splitmix64_signs(d, 42)
    kc, _ = o.codebook_f32(d, kb)
    vc, _ = o.codebook_f32(d, vb)
    kp = np.zeros((nblk, bs, h, o.row_bytes(d, kb)), dtype=np.uint8)
    vp = np.zeros((nblk, bs, h, o.row_bytes(d, vb)), dtype=np.uint8)
    for b, n in enumerate(lens):
        slots = np.array([bt[b, t // bs] * bs + t % bs for t in range(n)])
        kp = o.write_kv(rng.standard_normal((n, h, d)), kp, slots, signs, kc, kb)
        vp = o.write_kv(rng.standard_normal((n, h, d)), vp, slots, signs, vc, vb)
    return dict(d=d, h=h, hq=hq, kb=kb, vb=vb, bs=bs, lens=lens, bt=bt, signs=signs, kc=kc, vc=vc, kp=kp, vp=vp,
                rng=rng)


def test_prefill_rows_equal_per_query_brute_force():
    # each query row is softmax attention over the dequantised keys up to its position,
    # computed here directly (dense R built from signs and the Hadamard definition)
    c = _prefill_case()
    rng, d, bs = c["rng"], c["d"], c["bs"]
    # sequence 0: a 3-token chunk at positions 6, 7, 8; sequence 1: 2 tokens at 4, 5; seq 2: decode
    q_seq = np.array([0, 0, 0, 1, 1, 2])
    q_len = np.array([7, 8, 9, 5, 6, 1])
    q = rng.standard_normal((6, c["hq"], d))
    out = o.paged_prefill(q, q_seq, q_len, c["kp"], c["vp"], c["kb"], c["vb"], c["bt"], c["signs"], c["kc"], c["vc"])
    rt = (o.hadamard(d) * c["signs"][None, :]).T / math.sqrt(d)  # R^T, R = H diag(s) / sqrt(D)
    grp = c["hq"] // c["h"]
    for i in range(6):
        b, n = q_seq[i], q_len[i]
        for j in range(c["hq"]):
            kvh = j // grp
            keys, vals = [], []
            for t in range(n):
                blk, off = c["bt"][b, t // bs], t % bs
                for pages, bits, cents, dst in ((c["kp"], c["kb"], c["kc"], keys), (c["vp"], c["vb"], c["vc"], vals)):
                    row = pages[blk, off, kvh]
                    nb = o.index_bytes(d, bits)
                    idx = o.unpack_indices(row[None, :nb], d, bits)[0]
                    nu = float(np.frombuffer(row[nb:nb + 4].tobytes(), dtype="<f4")[0])
                    dst.append(nu * (rt @ cents.astype(np.float64)[idx]))
            s = np.array([np.dot(k, q[i, j]) for k in keys]) / math.sqrt(d)
            p = np.exp(s - s.max())
            p /= p.sum()
            want = sum(pi * v for pi, v in zip(p, vals))
            assert np.allclose(out[i, j], want, rtol=0, atol=1e-12)


def test_prefill_is_causal_and_reduces_to_decode():
    c = _prefill_case(22)
    rng = c["rng"]
    q_seq = np.array([0, 0, 1])
    q_len = np.array([5, 9, 6])
    q = rng.standard_normal((3, c["hq"], c["d"]))
    args = (c["kb"], c["vb"], c["bt"], c["signs"], c["kc"], c["vc"])
    out = o.paged_prefill(q, q_seq, q_len, c["kp"], c["vp"], *args)
    # tokens past a row's length do not change it: overwrite token 6..8 of sequence 0
    kp2 = c["kp"].copy()
    for t in (6, 7, 8):
        kp2[c["bt"][0, t // c["bs"]], t % c["bs"]] = 0x5A
    out2 = o.paged_prefill(q, q_seq, q_len, kp2, c["vp"], *args)
    assert np.array_equal(out[0], out2[0]) and not np.allclose(out[1], out2[1])
    # one row per sequence at the full length is the decode
    dec = o.paged_decode(q[[1, 2]], c["kp"], c["vp"], c["kb"], c["vb"], c["bt"][[0, 1]], np.array([9, 6]),
                         c["signs"], c["kc"], c["vc"])
    assert np.allclose(out[[1, 2]], dec, rtol=0, atol=1e-13)
