"""GPU parity of the product-quantised ("QJL residual") key path -- tq_write_kv_prod and
tq_paged_decode_prod through the C ABI -- against the fp64 oracle in oracle/qjl_oracle.py
("vLLM Reference Audit": File Map, MSE and QJL codecs; Feature Checklist, QJL residual).

Writer bars (fp32 kernel arithmetic against the fp64 oracle):
  * MSE indices: those of the MSE writer (bit-exact outside the 1e-6 decision band,
    in-band exceptions held to the rate bar, never more than one step);
  * nu: 1e-6 relative, as for the MSE rows;
  * sign bits, on rows whose indices all agree: bit-exact wherever the oracle's
    projection |(S r)_i| is at least SIGN_BAND = 1e-5.  The kernel's r carries the
    rounding of the fp32 rotation (a few 1e-8 per coordinate at |y_j| ~ D^-1/2), so
    (S dr)_i is of order sqrt(D) * 4e-8 < 1e-6: a flip needs the projection within a
    few 1e-7 of zero, and the band leaves an order of magnitude of headroom;
  * gamma, on the same rows: 5e-5 relative (||dr|| ~ sqrt(D) * 4e-8 against gamma >= 0.09,
    the 4-bit MSE distortion at D = 128, with the same headroom).
Decode bar: |gpu - oracle| <= 2e-3 + 2e-3 |oracle|, the MSE decode's, on pages the
oracle encoded (S rounded to fp32 once, the matrix both sides use).
"""

import numpy as np
import pytest
import torch

from oracle import qjl_oracle as qo
from oracle import tq_oracle as o
from parity import BAND, DEC_ATOL, DEC_RTOL, NORM_RTOL, OracleCodec, allowed_flips

pytestmark = pytest.mark.gpu

SIGN_BAND = 1e-5
GAMMA_RTOL = 5e-5
SKETCH_SEED = 43


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


def sketch(tq, d):
    s_lib = tq.tq_build_qjl_matrix(d, SKETCH_SEED)
    s_or = qo.normal_matrix(d, d, SKETCH_SEED).astype(np.float32)
    assert np.array_equal(s_lib.numpy(), s_or)
    return s_lib.cuda(), s_or.astype(np.float64)


@pytest.mark.parametrize("d,bits,dtype", [(64, 3, torch.float32), (64, 4, torch.float16), (64, 5, torch.bfloat16),
                                          (128, 3, torch.bfloat16), (128, 4, torch.float16), (128, 5, torch.float32),
                                          (128, 4, torch.bfloat16)])
def test_prod_writer_matches_oracle(tq, d, bits, dtype):
    rng = np.random.default_rng(2000 + 10 * d + bits)
    t, h, bs = 301, 4, 16
    nb = (t + bs - 1) // bs + 2
    raw32 = (rng.standard_normal((t, h, d)) * rng.lognormal(0.0, 0.5, (t, h, 1))).astype(np.float32)
    raw32[5, 1] = 0.0  # a zero row: nu = 0, every index at the lower middle centroid
    raw = torch.from_numpy(raw32).to(dtype)
    raw64 = raw.double().numpy()
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[::17] = -1
    rbp = tq.tq_prod_row_bytes(d, bits)
    pages = torch.full((nb, bs, h, rbp), 0xA5, dtype=torch.uint8, device="cuda")
    codec = OracleCodec(d)
    kc = codec.centroids(bits - 1)
    s_gpu, s64 = sketch(tq, d)
    st = tq.tq_write_kv_prod(raw.cuda(), pages, torch.from_numpy(slots).cuda(), tq.tq_build_rotation(d, 42, "cuda"),
                             torch.from_numpy(kc).cuda(), s_gpu, check=False)
    assert int(st.item()) == 0
    pg = pages.cpu().numpy().reshape(nb * bs, h, rbp)
    written = np.zeros(nb * bs, dtype=bool)
    written[slots[slots >= 0]] = True
    assert np.all(pg[~written] == 0xA5)

    tok = np.nonzero(slots >= 0)[0]
    rows = pg[slots[tok]].reshape(-1, rbp)
    x = raw64[tok].reshape(-1, d)
    enc = qo.encode_prod(x, codec.rot, kc, s64)
    _, _, margin = o.encode_rows(x, codec.rot, kc)
    gidx, gz, gnu, ggam = qo.unpack_prod_rows(rows, d, bits)

    diff = gidx != enc["idx"]
    assert int((diff & (margin >= BAND)).sum()) == 0
    assert diff.sum() <= allowed_flips(diff.size)
    assert np.abs(gidx - enc["idx"]).max() <= 1
    nu = enc["nu"].astype(np.float64)
    assert np.all(np.abs(gnu - nu) <= NORM_RTOL * nu)

    clean = ~diff.any(axis=1)
    assert clean.mean() > 0.99
    proj = enc["residual"] @ s64.T
    zbad = (gz != enc["z"]) & clean[:, None] & (np.abs(proj) >= SIGN_BAND)
    assert int(zbad.sum()) == 0
    g = enc["gamma"].astype(np.float64)[clean]
    assert np.all(np.abs(ggam[clean] - g) <= GAMMA_RTOL * g)


def test_prod_writer_bad_slot_writes_nothing(tq):
    d, bits, t, h, bs, nb = 64, 4, 40, 2, 16, 3
    rng = np.random.default_rng(7)
    raw = torch.from_numpy(rng.standard_normal((t, h, d)).astype(np.float32)).cuda()
    slots = torch.arange(t, dtype=torch.int64)
    slots[11] = nb * bs  # one past the pages
    pages = torch.full((nb, bs, h, tq.tq_prod_row_bytes(d, bits)), 0x3C, dtype=torch.uint8, device="cuda")
    s_gpu, _ = sketch(tq, d)
    kc = torch.from_numpy(OracleCodec(d).centroids(bits - 1)).cuda()
    st = tq.tq_write_kv_prod(raw, pages, slots.cuda(), tq.tq_build_rotation(d, 42, "cuda"), kc, s_gpu, check=False)
    assert int(st.item()) == tq.TQ_ERR_SLOT_OUT_OF_RANGE
    assert torch.all(pages == 0x3C)
    # no tokens: nothing launched past the status reset
    empty = torch.empty(0, h, d, dtype=torch.float32, device="cuda")
    st = tq.tq_write_kv_prod(empty, pages, torch.empty(0, dtype=torch.int64, device="cuda"),
                             tq.tq_build_rotation(d, 42, "cuda"), kc, s_gpu, check=False)
    assert int(st.item()) == 0


def build_pages(rng, codec, d, h, bs, nb, kb, vb, s64):
    n = nb * bs * h
    kx = rng.standard_normal((n, d)) * rng.lognormal(0.0, 0.5, (n, 1))
    enc = qo.encode_prod(kx, codec.rot, codec.centroids(kb - 1), s64)
    kp = qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], enc["gamma"], kb).reshape(nb, bs, h, -1)
    vx = rng.standard_normal((n, d))
    vidx, vnu, _ = o.encode_rows(vx, codec.rot, codec.centroids(vb))
    vp = o.make_rows(vidx, vnu, vb).reshape(nb, bs, h, -1)
    return np.ascontiguousarray(kp), np.ascontiguousarray(vp)


def tables(rng, lens, bs, extra=2):
    maxb = max(1, max((l + bs - 1) // bs for l in lens))
    need = sum((l + bs - 1) // bs for l in lens)
    nb = need + extra
    perm = rng.permutation(nb)
    bt = np.full((len(lens), maxb), -1, dtype=np.int32)
    k = 0
    for b, l in enumerate(lens):
        m = (l + bs - 1) // bs
        bt[b, :m] = perm[k:k + m]
        k += m
    return bt, nb


def run_prod_decode(tq, codec, q, kp, vp, bt, lens, kb, vb, out_dtype=torch.float32, status=None):
    """q: a CPU torch tensor (its dtype is the query dtype on the device) or a float32 array."""
    d = codec.d
    s_gpu, _ = sketch(tq, d)
    q = q if isinstance(q, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(q))
    out = tq.tq_paged_decode_prod(q.cuda(), torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda(),
                                  torch.from_numpy(bt).cuda(), torch.from_numpy(np.asarray(lens, np.int32)).cuda(),
                                  tq.tq_build_rotation(d, 42, "cuda"), torch.from_numpy(codec.centroids(kb - 1)).cuda(),
                                  torch.from_numpy(codec.centroids(vb)).cuda(), s_gpu, out_dtype=out_dtype,
                                  status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def oracle_prod(codec, q, kp, vp, bt, lens, kb, vb, s64):
    return qo.paged_decode_prod_keys(q, kp, vp, kb, vb, bt, np.asarray(lens), codec.signs, codec.centroids(kb - 1),
                                     codec.centroids(vb), s64)


def assert_close(got, want):
    err = np.abs(got - want) - (DEC_ATOL + DEC_RTOL * np.abs(want))
    assert err.max() <= 0.0, float(err.max())


# D 128, block size 16, GQA group 4 or 8 take the tensor-core decode (the sketch term as a
# second MMA over the +-1 sign pairs); the others the SIMT split decode
@pytest.mark.parametrize("d,hq,h,kb,vb,bs,lens,qdtype", [
    (64, 4, 4, 3, 2, 16, [1, 17, 200, 0], torch.float32),
    (64, 8, 4, 5, 5, 8, [33, 64, 5], torch.float16),
    (128, 32, 8, 4, 4, 16, [300, 129, 16, 1], torch.bfloat16),
    (128, 16, 2, 5, 3, 16, [257, 100], torch.float32),
    (128, 8, 1, 3, 4, 32, [500], torch.float16),
    (128, 32, 8, 3, 2, 16, [0, 45, 700, 1], torch.float16),
    (128, 64, 8, 4, 5, 16, [130, 17], torch.float32),
    (128, 16, 4, 5, 4, 16, [33, 0, 250], torch.bfloat16),
    (128, 16, 2, 3, 3, 16, [160, 31], torch.float16),
])
def test_prod_decode_matches_oracle(tq, d, hq, h, kb, vb, bs, lens, qdtype):
    rng = np.random.default_rng(3000 + d + hq + kb * 7 + vb)
    codec = OracleCodec(d)
    _, s64 = sketch(tq, d)
    bt, nb = tables(rng, lens, bs)
    kp, vp = build_pages(rng, codec, d, h, bs, nb, kb, vb, s64)
    q = torch.from_numpy(rng.standard_normal((len(lens), hq, d)).astype(np.float32)).to(qdtype)
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = run_prod_decode(tq, codec, q, kp, vp, bt, lens, kb, vb, status=st)
    assert int(st.item()) == 0
    want = oracle_prod(codec, q.double().numpy(), kp, vp, bt, lens, kb, vb, s64)
    assert_close(got, want)
    assert np.all(got[np.asarray(lens) == 0] == 0.0)


def test_prod_decode_sketch_term_matters(tq):
    # the same pages with gamma forced to zero decode differently: the kernel reads the signs
    d, hq, h, kb, vb, bs, lens = 128, 8, 2, 3, 4, 16, [96, 40]
    rng = np.random.default_rng(31)
    codec = OracleCodec(d)
    _, s64 = sketch(tq, d)
    bt, nb = tables(rng, lens, bs)
    kp, vp = build_pages(rng, codec, d, h, bs, nb, kb, vb, s64)
    q = (3.0 * rng.standard_normal((len(lens), hq, d))).astype(np.float32)
    got = run_prod_decode(tq, codec, q, kp, vp, bt, lens, kb, vb)
    kp0 = kp.copy()
    flat = kp0.reshape(-1, kp0.shape[-1])
    flat[:, -4:] = 0  # gamma = +0.0f
    got0 = run_prod_decode(tq, codec, q, kp0, vp, bt, lens, kb, vb)
    want = oracle_prod(codec, q, kp, vp, bt, lens, kb, vb, s64)
    want0 = oracle_prod(codec, q, kp0, vp, bt, lens, kb, vb, s64)
    assert_close(got, want)
    assert_close(got0, want0)
    assert np.abs(want - want0).max() > 20 * (DEC_ATOL + DEC_RTOL * np.abs(want).max())


def test_prod_decode_bad_block_and_long_length(tq):
    d, hq, h, kb, vb, bs, lens = 64, 8, 2, 4, 4, 16, [70, 50]
    rng = np.random.default_rng(41)
    codec = OracleCodec(d)
    _, s64 = sketch(tq, d)
    bt, nb = tables(rng, lens, bs)
    kp, vp = build_pages(rng, codec, d, h, bs, nb, kb, vb, s64)
    q = rng.standard_normal((2, hq, d)).astype(np.float32)
    bad = bt.copy()
    bad[0, 1] = nb + 5  # tokens 16..31 of sequence 0 point past the pages
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = run_prod_decode(tq, codec, q, kp, vp, bad, lens, kb, vb, status=st)
    assert int(st.item()) == tq.TQ_ERR_BLOCK_OUT_OF_RANGE
    assert_close(got, oracle_prod(codec, q, kp, vp, bad, lens, kb, vb, s64))
    # sequence 0 owns every block of its table row: past its capacity it is clamped to it
    cap = bt.shape[1] * bs
    assert np.all(bt[0] >= 0)
    got = run_prod_decode(tq, codec, q, kp, vp, bt, [cap + 3, lens[1]], kb, vb, status=st)
    assert int(st.item()) == tq.TQ_ERR_INVALID_ARG
    assert_close(got, oracle_prod(codec, q, kp, vp, bt, [cap, lens[1]], kb, vb, s64))
    # an empty batch launches nothing and returns an empty output
    s_gpu, _ = sketch(tq, d)
    out = tq.tq_paged_decode_prod(torch.empty(0, hq, d, device="cuda"), torch.from_numpy(kp).cuda(),
                                  torch.from_numpy(vp).cuda(), torch.empty(0, bt.shape[1], dtype=torch.int32,
                                                                           device="cuda"),
                                  torch.empty(0, dtype=torch.int32, device="cuda"), tq.tq_build_rotation(d, 42, "cuda"),
                                  torch.from_numpy(codec.centroids(kb - 1)).cuda(),
                                  torch.from_numpy(codec.centroids(vb)).cuda(), s_gpu, status=st)
    torch.cuda.synchronize()
    assert out.shape == (0, hq, d) and int(st.item()) == 0


@pytest.mark.parametrize("hq", [32, 64])
def test_prod_decode_tc_bad_block_and_large_norms(tq, hq):
    # the tensor-core form: a block id past the pages is skipped and reported; key rows of
    # norm up to 100 and value rows up to 1e4 take its exact paths.  (Larger keys make
    # scores of hundreds of log2 units, where fp32-level rounding of a score, ~1e-6 of its
    # terms, moves the weights of two near-tied tokens by ~1e-3; with values of norm 1e4
    # that exceeds the output bar even for fp32 arithmetic.)
    d, h, kb, vb, bs, lens = 128, 8, 4, 4, 16, [70, 300]
    rng = np.random.default_rng(53 + hq)
    codec = OracleCodec(d)
    _, s64 = sketch(tq, d)
    bt, nb = tables(rng, lens, bs)
    n = nb * bs * h
    kx = rng.standard_normal((n, d)) * (10.0 ** rng.uniform(-2, 2, (n, 1)))
    enc = qo.encode_prod(kx, codec.rot, codec.centroids(kb - 1), s64)
    kp = qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], enc["gamma"], kb).reshape(nb, bs, h, -1)
    vx = rng.standard_normal((n, d)) * (10.0 ** rng.uniform(-2, 4, (n, 1)))
    vidx, vnu, _ = o.encode_rows(vx, codec.rot, codec.centroids(vb))
    vp = o.make_rows(vidx, vnu, vb).reshape(nb, bs, h, -1)
    kp, vp = np.ascontiguousarray(kp), np.ascontiguousarray(vp)
    q = rng.standard_normal((2, hq, d)).astype(np.float32)
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = run_prod_decode(tq, codec, q, kp, vp, bt, lens, kb, vb, status=st)
    assert int(st.item()) == 0
    assert_close(got, oracle_prod(codec, q, kp, vp, bt, lens, kb, vb, s64))
    bad = bt.copy()
    bad[1, 3] = nb + 9
    got = run_prod_decode(tq, codec, q, kp, vp, bad, lens, kb, vb, status=st)
    assert int(st.item()) == tq.TQ_ERR_BLOCK_OUT_OF_RANGE
    assert_close(got, oracle_prod(codec, q, kp, vp, bad, lens, kb, vb, s64))
