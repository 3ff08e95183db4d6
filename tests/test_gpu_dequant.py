"""GPU parity of tq_dequant_rows (dense readback of packed rows) against the fp64 oracle.

Pages are built on the host (the oracle's packer, or seeded random bytes with finite
norms for the full-size case), never by the CUDA writer.  Tolerance, from the fp32
arithmetic of the kernel: log2(D) butterfly stages over at most D centroids (|c| < 0.35)
then 1/sqrt(D) give |error| <= ~2.3e-6 nu for D <= 256; the test allows 4e-6 * nu per
row, plus half an ulp of the output type when it is fp16 / bf16.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import tq_oracle as o  # noqa: E402

pytestmark = pytest.mark.gpu

ROUND = {torch.float32: 0.0, torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def _tq():
    import quantized_kv_cache_06_gb300 as tq

    return tq


def _random_pages(rng, nblk, bs, h, d, bits, norm_scale=1.0):
    n = nblk * bs * h
    idx = rng.integers(0, 1 << bits, size=(n, d))
    nu = (rng.lognormal(0.0, 1.0, size=n) * norm_scale).astype(np.float32)
    return o.make_rows(idx, nu, bits).reshape(nblk, bs, h, -1)


def _check(gpu, want, pages_rows_nu, dtype):
    got = gpu.float().cpu().numpy().astype(np.float64)
    tol = 4e-6 * pages_rows_nu[..., None] + ROUND[dtype] * np.abs(want) + 1e-30
    err = np.abs(got - want)
    assert np.all(err <= tol), float(np.max(err / tol))


def _norms_at(pages, slots):
    bs = pages.shape[1]
    rb = pages.shape[3]
    nu = np.zeros((len(slots), pages.shape[2]))
    for t, s in enumerate(slots):
        if s >= 0:
            nu[t] = pages[s // bs, s % bs, :, rb - 4:].copy().view("<f4").reshape(-1)
    return nu


@pytest.mark.parametrize("d", [32, 64, 128, 256])
@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_dequant_matches_oracle_every_shape(d, bits):
    tq = _tq()
    rng = np.random.default_rng(1000 + d + bits)
    nblk, bs, h, t = 7, 16, 3, 77
    pages = _random_pages(rng, nblk, bs, h, d, bits)
    slots = rng.permutation(nblk * bs)[:t].astype(np.int64)
    slots[rng.random(t) < 0.1] = -1
    signs = o.splitmix64_signs(d, 42)
    c32, _ = o.codebook_f32(d, bits)
    want = o.dequant_slots(pages, slots, signs, c32, bits)
    dev = torch.device("cuda")
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        out = tq.tq_dequant_rows(torch.from_numpy(pages).to(dev), torch.from_numpy(slots).to(dev),
                                 torch.from_numpy(signs.astype(np.float32)).to(dev), torch.from_numpy(c32).to(dev),
                                 out_dtype=dtype)
        torch.cuda.synchronize()
        assert out.shape == (t, h, d) and out.dtype == dtype
        _check(out, want, _norms_at(pages, slots), dtype)
        neg = slots < 0
        assert torch.all(out[torch.from_numpy(neg).to(dev)] == 0)


def test_dequant_out_of_range_slot_reports_and_zeroes():
    tq = _tq()
    rng = np.random.default_rng(5)
    d, bits, nblk, bs, h = 128, 4, 4, 16, 2
    pages = _random_pages(rng, nblk, bs, h, d, bits)
    slots = np.array([3, nblk * bs, 7, nblk * bs + 100, -2], dtype=np.int64)
    signs = o.splitmix64_signs(d, 42)
    c32, _ = o.codebook_f32(d, bits)
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = tq.tq_dequant_rows(torch.from_numpy(pages).to(dev), torch.from_numpy(slots).to(dev),
                             torch.from_numpy(signs.astype(np.float32)).to(dev), torch.from_numpy(c32).to(dev),
                             out_dtype=torch.float32, status=status, check=False)
    torch.cuda.synchronize()
    assert int(status.item()) == tq.TQ_ERR_SLOT_OUT_OF_RANGE
    assert torch.all(out[1] == 0) and torch.all(out[3] == 0) and torch.all(out[4] == 0)
    ok = slots.copy()
    ok[[1, 3]] = -1
    want = o.dequant_slots(pages, ok, signs, c32, bits)
    _check(out, want, _norms_at(pages, ok), torch.float32)
    with pytest.raises(tq.TQError):
        tq.tq_dequant_rows(torch.from_numpy(pages).to(dev), torch.from_numpy(slots).to(dev),
                           torch.from_numpy(signs.astype(np.float32)).to(dev), torch.from_numpy(c32).to(dev))


def test_dequant_zero_tokens_and_unsupported_dim():
    tq = _tq()
    dev = torch.device("cuda")
    d, bits = 64, 4
    pages = torch.zeros(2, 16, 1, o.row_bytes(d, bits), dtype=torch.uint8, device=dev)
    signs = torch.from_numpy(o.splitmix64_signs(d, 42).astype(np.float32)).to(dev)
    c32 = torch.from_numpy(o.codebook_f32(d, bits)[0]).to(dev)
    out = tq.tq_dequant_rows(pages, torch.zeros(0, dtype=torch.int64, device=dev), signs, c32)
    assert out.shape == (0, 1, d)
    # head_dim 8 is below the boundary's range (16 .. 256): refused on the host
    assert tq.lib().tq_dequant_rows(pages.data_ptr(), bits, 2, 16, 1, 8, pages.data_ptr(), 3, signs.data_ptr(),
                                    c32.data_ptr(), pages.data_ptr(), 1, None, None) == tq.TQ_ERR_UNSUPPORTED


def test_dequant_round_trip_of_oracle_written_rows():
    # rows written by the oracle's writer, read back on the GPU: equal to the oracle's
    # readback, and within the quantiser's distortion of the raw rows
    tq = _tq()
    rng = np.random.default_rng(9)
    d, bits, h, bs, nblk, t = 128, 4, 2, 16, 6, 90
    raw = rng.standard_normal((t, h, d)).astype(np.float32)
    signs = o.splitmix64_signs(d, 42)
    c32, _ = o.codebook_f32(d, bits)
    slots = rng.permutation(nblk * bs)[:t].astype(np.int64)
    pages = o.write_kv(raw, np.zeros((nblk, bs, h, o.row_bytes(d, bits)), dtype=np.uint8), slots, signs, c32, bits)
    dev = torch.device("cuda")
    out = tq.tq_dequant_rows(torch.from_numpy(pages).to(dev), torch.from_numpy(slots).to(dev),
                             torch.from_numpy(signs.astype(np.float32)).to(dev), torch.from_numpy(c32).to(dev),
                             out_dtype=torch.float32)
    want = o.dequant_slots(pages, slots, signs, c32, bits)
    _check(out, want, _norms_at(pages, slots), torch.float32)
    rel = np.linalg.norm(out.cpu().numpy() - raw, axis=-1) / np.linalg.norm(raw, axis=-1)
    assert float(np.mean(rel ** 2)) < 0.02  # 4-bit MSE distortion of a unit-norm direction is ~0.01


@pytest.mark.slow
def test_dequant_full_size_sampled():
    # the 64 x 8192 K4 D128 cache (32768 blocks x 16 x 8 heads): every row read back on the
    # GPU, 512 sampled tokens compared with the oracle
    tq = _tq()
    rng = np.random.default_rng(44)
    d, bits, h, bs, nblk = 128, 4, 8, 16, 32768
    rb = o.row_bytes(d, bits)
    pages = rng.integers(0, 256, size=(nblk, bs, h, rb), dtype=np.uint8)
    nu = rng.lognormal(0.0, 1.0, size=(nblk, bs, h)).astype(np.float32)
    pages[..., rb - 4:] = nu[..., None].view(np.uint8).reshape(nblk, bs, h, 4)
    t = nblk * bs
    slots = rng.permutation(t).astype(np.int64)
    signs = o.splitmix64_signs(d, 42)
    c32, _ = o.codebook_f32(d, bits)
    dev = torch.device("cuda")
    out = tq.tq_dequant_rows(torch.from_numpy(pages).to(dev), torch.from_numpy(slots).to(dev),
                             torch.from_numpy(signs.astype(np.float32)).to(dev), torch.from_numpy(c32).to(dev),
                             out_dtype=torch.float16)
    pick = rng.choice(t, size=512, replace=False)
    got = out[torch.from_numpy(pick).to(dev)]
    want = o.dequant_slots(pages, slots[pick], signs, c32, bits)
    _check(got, want, _norms_at(pages, slots[pick]), torch.float16)
