"""GPU tests of the status paths of the C ABI.

* A write called without a status word ("vLLM Usage", Slot Mapping: a slot outside the
  allocated pages raises) returns the slot error itself, having written nothing, and
  otherwise writes exactly what the asynchronous form writes.
* Failure detection without a fault: every device-side wait of the tensor-core decode is
  bounded.  With the tries of those waits set to 0 (tq_set_wait_limit) each one gives up
  at once, the decode reports TQ_ERR_TIMEOUT in its status word and returns, and the
  next decode with the default limit is correct (the context stays usable).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import tq_oracle as o  # noqa: E402
from parity import OracleCodec, assert_decode_close  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


def _raw_write(tq, fn, raw, slots, pages, signs, centroids, extra=()):
    """Calls the C entry point with status_dev = NULL on the current stream."""
    from quantized_kv_cache_06_gb300 import _lib

    t, h, d = raw.shape
    bits = centroids.numel().bit_length() - 1 + (1 if extra else 0)
    args = [raw.data_ptr(), _lib._DTYPES[raw.dtype], t, h, d, bits, slots.data_ptr(), pages.data_ptr(),
            pages.shape[0], pages.shape[1], signs.data_ptr(), centroids.data_ptr()]
    args += [e.data_ptr() for e in extra]
    args += [None, torch.cuda.current_stream().cuda_stream]
    return getattr(tq.lib(), fn)(*args)


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_write_without_status_word_returns_the_slot_error(tq, dtype):
    rng = np.random.default_rng(5)
    d, h, bits, nb, bs = 128, 4, 4, 6, 16
    raw = torch.from_numpy(rng.standard_normal((40, h, d)).astype(np.float32)).to(dtype).cuda()
    slots = torch.from_numpy(rng.permutation(nb * bs)[:40].astype(np.int64)).cuda()
    signs = tq.tq_build_rotation(d, 42, "cuda")
    cents = tq.tq_codebook(d, bits, "cuda")[0]
    ref = torch.zeros(nb, bs, h, tq.tq_row_bytes(d, bits), dtype=torch.uint8, device="cuda")
    tq.tq_write_kv(raw, ref, slots, signs, cents)
    pages = torch.zeros_like(ref)
    assert _raw_write(tq, "tq_write_kv", raw, slots, pages, signs, cents) == tq.TQ_OK
    assert torch.equal(pages, ref)
    bad = slots.clone()
    bad[17] = nb * bs  # one past the end
    before = torch.full_like(ref, 0x3C)
    pages = before.clone()
    assert _raw_write(tq, "tq_write_kv", raw, bad, pages, signs, cents) == tq.TQ_ERR_SLOT_OUT_OF_RANGE
    assert "no row was written" in tq.lib().tq_last_error().decode()
    assert torch.equal(pages, before)
    # the library's status word is reset by the next call
    assert _raw_write(tq, "tq_write_kv", raw, slots, pages, signs, cents) == tq.TQ_OK


def test_product_key_write_without_status_word(tq):
    rng = np.random.default_rng(6)
    d, h, bits, nb, bs = 64, 2, 4, 4, 16
    raw = torch.from_numpy(rng.standard_normal((30, h, d)).astype(np.float16)).cuda()
    slots = torch.from_numpy(rng.permutation(nb * bs)[:30].astype(np.int64)).cuda()
    signs = tq.tq_build_rotation(d, 42, "cuda")
    cents = tq.tq_codebook(d, bits - 1, "cuda")[0]
    s_mat = tq.tq_build_qjl_matrix(d, 43, "cuda")
    ref = torch.zeros(nb, bs, h, tq.tq_prod_row_bytes(d, bits), dtype=torch.uint8, device="cuda")
    tq.tq_write_kv_prod(raw, ref, slots, signs, cents, s_mat)
    pages = torch.zeros_like(ref)
    assert _raw_write(tq, "tq_write_kv_prod", raw, slots, pages, signs, cents, extra=(s_mat,)) == tq.TQ_OK
    assert torch.equal(pages, ref)
    bad = slots.clone()
    bad[0] = 10 ** 9
    pages = torch.full_like(ref, 0x11)
    assert _raw_write(tq, "tq_write_kv_prod", raw, bad, pages, signs, cents, extra=(s_mat,)) == \
        tq.TQ_ERR_SLOT_OUT_OF_RANGE
    assert bool(torch.all(pages == 0x11))


def test_decode_wait_timeout_is_reported_and_the_next_call_is_correct(tq):
    # tensor-core decode shape (D 128, K4/V4, group 4, block 16) over several blocks
    rng = np.random.default_rng(12)
    d, h, hq, bs, kb, vb = 128, 2, 8, 16, 4, 4
    lens = np.array([700, 333, 1024], dtype=np.int32)
    nblk = int(sum(-(-n // bs) for n in lens)) + 2
    perm = rng.permutation(nblk).astype(np.int32)
    maxb = max(-(-int(n) // bs) for n in lens)
    bt = np.zeros((len(lens), maxb), dtype=np.int32)
    slots, pos = [], 0
    for b, n in enumerate(lens):
        nbk = -(-int(n) // bs)
        bt[b, :nbk] = perm[pos:pos + nbk]
        pos += nbk
        t = np.arange(n)
        slots.append(bt[b, t // bs].astype(np.int64) * bs + t % bs)
    slots = np.concatenate(slots)
    codec = OracleCodec(d)
    signs = torch.from_numpy(codec.signs).float().cuda()
    kc, vc = torch.from_numpy(codec.centroids(kb)).cuda(), torch.from_numpy(codec.centroids(vb)).cuda()
    pages = []
    for c in (kc, vc):
        raw = torch.from_numpy(rng.standard_normal((slots.size, h, d)).astype(np.float16)).cuda()
        pg = torch.zeros(nblk, bs, h, tq.tq_row_bytes(d, 4), dtype=torch.uint8, device="cuda")
        tq.tq_write_kv(raw, pg, torch.from_numpy(slots).cuda(), signs, c)
        pages.append(pg)
    q = torch.from_numpy(rng.standard_normal((len(lens), hq, d)).astype(np.float32)).cuda()
    btt, lt = torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda()
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")

    def decode():
        out = tq.tq_paged_decode(q, pages[0], pages[1], btt, lt, signs, kc, vc, status=st)
        torch.cuda.synchronize()
        return out.cpu().numpy(), int(st.item())

    first, code = decode()
    assert code == tq.TQ_OK
    default = tq.tq_set_wait_limit(0)
    try:
        _, code = decode()
    finally:
        tq.tq_set_wait_limit(-1)
    assert code == tq.TQ_ERR_TIMEOUT
    again, code = decode()
    assert code == tq.TQ_OK
    assert np.array_equal(again, first)  # same launch, same arithmetic
    ref = o.paged_decode(q.cpu().numpy(), pages[0].cpu().numpy(), pages[1].cpu().numpy(), kb, vb, bt, lens,
                         codec.signs, codec.centroids(kb), codec.centroids(vb))
    assert_decode_close(again, ref)
    assert tq.tq_set_wait_limit(-1) == default
