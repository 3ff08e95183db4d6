"""GPU parity at head_dim 16, the smallest head size of the boundary ("vLLM Usage", TQ Byte
Layout: ceil(16 b / 8) + 4 bytes per row, 8 to 14 bytes -- rows of 3 and 5 bits are not a
whole number of 32-bit words).  Writer, decode, prefill, readback and the int8 query
quantiser against the oracle, with the bars of the other head sizes (tests/parity.py)."""

import numpy as np
import pytest
import torch

from oracle import int8q_oracle as iq
from oracle import tq_oracle as o
from parity import OracleCodec, assert_decode_close, assert_rows_match, compare_rows

pytestmark = pytest.mark.gpu

D = 16


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _layout(rng, lens, bs):
    nblk = int(sum(-(-n // bs) for n in lens)) + 2
    maxb = max(1, max(-(-n // bs) for n in lens))
    perm = rng.permutation(nblk).astype(np.int32)
    bt = np.zeros((len(lens), maxb), dtype=np.int32)
    slots, pos = [], 0
    for b, n in enumerate(lens):
        nb = -(-n // bs)
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
        t = np.arange(n)
        slots.append(bt[b, t // bs].astype(np.int64) * bs + t % bs)
    return nblk, bt, np.concatenate(slots)


@pytest.mark.parametrize("bits", [2, 3, 4, 5])
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_d16_writer_matches_oracle(tq, bits, dtype):
    rng = np.random.default_rng(16 + bits)
    t, h, bs = 400, 3, 16
    nb = -(-t // bs) + 2
    raw32 = (rng.standard_normal((t, h, D)) * rng.lognormal(0, 0.5, (1, h, D))).astype(np.float32)
    raw32[3, 1] = 0.0
    raw = torch.from_numpy(raw32).to(dtype)
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[::13] = -1
    codec = OracleCodec(D)
    rb = o.row_bytes(D, bits)
    pages = torch.full((nb, bs, h, rb), 0x5A, dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv(raw.cuda(), pages, _dev(slots), _dev(codec.signs.astype(np.float32)),
                        _dev(codec.centroids(bits)), check=False)
    assert int(st.item()) == 0
    pg = pages.cpu().numpy().reshape(nb * bs, h, rb)
    written = np.zeros(nb * bs, dtype=bool)
    written[slots[slots >= 0]] = True
    assert np.all(pg[~written] == 0x5A)
    tok = np.nonzero(slots >= 0)[0]
    stats = compare_rows(pg[slots[tok]].reshape(-1, rb), raw.double().numpy()[tok].reshape(-1, D), codec, bits)
    assert_rows_match(stats)
    # a slot past the pages: nothing written, the error reported
    bad = slots.copy()
    bad[7] = nb * bs
    before = pages.clone()
    st = tq.tq_write_kv(raw.cuda(), pages, _dev(bad), _dev(codec.signs.astype(np.float32)), _dev(codec.centroids(bits)),
                        check=False)
    assert int(st.item()) == tq.TQ_ERR_SLOT_OUT_OF_RANGE and torch.equal(pages, before)


@pytest.mark.parametrize("kb,vb,hq,h,bs", [(4, 4, 8, 2, 16), (3, 5, 4, 4, 5), (2, 3, 8, 1, 16), (5, 2, 2, 1, 8)])
def test_d16_decode_prefill_and_readback_match_oracle(tq, kb, vb, hq, h, bs):
    rng = np.random.default_rng(100 * kb + vb)
    lens = [0, 1, 29, 250, 1030]
    nblk, bt, slots = _layout(rng, lens, bs)
    codec = OracleCodec(D)
    signs = _dev(codec.signs.astype(np.float32))
    pages = []
    for bits in (kb, vb):
        raw = torch.from_numpy((rng.standard_normal((slots.size, h, D)) * rng.lognormal(0, .5, (1, h, D))).astype(np.float16))
        pg = torch.full((nblk, bs, h, o.row_bytes(D, bits)), 0xFF, dtype=torch.uint8, device="cuda")
        tq.tq_write_kv(raw.cuda(), pg, _dev(slots), signs, _dev(codec.centroids(bits)))
        pages.append(pg)
    kp, vp = pages[0].cpu().numpy(), pages[1].cpu().numpy()
    kc, vc = _dev(codec.centroids(kb)), _dev(codec.centroids(vb))
    q = rng.standard_normal((len(lens), hq, D)).astype(np.float32)
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = tq.tq_paged_decode(_dev(q), pages[0], pages[1], _dev(bt), _dev(np.array(lens, np.int32)), signs, kc, vc,
                             status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = o.paged_decode(q, kp, vp, kb, vb, bt, np.array(lens), codec.signs, codec.centroids(kb), codec.centroids(vb))
    assert_decode_close(got.cpu().numpy(), ref)
    # prefill rows: the last tokens of the longer sequences
    q_seq = np.array([3, 3, 3, 4, 4, 2], dtype=np.int32)
    q_len = np.array([248, 249, 250, 1, 1030, 29], dtype=np.int32)
    qp = rng.standard_normal((q_seq.size, hq, D)).astype(np.float32)
    got = tq.tq_paged_prefill(_dev(qp), _dev(q_seq), _dev(q_len), pages[0], pages[1], _dev(bt), signs, kc, vc)
    torch.cuda.synchronize()
    ref = o.paged_prefill(qp, q_seq, q_len, kp, vp, kb, vb, bt, codec.signs, codec.centroids(kb), codec.centroids(vb))
    assert_decode_close(got.cpu().numpy(), ref)
    # int8 query rows
    codes, scales = tq.tq_quantize_queries_int8(_dev(qp))
    want_c, want_s = iq.quantize_queries_int8(qp)
    assert np.array_equal(codes.cpu().numpy(), want_c) and np.array_equal(scales.cpu().numpy(), want_s)
    got = tq.tq_paged_prefill_int8q(codes, scales, _dev(q_seq), _dev(q_len), pages[0], pages[1], _dev(bt), signs, kc, vc,
                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = iq.paged_prefill_int8q(want_c, want_s, q_seq, q_len, kp, vp, kb, vb, bt, codec.signs, codec.centroids(kb),
                                 codec.centroids(vb))
    assert_decode_close(got.cpu().numpy(), ref)
    # readback of every written row
    out = tq.tq_dequant_rows(pages[0], _dev(slots), signs, kc, out_dtype=torch.float32)
    torch.cuda.synchronize()
    want = o.dequant_slots(kp, slots, codec.signs, codec.centroids(kb), kb)
    assert np.allclose(out.cpu().numpy(), want, rtol=2e-6, atol=2e-6 * np.abs(want).max())
    # a block id outside the pages: its tokens are left out, the status says so
    bad = bt.copy()
    bad[4, 3] = nblk + 9
    got = tq.tq_paged_decode(_dev(q), pages[0], pages[1], _dev(bad), _dev(np.array(lens, np.int32)), signs, kc, vc,
                             status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tq.TQ_ERR_BLOCK_OUT_OF_RANGE
    ref = o.paged_decode(q, kp, vp, kb, vb, bad, np.array(lens), codec.signs, codec.centroids(kb), codec.centroids(vb))
    assert_decode_close(got.cpu().numpy(), ref)
