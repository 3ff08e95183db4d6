"""GPU parity of tq_paged_prefill (mixed prefill/decode over the packed cache) against the
fp64 oracle.  Pages are written by the oracle's writer or drawn as seeded random rows;
tolerance |gpu - oracle| <= 2e-3 + 2e-3 |oracle| as for the decode.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import tq_oracle as o  # noqa: E402

pytestmark = pytest.mark.gpu


def _tq():
    import quantized_kv_cache_06_gb300 as tq

    return tq


def _cache(rng, lens, d, h, kb, vb, bs=16, random_rows=False):
    nblk = int(sum(-(-int(n) // bs) for n in lens)) + 3
    maxb = max(-(-int(n) // bs) for n in lens)
    bt = np.zeros((len(lens), maxb), dtype=np.int32)
    perm = rng.permutation(nblk).astype(np.int32)
    pos = 0
    for b, n in enumerate(lens):
        nb = -(-int(n) // bs)
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
    signs = o.splitmix64_signs(d, 42)
    kc, _ = o.codebook_f32(d, kb)
    vc, _ = o.codebook_f32(d, vb)
    pages = []
    for bits, cents in ((kb, kc), (vb, vc)):
        if random_rows:
            n = nblk * bs * h
            idx = rng.integers(0, 1 << bits, size=(n, d))
            nu = rng.lognormal(0.0, 0.5, size=n).astype(np.float32)
            pages.append(o.make_rows(idx, nu, bits).reshape(nblk, bs, h, -1))
        else:
            pg = np.zeros((nblk, bs, h, o.row_bytes(d, bits)), dtype=np.uint8)
            for b, n in enumerate(lens):
                slots = np.array([bt[b, t // bs] * bs + t % bs for t in range(n)], dtype=np.int64)
                raw = rng.standard_normal((n, h, d)) * rng.lognormal(0.0, 0.5, size=(1, h, d))
                pg = o.write_kv(raw.astype(np.float32), pg, slots, signs, cents, bits)
            pages.append(pg)
    return bt, signs, kc, vc, pages[0], pages[1]


def _rows_for(lens, chunks):
    """Query rows: the last chunks[b] tokens of sequence b (chunk 1 = a decode row)."""
    q_seq, q_len = [], []
    for b, (n, c) in enumerate(zip(lens, chunks)):
        for i in range(c):
            q_seq.append(b)
            q_len.append(n - c + 1 + i)
    return np.array(q_seq, dtype=np.int32), np.array(q_len, dtype=np.int32)


def _run(tq, q, q_seq, q_len, kp, vp, bt, signs, kc, vc, status=None):
    dev = torch.device("cuda")
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)  # noqa: E731
    out = tq.tq_paged_prefill(t(q), t(q_seq), t(q_len), t(kp), t(vp), t(bt), t(signs.astype(np.float32)), t(kc),
                              t(vc), out_dtype=torch.float32, status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def _close(got, want):
    err = np.abs(got - want)
    tol = 2e-3 + 2e-3 * np.abs(want)
    assert np.all(err <= tol), float(np.max(err / tol))


@pytest.mark.parametrize("d,kb,vb,hq,h", [(128, 4, 4, 32, 8), (128, 4, 2, 16, 2), (64, 4, 4, 8, 2),
                                          (128, 3, 3, 8, 2), (256, 4, 4, 8, 1)])
def test_prefill_matches_oracle(d, kb, vb, hq, h):
    tq = _tq()
    rng = np.random.default_rng(70 + d + kb + vb + hq)
    lens = [37, 16, 1, 70, 5]
    chunks = [9, 16, 1, 1, 3]  # chunks of several tokens and decode rows; a chunk of a whole sequence
    bt, signs, kc, vc, kp, vp = _cache(rng, lens, d, h, kb, vb)
    q_seq, q_len = _rows_for(lens, chunks)
    q = rng.standard_normal((len(q_seq), hq, d)).astype(np.float32)
    want = o.paged_prefill(q, q_seq, q_len, kp, vp, kb, vb, bt, signs, kc, vc)
    _close(_run(tq, q, q_seq, q_len, kp, vp, bt, signs, kc, vc), want)


def test_prefill_bad_row_and_empty_row():
    tq = _tq()
    rng = np.random.default_rng(81)
    d, kb, vb, hq, h = 128, 4, 4, 32, 8
    lens = [33, 20]
    bt, signs, kc, vc, kp, vp = _cache(rng, lens, d, h, kb, vb)
    q_seq = np.array([0, 5, 1, 1, -1], dtype=np.int32)  # rows 1 and 4 point outside the table
    q_len = np.array([33, 4, 0, 20, 7], dtype=np.int32)  # row 2 sees no token
    q = rng.standard_normal((5, hq, d)).astype(np.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(tq, q, q_seq, q_len, kp, vp, bt, signs, kc, vc, status=status)
    assert int(status.item()) == tq.TQ_ERR_INVALID_ARG
    assert np.all(got[[1, 2, 4]] == 0)
    ok = [0, 3]
    want = o.paged_prefill(q[ok], q_seq[ok], q_len[ok], kp, vp, kb, vb, bt, signs, kc, vc)
    _close(got[ok], want)


@pytest.mark.slow
def test_prefill_chunk_on_large_cache_sampled():
    # 16 sequences x 4096 tokens (random packed rows), a 64-token chunk at the end of each:
    # 1024 query rows on the GPU, 24 sampled rows checked against the oracle
    tq = _tq()
    rng = np.random.default_rng(90)
    d, kb, vb, hq, h = 128, 4, 4, 32, 8
    lens = [4096] * 16
    bt, signs, kc, vc, kp, vp = _cache(rng, lens, d, h, kb, vb, random_rows=True)
    q_seq, q_len = _rows_for(lens, [64] * 16)
    q = rng.standard_normal((len(q_seq), hq, d)).astype(np.float32)
    got = _run(tq, q, q_seq, q_len, kp, vp, bt, signs, kc, vc)
    pick = rng.choice(len(q_seq), size=24, replace=False)
    want = o.paged_prefill(q[pick], q_seq[pick], q_len[pick], kp, vp, kb, vb, bt, signs, kc, vc)
    _close(got[pick], want)


# ---- the multi-query kernel (D 64/128/256, 2/4-bit or equal 3/5-bit K and V, G 1/2/4/8, any
# block size; D 256 splits each row group's dimensions over two warps) ------------------------

@pytest.mark.parametrize("d,kb,vb,hq,h,bs", [(128, 4, 4, 8, 8, 16), (128, 4, 4, 16, 8, 16), (128, 2, 2, 32, 8, 16),
                                             (128, 2, 4, 32, 4, 16), (64, 2, 4, 16, 2, 8), (128, 4, 2, 64, 8, 32),
                                             (64, 4, 4, 8, 8, 5), (128, 3, 3, 32, 8, 16), (64, 5, 5, 16, 4, 16),
                                             (256, 4, 4, 32, 8, 16), (256, 3, 3, 16, 4, 16), (256, 5, 5, 8, 8, 8),
                                             (256, 2, 4, 64, 8, 16)])
def test_prefill_multi_query_shapes(d, kb, vb, hq, h, bs):
    # windows of 64 / G query rows hold rows of several sequences (segments), chunks of
    # several tokens, decode rows and a whole-sequence chunk
    tq = _tq()
    rng = np.random.default_rng(400 + d + 3 * kb + 5 * vb + hq + bs)
    lens = [37, 16, 1, 70, 5, 130]
    chunks = [9, 16, 1, 1, 3, 40]
    bt, signs, kc, vc, kp, vp = _cache(rng, lens, d, h, kb, vb, bs=bs)
    q_seq, q_len = _rows_for(lens, chunks)
    q = rng.standard_normal((len(q_seq), hq, d)).astype(np.float32)
    want = o.paged_prefill(q, q_seq, q_len, kp, vp, kb, vb, bt, signs, kc, vc)
    _close(_run(tq, q, q_seq, q_len, kp, vp, bt, signs, kc, vc), want)


def test_prefill_multi_query_unsorted_rows_and_token_splits():
    # 3 sequences of up to 3000 tokens in a 4096-token table: the kernel splits the
    # tokens (several partials per row); query rows in random order, so windows mix
    # sequences; fp16 query and output
    tq = _tq()
    rng = np.random.default_rng(77)
    d, kb, vb, hq, h = 128, 4, 4, 32, 8
    lens = [3000, 2100, 1500]
    bt, signs, kc, vc, kp, vp = _cache(rng, lens, d, h, kb, vb, random_rows=True)
    bt = np.concatenate([bt, np.zeros((3, 256 - bt.shape[1]), dtype=np.int32)], axis=1)  # 4096-token table
    q_seq, q_len = _rows_for(lens, [70, 33, 20])
    perm = rng.permutation(len(q_seq))
    q_seq, q_len = q_seq[perm], q_len[perm]
    q = rng.standard_normal((len(q_seq), hq, d)).astype(np.float16)
    dev = torch.device("cuda")
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)  # noqa: E731
    out = tq.tq_paged_prefill(t(q), t(q_seq), t(q_len), t(kp), t(vp), t(bt), t(signs.astype(np.float32)), t(kc),
                              t(vc), out_dtype=torch.float32)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    pick = rng.choice(len(q_seq), size=24, replace=False)
    want = o.paged_prefill(q[pick].astype(np.float32), q_seq[pick], q_len[pick], kp, vp, kb, vb, bt, signs, kc, vc)
    _close(got[pick], want)


def test_prefill_multi_query_large_norm_rows():
    # lognormal(0, 1) norms with 2% of rows x 8 and a query x 3: many tiles exceed the
    # fast-score bound and take the exact key path
    tq = _tq()
    rng = np.random.default_rng(12)
    d, kb, vb, hq, h, bs = 128, 4, 2, 32, 8, 16
    lens = [300, 77]
    nblk = sum(-(-n // bs) for n in lens) + 2
    bt = np.zeros((2, -(-max(lens) // bs)), dtype=np.int32)
    perm = rng.permutation(nblk).astype(np.int32)
    bt[0, :-(-lens[0] // bs)] = perm[:-(-lens[0] // bs)]
    bt[1, :-(-lens[1] // bs)] = perm[-(-lens[0] // bs):-(-lens[0] // bs) + -(-lens[1] // bs)]
    signs = o.splitmix64_signs(d, 42)
    kc, _ = o.codebook_f32(d, kb)
    vc, _ = o.codebook_f32(d, vb)
    pages = []
    for bits in (kb, vb):
        n = nblk * bs * h
        nu = rng.lognormal(0.0, 1.0, size=n) * np.where(rng.random(n) < 0.02, 8.0, 1.0)
        pages.append(o.make_rows(rng.integers(0, 1 << bits, size=(n, d)), nu.astype(np.float32), bits)
                     .reshape(nblk, bs, h, -1))
    q_seq, q_len = _rows_for(lens, [20, 7])
    q = 3.0 * rng.standard_normal((len(q_seq), hq, d)).astype(np.float32)
    want = o.paged_prefill(q, q_seq, q_len, pages[0], pages[1], kb, vb, bt, signs, kc, vc)
    _close(_run(tq, q, q_seq, q_len, pages[0], pages[1], bt, signs, kc, vc), want)


def test_prefill_multi_query_bad_block_is_skipped_and_reported():
    tq = _tq()
    rng = np.random.default_rng(31)
    d, kb, vb, hq, h = 128, 4, 4, 32, 8
    lens = [90, 40]
    bt, signs, kc, vc, kp, vp = _cache(rng, lens, d, h, kb, vb)
    bt[0, 2] = kp.shape[0] + 7  # tokens 32..47 of sequence 0 point outside the pages
    q_seq, q_len = _rows_for(lens, [12, 5])
    q = rng.standard_normal((len(q_seq), hq, d)).astype(np.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(tq, q, q_seq, q_len, kp, vp, bt, signs, kc, vc, status=status)
    assert int(status.item()) == tq.TQ_ERR_BLOCK_OUT_OF_RANGE
    want, bad = o.paged_prefill(q, q_seq, q_len, kp, vp, kb, vb, bt, signs, kc, vc, return_flags=True)
    assert bad
    _close(got, want)
