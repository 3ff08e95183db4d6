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
