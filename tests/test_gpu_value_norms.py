"""GPU parity for rows of any norm ("vLLM Usage", TQ Packed Page Contract: the writer takes
arbitrary K/V tensors, so nothing bounds a row's norm).

Value rows whose norms span 1e-3 .. 1e5 (and key rows over a wide range too) are written
from fp32 and bf16 raw rows by tq_write_kv, then read by tq_paged_decode and
tq_paged_prefill and compared element by element with the oracle on the very page bytes
the GPU wrote, at |gpu - oracle| <= 2e-3 + 2e-3 |oracle|.  The shapes route to every
decode kernel: the tensor-core decode (D 64/128/256, G 4/8), the multi-query kernel (3-
and 5-bit rows, G 2) and the SIMT decode (D 256 at 5 bits).

The pages start as 0xFF bytes and the sequence lengths are not multiples of the block
size, so the rows past a sequence's end inside its last block hold NaN norms: the decode
must mask them out, score and value alike.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import tq_oracle as o  # noqa: E402
from parity import OracleCodec, assert_decode_close, assert_rows_match, compare_rows  # noqa: E402

pytestmark = pytest.mark.gpu

LENS = [37, 301, 1000, 16, 5]
BS = 16

# (D, k_bits, v_bits, Hq, H): tensor-core decode (4/4 G4, 4/2 G8, D256 2/4, D64 4/4, 3/3 G4,
# D256 5/5 G4, 5/5 G8, D256 3/3 G8, D64 3/2 G8, D64 5/3 G4), multi-query kernel (D64 5/5 G2),
# SIMT decode (D256 5/5 G2)
SHAPES = [(128, 4, 4, 8, 2), (128, 4, 2, 16, 2), (256, 2, 4, 8, 2), (64, 4, 4, 8, 2),
          (128, 3, 3, 8, 2), (64, 5, 5, 4, 2), (256, 5, 5, 8, 2), (128, 5, 5, 16, 2), (256, 3, 3, 16, 2),
          (256, 5, 5, 4, 2), (64, 3, 2, 16, 2), (64, 5, 3, 8, 2)]


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


def _rows(rng, n, h, d, lo, hi):
    """Rows with uniformly random directions and norms 10^U(lo, hi)."""
    x = rng.standard_normal((n, h, d))
    x /= np.linalg.norm(x, axis=2, keepdims=True)
    return x * 10.0 ** rng.uniform(lo, hi, size=(n, h, 1))


def _layout(rng):
    nblk = sum(-(-n // BS) for n in LENS) + 4
    maxb = max(-(-n // BS) for n in LENS)
    perm = rng.permutation(nblk).astype(np.int32)
    bt = np.zeros((len(LENS), maxb), dtype=np.int32)
    slots, pos = [], 0
    for b, n in enumerate(LENS):
        nb = -(-n // BS)
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
        t = np.arange(n)
        slots.append(bt[b, t // BS].astype(np.int64) * BS + t % BS)
    return nblk, bt, np.concatenate(slots)


def _write(tq, raw_t, slots, nblk, bits, codec):
    d = raw_t.shape[2]
    pages = torch.full((nblk, BS, raw_t.shape[1], o.row_bytes(d, bits)), 0xFF, dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv(raw_t.cuda(), pages, torch.from_numpy(slots).cuda(), torch.from_numpy(codec.signs).float().cuda(),
                        torch.from_numpy(codec.centroids(bits)).cuda())
    assert int(st.item()) == 0
    return pages


def _case(tq, d, kb, vb, hq, h, dtype, key_range, seed):
    rng = np.random.default_rng(seed)
    codec = OracleCodec(d)
    nblk, bt, slots = _layout(rng)
    t = slots.shape[0]
    k32 = _rows(rng, t, h, d, *key_range).astype(np.float32)
    v32 = _rows(rng, t, h, d, -3.0, 5.0).astype(np.float32)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    k_t, v_t = torch.from_numpy(k32).to(tdt), torch.from_numpy(v32).to(tdt)
    kp = _write(tq, k_t, slots, nblk, kb, codec)
    vp = _write(tq, v_t, slots, nblk, vb, codec)
    kp_np, vp_np = kp.cpu().numpy(), vp.cpu().numpy()
    # the writer on these rows: indices and norms against the oracle (exact raw values)
    flat_k = kp_np.reshape(nblk * BS, h, -1)[slots].reshape(t * h, -1)
    flat_v = vp_np.reshape(nblk * BS, h, -1)[slots].reshape(t * h, -1)
    assert_rows_match(compare_rows(flat_k, k_t.float().numpy().astype(np.float64).reshape(t * h, d), codec, kb))
    assert_rows_match(compare_rows(flat_v, v_t.float().numpy().astype(np.float64).reshape(t * h, d), codec, vb))
    return codec, bt, kp, vp, kp_np, vp_np


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,kb,vb,hq,h", SHAPES, ids=[f"d{s[0]}_k{s[1]}v{s[2]}_g{s[3] // s[4]}" for s in SHAPES])
def test_decode_any_value_norm(tq, d, kb, vb, hq, h, dtype):
    codec, bt, kp, vp, kp_np, vp_np = _case(tq, d, kb, vb, hq, h, dtype, (-1.0, 2.0), seed=d + 10 * kb + vb)
    rng = np.random.default_rng(7)
    q = rng.standard_normal((len(LENS), hq, d)).astype(np.float32)
    lens = np.array(LENS, dtype=np.int32)
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = tq.tq_paged_decode(torch.from_numpy(q).cuda(), kp, vp, torch.from_numpy(bt).cuda(),
                             torch.from_numpy(lens).cuda(), torch.from_numpy(codec.signs).float().cuda(),
                             torch.from_numpy(codec.centroids(kb)).cuda(), torch.from_numpy(codec.centroids(vb)).cuda(),
                             status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = o.paged_decode(q, kp_np, vp_np, kb, vb, bt, lens, codec.signs, codec.centroids(kb), codec.centroids(vb))
    assert np.abs(ref).max() > 1e3  # the large-norm rows do reach the outputs
    assert_decode_close(got.cpu().numpy(), ref)


@pytest.mark.parametrize("d,kb,vb,hq,h", [(128, 4, 4, 8, 2), (128, 4, 2, 16, 2), (64, 5, 5, 4, 2), (256, 2, 4, 8, 2)])
def test_decode_wide_key_and_value_norms(tq, d, kb, vb, hq, h):
    # keys as wide as the values: scores from ~0 to ~1e5 (the exact key and value paths
    # together, and tiles that are almost one-hot)
    codec, bt, kp, vp, kp_np, vp_np = _case(tq, d, kb, vb, hq, h, "f32", (-3.0, 5.0), seed=99 + d)
    rng = np.random.default_rng(8)
    q = rng.standard_normal((len(LENS), hq, d)).astype(np.float32)
    lens = np.array(LENS, dtype=np.int32)
    got = tq.tq_paged_decode(torch.from_numpy(q).cuda(), kp, vp, torch.from_numpy(bt).cuda(),
                             torch.from_numpy(lens).cuda(), torch.from_numpy(codec.signs).float().cuda(),
                             torch.from_numpy(codec.centroids(kb)).cuda(), torch.from_numpy(codec.centroids(vb)).cuda())
    torch.cuda.synchronize()
    ref = o.paged_decode(q, kp_np, vp_np, kb, vb, bt, lens, codec.signs, codec.centroids(kb), codec.centroids(vb))
    assert_decode_close(got.cpu().numpy(), ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d,kb,vb,hq,h", [(128, 4, 4, 8, 2), (128, 4, 2, 16, 2), (128, 3, 3, 8, 2),
                                          (64, 5, 5, 4, 2), (256, 4, 4, 8, 2)])
def test_prefill_any_value_norm(tq, d, kb, vb, hq, h, dtype):
    codec, bt, kp, vp, kp_np, vp_np = _case(tq, d, kb, vb, hq, h, dtype, (-1.0, 2.0), seed=3 * d + kb)
    # the last tokens of every sequence as a prefill chunk (one row: a decode row)
    chunks = [5, 17, 33, 1, 3]
    q_seq = np.concatenate([np.full(c, b) for b, c in enumerate(chunks)]).astype(np.int32)
    q_len = np.concatenate([np.arange(n - c + 1, n + 1) for n, c in zip(LENS, chunks)]).astype(np.int32)
    rng = np.random.default_rng(11)
    q = rng.standard_normal((q_seq.shape[0], hq, d)).astype(np.float32)
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = tq.tq_paged_prefill(torch.from_numpy(q).cuda(), torch.from_numpy(q_seq).cuda(),
                              torch.from_numpy(q_len).cuda(), kp, vp, torch.from_numpy(bt).cuda(),
                              torch.from_numpy(codec.signs).float().cuda(), torch.from_numpy(codec.centroids(kb)).cuda(),
                              torch.from_numpy(codec.centroids(vb)).cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = o.paged_prefill(q, q_seq, q_len, kp_np, vp_np, kb, vb, bt, codec.signs, codec.centroids(kb),
                          codec.centroids(vb))
    assert np.abs(ref).max() > 1e3
    assert_decode_close(got.cpu().numpy(), ref)
