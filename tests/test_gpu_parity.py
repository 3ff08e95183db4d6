"""GPU parity: the CUDA writer and decode (through the C ABI) against the CPU oracle
on the same seeded inputs, for the five workloads and the edge cases.

Writer: packed index bytes bit-exact except near-boundary coordinates (counted),
norms to 1e-6 relative.  Decode: |gpu - oracle| <= 2e-3 + 2e-3 |oracle|; the oracle
decodes the very page bytes the GPU wrote.
"""

import numpy as np
import pytest
import torch

from oracle import tq_oracle as o
from parity import MAX_FLIP_FRACTION, OracleCodec, assert_decode_close, assert_rows_match, compare_rows
from quantized_kv_cache_06_gb300.workloads import SWEEP, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


def lib_codebook(tq, d, bits):
    return tq.tq_codebook(d, bits, "cuda")[0]


def gpu_write(tq, raw_np, slots_np, num_blocks, block_size, bits, pages=None):
    t, h, d = raw_np.shape
    raw = torch.from_numpy(np.ascontiguousarray(raw_np)).cuda()
    slots = torch.from_numpy(np.ascontiguousarray(slots_np)).cuda()
    if pages is None:
        pages = torch.zeros(num_blocks, block_size, h, tq.tq_row_bytes(d, bits), dtype=torch.uint8, device="cuda")
    signs = tq.tq_build_rotation(d, 42, "cuda")
    st = tq.tq_write_kv(raw, pages, slots, signs, lib_codebook(tq, d, bits), check=False)
    return pages, int(st.item())


def check_written_rows(pages_np, raw_np, slots_np, bits, codec, sample_tokens=None):
    nb, bs, h, rb = pages_np.shape
    flat = pages_np.reshape(nb * bs, h, rb)
    tok = np.nonzero(slots_np >= 0)[0]
    if sample_tokens is not None and tok.size > sample_tokens:
        tok = np.sort(np.random.default_rng(123).choice(tok, sample_tokens, replace=False))
    rows = flat[slots_np[tok]].reshape(-1, rb)
    raw = np.asarray(raw_np[tok], dtype=np.float64).reshape(-1, raw_np.shape[2])
    stats = compare_rows(rows, raw, codec, bits)
    assert_rows_match(stats)
    return stats


def check_untouched(pages_np, slots_np, fill=0):
    nb, bs = pages_np.shape[:2]
    written = np.zeros(nb * bs, dtype=bool)
    written[slots_np[slots_np >= 0]] = True
    assert np.all(pages_np.reshape(nb * bs, -1)[~written] == fill)


def gpu_decode(tq, w, kp, vp, q=None, seq_lens=None, block_table=None, scale=None, out_dtype=None):
    d = w.head_dim
    q = torch.from_numpy(np.ascontiguousarray(w.q if q is None else q)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(w.block_table if block_table is None else block_table)).cuda()
    lens = torch.from_numpy(np.ascontiguousarray(w.seq_lens if seq_lens is None else seq_lens)).cuda()
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    out = tq.tq_paged_decode(q, kp, vp, bt, lens, tq.tq_build_rotation(d, 42, "cuda"), lib_codebook(tq, d, w.k_bits),
                             lib_codebook(tq, d, w.v_bits), scale=scale, out_dtype=out_dtype, status=st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(st.item())


def oracle_decode(w, kp_np, vp_np, codec, heads=None, **kw):
    args = dict(q=w.q, k_pages=kp_np, v_pages=vp_np, k_bits=w.k_bits, v_bits=w.v_bits, block_table=w.block_table,
                seq_lens=w.seq_lens, signs=codec.signs, k_centroids32=codec.centroids(w.k_bits),
                v_centroids32=codec.centroids(w.v_bits), heads=heads)
    args.update(kw)
    return o.paged_decode(**args)


def run_workload(tq, w, sample_tokens=None, heads=None):
    codec = OracleCodec(w.head_dim)
    kp, st = gpu_write(tq, w.k_raw, w.slots, w.num_blocks, w.block_size, w.k_bits)
    assert st == 0
    vp, st = gpu_write(tq, w.v_raw, w.slots, w.num_blocks, w.block_size, w.v_bits)
    assert st == 0
    kp_np, vp_np = kp.cpu().numpy(), vp.cpu().numpy()
    ks = check_written_rows(kp_np, w.k_raw, w.slots, w.k_bits, codec, sample_tokens)
    vs = check_written_rows(vp_np, w.v_raw, w.slots, w.v_bits, codec, sample_tokens)
    check_untouched(kp_np, w.slots)
    check_untouched(vp_np, w.slots)
    got, st = gpu_decode(tq, w, kp, vp)
    assert st == 0
    ref = oracle_decode(w, kp_np, vp_np, codec, heads=heads)
    if heads is not None:
        sel = tuple(np.array(heads).T)
        got, ref = got[sel], ref[sel]
    worst = assert_decode_close(got, ref)
    return ks, vs, worst


# ---------------------------------------------------------------- the five workloads

def test_workload1_tiny(tq):
    w = make_workload(1)
    ks, vs, worst = run_workload(tq, w)
    assert ks["coords"] == 64 * 2 * 128


def test_workload1_rotated_form_and_contract_shape(tq):
    # the contract example: pages [32, 16, 2, 68] at dim 128 / 4 bits
    w = make_workload(1)
    kp, _ = gpu_write(tq, w.k_raw, w.slots, 32, 16, 4)
    assert tuple(kp.shape) == (32, 16, 2, 68)


def test_workload2_mixed_bits(tq):
    w = make_workload(2)
    assert (w.slots < 0).mean() > 0.05
    run_workload(tq, w)


# Full-size workloads: every (sequence, q head) output is compared with the oracle (the
# oracle's cost is per (sequence, kv head), the same for one q head or all of them).  The
# writer is checked on sampled tokens: >= 1e7 coordinates per component for workloads 4
# and 5, where the in-band flip count is held to the strict 1e-5 n.

@pytest.mark.parametrize("sub", range(len(SWEEP)), ids=[f"b{b}_d{d}" for b, d in SWEEP])
def test_workload3_sweep(tq, sub):
    w = make_workload(3, sub=sub)
    run_workload(tq, w, sample_tokens=3000)


def test_workload4_full_size(tq):
    w = make_workload(4)
    ks, vs, _ = run_workload(tq, w, sample_tokens=10000)
    assert ks["coords"] >= 10_000_000 and vs["coords"] >= 10_000_000


def test_workload5_full_size_with_prefill_write(tq):
    w = make_workload(5)
    codec = OracleCodec(w.head_dim)
    ks, vs, _ = run_workload(tq, w, sample_tokens=10000)
    assert ks["coords"] >= 10_000_000 and vs["coords"] >= 10_000_000
    # prefill-style re-write of sequence 0 with 5% negative slots: the skipped rows keep the
    # bytes of the first write, the others hold the new rows
    kp, _ = gpu_write(tq, w.k_raw, w.slots, w.num_blocks, w.block_size, w.k_bits)
    before = kp.cpu().numpy()
    kp, st = gpu_write(tq, w.write_k, w.write_slots, w.num_blocks, w.block_size, w.k_bits, pages=kp)
    assert st == 0
    after = kp.cpu().numpy()
    skipped = w.slots[: w.write_slots.shape[0]][w.write_slots < 0]
    flat_b = before.reshape(-1, before.shape[2], before.shape[3])
    flat_a = after.reshape(-1, after.shape[2], after.shape[3])
    assert np.array_equal(flat_a[skipped], flat_b[skipped])
    st = check_written_rows(after, w.write_k, w.write_slots, w.k_bits, codec, sample_tokens=10000)
    assert st["coords"] >= 10_000_000


# ---------------------------------------------------------------- writer edge cases

def test_write_empty_batch(tq):
    raw = np.zeros((0, 2, 64), dtype=np.float16)
    pages, st = gpu_write(tq, raw, np.zeros(0, dtype=np.int64), 2, 4, 4)
    assert st == 0 and int(pages.sum()) == 0


def test_write_out_of_range_slot_writes_nothing(tq):
    rng = np.random.default_rng(9)
    raw = rng.standard_normal((10, 2, 64)).astype(np.float16)
    slots = np.arange(10, dtype=np.int64)
    slots[7] = 2 * 4  # == num_blocks * block_size: one past the end
    pages = torch.full((2, 4, 2, o.row_bytes(64, 3)), 0x5A, dtype=torch.uint8, device="cuda")
    pages, st = gpu_write(tq, raw, slots, 2, 4, 3, pages=pages)
    assert st == tq.TQ_ERR_SLOT_OUT_OF_RANGE
    assert torch.all(pages == 0x5A)
    with pytest.raises(tq.TQError) as e:
        tq.tq_write_kv(torch.from_numpy(raw).cuda(), pages, torch.from_numpy(slots).cuda(),
                       tq.tq_build_rotation(64, 42, "cuda"), lib_codebook(tq, 64, 3))
    assert e.value.status == tq.TQ_ERR_SLOT_OUT_OF_RANGE


def test_write_all_negative_slots(tq):
    raw = np.random.default_rng(1).standard_normal((6, 2, 128)).astype(np.float16)
    pages, st = gpu_write(tq, raw, -np.ones(6, dtype=np.int64), 2, 4, 4)
    assert st == 0 and int(pages.sum()) == 0


@pytest.mark.parametrize("dtype", [np.float32, "bf16"])
@pytest.mark.parametrize("d,bits", [(32, 5), (64, 3), (256, 2)])
def test_write_dtypes_and_dims(tq, dtype, d, bits):
    rng = np.random.default_rng(d + bits)
    raw32 = (rng.standard_normal((37, 3, d)) * rng.lognormal(0, 0.5, (3, d))).astype(np.float32)
    slots = rng.permutation(40)[:37].astype(np.int64)
    codec = OracleCodec(d)
    if dtype == "bf16":
        raw_t = torch.from_numpy(raw32).to(torch.bfloat16)
        raw_exact = raw_t.float().numpy()
        pages = torch.zeros(10, 4, 3, o.row_bytes(d, bits), dtype=torch.uint8, device="cuda")
        st = tq.tq_write_kv(raw_t.cuda(), pages, torch.from_numpy(slots).cuda(), tq.tq_build_rotation(d, 42, "cuda"),
                            lib_codebook(tq, d, bits), check=False)
        st = int(st.item())
    else:
        raw_exact = raw32
        pages, st = gpu_write(tq, raw32, slots, 10, 4, bits)
    assert st == 0
    check_written_rows(pages.cpu().numpy(), raw_exact, slots, bits, codec)


def test_write_zero_row(tq):
    raw = np.zeros((1, 1, 128), dtype=np.float16)
    pages, st = gpu_write(tq, raw, np.array([0], dtype=np.int64), 1, 1, 4)
    row = pages.cpu().numpy()[0, 0, 0]
    # u = 0 sits on the middle decision point (exactly 0): every index is the lower middle one
    assert np.all(o.unpack_indices(row[None, :64], 128, 4) == 7)
    assert row[64:].tobytes() == b"\0\0\0\0"


# ---------------------------------------------------------------- decode edge cases

def _small_case(tq, d=64, h=2, hq=8, kb=3, vb=5, lens=(5, 0, 33, 16), bs=8, seed=4):
    rng = np.random.default_rng(seed)
    from quantized_kv_cache_06_gb300.workloads import Workload, _block_table, _slots

    lens = np.array(lens, dtype=np.int32)
    nb = int(sum(-(-int(n) // bs) for n in lens)) + 3
    bt = _block_table(rng, lens, bs, nb)
    slots = _slots(lens, bt, bs)
    k = rng.standard_normal((slots.size, h, d)).astype(np.float16)
    v = rng.standard_normal((slots.size, h, d)).astype(np.float16)
    q = rng.standard_normal((lens.size, hq, d)).astype(np.float16)
    w = Workload("small", d, kb, vb, hq, h, bs, nb, lens, bt, k, v, slots, q)
    kp, st = gpu_write(tq, k, slots, nb, bs, kb)
    vp, st2 = gpu_write(tq, v, slots, nb, bs, vb)
    assert st == 0 and st2 == 0
    return w, kp, vp


@pytest.mark.parametrize("d,h,hq", [(32, 4, 4), (64, 2, 4), (128, 1, 8), (256, 2, 4)])
def test_decode_groups_and_dims(tq, d, h, hq):
    w, kp, vp = _small_case(tq, d=d, h=h, hq=hq)
    got, st = gpu_decode(tq, w, kp, vp)
    assert st == 0
    ref = oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(d))
    assert_decode_close(got, ref)
    assert np.all(got[1] == 0)  # seq_len 0


def test_decode_scale_and_out_dtype(tq):
    w, kp, vp = _small_case(tq)
    got, st = gpu_decode(tq, w, kp, vp, scale=0.05, out_dtype=torch.float32)
    ref = oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(64), scale=0.05)
    assert st == 0
    assert_decode_close(got, ref)


def test_decode_bad_block_id_is_skipped_and_reported(tq):
    w, kp, vp = _small_case(tq)
    bt = w.block_table.copy()
    bt[2, 1] = w.num_blocks + 11
    bt[3, 0] = -2
    got, st = gpu_decode(tq, w, kp, vp, block_table=bt)
    assert st == tq.TQ_ERR_BLOCK_OUT_OF_RANGE
    ref, flag = oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(64), block_table=bt,
                              return_flags=True)
    assert flag
    assert_decode_close(got, ref)


def test_decode_seq_len_over_capacity_is_clamped_and_reported(tq):
    w, kp, vp = _small_case(tq)
    lens = w.seq_lens.copy()
    cap = w.block_table.shape[1] * w.block_size
    lens[0] = cap + 100
    got, st = gpu_decode(tq, w, kp, vp, seq_lens=lens)
    assert st == tq.TQ_ERR_INVALID_ARG
    lens[0] = cap
    ref = oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(64), seq_lens=lens)
    assert_decode_close(got, ref)


def test_decode_empty_batch(tq):
    w, kp, vp = _small_case(tq)
    q = torch.zeros((0, 8, 64), dtype=torch.float16, device="cuda")
    out = tq.tq_paged_decode(q, kp, vp, torch.zeros((0, 4), dtype=torch.int32, device="cuda"),
                             torch.zeros(0, dtype=torch.int32, device="cuda"), tq.tq_build_rotation(64, 42, "cuda"),
                             lib_codebook(tq, 64, 3), lib_codebook(tq, 64, 5))
    torch.cuda.synchronize()
    assert out.shape == (0, 8, 64)


# ---------------------------------------------------------------- tensor-core decode edge cases
# (block size 16, K and V widths 2 to 5 bits each, GQA group 4 or 8: the shapes the
# tensor-core kernel takes; 3- and 5-bit widths use its window mode, independently for K
# and V)

@pytest.mark.parametrize("kb,vb,hq", [(4, 4, 32), (4, 2, 32), (2, 4, 64), (2, 2, 64), (4, 2, 64), (3, 3, 32),
                                      (3, 3, 64), (5, 5, 32), (5, 5, 64), (3, 4, 32), (4, 3, 64), (5, 2, 32),
                                      (2, 5, 64), (3, 5, 32), (5, 3, 64)])
def test_tc_decode_ragged_and_empty_sequences(tq, kb, vb, hq):
    # lengths with empty sequences in the middle, ragged last blocks, a single token, and
    # fewer blocks in total than there are SMs (some CTAs own no block)
    w, kp, vp = _small_case(tq, d=128, h=8, hq=hq, kb=kb, vb=vb, lens=(5, 0, 33, 16, 1, 0, 200, 17), bs=16, seed=kb * 10 + vb)
    got, st = gpu_decode(tq, w, kp, vp)
    assert st == 0
    ref = oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(128))
    assert_decode_close(got, ref)
    assert np.all(got[1] == 0) and np.all(got[5] == 0)


@pytest.mark.parametrize("d,kb,vb,hq", [(64, 4, 4, 16), (256, 4, 4, 16), (256, 3, 3, 16), (256, 3, 3, 32),
                                         (256, 5, 5, 16), (256, 5, 5, 32), (256, 3, 4, 16), (256, 5, 2, 32),
                                         (64, 2, 2, 16), (64, 3, 3, 32), (64, 5, 5, 16), (64, 2, 5, 32),
                                         (64, 3, 4, 16), (64, 5, 2, 32), (64, 4, 3, 32), (64, 2, 4, 16)])
def test_tc_decode_other_head_dims(tq, d, kb, vb, hq):
    w, kp, vp = _small_case(tq, d=d, h=4, hq=hq, kb=kb, vb=vb, lens=(70, 3, 129), bs=16, seed=d + kb + 7 * vb)
    got, st = gpu_decode(tq, w, kp, vp)
    assert st == 0
    assert_decode_close(got, oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(d)))


def test_tc_decode_bad_block_and_over_capacity(tq):
    w, kp, vp = _small_case(tq, d=128, h=8, hq=32, kb=4, vb=2, lens=(40, 64, 7), bs=16, seed=5)
    bt = w.block_table.copy()
    bt[1, 2] = w.num_blocks + 3
    got, st = gpu_decode(tq, w, kp, vp, block_table=bt)
    assert st == tq.TQ_ERR_BLOCK_OUT_OF_RANGE
    ref, flag = oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(128), block_table=bt,
                              return_flags=True)
    assert flag
    assert_decode_close(got, ref)
    lens = w.seq_lens.copy()
    lens[2] = w.block_table.shape[1] * 16 + 40
    got, st = gpu_decode(tq, w, kp, vp, seq_lens=lens)
    assert st == tq.TQ_ERR_INVALID_ARG
    lens[2] = w.block_table.shape[1] * 16
    assert_decode_close(got, oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(128), seq_lens=lens))


def test_tc_decode_many_short_sequences(tq):
    # more sequences than SMs: CTAs cover several sequences each
    rng = np.random.default_rng(17)
    lens = tuple(int(x) for x in rng.integers(0, 50, size=300))
    w, kp, vp = _small_case(tq, d=128, h=8, hq=32, kb=4, vb=4, lens=lens, bs=16, seed=17)
    got, st = gpu_decode(tq, w, kp, vp)
    assert st == 0
    heads = [(b, j) for b in range(0, 300, 7) for j in (0, 9, 31)]
    ref = oracle_decode(w, kp.cpu().numpy(), vp.cpu().numpy(), OracleCodec(128), heads=heads)
    sel = tuple(np.array(heads).T)
    assert_decode_close(got[sel], ref[sel])
    empty = [b for b, n in enumerate(lens) if n == 0]
    assert np.all(got[empty] == 0)


# ---------------------------------------------------------------- tensor-core writer shapes
# (fp16 / bf16 rows, head_dim 64, 128 or 256, 2 to 5 bits; H dividing the 16-row tile or
# not; 3- and 5-bit fields cross bytes; D 256 puts the signs on the A operand)

# fp32 rows: the tensor-core writer at D 64 / 128 (three exact bf16 parts), the SIMT writer at
# D 256
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("d,bits", [(64, 2), (64, 3), (64, 4), (64, 5), (128, 2), (128, 3), (128, 4), (128, 5),
                                    (256, 2), (256, 3), (256, 4), (256, 5)])
@pytest.mark.parametrize("h", [1, 3, 8, 16])
def test_tc_writer_shapes(tq, dtype, d, bits, h):
    rng = np.random.default_rng(d * 7 + bits * 3 + h)
    t = 37  # rows not a multiple of the 16-row tile
    raw32 = (rng.standard_normal((t, h, d)) * rng.lognormal(0, 0.5, (h, d))).astype(np.float32)
    raw32[5] = 0.0  # an all-zero token
    slots = rng.permutation(48)[:t].astype(np.int64)
    slots[rng.random(t) < 0.2] = -1
    raw_t = torch.from_numpy(raw32).to({"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dtype])
    raw_exact = raw_t.float().numpy()
    pages = torch.zeros(12, 4, h, o.row_bytes(d, bits), dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv(raw_t.cuda(), pages, torch.from_numpy(slots).cuda(), tq.tq_build_rotation(d, 42, "cuda"),
                        lib_codebook(tq, d, bits), check=False)
    assert int(st.item()) == 0
    pages_np = pages.cpu().numpy()
    check_written_rows(pages_np, raw_exact, slots, bits, OracleCodec(d))
    check_untouched(pages_np, slots)


@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (128, torch.float32), (256, torch.float32),
                                     (64, torch.bfloat16), (128, torch.bfloat16), (256, torch.bfloat16)])
def test_writer_rows_across_the_fp32_range(tq, d, dtype):
    # rows from 1e-25 to 1e30 in scale, and one along an axis at 3e38 (far outside fp16's
    # range, inside bf16's and fp32's): their sums of squares leave fp32's range, so the
    # writers rescale them by an exact power of two first; u is scale free.  fp32 at D 64 /
    # 128 and bf16 take the tensor-core writer (fp32 rows as three exact bf16 parts, all
    # normal numbers at these scales), fp32 at D 256 the SIMT writer.
    rng = np.random.default_rng(11 + d)
    t, h = 61, 4
    raw32 = rng.standard_normal((t, h, d)).astype(np.float32)
    raw32 *= (10.0 ** rng.uniform(-25, 30, (t, h, 1))).astype(np.float32)
    raw32[7, 2, :] = 0.0
    raw32[9, 1, :] = 0.0
    raw32[9, 1, 3] = 3e38  # a row along one axis, near the top of the range
    raw_t = torch.from_numpy(raw32).to(dtype)
    slots = np.arange(t, dtype=np.int64)
    pages = torch.zeros(4, 16, h, o.row_bytes(d, 4), dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv(raw_t.cuda(), pages, torch.from_numpy(slots).cuda(), tq.tq_build_rotation(d, 42, "cuda"),
                        lib_codebook(tq, d, 4), check=False)
    assert int(st.item()) == 0
    check_written_rows(pages.cpu().numpy(), raw_t.float().numpy(), slots, 4, OracleCodec(d))


@pytest.mark.parametrize("d,dtype", [(128, torch.float32), (128, torch.float16), (128, torch.bfloat16),
                                     (64, torch.float32), (256, torch.float16), (256, torch.float32)])
def test_writer_non_finite_rows_are_zero_rows(tq, d, dtype):
    # a row with a NaN or infinite coordinate is stored with the zero row's indices and a
    # non-finite norm; the rows around it (same 16-row tiles) are unaffected
    t, h = 40, 4
    rng = np.random.default_rng(71 + d)
    raw32 = rng.standard_normal((t, h, d)).astype(np.float32)
    raw32[3, 1, 7] = np.nan
    raw32[10, 0, :] = np.inf
    raw32[17, 2, 5] = -np.inf
    raw32[21, 3, :] = 0.0
    raw_t = torch.from_numpy(raw32).to(dtype)
    slots = np.arange(t, dtype=np.int64)
    pages = torch.zeros(3, 16, h, o.row_bytes(d, 4), dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv(raw_t.cuda(), pages, torch.from_numpy(slots).cuda(), tq.tq_build_rotation(d, 42, "cuda"),
                        lib_codebook(tq, d, 4), check=False)
    assert int(st.item()) == 0
    rows = pages.cpu().numpy().reshape(-1, h, o.row_bytes(d, 4))[:t]
    nb = o.index_bytes(d, 4)
    nu = np.ascontiguousarray(rows[..., nb:nb + 4]).view("<f4")[..., 0]
    bad = ~np.isfinite(raw_t.float().numpy()).all(axis=2)
    assert bad.sum() == 3
    assert np.all(~np.isfinite(nu[bad]))
    zero_idx = rows[21, 3, :nb]
    for i, j in np.argwhere(bad):
        assert np.array_equal(rows[i, j, :nb], zero_idx)
    good = ~bad
    stats = compare_rows(rows[good], raw_t.float().numpy().astype(np.float64)[good], OracleCodec(d), 4)
    assert_rows_match(stats)


def test_tc_writer_large_values_and_tiny_rows(tq):
    # rows spanning many binades (tiny, huge) still quantise exactly: u is scale free
    rng = np.random.default_rng(3)
    raw32 = rng.standard_normal((64, 8, 128)).astype(np.float32)
    raw32[:16] *= 1e-3
    raw32[16:32] *= 3e3
    raw_t = torch.from_numpy(raw32).half()
    slots = np.arange(64, dtype=np.int64)
    pages = torch.zeros(4, 16, 8, 68, dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv(raw_t.cuda(), pages, torch.from_numpy(slots).cuda(), tq.tq_build_rotation(128, 42, "cuda"),
                        lib_codebook(tq, 128, 4), check=False)
    assert int(st.item()) == 0
    check_written_rows(pages.cpu().numpy(), raw_t.float().numpy(), slots, 4, OracleCodec(128))


@pytest.mark.parametrize("d,bits,dt", [(256, 5, np.float16), (256, 3, np.float16), (128, 5, np.float16),
                                       (64, 5, np.float16), (128, 5, np.float32), (64, 3, np.float32)])
def test_index_flip_rate_at_scale(tq, d, bits, dt):
    # the index-byte bar measured as a rate: 3.4e7 coordinates of the densest codebooks
    # (rows N(0,1) times a lognormal(0, 0.5) scale per (head, channel), 8 heads, fp16 or
    # fp32), every exception within 1e-6 of a decision point and fewer than 1e-5 of all
    rng = np.random.default_rng(7 + d + bits)
    ntok, h = 33_554_432 // (8 * d), 8
    raw = (rng.standard_normal((ntok, h, d)) * rng.lognormal(0, 0.5, (h, d))).astype(dt)
    slots = np.arange(ntok, dtype=np.int64)
    pages, st = gpu_write(tq, raw, slots, ntok // 16, 16, bits)
    assert st == 0
    rows = pages.cpu().numpy().reshape(ntok * h, -1)
    flat = raw.reshape(-1, d)
    codec = OracleCodec(d)
    tot = dict(coords=0, flips=0, flips_outside_band=0)
    for s0 in range(0, ntok * h, 16384):
        part = compare_rows(rows[s0:s0 + 16384], flat[s0:s0 + 16384].astype(np.float64), codec, bits)
        for k in tot:
            tot[k] += part[k]
    assert tot["flips_outside_band"] == 0, tot
    assert tot["flips"] < MAX_FLIP_FRACTION * tot["coords"], tot
