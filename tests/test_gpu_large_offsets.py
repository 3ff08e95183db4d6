"""Page tensors past 2 GiB: every row the calls write or read lies more than 2^31 bytes into
its page tensor ("vLLM Usage", TQ Packed Page Contract: pages [num_blocks, block_size, H,
row_bytes] of any size; Slot Mapping: slots index the whole tensor).

The K and V pages hold 2^31 bytes plus 256 blocks each, and the sequences live in blocks
drawn from the top 256, so the byte offsets of their rows exceed 2^31 in both tensors.
The writer, the tensor-core decode, the mixed prefill/decode, the readback and the
product-key write and decode are compared with the oracle, which sees the same rows gathered
into compact pages (block ids remapped).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import tq_oracle as o  # noqa: E402
from parity import OracleCodec, assert_decode_close, assert_rows_match, compare_rows  # noqa: E402

pytestmark = pytest.mark.gpu

D, H, BS, KB, VB, HQ = 128, 8, 16, 4, 4, 32
LENS = [37, 300, 1000, 16]
TOP = 256


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


@pytest.fixture(scope="module")
def case(tq):
    rng = np.random.default_rng(2031)
    codec = OracleCodec(D)
    rbk, rbv = o.row_bytes(D, KB), o.row_bytes(D, VB)
    nblk = -(-(1 << 31) // (BS * H * min(rbk, rbv))) + TOP
    assert (nblk - TOP) * BS * H * min(rbk, rbv) >= 1 << 31  # every top block starts past 2^31
    nb_seq = [-(-n // BS) for n in LENS]
    used = rng.permutation(np.arange(nblk - TOP, nblk))[:sum(nb_seq)].astype(np.int32)
    maxb = max(nb_seq)
    bt = np.zeros((len(LENS), maxb), dtype=np.int32)
    slots, pos = [], 0
    for b, n in enumerate(LENS):
        bt[b, :nb_seq[b]] = used[pos:pos + nb_seq[b]]
        pos += nb_seq[b]
        t = np.arange(n)
        slots.append(bt[b, t // BS].astype(np.int64) * BS + t % BS)
    slots = np.concatenate(slots)
    t = slots.shape[0]
    k32 = rng.standard_normal((t, H, D)).astype(np.float32)
    v32 = rng.standard_normal((t, H, D)).astype(np.float32)
    dev = torch.device("cuda")
    kp = torch.zeros(nblk, BS, H, rbk, dtype=torch.uint8, device=dev)
    vp = torch.zeros(nblk, BS, H, rbv, dtype=torch.uint8, device=dev)
    signs = torch.from_numpy(codec.signs).float().to(dev)
    ck, cv = torch.from_numpy(codec.centroids(KB)).to(dev), torch.from_numpy(codec.centroids(VB)).to(dev)
    slots_t = torch.from_numpy(slots).to(dev)
    k_h, v_h = torch.from_numpy(k32).half(), torch.from_numpy(v32).half()
    for raw, pages, cents in ((k_h, kp, ck), (v_h, vp, cv)):
        st = tq.tq_write_kv(raw.to(dev), pages, slots_t, signs, cents)
        assert int(st.item()) == 0
    torch.cuda.synchronize()
    # compact copies of the used blocks, in `used` order, and the remapped table
    used_t = torch.from_numpy(used.astype(np.int64)).to(dev)
    kc, vc = kp[used_t].cpu().numpy(), vp[used_t].cpu().numpy()
    remap = {int(bid): i for i, bid in enumerate(used)}
    bt_c = np.zeros_like(bt)
    for b, n in enumerate(nb_seq):
        bt_c[b, :n] = [remap[int(x)] for x in bt[b, :n]]
    slots_c = np.concatenate([bt_c[b, np.arange(n) // BS].astype(np.int64) * BS + np.arange(n) % BS
                              for b, n in enumerate(LENS)])
    return dict(codec=codec, nblk=nblk, bt=bt, bt_c=bt_c, slots=slots, slots_c=slots_c, k_h=k_h, v_h=v_h, kp=kp,
                vp=vp, kc=kc, vc=vc, signs=signs, ck=ck, cv=cv, dev=dev)


def test_writer_rows_past_2gib(case):
    c = case
    t = c["slots"].shape[0]
    for raw, pages, bits in ((c["k_h"], c["kc"], KB), (c["v_h"], c["vc"], VB)):
        rows = pages.reshape(-1, H, pages.shape[3])[c["slots_c"]].reshape(t * H, -1)
        assert_rows_match(compare_rows(rows, raw.float().numpy().astype(np.float64).reshape(t * H, D), c["codec"],
                                       bits))


def test_decode_and_prefill_past_2gib(tq, case):
    c = case
    rng = np.random.default_rng(7)
    q = rng.standard_normal((len(LENS), HQ, D)).astype(np.float32)
    lens = np.array(LENS, dtype=np.int32)
    dev = c["dev"]
    st = torch.full((1,), -7, dtype=torch.int32, device=dev)
    got = tq.tq_paged_decode(torch.from_numpy(q).to(dev), c["kp"], c["vp"], torch.from_numpy(c["bt"]).to(dev),
                             torch.from_numpy(lens).to(dev), c["signs"], c["ck"], c["cv"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    codec = c["codec"]
    ref = o.paged_decode(q, c["kc"], c["vc"], KB, VB, c["bt_c"], lens, codec.signs, codec.centroids(KB),
                         codec.centroids(VB))
    assert_decode_close(got.cpu().numpy(), ref)
    # mixed prefill/decode: the last 5 tokens of each sequence as query rows
    q_seq = np.repeat(np.arange(len(LENS)), 5).astype(np.int32)
    q_len = np.concatenate([np.arange(n - 4, n + 1) for n in LENS]).astype(np.int32)
    qp = rng.standard_normal((q_seq.shape[0], HQ, D)).astype(np.float32)
    st.fill_(-7)
    gotp = tq.tq_paged_prefill(torch.from_numpy(qp).to(dev), torch.from_numpy(q_seq).to(dev),
                               torch.from_numpy(q_len).to(dev), c["kp"], c["vp"], torch.from_numpy(c["bt"]).to(dev),
                               c["signs"], c["ck"], c["cv"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    refp = o.paged_prefill(qp, q_seq, q_len, c["kc"], c["vc"], KB, VB, c["bt_c"], codec.signs, codec.centroids(KB),
                           codec.centroids(VB))
    assert_decode_close(gotp.cpu().numpy(), refp)


def test_readback_past_2gib(tq, case):
    c = case
    sel = np.random.default_rng(3).permutation(c["slots"].shape[0])[:200]
    out = tq.tq_dequant_rows(c["kp"], torch.from_numpy(c["slots"][sel]).to(c["dev"]), c["signs"], c["ck"],
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    codec = c["codec"]
    want = o.dequant_slots(c["kc"], c["slots_c"][sel], codec.signs, codec.centroids(KB), KB)
    nu = np.stack([c["kc"][s // BS, s % BS, :, -4:].copy().view("<f4").reshape(-1) for s in c["slots_c"][sel]])
    err = np.abs(out.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= 4e-6 * nu[..., None] + 1e-30), float(np.max(err))


def test_product_keys_past_2gib(tq, case):
    # product-quantised key rows ("QJL residual", 72 B at K4) in a third page tensor with the
    # same block count: the same blocks start past 2^31 bytes there too; written, then decoded
    # with the V pages above, against the oracle of the product-key path
    from oracle import qjl_oracle as qo
    from parity import BAND, NORM_RTOL, allowed_flips

    c = case
    dev, codec = c["dev"], c["codec"]
    rbp = tq.tq_prod_row_bytes(D, KB)
    assert (c["nblk"] - TOP) * BS * H * rbp >= 1 << 31
    kpp = torch.zeros(c["nblk"], BS, H, rbp, dtype=torch.uint8, device=dev)
    s_lib = tq.tq_build_qjl_matrix(D, 43)
    s64 = qo.normal_matrix(D, D, 43).astype(np.float32).astype(np.float64)
    kc = codec.centroids(KB - 1)
    st = tq.tq_write_kv_prod(c["k_h"].to(dev), kpp, torch.from_numpy(c["slots"]).to(dev), c["signs"],
                             torch.from_numpy(kc).to(dev), s_lib.to(dev))
    assert int(st.item()) == 0
    # the compact copy in the order the case fixture used (block ids remapped the same way)
    order = np.zeros(int(c["bt_c"].max()) + 1, dtype=np.int64)
    for b in range(len(LENS)):
        n = -(-LENS[b] // BS)
        order[c["bt_c"][b, :n]] = c["bt"][b, :n]
    kpc = kpp[torch.from_numpy(order).to(dev)].cpu().numpy()
    t = c["slots"].shape[0]
    rows = kpc.reshape(-1, H, rbp)[c["slots_c"]].reshape(t * H, rbp)
    x = c["k_h"].float().numpy().astype(np.float64).reshape(t * H, D)
    enc = qo.encode_prod(x, codec.rot, kc, s64)
    _, _, margin = o.encode_rows(x, codec.rot, kc)
    gidx, gz, gnu, ggam = qo.unpack_prod_rows(rows, D, KB)
    diff = gidx != enc["idx"]
    assert int((diff & (margin >= BAND)).sum()) == 0 and diff.sum() <= allowed_flips(diff.size)
    assert np.all(np.abs(gnu - enc["nu"]) <= NORM_RTOL * enc["nu"])
    clean = ~diff.any(axis=1)
    proj = enc["residual"] @ s64.T
    assert int(((gz != enc["z"]) & clean[:, None] & (np.abs(proj) >= 1e-5)).sum()) == 0
    q = np.random.default_rng(17).standard_normal((len(LENS), HQ, D)).astype(np.float32)
    lens = np.array(LENS, dtype=np.int32)
    st = torch.full((1,), -7, dtype=torch.int32, device=dev)
    got = tq.tq_paged_decode_prod(torch.from_numpy(q).to(dev), kpp, c["vp"], torch.from_numpy(c["bt"]).to(dev),
                                  torch.from_numpy(lens).to(dev), c["signs"], torch.from_numpy(kc).to(dev), c["cv"],
                                  s_lib.to(dev), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = qo.paged_decode_prod_keys(q, kpc, c["vc"], KB, VB, c["bt_c"], lens, codec.signs, kc, codec.centroids(VB), s64)
    assert_decode_close(got.cpu().numpy(), ref)
