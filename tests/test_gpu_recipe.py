"""GPU parity of the recipe cache modes turboquant25 / turboquant35 -- tq_write_kv_recipe
and tq_paged_decode_recipe through the C ABI -- against the fp64 oracle
(oracle/recipe_oracle.py; "vLLM Usage", Cache Dtypes; "Architecture", vLLM Runtime
Mapping: grouped MSE+QJL rows).

Each group of a row is a product-quantised vector of dimension D/2, so the writer bars are
those of the product-key writer (tests/test_gpu_qjl.py) applied per group: MSE indices
bit-exact outside the 1e-6 decision band (in-band exceptions held to the rate bar), nu to
1e-6 relative, and on rows whose indices all agree the sign bits exact wherever the
oracle's |(S r)_i| >= 1e-5 and gamma to 5e-5 relative.  Decode bar:
|gpu - oracle| <= 2e-3 + 2e-3 |oracle| on the page bytes being decoded, with S rounded to
fp32 once, the matrix both sides use.
"""

import numpy as np
import pytest
import torch

from oracle import qjl_oracle as qo
from oracle import recipe_oracle as ro
from oracle import tq_oracle as o
from parity import BAND, NORM_RTOL, allowed_flips, assert_decode_close

pytestmark = pytest.mark.gpu

SIGN_BAND = 1e-5
GAMMA_RTOL = 5e-5
RECIPES = ["turboquant25", "turboquant35"]


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


def codecs(tq, recipe, d):
    gpu = tq.RecipeCodec(recipe, d, "cuda")
    s32 = gpu.smat.cpu().numpy()
    assert np.array_equal(s32, qo.normal_matrix(d // 2, d // 2, ro.SKETCH_SEED).astype(np.float32))
    return gpu, ro.RecipeCodec(recipe, d, smat=s32.astype(np.float64))


def _layout(rng, lens, bs, spare=3):
    nblk = int(sum(-(-int(n) // bs) for n in lens)) + spare
    maxb = max(1, max(-(-int(n) // bs) for n in lens))
    perm = rng.permutation(nblk).astype(np.int32)
    bt = np.zeros((len(lens), maxb), dtype=np.int32)
    slots, pos = [], 0
    for b, n in enumerate(lens):
        nb = -(-int(n) // bs)
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
        t = np.arange(int(n))
        slots.append(bt[b, t // bs].astype(np.int64) * bs + t % bs)
    return nblk, bt, np.concatenate(slots)


def check_group_rows(rows, x, bits, oc):
    """rows uint8[N, RBg] of one group written by the GPU for gathered rows x[N, d]."""
    d = oc.d
    mse = oc.mse[0] if bits == oc.bits[0] else oc.mse[1]
    enc = qo.encode_prod(x, oc.rot, mse, oc.smat)
    _, _, margin = o.encode_rows(x, oc.rot, mse)
    gidx, gz, gnu, ggam = qo.unpack_prod_rows(rows, d, bits)
    diff = gidx != enc["idx"]
    assert int((diff & (margin >= BAND)).sum()) == 0
    assert diff.sum() <= allowed_flips(diff.size)
    assert np.abs(gidx - enc["idx"]).max() <= 1
    nu = enc["nu"].astype(np.float64)
    assert np.all(np.abs(gnu - nu) <= NORM_RTOL * nu)
    clean = ~diff.any(axis=1)
    assert clean.mean() > 0.98
    proj = enc["residual"] @ oc.smat.T
    assert int(((gz != enc["z"]) & clean[:, None] & (np.abs(proj) >= SIGN_BAND)).sum()) == 0
    g = enc["gamma"].astype(np.float64)[clean]
    assert np.all(np.abs(ggam[clean] - g) <= GAMMA_RTOL * np.maximum(g, 1e-30))


@pytest.mark.parametrize("recipe", RECIPES)
@pytest.mark.parametrize("d,dtype", [(128, torch.float16), (128, torch.bfloat16), (128, torch.float32),
                                     (64, torch.float32), (64, torch.float16)])
def test_recipe_writer_matches_oracle(tq, recipe, d, dtype):
    rng = np.random.default_rng(500 + d + (0 if recipe == "turboquant25" else 7))
    t, h, bs = 301, 3, 16
    nb = (t + bs - 1) // bs + 2
    raw32 = (rng.standard_normal((t, h, d)) * rng.lognormal(0.0, 0.6, (1, h, d))).astype(np.float32)
    raw32[7, 2] = 0.0  # a zero row: nu = 0 in both groups
    raw = torch.from_numpy(raw32).to(dtype)
    raw64 = raw.double().numpy()
    high = tq.tq_recipe_calibrate(recipe, raw.float().numpy()[:100])
    order = tq.tq_recipe_channel_order(recipe, d, high)
    gpu, oc = codecs(tq, recipe, d)
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[::17] = -1
    rb = gpu.row_bytes
    pages = torch.full((nb, bs, h, rb), 0xA5, dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv_recipe(raw.cuda(), pages, torch.from_numpy(slots).cuda(), order.cuda(), gpu, check=False)
    assert int(st.item()) == 0
    pg = pages.cpu().numpy().reshape(nb * bs, h, rb)
    written = np.zeros(nb * bs, dtype=bool)
    written[slots[slots >= 0]] = True
    assert np.all(pg[~written] == 0xA5)
    tok = np.nonzero(slots >= 0)[0]
    nh = qo.prod_row_bytes(d // 2, oc.bits[0])
    ordn = order.numpy()
    for k in range(h):
        rows = pg[slots[tok], k]
        for g, (lo, hi) in enumerate(((0, nh), (nh, rb))):
            chans = ordn[k, g * (d // 2):(g + 1) * (d // 2)]
            check_group_rows(rows[:, lo:hi], raw64[tok, k][:, chans], oc.bits[g], oc)


def test_recipe_writer_bad_slot_and_empty_batch(tq):
    d, t, h, bs, nb = 64, 40, 2, 16, 3
    rng = np.random.default_rng(8)
    raw = torch.from_numpy(rng.standard_normal((t, h, d)).astype(np.float32)).cuda()
    order = tq.tq_recipe_channel_order("turboquant35", d, np.tile(np.arange(d // 2), (h, 1))).cuda()
    gpu = tq.RecipeCodec("turboquant35", d, "cuda")
    slots = torch.arange(t, dtype=torch.int64)
    slots[9] = nb * bs
    pages = torch.full((nb, bs, h, gpu.row_bytes), 0x3C, dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv_recipe(raw, pages, slots.cuda(), order, gpu, check=False)
    assert int(st.item()) == tq.TQ_ERR_SLOT_OUT_OF_RANGE
    assert bool(torch.all(pages == 0x3C))
    empty = torch.empty(0, h, d, dtype=torch.float32, device="cuda")
    st = tq.tq_write_kv_recipe(empty, pages, torch.empty(0, dtype=torch.int64, device="cuda"), order, gpu, check=False)
    assert int(st.item()) == 0


@pytest.mark.parametrize("recipe", RECIPES)
@pytest.mark.parametrize("d,hq,h,bs,qdt", [(128, 32, 8, 16, np.float16), (128, 8, 8, 16, np.float32),
                                           (64, 8, 4, 8, np.float32), (128, 16, 2, 32, np.float16),
                                           (128, 8, 2, 12, np.float32)])
def test_recipe_decode_matches_oracle(tq, recipe, d, hq, h, bs, qdt):
    rng = np.random.default_rng(77 + hq + d)
    lens = [0, 1, 37, 300, 1000]
    nblk, bt, slots = _layout(rng, lens, bs)
    gpu, oc = codecs(tq, recipe, d)
    t = slots.shape[0]
    kraw = rng.standard_normal((t, h, d)) * rng.lognormal(0.0, 0.5, (1, h, d))
    vraw = rng.standard_normal((t, h, d)) * rng.lognormal(0.0, 0.5, (1, h, d))
    high = ro.calibrate_high_groups(kraw[:200], recipe)
    rb = gpu.row_bytes
    kp = ro.write_recipe_kv(kraw, np.zeros((nblk, bs, h, rb), np.uint8), slots, high, oc)
    vp = ro.write_recipe_kv(vraw, np.zeros((nblk, bs, h, rb), np.uint8), slots, high, oc)
    order = tq.tq_recipe_channel_order(recipe, d, high).cuda()
    q = rng.standard_normal((len(lens), hq, d)).astype(qdt)
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = tq.tq_paged_decode_recipe(torch.from_numpy(q).cuda(), torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda(),
                                    torch.from_numpy(bt).cuda(), torch.from_numpy(np.array(lens, np.int32)).cuda(),
                                    order, gpu, out_dtype=torch.float32, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = ro.paged_decode_recipe(q, kp, vp, bt, np.array(lens), high, oc)
    assert_decode_close(got.cpu().numpy(), ref)
    assert np.all(got[0].cpu().numpy() == 0)  # an empty sequence gives zeros


@pytest.mark.parametrize("recipe", RECIPES)
def test_recipe_write_then_decode_end_to_end(tq, recipe):
    # the GPU writer's pages decoded by the GPU, against the oracle decode of those bytes
    rng = np.random.default_rng(31)
    d, hq, h, bs = 128, 16, 4, 16
    lens = [513, 64, 2048]
    nblk, bt, slots = _layout(rng, lens, bs)
    gpu, oc = codecs(tq, recipe, d)
    t = slots.shape[0]
    raw = [torch.from_numpy((rng.standard_normal((t, h, d)) * rng.lognormal(0, 0.5, (1, h, d))).astype(np.float16))
           for _ in range(2)]
    high = tq.tq_recipe_calibrate(recipe, raw[0].float().numpy()[:256])
    order = tq.tq_recipe_channel_order(recipe, d, high).cuda()
    pages = []
    for x in raw:
        pg = torch.zeros(nblk, bs, h, gpu.row_bytes, dtype=torch.uint8, device="cuda")
        tq.tq_write_kv_recipe(x.cuda(), pg, torch.from_numpy(slots).cuda(), order, gpu)
        pages.append(pg)
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float16)
    got = tq.tq_paged_decode_recipe(torch.from_numpy(q).cuda(), pages[0], pages[1], torch.from_numpy(bt).cuda(),
                                    torch.from_numpy(np.array(lens, np.int32)).cuda(), order, gpu,
                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = ro.paged_decode_recipe(q, pages[0].cpu().numpy(), pages[1].cpu().numpy(), bt, np.array(lens), high.numpy(), oc)
    assert_decode_close(got.cpu().numpy(), ref)


def test_recipe_decode_bad_block_and_over_long_length(tq):
    rng = np.random.default_rng(5)
    d, hq, h, bs = 64, 4, 2, 16
    lens = [100, 40]
    nblk, bt, slots = _layout(rng, lens, bs)
    gpu, oc = codecs(tq, "turboquant25", d)
    kraw = rng.standard_normal((slots.shape[0], h, d))
    high = ro.calibrate_high_groups(kraw, "turboquant25")
    kp = ro.write_recipe_kv(kraw, np.zeros((nblk, bs, h, gpu.row_bytes), np.uint8), slots, high, oc)
    order = tq.tq_recipe_channel_order("turboquant25", d, high).cuda()
    q = rng.standard_normal((2, hq, d)).astype(np.float32)
    bad = bt.copy()
    bad[0, 2] = nblk + 5  # block id outside the pages: its tokens are left out and reported
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = tq.tq_paged_decode_recipe(torch.from_numpy(q).cuda(), torch.from_numpy(kp).cuda(), torch.from_numpy(kp).cuda(),
                                    torch.from_numpy(bad).cuda(), torch.from_numpy(np.array(lens, np.int32)).cuda(),
                                    order, gpu, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tq.TQ_ERR_BLOCK_OUT_OF_RANGE
    ref = ro.paged_decode_recipe(q, kp, kp, bad, np.array(lens), high, oc)  # the oracle leaves it out too
    assert_decode_close(got.cpu().numpy(), ref)
    long = np.array([100, bt.shape[1] * bs + 1], dtype=np.int32)
    tq.tq_paged_decode_recipe(torch.from_numpy(q).cuda(), torch.from_numpy(kp).cuda(), torch.from_numpy(kp).cuda(),
                              torch.from_numpy(bt).cuda(), torch.from_numpy(long).cuda(), order, gpu, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tq.TQ_ERR_INVALID_ARG


@pytest.mark.parametrize("recipe", RECIPES)
def test_recipe_decode_wide_value_norms(tq, recipe):
    # value rows whose norms span 1e-3 .. 1e5 within every 16-token tile (the weights' power-of-
    # two scale follows the largest value norm seen; no weight may leave fp16 range), keys of
    # moderate norm so that many tokens carry weight; fp32 and fp16 queries
    rng = np.random.default_rng(41)
    d, hq, h, bs = 128, 8, 2, 16
    lens = [700, 33, 16]
    nblk, bt, slots = _layout(rng, lens, bs)
    gpu, oc = codecs(tq, recipe, d)
    t = slots.shape[0]
    kraw = rng.standard_normal((t, h, d)) * 0.3
    vraw = rng.standard_normal((t, h, d)) * 10.0 ** rng.uniform(-3.0, 5.0, (t, h, 1))
    high = ro.calibrate_high_groups(kraw[:200], recipe)
    rb = gpu.row_bytes
    kp = ro.write_recipe_kv(kraw, np.zeros((nblk, bs, h, rb), np.uint8), slots, high, oc)
    vp = ro.write_recipe_kv(vraw, np.zeros((nblk, bs, h, rb), np.uint8), slots, high, oc)
    order = tq.tq_recipe_channel_order(recipe, d, high).cuda()
    for qdt in (np.float32, np.float16):
        q = rng.standard_normal((len(lens), hq, d)).astype(qdt)
        st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        got = tq.tq_paged_decode_recipe(torch.from_numpy(q).cuda(), torch.from_numpy(kp).cuda(),
                                        torch.from_numpy(vp).cuda(), torch.from_numpy(bt).cuda(),
                                        torch.from_numpy(np.array(lens, np.int32)).cuda(), order, gpu,
                                        out_dtype=torch.float32, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref = ro.paged_decode_recipe(q, kp, vp, bt, np.array(lens), high, oc)
        assert np.abs(ref).max() > 1e3  # the large norms reach the output
        assert_decode_close(got.cpu().numpy(), ref)


def test_recipe_writer_many_tiles_per_warp(tq):
    # 16384 tokens x 8 heads: 4096 tiles of 32 rows, more than the resident warps take at once,
    # so warps stage the next tile while they encode the current one; rows checked on a sample
    recipe, d, t, h, bs = "turboquant35", 128, 16384, 8, 16
    rng = np.random.default_rng(909)
    nb = t // bs + 4
    raw32 = (rng.standard_normal((t, h, d)) * rng.lognormal(0.0, 0.6, (1, h, d))).astype(np.float32)
    raw = torch.from_numpy(raw32).half()
    raw64 = raw.double().numpy()
    high = tq.tq_recipe_calibrate(recipe, raw.float().numpy()[:256])
    order = tq.tq_recipe_channel_order(recipe, d, high)
    gpu, oc = codecs(tq, recipe, d)
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[5::97] = -1
    rb = gpu.row_bytes
    pages = torch.full((nb, bs, h, rb), 0x5A, dtype=torch.uint8, device="cuda")
    st = tq.tq_write_kv_recipe(raw.cuda(), pages, torch.from_numpy(slots).cuda(), order.cuda(), gpu, check=False)
    assert int(st.item()) == 0
    pg = pages.cpu().numpy().reshape(nb * bs, h, rb)
    written = np.zeros(nb * bs, dtype=bool)
    written[slots[slots >= 0]] = True
    assert np.all(pg[~written] == 0x5A)
    tok = rng.choice(np.nonzero(slots >= 0)[0], size=1500, replace=False)
    nh = qo.prod_row_bytes(d // 2, oc.bits[0])
    ordn = order.numpy()
    for k in range(h):
        rows = pg[slots[tok], k]
        for g, (lo, hi) in enumerate(((0, nh), (nh, rb))):
            chans = ordn[k, g * (d // 2):(g + 1) * (d // 2)]
            check_group_rows(rows[:, lo:hi], raw64[tok, k][:, chans], oc.bits[g], oc)
