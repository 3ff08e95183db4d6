"""GPU parity of the INT8-query prefill ("vLLM Usage", Runtime Dispatch: the int8 query
path; "vLLM Reference Audit", File Map: INT8-Q prefill) against oracle/int8q_oracle.py.

* tq_quantize_queries_int8: codes and scales bit-exact (both sides decide in fp32, the
  precision the reading fixes for the quantiser).
* tq_paged_prefill_int8q: |gpu - oracle| <= 2e-3 + 2e-3 |oracle| against the oracle's
  prefill on the same codes and scales, over the multi-query kernel's shapes and shapes that
  run the SIMT kernels.
"""

import numpy as np
import pytest
import torch

from oracle import int8q_oracle as iq
from oracle import tq_oracle as o
from parity import assert_decode_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_quantizer_matches_oracle_bit_exact(tq, dtype, d):
    rng = np.random.default_rng(d)
    q = torch.from_numpy((rng.standard_normal((37, 8, d)) * rng.lognormal(0, 2, (37, 8, 1))).astype(np.float32))
    q[3, 2] = 0.0  # a zero row
    q[5, 1, :4] = torch.tensor([127.0, -63.5, 0.5, 1.5])  # ties once scaled by 1
    q[5, 1, 4:] = 0.0
    q = q.to(dtype)
    codes, scales = tq.tq_quantize_queries_int8(q.cuda())
    torch.cuda.synchronize()
    want_c, want_s = iq.quantize_queries_int8(q.float().numpy())
    assert np.array_equal(scales.cpu().numpy(), want_s)
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert scales[3, 2].item() == 0.0 and int(codes[3, 2].abs().max()) == 0


def _cache(rng, lens, d, h, kb, vb, bs=16):
    nblk = int(sum(-(-n // bs) for n in lens)) + 2
    maxb = max(-(-n // bs) for n in lens)
    perm = rng.permutation(nblk).astype(np.int32)
    bt = np.zeros((len(lens), maxb), dtype=np.int32)
    signs = o.splitmix64_signs(d, 42)
    kc, vc = o.codebook_f32(d, kb)[0], o.codebook_f32(d, vb)[0]
    kp = np.zeros((nblk, bs, h, o.row_bytes(d, kb)), np.uint8)
    vp = np.zeros((nblk, bs, h, o.row_bytes(d, vb)), np.uint8)
    pos = 0
    for b, n in enumerate(lens):
        nb = -(-n // bs)
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
        slots = np.array([bt[b, t // bs] * bs + t % bs for t in range(n)], dtype=np.int64)
        scl = rng.lognormal(0, 0.5, (1, h, d))
        kp = o.write_kv(rng.standard_normal((n, h, d)) * scl, kp, slots, signs, kc, kb)
        vp = o.write_kv(rng.standard_normal((n, h, d)) * scl, vp, slots, signs, vc, vb)
    return bt, signs, kc, vc, kp, vp


# multi-query kernel shapes (D 64/128/256, 2/4 or equal 3/5 bits) and SIMT shapes (D 32,
# unequal 3/5-bit K/V)
@pytest.mark.parametrize("d,kb,vb,hq,h", [(128, 4, 4, 32, 8), (128, 4, 2, 16, 2), (64, 3, 3, 8, 4),
                                          (256, 2, 4, 8, 2), (32, 4, 4, 8, 2), (128, 3, 5, 8, 2)])
def test_int8q_prefill_matches_oracle(tq, d, kb, vb, hq, h):
    rng = np.random.default_rng(100 + d + kb)
    lens = [300, 17, 90]
    bt, signs, kc, vc, kp, vp = _cache(rng, lens, d, h, kb, vb)
    chunks = [24, 1, 5]
    q_seq = np.concatenate([np.full(c, b) for b, c in enumerate(chunks)]).astype(np.int32)
    q_len = np.concatenate([np.arange(n - c + 1, n + 1) for n, c in zip(lens, chunks)]).astype(np.int32)
    q = torch.from_numpy(rng.standard_normal((q_seq.size, hq, d)).astype(np.float16)).cuda()
    codes, scales = tq.tq_quantize_queries_int8(q)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    got = tq.tq_paged_prefill_int8q(codes, scales, dev(q_seq), dev(q_len), dev(kp), dev(vp), dev(bt),
                                    dev(signs.astype(np.float32)), dev(kc), dev(vc), out_dtype=torch.float32,
                                    status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = iq.paged_prefill_int8q(codes.cpu().numpy(), scales.cpu().numpy(), q_seq, q_len, kp, vp, kb, vb, bt, signs,
                                 kc, vc)
    assert_decode_close(got.cpu().numpy(), ref)
    # the int8 path stays near the fp16 query's prefill (quantisation error of the query only)
    flt = tq.tq_paged_prefill(q, dev(q_seq), dev(q_len), dev(kp), dev(vp), dev(bt), dev(signs.astype(np.float32)),
                              dev(kc), dev(vc), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert float((got - flt).abs().max()) < 0.05 * float(flt.abs().max())


def test_int8q_refuses_inconsistent_arguments(tq):
    codes = torch.zeros(2, 4, 64, dtype=torch.int8, device="cuda")
    lib = tq.lib()
    assert lib.tq_paged_prefill_int8q(codes.data_ptr(), None, 2, 4, 2, 64, 1 << 20, 4, 1 << 20, 4, 4, 16, 1 << 20, 1,
                                      4, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 0.0, 1 << 20, 1, 1 << 20,
                                      1 << 30, None, None) == tq.TQ_ERR_INVALID_ARG  # no scales
