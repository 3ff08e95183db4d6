"""tq_paged_decode_static: the allocation-free decode for callers that cannot call
cudaMalloc (a plugin whose host owns all device memory, a fixed memory budget, a loop
that must not synchronise on cudaMalloc/cudaFree).  Its split-K partials live in the
library's fixed device array instead of a caller workspace.

Checked through the C ABI against tq_paged_decode (the entry point with a caller
workspace) on two calls in a row with different queries, so stale scratch contents
from the first call cannot leak into the second.  Runs last (file name) and passes
both alone in a fresh process and after the other tests.
"""

import numpy as np
import pytest
import torch

from parity import assert_decode_close
from quantized_kv_cache_06_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for the gpu tests")
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


def test_static_scratch_decode_matches_workspace_decode(tq):
    w = make_workload(2)
    dev = torch.device("cuda")
    d = w.head_dim
    signs = tq.tq_build_rotation(d, 42, dev)
    ck = tq.tq_codebook(d, w.k_bits, dev)[0]
    cv = tq.tq_codebook(d, w.v_bits, dev)[0]
    kp = torch.zeros(w.num_blocks, w.block_size, w.num_kv_heads, tq.tq_row_bytes(d, w.k_bits), dtype=torch.uint8,
                     device=dev)
    vp = torch.zeros(w.num_blocks, w.block_size, w.num_kv_heads, tq.tq_row_bytes(d, w.v_bits), dtype=torch.uint8,
                     device=dev)
    slots = torch.from_numpy(w.slots).to(dev)
    tq.tq_write_kv(torch.from_numpy(w.k_raw).to(dev), kp, slots, signs, ck)
    tq.tq_write_kv(torch.from_numpy(w.v_raw).to(dev), vp, slots, signs, cv)
    bt = torch.from_numpy(w.block_table).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)

    queries = [torch.from_numpy(w.q).to(dev),
               torch.from_numpy(np.random.default_rng(77).standard_normal(w.q.shape).astype(np.float16)).to(dev)]
    for q in queries:
        ref = tq.tq_paged_decode(q, kp, vp, bt, lens, signs, ck, cv)
        out = torch.full_like(q, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        tq.tq_paged_decode_static(q, kp, vp, bt, lens, signs, ck, cv, out, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == tq.TQ_OK
        assert_decode_close(out.float().cpu().numpy(), ref.float().cpu().numpy().astype(np.float64))


def test_static_scratch_rejects_shapes_beyond_its_capacity(tq):
    dev = torch.device("cuda")
    b, hq, h, d = 4096, 64, 8, 256
    need = tq.tq_paged_decode_workspace(b, hq, h, d, 1, 16)
    assert need > 16 << 20
    q = torch.zeros((b, hq, d), dtype=torch.float16, device=dev)
    pages = torch.zeros((1, 16, h, tq.tq_row_bytes(d, 4)), dtype=torch.uint8, device=dev)
    with pytest.raises(tq.TQError) as e:
        tq.tq_paged_decode_static(q, pages, pages, torch.zeros((b, 1), dtype=torch.int32, device=dev),
                                  torch.zeros(b, dtype=torch.int32, device=dev), tq.tq_build_rotation(d, 42, dev),
                                  tq.tq_codebook(d, 4, dev)[0], tq.tq_codebook(d, 4, dev)[0], torch.empty_like(q))
    assert e.value.status == tq.TQ_ERR_INVALID_ARG
    assert "16777216" in str(e.value)
