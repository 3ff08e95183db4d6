"""The calls are graph-capturable ("vLLM Usage", plugin backend: CUDA-graph buffer
ownership): write, decode, readback and mixed prefill/decode are captured into one CUDA
graph after an eager first call, replayed on new inputs copied into the captured
buffers, and must give the same bytes as eager calls on those inputs."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def test_capture_and_replay_matches_eager():
    import quantized_kv_cache_06_gb300 as tq

    dev = torch.device("cuda")
    rng = np.random.default_rng(123)
    d, h, hq, bs, b, n = 128, 8, 32, 16, 4, 100
    nblk = b * (-(-n // bs))
    bt = torch.from_numpy(rng.permutation(nblk).astype(np.int32).reshape(b, -1)).to(dev)
    lens = torch.full((b,), n, dtype=torch.int32, device=dev)
    slots = torch.from_numpy(np.concatenate(
        [bt[i].cpu().numpy().astype(np.int64)[np.arange(n) // bs] * bs + np.arange(n) % bs for i in range(b)])).to(dev)
    signs = tq.tq_build_rotation(d, 42, dev)
    ck, cv = tq.tq_codebook(d, 4, dev)[0], tq.tq_codebook(d, 4, dev)[0]
    rb = tq.tq_row_bytes(d, 4)
    kraw = torch.empty(b * n, h, d, dtype=torch.float16, device=dev)
    vraw = torch.empty_like(kraw)
    q = torch.empty(b, hq, d, dtype=torch.float16, device=dev)
    q_seq = torch.arange(b, dtype=torch.int32, device=dev).repeat_interleave(3)
    q_len = (lens.repeat_interleave(3) - torch.tensor([2, 1, 0] * b, dtype=torch.int32, device=dev)).int()
    qp = torch.empty(3 * b, hq, d, dtype=torch.float16, device=dev)
    kp = torch.zeros(nblk, bs, h, rb, dtype=torch.uint8, device=dev)
    vp = torch.zeros_like(kp)
    out = torch.empty(b, hq, d, dtype=torch.float16, device=dev)
    outp = torch.empty(3 * b, hq, d, dtype=torch.float16, device=dev)
    back = torch.empty(b * n, h, d, dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_paged_decode_workspace(b, hq, h, d, bt.shape[1], bs), dtype=torch.uint8, device=dev)
    wsp = torch.empty(int(tq.lib().tq_paged_prefill_workspace(3 * b, hq, h, d, bt.shape[1], bs)), dtype=torch.uint8,
                      device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)

    def fill(seed):
        g = torch.Generator(device="cpu").manual_seed(seed)
        for t in (kraw, vraw, q, qp):
            t.copy_(torch.randn(t.shape, generator=g).to(torch.float16))

    def work():
        tq.tq_write_kv(kraw, kp, slots, signs, ck, status=st[0:1], check=False)
        tq.tq_write_kv(vraw, vp, slots, signs, cv, status=st[1:2], check=False)
        tq.tq_paged_decode(q, kp, vp, bt, lens, signs, ck, cv, out=out, workspace=ws, status=st[2:3])
        tq.tq_dequant_rows(kp, slots, signs, ck, out=back, status=st[3:4], check=False)
        tq.tq_paged_prefill(qp, q_seq, q_len, kp, vp, bt, signs, ck, cv, out=outp, workspace=wsp)

    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        fill(1)
        work()  # first calls outside capture (one-time set-up such as kernel attributes)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            work()
        fill(2)
        graph.replay()
        stream.synchronize()
        got = [t.clone() for t in (kp, vp, out, back, outp)]
        assert int(st.abs().sum().item()) == 0
        fill(2)
        work()
        stream.synchronize()
        want = [kp, vp, out, back, outp]
    for g, w in zip(got, want):
        assert torch.equal(g, w)
