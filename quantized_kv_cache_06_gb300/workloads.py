"""Seeded synthetic inputs for the five TurboQuant packed-KV workloads.

Shared by the tests, the benchmark and the CPU oracle runs.  This module only draws
random numbers and lays out sequences, block tables and slots; it holds none of the
method's arithmetic (no rotation, codebook, quantisation or attention).

Workloads (sizes of the pages' contract example and of the benchmark configurations):
  1  tiny: D=128, K4/V4, Hq=16 / H=2, block 16, 64 fp32 tokens N(0,1) at slots
     0..63 in 32 blocks, one fp32 query, identity block table.
  2  mixed bits K4/V2: D=128, Hq=32 / H=8, block 16, 8 sequences with lengths
     uniform in [1, 2048] (seed 0), randomly permuted block table, 10% of write
     slots -1, fp16 K/V N(0,1) times a lognormal(0, 0.5) scale per (kv head,
     channel) and component, fp16 q N(0,1).
  3  sweep: bits in {2, 3, 5} x D in {64, 128, 256}, Hq=32 / H=8, block 16,
     16 sequences x 4096 tokens, 4096 blocks, fp16 K/V and q as in 2.
  4  large decode batch: 64 sequences x 8192, D=128, Hq=32 / H=8, K4/V4, block 16,
     32768 blocks in a random permutation, fp16 as in 2; all 524288 tokens written.
  5  long context: 4 sequences x 131072, D=128, Hq=64 / H=8 (group 8), K4/V2,
     block 16, 32768 blocks, fp16 K/V with the lognormal scale and 1% of the
     token-head rows multiplied by 8; plus a prefill-style batch re-writing
     sequence 0 (131072 tokens = 1,048,576 head-rows per component) with 5% of its
     slots -1.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SWEEP = [(bits, d) for bits in (2, 3, 5) for d in (64, 128, 256)]


@dataclass
class Workload:
    name: str
    head_dim: int
    k_bits: int
    v_bits: int
    num_q_heads: int
    num_kv_heads: int
    block_size: int
    num_blocks: int
    seq_lens: np.ndarray      # int32 [B]
    block_table: np.ndarray   # int32 [B, max_blocks]
    k_raw: np.ndarray         # [T, H, D] float32 or float16, tokens of all sequences in order
    v_raw: np.ndarray
    slots: np.ndarray         # int64 [T]
    q: np.ndarray             # [B, Hq, D]
    write_k: np.ndarray | None = None      # optional separate write batch
    write_v: np.ndarray | None = None
    write_slots: np.ndarray | None = None
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.slots.shape[0])

    def seq_token_offsets(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seq_lens.astype(np.int64))])


def _block_table(rng, seq_lens, block_size, num_blocks):
    nblk = [-(-int(n) // block_size) for n in seq_lens]
    width = max(max(nblk), 1)
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.zeros((len(seq_lens), width), dtype=np.int32)
    pos = 0
    for b, nb in enumerate(nblk):
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
    assert pos <= num_blocks
    return bt


def _slots(seq_lens, block_table, block_size):
    out = []
    for b, n in enumerate(seq_lens):
        t = np.arange(int(n), dtype=np.int64)
        out.append(block_table[b, t // block_size].astype(np.int64) * block_size + t % block_size)
    return np.concatenate(out) if out else np.zeros(0, dtype=np.int64)


def _scaled_normal(rng, shape, dtype, scale=None, outlier_p=0.0, chunk=1 << 16):
    """N(0,1) rows times a per-(head, channel) scale, optionally x8 outlier rows, in chunks."""
    t = shape[0]
    out = np.empty(shape, dtype=dtype)
    for s in range(0, t, chunk):
        e = min(t, s + chunk)
        x = rng.standard_normal((e - s,) + tuple(shape[1:]), dtype=np.float32)
        if scale is not None:
            x *= scale[None]
        if outlier_p > 0:
            hit = rng.random((e - s, shape[1]), dtype=np.float32) < outlier_p
            x[hit] *= 8.0
        out[s:e] = x.astype(dtype, copy=False)
    return out


def make_workload(cfg: int, sub: int = 0, batch: int | None = None, shard: int = 0) -> Workload:
    """Workload `cfg` (1..5); `sub` picks the sweep point of workload 3 (index into SWEEP);
    `batch` optionally keeps only the first sequences (same per-sequence structure);
    `shard` > 0 draws another independent batch of the same shape (one per rank when the
    batch is replicated across GPUs; shard 0 is the workload itself)."""
    if cfg == 1:
        rng = np.random.default_rng(1)
        d, h, hq, bs, nb = 128, 2, 16, 16, 32
        seq_lens = np.array([64], dtype=np.int32)
        bt = np.arange(32, dtype=np.int32)[None, :]
        k = rng.standard_normal((64, h, d), dtype=np.float32)
        v = rng.standard_normal((64, h, d), dtype=np.float32)
        q = rng.standard_normal((1, hq, d), dtype=np.float32)
        return Workload("tiny D128 K4/V4 Hq16/H2 64 tokens", d, 4, 4, hq, h, bs, nb, seq_lens, bt, k, v,
                        np.arange(64, dtype=np.int64), q)

    if cfg == 2:
        seq_lens = np.random.default_rng(0).integers(1, 2049, size=8).astype(np.int32)
        rng = np.random.default_rng(2 if shard == 0 else (2, shard))
        d, h, hq, bs, kb, vb = 128, 8, 32, 16, 4, 2
        name = "mixed K4/V2 D128 Hq32/H8 8 seqs len U[1,2048]"
    elif cfg == 3:
        kb, d = SWEEP[sub]
        vb = kb
        seq_lens = np.full(16, 4096, dtype=np.int32)
        rng = np.random.default_rng(300 + sub if shard == 0 else (300 + sub, shard))
        h, hq, bs = 8, 32, 16
        name = f"sweep K{kb}/V{vb} D{d} Hq32/H8 16x4096"
    elif cfg == 4:
        seq_lens = np.full(64, 8192, dtype=np.int32)
        rng = np.random.default_rng(4 if shard == 0 else (4, shard))
        d, h, hq, bs, kb, vb = 128, 8, 32, 16, 4, 4
        name = "decode batch K4/V4 D128 Hq32/H8 64x8192"
    elif cfg == 5:
        seq_lens = np.full(4, 131072, dtype=np.int32)
        rng = np.random.default_rng(5 if shard == 0 else (5, shard))
        d, h, hq, bs, kb, vb = 128, 8, 64, 16, 4, 2
        name = "long context K4/V2 D128 Hq64/H8 4x131072"
    else:
        raise ValueError(f"unknown workload {cfg}")

    full_blocks = {2: int(sum(-(-int(n) // 16) for n in seq_lens)), 3: 4096, 4: 32768, 5: 32768}[cfg]
    bt = _block_table(rng, seq_lens, bs, full_blocks)
    if batch is not None:
        seq_lens, bt = seq_lens[:batch].copy(), bt[:batch].copy()
    slots = _slots(seq_lens, bt, bs)
    t = slots.shape[0]
    k_scale = rng.lognormal(0.0, 0.5, size=(h, d)).astype(np.float32)
    v_scale = rng.lognormal(0.0, 0.5, size=(h, d)).astype(np.float32)
    outlier = 0.01 if cfg == 5 else 0.0
    k = _scaled_normal(rng, (t, h, d), np.float16, k_scale, outlier)
    v = _scaled_normal(rng, (t, h, d), np.float16, v_scale, outlier)
    if cfg == 2:
        slots = np.where(rng.random(t) < 0.10, -1, slots)
    q = rng.standard_normal((len(seq_lens), hq, d), dtype=np.float32).astype(np.float16)
    w = Workload(name, d, kb, vb, hq, h, bs, full_blocks, seq_lens, bt, k, v, slots, q)
    if cfg == 5:
        n0 = int(seq_lens[0])
        ws = slots[:n0].copy()
        ws[rng.random(n0) < 0.05] = -1
        w.write_k = _scaled_normal(rng, (n0, h, d), np.float16, k_scale, outlier)
        w.write_v = _scaled_normal(rng, (n0, h, d), np.float16, v_scale, outlier)
        w.write_slots = ws
    return w
