"""Benchmark of the TurboQuant packed-KV hot path on GB300.

One step = the whole hot path over one batch of the 64 x 8192 K4/V4 decode-batch
workload: tq_write_kv of all 524,288 token rows for K, the same for V, an L2 flush,
then tq_paged_decode of 64 queries (32 q heads, 8 kv heads, D=128) over the pages.

Prints ONE JSON line (rank 0).  `value` is the decode's packed-KV throughput in GB/s
(algorithmic bytes: packed K and V rows read plus q and out, over the decode's
CUDA-event time); the writer's rows/s and the decode's seq/s ride along.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--batch B]

--impl reference times the CPU oracle (the only other implementation: the pages
publish no code to run) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TQ paged decode KV GB/s (% of HBM peak) and seq/s; tq_write_kv rows/s"
WORKLOAD_CFG = 4
# What "dtype" stands for: the arithmetic of the path, kernel by kernel.
DTYPE_NOTE = ("writer: fp16/bf16 raw rows rotated by m16n8k16 MMAs with fp32 accumulation (fp32 rows on the "
              "SIMT writer), norms and quantiser decisions in fp32; decode: m16n8k16 fp16 MMA operands with fp32 "
              "accumulation (query split into fp16 hi + lo, fp16 centroid table entries, fp16 value weights; the "
              "fp16 remainders of keys and values added on tiles of large norm), softmax and split-K merge in fp32")
THREADS_NOTE = ("cores = the BLAS threads the oracle's matrix products use; its unpacking, gathers and softmax "
                "run in one thread; host_cores = os.cpu_count()")
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--batch", type=int, default=None, help="keep only the first B sequences (profiling runs)")
    p.add_argument("--workload", type=int, default=WORKLOAD_CFG, help="workload number 1..5 (default 4)")
    p.add_argument("--sub", type=int, default=0, help="sweep point of workload 3 (0..8)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def init_dist(world, local_rank, backend):
    """One process per GPU (torchrun env); no-op for a single rank."""
    if world > 1:
        import torch
        import torch.distributed as dist

        if backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        else:
            dist.init_process_group(backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(values, world, device="cpu"):
    """Element-wise max of `values` over all ranks (the slowest rank sets the time)."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def weak_scaling_rate(world, units_per_rank, max_seconds):
    """Whole-job throughput: every rank processed `units_per_rank` within `max_seconds`."""
    return world * units_per_rank / max_seconds


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def row_bytes(d, b):
    return -(-d * b // 8) + 4


def decode_bytes(w):
    """Algorithmic decode bytes: packed K+V rows of every attended token-head, plus q and out."""
    kv = int(w.seq_lens.astype(np.int64).sum()) * w.num_kv_heads * (row_bytes(w.head_dim, w.k_bits) +
                                                                     row_bytes(w.head_dim, w.v_bits))
    qo = 2 * w.q.size * w.q.itemsize
    return kv + qo


def write_bytes(w, raw, slots, bits):
    """Algorithmic writer bytes for one component: raw rows read, packed rows written, slots read."""
    written = int((slots >= 0).sum()) * w.num_kv_heads
    return raw.size * raw.itemsize + written * row_bytes(w.head_dim, bits) + slots.size * 8


def kernel_source_hash(files):
    """Hash of the kernel source files a traffic figure was taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_kv_cache_06_gb300", "csrc")
    for name in sorted(files):
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
        except OSError:
            return None
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """Per-launch DRAM bytes from the committed ncu summary, if taken on the kernel's current sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get("kernels", {}).get(kernel_key)
    if ent is None or ent.get("source_hash") != kernel_source_hash(ent.get("sources", [])):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle timing

class OracleSample:
    """Times the oracle (as it stands) on a bounded sample of the workload: the write of
    the first n_write_tokens tokens (K and V) and the decode of the first n_seq
    sequences.  The pages the decode reads are written by the oracle once, untimed."""

    def __init__(self, w, n_seq, n_write_tokens):
        from oracle import tq_oracle as o

        self.o, self.w, self.n_seq = o, w, n_seq
        d = w.head_dim
        self.signs = o.splitmix64_signs(d, 42)
        self.ck = o.codebook_f32(d, w.k_bits)[0]
        self.cv = o.codebook_f32(d, w.v_bits)[0]
        rb_k, rb_v = row_bytes(d, w.k_bits), row_bytes(d, w.v_bits)
        ntok = int(w.seq_token_offsets()[n_seq])
        self.nw = min(n_write_tokens, ntok)
        kp = np.zeros((w.num_blocks, w.block_size, w.num_kv_heads, rb_k), dtype=np.uint8)
        vp = np.zeros((w.num_blocks, w.block_size, w.num_kv_heads, rb_v), dtype=np.uint8)
        self.kp = o.write_kv(w.k_raw[:ntok], kp, w.slots[:ntok], self.signs, self.ck, w.k_bits)
        self.vp = o.write_kv(w.v_raw[:ntok], vp, w.slots[:ntok], self.signs, self.cv, w.v_bits)
        self.dec_bytes = int(w.seq_lens[:n_seq].astype(np.int64).sum()) * w.num_kv_heads * (rb_k + rb_v) + \
            2 * w.q[:n_seq].size * w.q.itemsize

    def run(self):
        o, w, nw = self.o, self.w, self.nw
        t0 = time.perf_counter()
        o.write_kv(w.k_raw[:nw], self.kp, w.slots[:nw], self.signs, self.ck, w.k_bits)
        o.write_kv(w.v_raw[:nw], self.vp, w.slots[:nw], self.signs, self.cv, w.v_bits)
        t_write = time.perf_counter() - t0
        t0 = time.perf_counter()
        o.paged_decode(w.q[:self.n_seq], self.kp, self.vp, w.k_bits, w.v_bits, w.block_table[:self.n_seq],
                       w.seq_lens[:self.n_seq], self.signs, self.ck, self.cv)
        t_dec = time.perf_counter() - t0
        return {"decode_gbs": self.dec_bytes / t_dec / 1e9, "decode_seq_per_s": self.n_seq / t_dec,
                "write_rows_per_s": 2 * nw * w.num_kv_heads / t_write, "t_decode_s": t_dec, "t_write_s": t_write}


def next_rows_cpu_baselines(w, n_write_tokens=2048, chunk=4):
    """The oracle (as it stands) timed on bounded samples of the next rows' work, on this host's
    cores, in the units of each row's GPU figure: the readback of sequence 0's K rows, a
    `chunk`-row prefill chunk at the end of sequence 0, and for product-quantised keys the
    write of `n_write_tokens` tokens' K rows plus the decode of sequence 0 over them.  The
    pages hold sequence 0 only (its tokens at slots 0..n-1), written by the oracle, untimed."""
    from oracle import qjl_oracle as qo
    from oracle import tq_oracle as o

    d, h, bs, hq = w.head_dim, w.num_kv_heads, w.block_size, w.num_q_heads
    n0 = int(w.seq_lens[0])
    nblk = max(1, -(-n0 // bs))
    bt = np.arange(nblk, dtype=np.int32)[None]
    slots = np.arange(n0, dtype=np.int64)
    signs = o.splitmix64_signs(d, 42)
    ck, cv = o.codebook_f32(d, w.k_bits)[0], o.codebook_f32(d, w.v_bits)[0]
    rb_k, rb_v = row_bytes(d, w.k_bits), row_bytes(d, w.v_bits)
    kraw, vraw = w.k_raw[:n0], w.v_raw[:n0]
    kp = o.write_kv(kraw, np.zeros((nblk, bs, h, rb_k), np.uint8), slots, signs, ck, w.k_bits)
    vp = o.write_kv(vraw, np.zeros((nblk, bs, h, rb_v), np.uint8), slots, signs, cv, w.v_bits)
    cores = blas_threads()

    def entry(value, sample):
        return {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}

    out = {}
    t0 = time.perf_counter()
    o.dequant_slots(kp, slots, signs, ck, w.k_bits)
    t = time.perf_counter() - t0
    out["tq_dequant_rows"] = entry((n0 * h * (rb_k + 2 * d) + n0 * 8) / t / 1e9,
                                   f"readback of the {n0 * h} K rows of sequence 0 (fp64 out)")

    c = min(chunk, n0)
    q = np.random.default_rng(7).standard_normal((c, hq, d)).astype(np.float16)
    q_len = (n0 - c + 1 + np.arange(c)).astype(np.int64)
    t0 = time.perf_counter()
    o.paged_prefill(q, np.zeros(c, np.int64), q_len, kp, vp, w.k_bits, w.v_bits, bt, signs, ck, cv)
    t = time.perf_counter() - t0
    unique = n0 * h * (rb_k + rb_v) + 2 * q.size * 2
    out["tq_paged_prefill"] = entry(unique / t / 1e9, f"{c} query rows at the end of sequence 0 ({n0} tokens), "
                                                      "GB/s of unique bytes")

    kb = w.k_bits
    if d in (64, 128) and 3 <= kb <= 5:
        rot = o.rotation_matrix(signs)
        kc = o.codebook_f32(d, kb - 1)[0]
        smat = qo.normal_matrix(d, d, 43).astype(np.float32).astype(np.float64)
        rbp = qo.prod_row_bytes(d, kb)
        nw = min(n_write_tokens, n0)
        x = np.asarray(kraw[:nw], dtype=np.float64).reshape(-1, d)
        t0 = time.perf_counter()
        enc = qo.encode_prod(x, rot, kc, smat)
        qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], enc["gamma"], kb)
        t_w = time.perf_counter() - t0
        enc = qo.encode_prod(np.asarray(kraw, dtype=np.float64).reshape(-1, d), rot, kc, smat)
        rows = qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], enc["gamma"], kb).reshape(n0, h, rbp)
        kpp = np.zeros((nblk * bs, h, rbp), np.uint8)
        kpp[:n0] = rows
        kpp = kpp.reshape(nblk, bs, h, rbp)
        t0 = time.perf_counter()
        qo.paged_decode_prod_keys(w.q[:1], kpp, vp, kb, w.v_bits, bt, np.array([n0]), signs, kc, cv, smat)
        t_d = time.perf_counter() - t0
        wr_bytes = nw * h * (d * kraw.itemsize + rbp) + nw * 8
        dec_bytes = n0 * h * (rbp + rb_v) + 2 * w.q[:1].size * w.q.itemsize
        out["qjl_residual_keys"] = {
            "write": entry(wr_bytes / t_w / 1e9, f"product-key write of {nw} tokens x {h} K rows"),
            "decode": entry(dec_bytes / t_d / 1e9, f"decode of sequence 0 ({n0} tokens) over product keys")}

    # INT8-query prefill: the same chunk as the float prefill, on int8 codes and scales
    from oracle import int8q_oracle as iq
    codes, scales = iq.quantize_queries_int8(q)
    t0 = time.perf_counter()
    iq.paged_prefill_int8q(codes, scales, np.zeros(c, np.int64), q_len, kp, vp, w.k_bits, w.v_bits, bt, signs, ck, cv)
    t = time.perf_counter() - t0
    out["int8q_prefill"] = entry((n0 * h * (rb_k + rb_v) + codes.size + 4 * scales.size + 2 * q.size) / t / 1e9,
                                 f"{c} int8 query rows at the end of sequence 0 ({n0} tokens), GB/s of unique bytes")

    # recipe modes: the recipe write of n_write_tokens tokens' K rows, and the decode of
    # sequence 0 over K and V recipe pages (channel groups calibrated on those K rows)
    if d in (64, 128):
        from oracle import recipe_oracle as ro
        nw = min(n_write_tokens, n0)
        rec = {}
        for recipe in ("turboquant25", "turboquant35"):
            smat = qo.normal_matrix(d // 2, d // 2, ro.SKETCH_SEED).astype(np.float32).astype(np.float64)
            codec = ro.RecipeCodec(recipe, d, smat=smat)
            rb = ro.recipe_row_bytes(recipe, d)
            high = ro.calibrate_high_groups(np.asarray(kraw[:nw], dtype=np.float64), recipe)
            pages = np.zeros((nblk, bs, h, rb), np.uint8)
            t0 = time.perf_counter()
            ro.write_recipe_kv(kraw[:nw], pages, slots[:nw], high, codec)
            t_w = time.perf_counter() - t0
            kpr = ro.write_recipe_kv(kraw, pages, slots, high, codec)
            vpr = ro.write_recipe_kv(vraw, pages, slots, high, codec)
            t0 = time.perf_counter()
            ro.paged_decode_recipe(w.q[:1], kpr, vpr, bt, np.array([n0]), high, codec)
            t_d = time.perf_counter() - t0
            rec[recipe] = {
                "write": entry((nw * h * (d * kraw.itemsize + rb) + nw * 8) / t_w / 1e9,
                               f"recipe write of {nw} tokens x {h} K rows"),
                "decode": entry((n0 * h * 2 * rb + 2 * w.q[:1].size * w.q.itemsize) / t_d / 1e9,
                                f"decode of sequence 0 ({n0} tokens) over K and V recipe pages")}
        out["recipe_modes"] = rec
    return out


def blas_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def write_batch(w):
    """(K rows, V rows, slots) the step writes: the workload's separate write batch when it has
    one (workload 5: a prefill-style re-write of sequence 0), else the whole cache."""
    if w.write_k is not None:
        return w.write_k, w.write_v, w.write_slots
    return w.k_raw, w.v_raw, w.slots


def workload_config(w, batch_override):
    wk, _, _ = write_batch(w)
    raw_gb = wk.size * wk.itemsize / 1e9
    return {"workload": f"{w.name}: write {wk.shape[0]} tokens K+V, then decode", "batch": w.batch,
            "seq_len": int(w.seq_lens.max()), "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "k_bits": w.k_bits, "v_bits": w.v_bits, "block_size": w.block_size,
            "num_blocks": w.num_blocks, "raw_dtype": str(w.k_raw.dtype),
            "l2": f"256 MB L2 flush before each decode ({raw_gb:.2f} GB raw rows written per component)",
            "batch_override": batch_override}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from quantized_kv_cache_06_gb300.workloads import make_workload

    w = make_workload(args.workload, sub=args.sub, batch=args.batch)
    n_seq, n_write = min(2, w.batch), 4096
    sampler = OracleSample(w, n_seq, n_write)
    for _ in range(args.warmup):
        sampler.run()
    vals, secs = [], []
    for _ in range(args.steps):
        r = sampler.run()
        vals.append(r["decode_gbs"])
        secs.append(r["t_decode_s"] + r["t_write_s"])
    value = statistics.median(vals)
    cores = blas_threads()
    sample = (f"oracle decode of {n_seq} of {w.batch} sequences (all {w.num_q_heads} q heads, full context) and "
              f"write of {n_write} tokens x {w.num_kv_heads} heads for K and V, per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.batch),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "host_cores": os.cpu_count(),
                             "threads_note": THREADS_NOTE, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch

    import quantized_kv_cache_06_gb300 as tq
    from quantized_kv_cache_06_gb300.workloads import make_workload

    rank, world, local_rank = dist_env()
    init_dist(world, local_rank, "nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    tq.lib()

    w = make_workload(args.workload, sub=args.sub, batch=args.batch, shard=rank)  # each rank its own batch
    d = w.head_dim
    signs = tq.tq_build_rotation(d, 42, dev)
    ck = tq.tq_codebook(d, w.k_bits, dev)[0]
    cv = tq.tq_codebook(d, w.v_bits, dev)[0]
    rb_k, rb_v = tq.tq_row_bytes(d, w.k_bits), tq.tq_row_bytes(d, w.v_bits)
    wk_np, wv_np, ws_np = write_batch(w)
    kraw = torch.from_numpy(wk_np).to(dev)
    vraw = torch.from_numpy(wv_np).to(dev)
    slots = torch.from_numpy(ws_np).to(dev)
    cache_slots = torch.from_numpy(w.slots).to(dev)  # every token of the cache, for the readback
    q = torch.from_numpy(w.q).to(dev)
    bt = torch.from_numpy(w.block_table).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    kp = torch.zeros(w.num_blocks, w.block_size, w.num_kv_heads, rb_k, dtype=torch.uint8, device=dev)
    vp = torch.zeros(w.num_blocks, w.block_size, w.num_kv_heads, rb_v, dtype=torch.uint8, device=dev)
    out = torch.empty(w.q.shape, dtype=q.dtype, device=dev)
    ws = torch.empty(max(16, tq.tq_paged_decode_workspace(w.batch, w.num_q_heads, w.num_kv_heads, d,
                                                           w.block_table.shape[1], w.block_size)),
                     dtype=torch.uint8, device=dev)
    st_k = torch.zeros(1, dtype=torch.int32, device=dev)
    st_v = torch.zeros(1, dtype=torch.int32, device=dev)
    st_d = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        tq.tq_write_kv(kraw, kp, slots, signs, ck, status=st_k, check=False)
        if ev is not None:
            ev[1].record(stream)
        tq.tq_write_kv(vraw, vp, slots, signs, cv, status=st_v, check=False)
        if ev is not None:
            ev[2].record(stream)
        flush.zero_()
        if ev is not None:
            ev[3].record(stream)
        tq.tq_paged_decode(q, kp, vp, bt, lens, signs, ck, cv, out=out, workspace=ws, status=st_d)
        if ev is not None:
            ev[4].record(stream)

    if w.write_k is not None:  # the cache the decode reads: every token written once, untimed
        for raw, pages, cents, st in ((w.k_raw, kp, ck, st_k), (w.v_raw, vp, cv, st_v)):
            tq.tq_write_kv(torch.from_numpy(raw).to(dev), pages, cache_slots, signs, cents, status=st, check=False)
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for s in (st_k, st_v, st_d):
        tq.raise_for_device_status(s)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = tq.tq_launch_count()
    t0.record(stream)
    for i in range(args.steps):
        step(events[i])
    t1.record(stream)
    torch.cuda.synchronize()
    launches = tq.tq_launch_count() - launches0
    barrier(world)
    clk = clocks.stop()
    for s in (st_k, st_v, st_d):  # the status words of the last timed step
        tq.raise_for_device_status(s)
    total_ms = t0.elapsed_time(t1)
    wk = [e[0].elapsed_time(e[1]) for e in events]
    wv = [e[1].elapsed_time(e[2]) for e in events]
    dec = [e[3].elapsed_time(e[4]) for e in events]
    ms_step, dec_max, wr_max = max_over_ranks(
        [total_ms / args.steps, statistics.mean(dec), statistics.mean(wk) + statistics.mean(wv)], world, dev)

    dbytes = decode_bytes(w)
    kbytes = write_bytes(w, wk_np, ws_np, w.k_bits)
    vbytes = write_bytes(w, wv_np, ws_np, w.v_bits)
    dec_s = dec_max / 1e3
    value = weak_scaling_rate(world, dbytes, dec_s) / 1e9
    write_tokens = int(ws_np.shape[0])
    head_rows = 2 * write_tokens * w.num_kv_heads
    write_s = wr_max / 1e3
    peak, peak_kind = peaks()
    dec_gbs = dbytes / dec_s / 1e9
    wr_gbs = (kbytes + vbytes) / write_s / 1e9
    roof_dec = {"kernel": "tq_paged_decode (split + combine kernels)", "bound": "hbm", "achieved": dec_gbs,
                "peak": peak, "unit": "GB/s", "frac": dec_gbs / peak, "peak_source": peak_kind,
                "algorithmic_bytes_per_launch": dbytes, "traffic": ncu_traffic("decode")}
    roof_wr = {"kernel": "tq_write_kv (validate + write kernels)", "bound": "hbm", "achieved": wr_gbs, "peak": peak,
               "unit": "GB/s", "frac": wr_gbs / peak, "peak_source": peak_kind,
               "algorithmic_bytes_per_launch": (kbytes + vbytes) / 2, "traffic": ncu_traffic("write")}
    dominant = roof_dec if dec_max / 1e3 > write_s / 2 else roof_wr

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16/f32", "dtype_note": DTYPE_NOTE, "data": "synthetic",
            "config": workload_config(w, args.batch),
            "decode_us": dec_max * 1e3, "decode_gbs_per_gpu": dec_gbs, "decode_frac_of_peak": dec_gbs / peak,
            "decode_seq_per_s": weak_scaling_rate(world, w.batch, dec_s),
            "write_us_per_component": write_s / 2 * 1e6, "write_rows_per_s": weak_scaling_rate(world, head_rows, write_s),
            "write_token_rows_per_s": weak_scaling_rate(world, 2 * write_tokens, write_s), "write_gbs_per_gpu": wr_gbs,
            "roofline": dominant, "roofline_decode": roof_dec, "roofline_write": roof_wr,
            "gpu_launches": launches, "clocks": clk}
    line["next_rows"] = {"tq_dequant_rows": dequant_measure(tq, w, dev, kp, cache_slots, signs, ck, flush, stream, peak,
                                                             peak_kind, world),
                         "tq_paged_prefill": prefill_measure(tq, w, dev, kp, vp, bt, signs, ck, cv, flush, stream,
                                                             peak, peak_kind, world),
                         "qjl_residual_keys": qjl_measure(tq, w, dev, kraw, slots, ws_np, vp, bt, lens, q, signs, cv,
                                                          flush, stream, peak, peak_kind, world),
                         "int8q_prefill": int8q_measure(tq, w, dev, kp, vp, bt, signs, ck, cv, flush, stream, peak,
                                                        peak_kind, world),
                         "recipe_modes": recipe_measure(tq, w, dev, kraw, vraw, slots, ws_np, bt, lens, q, flush,
                                                        stream, peak, peak_kind, world)}

    if not args.no_e2e:
        line["e2e"] = e2e_measure(tq, w, dev, signs, ck, cv, kp, vp, ws, dbytes, world)
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        sampler = OracleSample(w, min(2, w.batch), 4096)
        r = sampler.run()
        line["cpu_baseline"] = {"value": r["decode_gbs"], "unit": "GB/s", "cores": blas_threads(),
                                "host_cores": os.cpu_count(), "threads_note": THREADS_NOTE, "kind": "oracle",
                                "sample": f"oracle decode of {sampler.n_seq} sequences ({w.num_q_heads} q heads, "
                                          f"{int(w.seq_lens[:sampler.n_seq].max())} tokens) and write of {sampler.nw} "
                                          f"tokens x {w.num_kv_heads} heads for K and V",
                                "decode_seq_per_s": r["decode_seq_per_s"], "write_rows_per_s": r["write_rows_per_s"]}
        for key, base in next_rows_cpu_baselines(w).items():
            if key in line["next_rows"]:
                line["next_rows"][key]["cpu_baseline"] = base
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def dequant_measure(tq, w, dev, kp, cache_slots, signs, ck, flush, stream, peak, peak_kind, world, steps=5):
    """Dense readback of every K row of the workload (tq_dequant_rows, fp16 out), timed
    apart from the step with CUDA events, an L2 flush before each call."""
    import torch

    out = torch.empty(w.num_tokens, w.num_kv_heads, w.head_dim, dtype=torch.float16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):
        tq.tq_dequant_rows(kp, cache_slots, signs, ck, out=out, status=st, check=False)
    times = []
    for i in range(steps):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        tq.tq_dequant_rows(kp, cache_slots, signs, ck, out=out, status=st, check=False)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    tq.raise_for_device_status(st)
    t_s = max_over_ranks([statistics.mean(times)], world, dev)[0] / 1e3
    written = int((w.slots >= 0).sum()) * w.num_kv_heads
    rows = w.num_tokens * w.num_kv_heads
    nbytes = written * row_bytes(w.head_dim, w.k_bits) + rows * w.head_dim * 2 + w.num_tokens * 8
    gbs = nbytes / t_s / 1e9
    return {"workload": f"read back all {rows} K rows (K{w.k_bits} D{w.head_dim}) to fp16", "us": t_s * 1e6,
            "rows_per_s": weak_scaling_rate(world, rows, t_s), "gbs_per_gpu": gbs,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_source": peak_kind, "algorithmic_bytes_per_launch": nbytes,
                         "traffic": ncu_traffic("dequant")},
            "gpu_launches": steps + 2}


def prefill_measure(tq, w, dev, kp, vp, bt, signs, ck, cv, flush, stream, peak, peak_kind, world, chunk=16,
                    steps=5):
    """Mixed prefill/decode over the workload's cache: a chunk of the last `chunk` tokens of
    every sequence as query rows (each sees its causal prefix), timed apart from the step."""
    import numpy as np
    import torch

    lens = w.seq_lens.astype(np.int64)
    q_seq = np.repeat(np.arange(w.batch, dtype=np.int32), chunk)
    q_len = (np.repeat(lens, chunk) - chunk + 1 + np.tile(np.arange(chunk), w.batch)).astype(np.int32)
    rows = len(q_seq)
    gen = torch.Generator().manual_seed(7)
    q = torch.randn(rows, w.num_q_heads, w.head_dim, generator=gen).to(torch.float16).to(dev)
    dq_seq, dq_len = torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_len).to(dev)
    out = torch.empty_like(q)
    need = int(tq.lib().tq_paged_prefill_workspace(rows, w.num_q_heads, w.num_kv_heads, w.head_dim, bt.shape[1],
                                                  w.block_size))
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):
        tq.tq_paged_prefill(q, dq_seq, dq_len, kp, vp, bt, signs, ck, cv, out=out, workspace=ws, status=st)
    launches0 = tq.tq_launch_count()
    times = []
    for i in range(steps):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        tq.tq_paged_prefill(q, dq_seq, dq_len, kp, vp, bt, signs, ck, cv, out=out, workspace=ws, status=st)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    tq.raise_for_device_status(st)
    launches = tq.tq_launch_count() - launches0
    t_s = max_over_ranks([statistics.mean(times)], world, dev)[0] / 1e3
    rb = row_bytes(w.head_dim, w.k_bits) + row_bytes(w.head_dim, w.v_bits)
    unique = int(lens.sum()) * w.num_kv_heads * rb + 2 * rows * w.num_q_heads * w.head_dim * 2
    streamed = int(q_len.astype(np.int64).sum()) * w.num_kv_heads * rb
    gbs = unique / t_s / 1e9
    return {"workload": f"{rows} query rows: the last {chunk} tokens of each of the {w.batch} sequences "
                        f"(K{w.k_bits}/V{w.v_bits} D{w.head_dim}), each over its causal prefix",
            "us": t_s * 1e6, "rows_per_s": weak_scaling_rate(world, rows, t_s),
            "streamed_kv_gbs": streamed / t_s / 1e9, "streamed_kv_bytes": streamed,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_source": peak_kind, "algorithmic_bytes_per_launch": unique,
                         "traffic": ncu_traffic("prefill")},
            "gpu_launches": launches}


def qjl_measure(tq, w, dev, kraw, slots, slots_np, vp, bt, lens, q, signs, cv, flush, stream, peak, peak_kind,
                world, steps=3):
    """Product-quantised (QJL residual) keys at the workload's key width: the step's K rows
    written as product rows (tq_write_kv_prod), then the decode over them with the MSE value
    pages (tq_paged_decode_prod); each timed apart with CUDA events, an L2 flush before
    each call."""
    import torch

    d, kb = w.head_dim, w.k_bits
    if d not in (64, 128) or not 3 <= kb <= 5:
        return {"skipped": f"product-key kernels take head_dim 64/128 and 3..5 key bits (D{d}, K{kb})"}
    rbp = tq.tq_prod_row_bytes(d, kb)
    kmse = tq.tq_codebook(d, kb - 1, dev)[0]
    smat = tq.tq_build_qjl_matrix(d, 43, dev)
    kpp = torch.zeros(w.num_blocks, w.block_size, w.num_kv_heads, rbp, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    need = int(tq.lib().tq_paged_decode_prod_workspace(w.batch, w.num_q_heads, w.num_kv_heads, d, bt.shape[1],
                                                       w.block_size))
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

    def timed(fn):
        fn()
        times = []
        for i in range(steps):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        tq.raise_for_device_status(st)
        return max_over_ranks([statistics.mean(times)], world, dev)[0] / 1e3

    launches0 = tq.tq_launch_count()
    wr_s = timed(lambda: tq.tq_write_kv_prod(kraw, kpp, slots, signs, kmse, smat, status=st, check=False))
    dec_s = timed(lambda: tq.tq_paged_decode_prod(q, kpp, vp, bt, lens, signs, kmse, cv, smat, out=out, workspace=ws,
                                                  status=st))
    rows = int((slots_np >= 0).sum()) * w.num_kv_heads
    wr_bytes = kraw.numel() * kraw.element_size() + rows * rbp + slots_np.size * 8
    dec_bytes = int(w.seq_lens.astype(np.int64).sum()) * w.num_kv_heads * (rbp + row_bytes(d, w.v_bits)) + \
        2 * q.numel() * q.element_size()
    wr_gbs, dec_gbs = wr_bytes / wr_s / 1e9, dec_bytes / dec_s / 1e9
    return {"workload": f"{rows} K rows written as product rows (K{kb} = {kb - 1}-bit MSE + 1 sign bit, D{d}), "
                        f"then the decode of the {w.batch} sequences over them with the V{w.v_bits} pages",
            "write_us": wr_s * 1e6, "write_rows_per_s": weak_scaling_rate(world, rows, wr_s), "write_gbs": wr_gbs,
            "write_frac_of_hbm": wr_gbs / peak, "sketch_tflops": rows * 2.0 * d * d / wr_s / 1e12,
            "decode_us": dec_s * 1e6, "decode_gbs": dec_gbs, "decode_frac_of_hbm": dec_gbs / peak,
            "algorithmic_bytes": {"write": wr_bytes, "decode": dec_bytes}, "peak": peak, "peak_source": peak_kind,
            "kernels": ("write_tc_kernel<fp16, 128, 3, PROD> (mma.sync rotation, tcgen05 sketch S r); "
                        "qjl_project_kernel (p = S q~) + decode_tc_kernel<128, 3, 4, 4, 2, PROD> "
                        "(mma.sync, sketch term as a second MMA) + combine_tc_kernel"),
            "gpu_launches": tq.tq_launch_count() - launches0}


def recipe_measure(tq, w, dev, kraw, vraw, slots, slots_np, bt, lens, q, flush, stream, peak, peak_kind, world,
                   steps=3):
    """Recipe cache modes turboquant25 / turboquant35 on the workload's cache: the step's K and
    V rows written as recipe rows (channel groups calibrated on the first 4096 tokens' K rows),
    then the decode of the batch over them; each call timed apart with CUDA events, an L2
    flush before each."""
    import torch

    d = w.head_dim
    if d not in (64, 128):
        return {"skipped": f"recipe kernels take head_dim 64/128 (D{d})"}
    out = {}
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    res = torch.empty_like(q)

    def timed(fn):
        fn()
        times = []
        for i in range(steps):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        tq.raise_for_device_status(st)
        return max_over_ranks([statistics.mean(times)], world, dev)[0] / 1e3

    for recipe in ("turboquant25", "turboquant35"):
        codec = tq.RecipeCodec(recipe, d, dev)
        high = tq.tq_recipe_calibrate(recipe, kraw[:4096].float().cpu())
        order = tq.tq_recipe_channel_order(recipe, d, high).to(dev)
        kp = torch.zeros(w.num_blocks, w.block_size, w.num_kv_heads, codec.row_bytes, dtype=torch.uint8, device=dev)
        vp = torch.zeros_like(kp)
        tq.tq_write_kv_recipe(vraw, vp, slots, order, codec, status=st, check=False)
        need = int(tq.lib().tq_paged_decode_recipe_workspace(w.batch, w.num_q_heads, w.num_kv_heads, d, bt.shape[1],
                                                             w.block_size))
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        launches0 = tq.tq_launch_count()
        wr_s = timed(lambda: tq.tq_write_kv_recipe(kraw, kp, slots, order, codec, status=st, check=False))
        dec_s = timed(lambda: tq.tq_paged_decode_recipe(q, kp, vp, bt, lens, order, codec, out=res, workspace=ws,
                                                        status=st))
        launches = tq.tq_launch_count() - launches0
        rows = int((slots_np >= 0).sum()) * w.num_kv_heads
        wr_bytes = kraw.numel() * kraw.element_size() + rows * codec.row_bytes + slots_np.size * 8
        dec_bytes = int(w.seq_lens.astype(np.int64).sum()) * w.num_kv_heads * 2 * codec.row_bytes + \
            2 * q.numel() * q.element_size()
        wr_gbs, dec_gbs = wr_bytes / wr_s / 1e9, dec_bytes / dec_s / 1e9
        out[recipe] = {"row_bytes": codec.row_bytes, "write_us": wr_s * 1e6,
                       "write_rows_per_s": weak_scaling_rate(world, rows, wr_s), "write_gbs": wr_gbs,
                       "write_frac_of_hbm": wr_gbs / peak, "decode_us": dec_s * 1e6, "decode_gbs": dec_gbs,
                       "decode_frac_of_hbm": dec_gbs / peak,
                       "algorithmic_bytes": {"write": wr_bytes, "decode": dec_bytes}, "gpu_launches": launches}
    out.update({"workload": f"the step's {int((slots_np >= 0).sum()) * w.num_kv_heads} K rows (and V rows, untimed) "
                            f"as recipe rows at D{d}, then the decode of the {w.batch} sequences over K and V recipe "
                            "pages", "peak": peak, "peak_source": peak_kind,
                "kernels": "write_recipe_kernel (SIMT rotation and quantiser, m16n8k16 sketch); "
                           "recipe_project_kernel + decode_recipe_tc_kernel (m16n8k16 scores and values) + "
                           "combine_recipe_kernel"})
    return out


def int8q_measure(tq, w, dev, kp, vp, bt, signs, ck, cv, flush, stream, peak, peak_kind, world, chunk=16, steps=5):
    """The INT8-query prefill on the prefill chunk of prefill_measure: the queries quantised to
    int8 codes and scales once (untimed), then tq_paged_prefill_int8q timed with CUDA events,
    an L2 flush before each call."""
    import torch

    lens = w.seq_lens.astype(np.int64)
    q_seq = np.repeat(np.arange(w.batch, dtype=np.int32), chunk)
    q_len = (np.repeat(lens, chunk) - chunk + 1 + np.tile(np.arange(chunk), w.batch)).astype(np.int32)
    rows = len(q_seq)
    gen = torch.Generator().manual_seed(7)
    q = torch.randn(rows, w.num_q_heads, w.head_dim, generator=gen).to(torch.float16).to(dev)
    codes, scales = tq.tq_quantize_queries_int8(q)
    dq_seq, dq_len = torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_len).to(dev)
    out = torch.empty_like(q)
    need = int(tq.lib().tq_paged_prefill_workspace(rows, w.num_q_heads, w.num_kv_heads, w.head_dim, bt.shape[1],
                                                  w.block_size))
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        tq.tq_paged_prefill_int8q(codes, scales, dq_seq, dq_len, kp, vp, bt, signs, ck, cv, out=out, workspace=ws,
                                  status=st)

    for _ in range(2):
        call()
    launches0 = tq.tq_launch_count()
    times = []
    for i in range(steps):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    tq.raise_for_device_status(st)
    launches = tq.tq_launch_count() - launches0
    t_s = max_over_ranks([statistics.mean(times)], world, dev)[0] / 1e3
    rb = row_bytes(w.head_dim, w.k_bits) + row_bytes(w.head_dim, w.v_bits)
    unique = int(lens.sum()) * w.num_kv_heads * rb + codes.numel() + scales.numel() * 4 + out.numel() * 2
    gbs = unique / t_s / 1e9
    return {"workload": f"{rows} int8 query rows (one scale per row and q head): the last {chunk} tokens of each of "
                        f"the {w.batch} sequences, each over its causal prefix",
            "us": t_s * 1e6, "rows_per_s": weak_scaling_rate(world, rows, t_s),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "peak_source": peak_kind, "algorithmic_bytes_per_launch": unique, "traffic": None},
            "gpu_launches": launches}


def e2e_measure(tq, w, dev, signs, ck, cv, kp, vp, ws, dbytes, world, steps=5, chunks=8):
    """Same step from pinned host buffers: H2D of the step's inputs, write K, write V,
    decode, D2H of the output, all inside the timed region.  The raw rows go over in
    `chunks` token ranges on a copy stream, and each range is written as soon as it has
    landed, so the writes run under the remaining copies (the host link is the bound)."""
    import torch

    wk_np, wv_np, ws_np = write_batch(w)
    hk = torch.from_numpy(wk_np).pin_memory()
    hv = torch.from_numpy(wv_np).pin_memory()
    hs = torch.from_numpy(ws_np).pin_memory()
    hq = torch.from_numpy(w.q).pin_memory()
    hbt = torch.from_numpy(w.block_table).pin_memory()
    hl = torch.from_numpy(w.seq_lens).pin_memory()
    hout = torch.empty(w.q.shape, dtype=hq.dtype).pin_memory()
    dk, dv = torch.empty_like(hk, device=dev), torch.empty_like(hv, device=dev)
    ds, dq = torch.empty_like(hs, device=dev), torch.empty_like(hq, device=dev)
    dbt, dl = torch.empty_like(hbt, device=dev), torch.empty_like(hl, device=dev)
    dout = torch.empty_like(hq, device=dev)
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    t = hk.shape[0]
    bounds = [(t * i // chunks, t * (i + 1) // chunks) for i in range(chunks)]
    landed = [torch.cuda.Event() for _ in bounds]
    done = torch.cuda.Event()
    done.record(stream)

    def one():
        copy_stream.wait_event(done)  # the previous step no longer reads the device buffers
        with torch.cuda.stream(copy_stream):
            for h, dd in ((hq, dq), (hbt, dbt), (hl, dl)):
                dd.copy_(h, non_blocking=True)
            for (lo, hi), ev in zip(bounds, landed):
                for h, dd in ((hk, dk), (hv, dv), (hs, ds)):
                    dd[lo:hi].copy_(h[lo:hi], non_blocking=True)
                ev.record(copy_stream)
        for (lo, hi), ev in zip(bounds, landed):
            stream.wait_event(ev)
            if hi > lo:
                tq.tq_write_kv(dk[lo:hi], kp, ds[lo:hi], signs, ck, status=st, check=False)
                tq.tq_write_kv(dv[lo:hi], vp, ds[lo:hi], signs, cv, status=st, check=False)
        tq.tq_paged_decode(dq, kp, vp, dbt, dl, signs, ck, cv, out=dout, workspace=ws)
        hout.copy_(dout, non_blocking=True)
        done.record(stream)

    one()
    torch.cuda.synchronize()
    # the host link on its own, right before the steps: plain copies of the step's raw rows
    # (the link is shared with whatever else uses this host's memory, so it is taken per run)
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(copy_stream):
        l0.record(copy_stream)
        for _ in range(2):
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
        l1.record(copy_stream)
    torch.cuda.synchronize()
    link_gbs = 2 * (hk.numel() * hk.element_size() + hv.numel() * hv.element_size()) / (l0.elapsed_time(l1) / 1e3) / 1e9
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    tq.raise_for_device_status(st)
    sec = e0.elapsed_time(e1) / 1e3 / steps
    h2d = sum(t_.numel() * t_.element_size() for t_ in (hk, hv, hs, hq, hbt, hl))
    return {"value": world * dbytes / sec / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": hout.numel() * hout.element_size(), "ms_per_step": sec * 1e3,
            "h2d_chunks": chunks, "host_link_gbs": link_gbs,
            "h2d_frac_of_link": h2d / sec / 1e9 / link_gbs}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
