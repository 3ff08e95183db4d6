"""ctypes binding of libtq_gb300.so (include/tq.h): argument marshalling only.

Every computation runs in the library's CUDA kernels (or, for the rotation signs
and the codebook, in its host C++).  If the library has not been built these
functions raise: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

TQ_OK = 0
TQ_ERR_INVALID_ARG = 1
TQ_ERR_UNSUPPORTED = 2
TQ_ERR_SLOT_OUT_OF_RANGE = 3
TQ_ERR_BLOCK_OUT_OF_RANGE = 4
TQ_ERR_CUDA = 5
TQ_ERR_TIMEOUT = 6

STATUS_NAMES = {
    TQ_OK: "TQ_OK",
    TQ_ERR_INVALID_ARG: "TQ_ERR_INVALID_ARG",
    TQ_ERR_UNSUPPORTED: "TQ_ERR_UNSUPPORTED",
    TQ_ERR_SLOT_OUT_OF_RANGE: "TQ_ERR_SLOT_OUT_OF_RANGE",
    TQ_ERR_BLOCK_OUT_OF_RANGE: "TQ_ERR_BLOCK_OUT_OF_RANGE",
    TQ_ERR_CUDA: "TQ_ERR_CUDA",
    TQ_ERR_TIMEOUT: "TQ_ERR_TIMEOUT",
}

_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

TQ_RECIPE_TURBOQUANT25 = 25
TQ_RECIPE_TURBOQUANT35 = 35
RECIPES = {"turboquant25": TQ_RECIPE_TURBOQUANT25, "turboquant35": TQ_RECIPE_TURBOQUANT35}
RECIPE_ROTATION_SEED = 42
RECIPE_SKETCH_SEED = 43

# Every symbol include/tq.h declares, with (restype, argtypes).
_c_int, _c_i64, _c_u64, _c_f, _c_p, _c_sz = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float,
                                            ctypes.c_void_p, ctypes.c_size_t)
SIGNATURES = {
    "tq_last_error": (ctypes.c_char_p, []),
    "tq_set_wait_limit": (_c_i64, [_c_i64]),
    "tq_launch_count": (ctypes.c_uint64, []),
    "tq_row_bytes": (_c_i64, [_c_int, _c_int]),
    "tq_build_rotation": (_c_int, [_c_int, _c_u64, _c_p]),
    "tq_codebook": (_c_int, [_c_int, _c_int, _c_p, _c_p]),
    "tq_write_kv": (_c_int, [_c_p, _c_int, _c_i64, _c_int, _c_int, _c_int, _c_p, _c_p, _c_i64, _c_int,
                             _c_p, _c_p, _c_p, _c_p]),
    "tq_dequant_rows": (_c_int, [_c_p, _c_int, _c_i64, _c_int, _c_int, _c_int, _c_p, _c_i64, _c_p, _c_p, _c_p,
                                 _c_int, _c_p, _c_p]),
    "tq_paged_decode_workspace": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "tq_paged_prefill_workspace": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "tq_paged_prefill": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_int, _c_p, _c_int, _c_i64,
                                  _c_int, _c_p, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_p, _c_int,
                                  _c_p, _c_sz, _c_p, _c_p]),
    "tq_paged_decode": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_int, _c_p, _c_int,
                                 _c_i64, _c_int, _c_p, _c_int, _c_p, _c_p, _c_p, _c_p, _c_f, _c_p, _c_int,
                                 _c_p, _c_sz, _c_p, _c_p]),
    "tq_paged_decode_static": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_int, _c_p,
                                        _c_int, _c_i64, _c_int, _c_p, _c_int, _c_p, _c_p, _c_p, _c_p, _c_f,
                                        _c_p, _c_int, _c_p, _c_p]),
    "tq_prod_row_bytes": (_c_i64, [_c_int, _c_int]),
    "tq_build_qjl_matrix": (_c_int, [_c_int, _c_u64, _c_p]),
    "tq_write_kv_prod": (_c_int, [_c_p, _c_int, _c_i64, _c_int, _c_int, _c_int, _c_p, _c_p, _c_i64, _c_int,
                                  _c_p, _c_p, _c_p, _c_p, _c_p]),
    "tq_paged_decode_prod_workspace": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "tq_paged_decode_prod": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_int, _c_p, _c_int,
                                      _c_i64, _c_int, _c_p, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_p,
                                      _c_int, _c_p, _c_sz, _c_p, _c_p]),
    "tq_quantize_queries_int8": (_c_int, [_c_p, _c_int, _c_i64, _c_int, _c_int, _c_p, _c_p, _c_p]),
    "tq_paged_prefill_int8q": (_c_int, [_c_p, _c_p, _c_int, _c_int, _c_int, _c_int, _c_p, _c_int, _c_p, _c_int,
                                        _c_i64, _c_int, _c_p, _c_int, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_f,
                                        _c_p, _c_int, _c_p, _c_sz, _c_p, _c_p]),
    "tq_recipe_row_bytes": (_c_i64, [_c_int, _c_int]),
    "tq_recipe_channel_order": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p]),
    "tq_recipe_calibrate": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_i64, _c_p]),
    "tq_write_kv_recipe": (_c_int, [_c_p, _c_int, _c_i64, _c_int, _c_int, _c_int, _c_p, _c_p, _c_i64, _c_int, _c_p,
                                    _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "tq_paged_decode_recipe_workspace": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "tq_paged_decode_recipe": (_c_int, [_c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_p, _c_p, _c_int, _c_i64,
                                        _c_int, _c_p, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_f, _c_p, _c_int,
                                        _c_p, _c_sz, _c_p, _c_p]),
}

_lib = None
_lock = threading.Lock()


class TQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                                       "(python -m quantized_kv_cache_06_gb300.build, needs nvcc for sm_103a)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def _check(status: int) -> None:
    if status != TQ_OK:
        msg = lib().tq_last_error().decode(errors="replace")
        raise TQError(status, msg)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(name: str, *tensors: torch.Tensor) -> torch.device:
    dev = tensors[0].device
    for t in tensors:
        if t.device.type != "cuda" or t.device != dev:
            raise ValueError(f"{name}: all tensors must be on the same CUDA device")
        if not t.is_contiguous():
            raise ValueError(f"{name}: tensors must be contiguous")
    return dev


_status_bufs: dict = {}


def _status_buffer(device: torch.device) -> torch.Tensor:
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    buf = _status_bufs.get(key)
    if buf is None:
        buf = torch.zeros(1, dtype=torch.int32, device=device)
        _status_bufs[key] = buf
    return buf


def raise_for_device_status(status: torch.Tensor) -> None:
    """Synchronises on `status` (a device int32 the library wrote) and raises on a non-zero code."""
    code = int(status.item())
    if code != TQ_OK:
        raise TQError(code, "reported by the device status word")


# ---------------------------------------------------------------- host set-up

def tq_set_wait_limit(tries: int) -> int:
    """Failure-path testing hook: tries of the decode's bounded device waits for later
    launches (>= 0), or the default (< 0).  Returns the previous value."""
    return int(lib().tq_set_wait_limit(int(tries)))


def tq_launch_count() -> int:
    """Kernel launches the library has enqueued in this process so far."""
    return int(lib().tq_launch_count())


def tq_row_bytes(head_dim: int, bits: int) -> int:
    n = lib().tq_row_bytes(int(head_dim), int(bits))
    if n < 0:
        raise TQError(TQ_ERR_UNSUPPORTED, f"head_dim {head_dim} / bits {bits} unsupported")
    return int(n)


def tq_build_rotation(head_dim: int, seed: int = 42, device=None) -> torch.Tensor:
    """RHT signs (float32 [head_dim], +-1) for build_rotation(dim, RHT, seed)."""
    out = torch.empty(int(head_dim), dtype=torch.float32)
    _check(lib().tq_build_rotation(int(head_dim), int(seed) & ((1 << 64) - 1), out.data_ptr()))
    return out if device is None else out.to(device)


def tq_codebook(head_dim: int, bits: int, device=None):
    """(centroids float32 [2^bits], boundaries float32 [2^bits - 1])."""
    n = 1 << int(bits)
    c = torch.empty(n, dtype=torch.float32)
    b = torch.empty(n - 1, dtype=torch.float32)
    _check(lib().tq_codebook(int(head_dim), int(bits), c.data_ptr(), b.data_ptr()))
    if device is not None:
        c, b = c.to(device), b.to(device)
    return c, b


def _need_f32(name: str, head_dim: int, signs: torch.Tensor, *others: torch.Tensor) -> None:
    """The rotation signs, codebooks and sketch matrix are read by the kernels as fp32 arrays
    of known length: another dtype, or fewer than head_dim signs, would make them read past
    the buffer."""
    for t in (signs, *others):
        if t.dtype != torch.float32:
            raise ValueError(f"{name}: signs, codebooks and the sketch matrix must be float32, got {t.dtype}")
    if signs.numel() != head_dim:
        raise ValueError(f"{name}: signs must hold head_dim = {head_dim} values, got {signs.numel()}")


def _need_out(name: str, out: torch.Tensor, shape: tuple, device: torch.device) -> None:
    """A caller-supplied output must have exactly the rows the kernels write."""
    if tuple(out.shape) != tuple(shape) or out.dtype not in _DTYPES:
        raise ValueError(f"{name}: out must be {list(shape)} f32/f16/bf16, got {list(out.shape)} {out.dtype}")
    _need_cuda(name, out)
    if out.device != device:
        raise ValueError(f"{name}: out must be on {device}")


def _need_status(name: str, status: torch.Tensor | None, device: torch.device | None = None) -> None:
    """A caller-supplied status word: one int32 (at least) on the call's device."""
    if status is None:
        return
    if status.dtype != torch.int32 or status.numel() < 1 or status.device.type != "cuda" or \
            (device is not None and status.device != device):
        raise ValueError(f"{name}: status must be an int32 tensor of at least one element on the call's device")


def _bits_from_centroids(centroids: torch.Tensor) -> int:
    n = centroids.numel()
    bits = n.bit_length() - 1
    if n < 4 or (1 << bits) != n:
        raise ValueError(f"centroids must hold 2^bits values, got {n}")
    return bits


# ---------------------------------------------------------------- writer

def tq_write_kv(raw: torch.Tensor, pages: torch.Tensor, slots: torch.Tensor, signs: torch.Tensor,
                centroids: torch.Tensor, status: torch.Tensor | None = None, check: bool = True) -> torch.Tensor:
    """write_tq4_kv(raw, pages, slots, rotation, centroids): encode raw[T, H, D] into pages[NB, bs, H, RB].

    Returns the device status word.  With check=True the call synchronises on it and
    raises TQError(TQ_ERR_SLOT_OUT_OF_RANGE) when a slot was out of range (then no row
    was written).
    """
    dev = _need_cuda("tq_write_kv", raw, pages, slots, signs, centroids)
    if raw.dim() != 3 or pages.dim() != 4 or slots.dim() != 1 or slots.numel() != raw.shape[0]:
        raise ValueError("tq_write_kv: raw [T, H, D], pages [NB, bs, H, RB], slots [T] expected")
    if raw.dtype not in _DTYPES or pages.dtype != torch.uint8 or slots.dtype != torch.int64:
        raise ValueError("tq_write_kv: raw f32/f16/bf16, pages uint8, slots int64 expected")
    t, h, d = raw.shape
    bits = _bits_from_centroids(centroids)
    _need_f32("tq_write_kv", d, signs, centroids)
    if pages.shape[2] != h or pages.shape[3] != tq_row_bytes(d, bits):
        raise ValueError(f"tq_write_kv: pages {tuple(pages.shape)} do not match H={h}, RB={tq_row_bytes(d, bits)}")
    _need_status("tq_write_kv", status, dev)
    if status is None:
        status = _status_buffer(dev)
    with torch.cuda.device(dev):
        _check(lib().tq_write_kv(_ptr(raw), _DTYPES[raw.dtype], t, h, d, bits, _ptr(slots), _ptr(pages),
                                 pages.shape[0], pages.shape[1], _ptr(signs), _ptr(centroids), _ptr(status),
                                 _stream(dev)))
    if check:
        raise_for_device_status(status)
    return status


# ---------------------------------------------------------------- readback

def tq_dequant_rows(pages: torch.Tensor, slots: torch.Tensor, signs: torch.Tensor, centroids: torch.Tensor,
                    out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float16,
                    status: torch.Tensor | None = None, check: bool = True) -> torch.Tensor:
    """Dense readback (tq4_decompress) of the rows written at `slots`: out[T, H, D] =
    nu * R^T c[idx] for slot >= 0, zeros for slot < 0.  pages [NB, bs, H, RB] uint8,
    slots [T] int64.  With check=True the call synchronises and raises
    TQError(TQ_ERR_SLOT_OUT_OF_RANGE) when a slot lies past the pages.  Returns `out`."""
    dev = _need_cuda("tq_dequant_rows", pages, slots, signs, centroids)
    if pages.dim() != 4 or slots.dim() != 1 or pages.dtype != torch.uint8 or slots.dtype != torch.int64:
        raise ValueError("tq_dequant_rows: pages uint8 [NB, bs, H, RB] and slots int64 [T] expected")
    nb, bs, h, rb = pages.shape
    d = signs.numel()
    bits = _bits_from_centroids(centroids)
    _need_f32("tq_dequant_rows", d, signs, centroids)
    if rb != tq_row_bytes(d, bits):
        raise ValueError(f"tq_dequant_rows: pages row bytes {rb} != RB({d}, {bits})")
    t = slots.numel()
    if out is None:
        out = torch.empty(t, h, d, dtype=out_dtype, device=dev)
    if tuple(out.shape) != (t, h, d) or out.dtype not in _DTYPES:
        raise ValueError(f"tq_dequant_rows: out must be [{t}, {h}, {d}] f32/f16/bf16")
    _need_cuda("tq_dequant_rows", pages, out)
    _need_status("tq_dequant_rows", status, dev)
    if status is None:
        status = _status_buffer(dev)
    with torch.cuda.device(dev):
        _check(lib().tq_dequant_rows(_ptr(pages), bits, nb, bs, h, d, _ptr(slots), t, _ptr(signs), _ptr(centroids),
                                     _ptr(out), _DTYPES[out.dtype], _ptr(status), _stream(dev)))
    if check:
        raise_for_device_status(status)
    return out


# ---------------------------------------------------------------- decode

def tq_paged_decode_workspace(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                              max_blocks_per_seq: int, block_size: int) -> int:
    return int(lib().tq_paged_decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                               block_size))


def tq_paged_decode(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                    seq_lens: torch.Tensor, signs: torch.Tensor, k_centroids: torch.Tensor,
                    v_centroids: torch.Tensor, scale: float | None = None, out: torch.Tensor | None = None,
                    out_dtype: torch.dtype | None = None, workspace: torch.Tensor | None = None,
                    status: torch.Tensor | None = None, check: bool = False) -> torch.Tensor:
    """decode_tq4_paged: attention of q[B, Hq, D] over packed K/V pages through block_table[B, maxblk]."""
    dev = _need_cuda("tq_paged_decode", q, k_pages, v_pages, block_table, seq_lens, signs, k_centroids,
                     v_centroids)
    if q.dim() != 3 or k_pages.dim() != 4 or v_pages.dim() != 4 or block_table.dim() != 2:
        raise ValueError("tq_paged_decode: q [B, Hq, D], pages [NB, bs, H, RB], block_table [B, maxblk] expected")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32 or q.dtype not in _DTYPES:
        raise ValueError("tq_paged_decode: block_table / seq_lens int32, q f32/f16/bf16 expected")
    b, hq, d = q.shape
    nb, bs, h, _ = k_pages.shape
    kb, vb = _bits_from_centroids(k_centroids), _bits_from_centroids(v_centroids)
    _need_f32("tq_paged_decode", d, signs, k_centroids, v_centroids)
    if k_pages.shape[3] != tq_row_bytes(d, kb) or v_pages.shape[3] != tq_row_bytes(d, vb) or \
            tuple(v_pages.shape[:3]) != (nb, bs, h) or block_table.shape[0] != b or seq_lens.numel() != b:
        raise ValueError("tq_paged_decode: page / table shapes inconsistent with q and the codebooks")
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((b, hq, d), dtype=out_dtype, device=dev)
    _need_out("tq_paged_decode", out, (b, hq, d), dev)
    _need_status("tq_paged_decode", status, dev)
    maxb = block_table.shape[1]
    need = tq_paged_decode_workspace(b, hq, h, d, maxb, bs)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().tq_paged_decode(_ptr(q), _DTYPES[q.dtype], b, hq, h, d, _ptr(k_pages), kb, _ptr(v_pages), vb,
                                     nb, bs, _ptr(block_table), maxb, _ptr(seq_lens), _ptr(signs),
                                     _ptr(k_centroids), _ptr(v_centroids), float(scale or 0.0), _ptr(out),
                                     _DTYPES[out.dtype], _ptr(workspace), workspace.numel(), _ptr(status),
                                     _stream(dev)))
    if check and status is not None:
        raise_for_device_status(status)
    return out


def tq_paged_prefill(q: torch.Tensor, q_seq: torch.Tensor, q_len: torch.Tensor, k_pages: torch.Tensor,
                     v_pages: torch.Tensor, block_table: torch.Tensor, signs: torch.Tensor, k_centroids: torch.Tensor,
                     v_centroids: torch.Tensor, scale: float | None = None, out: torch.Tensor | None = None,
                     out_dtype: torch.dtype | None = None, workspace: torch.Tensor | None = None,
                     status: torch.Tensor | None = None, check: bool = False) -> torch.Tensor:
    """Mixed prefill/decode over the packed pages: row i of q[T, Hq, D] is a query of sequence
    q_seq[i] that sees that sequence's first q_len[i] tokens (block_table[S, maxblk])."""
    dev = _need_cuda("tq_paged_prefill", q, q_seq, q_len, k_pages, v_pages, block_table, signs, k_centroids,
                     v_centroids)
    if q.dim() != 3 or k_pages.dim() != 4 or v_pages.dim() != 4 or block_table.dim() != 2:
        raise ValueError("tq_paged_prefill: q [T, Hq, D], pages [NB, bs, H, RB], block_table [S, maxblk] expected")
    if block_table.dtype != torch.int32 or q_seq.dtype != torch.int32 or q_len.dtype != torch.int32 or \
            q.dtype not in _DTYPES:
        raise ValueError("tq_paged_prefill: block_table / q_seq / q_len int32, q f32/f16/bf16 expected")
    t, hq, d = q.shape
    nb, bs, h, _ = k_pages.shape
    kb, vb = _bits_from_centroids(k_centroids), _bits_from_centroids(v_centroids)
    _need_f32("tq_paged_prefill", d, signs, k_centroids, v_centroids)
    if k_pages.shape[3] != tq_row_bytes(d, kb) or v_pages.shape[3] != tq_row_bytes(d, vb) or \
            tuple(v_pages.shape[:3]) != (nb, bs, h) or q_seq.numel() != t or q_len.numel() != t:
        raise ValueError("tq_paged_prefill: page / row shapes inconsistent with q and the codebooks")
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((t, hq, d), dtype=out_dtype, device=dev)
    _need_out("tq_paged_prefill", out, (t, hq, d), dev)
    _need_status("tq_paged_prefill", status, dev)
    s_rows, maxb = block_table.shape
    need = int(lib().tq_paged_prefill_workspace(t, hq, h, d, maxb, bs))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().tq_paged_prefill(_ptr(q), _DTYPES[q.dtype], t, hq, h, d, _ptr(k_pages), kb, _ptr(v_pages), vb,
                                      nb, bs, _ptr(block_table), s_rows, maxb, _ptr(q_seq), _ptr(q_len), _ptr(signs),
                                      _ptr(k_centroids), _ptr(v_centroids), float(scale or 0.0), _ptr(out),
                                      _DTYPES[out.dtype], _ptr(workspace), workspace.numel(), _ptr(status),
                                      _stream(dev)))
    if check and status is not None:
        raise_for_device_status(status)
    return out


def tq_quantize_queries_int8(q: torch.Tensor):
    """int8 codes [T, Hq, D] and fp32 scales [T, Hq] of queries q[T, Hq, D] (one symmetric
    scale per (row, q head))."""
    dev = _need_cuda("tq_quantize_queries_int8", q)
    if q.dim() != 3 or q.dtype not in _DTYPES or not q.is_contiguous():
        raise ValueError("tq_quantize_queries_int8: contiguous q [T, Hq, D] f32/f16/bf16 expected")
    t, hq, d = q.shape
    codes = torch.empty((t, hq, d), dtype=torch.int8, device=dev)
    scales = torch.empty((t, hq), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _check(lib().tq_quantize_queries_int8(_ptr(q), _DTYPES[q.dtype], t, hq, d, _ptr(codes), _ptr(scales),
                                              _stream(dev)))
    return codes, scales


def tq_paged_prefill_int8q(q_codes: torch.Tensor, q_scales: torch.Tensor, q_seq: torch.Tensor, q_len: torch.Tensor,
                           k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                           signs: torch.Tensor, k_centroids: torch.Tensor, v_centroids: torch.Tensor,
                           scale: float | None = None, out: torch.Tensor | None = None,
                           out_dtype: torch.dtype = torch.float16, workspace: torch.Tensor | None = None,
                           status: torch.Tensor | None = None, check: bool = False) -> torch.Tensor:
    """tq_paged_prefill with int8 query codes [T, Hq, D] and their fp32 scales [T, Hq]."""
    dev = _need_cuda("tq_paged_prefill_int8q", q_codes, q_scales, q_seq, q_len, k_pages, v_pages, block_table, signs,
                     k_centroids, v_centroids)
    if q_codes.dim() != 3 or q_codes.dtype != torch.int8 or q_scales.dtype != torch.float32 or \
            tuple(q_scales.shape) != tuple(q_codes.shape[:2]) or not q_codes.is_contiguous() or \
            not q_scales.is_contiguous():
        raise ValueError("tq_paged_prefill_int8q: contiguous int8 codes [T, Hq, D] and float32 scales [T, Hq] "
                         "expected")
    if block_table.dtype != torch.int32 or q_seq.dtype != torch.int32 or q_len.dtype != torch.int32:
        raise ValueError("tq_paged_prefill_int8q: block_table / q_seq / q_len int32 expected")
    t, hq, d = q_codes.shape
    nb, bs, h, _ = k_pages.shape
    kb, vb = _bits_from_centroids(k_centroids), _bits_from_centroids(v_centroids)
    _need_f32("tq_paged_prefill_int8q", d, signs, k_centroids, v_centroids)
    if k_pages.shape[3] != tq_row_bytes(d, kb) or v_pages.shape[3] != tq_row_bytes(d, vb) or \
            tuple(v_pages.shape[:3]) != (nb, bs, h) or q_seq.numel() != t or q_len.numel() != t:
        raise ValueError("tq_paged_prefill_int8q: page / row shapes inconsistent with q and the codebooks")
    if out is None:
        out = torch.empty((t, hq, d), dtype=out_dtype, device=dev)
    _need_out("tq_paged_prefill_int8q", out, (t, hq, d), dev)
    _need_status("tq_paged_prefill_int8q", status, dev)
    s_rows, maxb = block_table.shape
    need = int(lib().tq_paged_prefill_workspace(t, hq, h, d, maxb, bs))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().tq_paged_prefill_int8q(_ptr(q_codes), _ptr(q_scales), t, hq, h, d, _ptr(k_pages), kb,
                                            _ptr(v_pages), vb, nb, bs, _ptr(block_table), s_rows, maxb, _ptr(q_seq),
                                            _ptr(q_len), _ptr(signs), _ptr(k_centroids), _ptr(v_centroids),
                                            float(scale or 0.0), _ptr(out), _DTYPES[out.dtype], _ptr(workspace),
                                            workspace.numel(), _ptr(status), _stream(dev)))
    if check and status is not None:
        raise_for_device_status(status)
    return out


def tq_paged_decode_static(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                           seq_lens: torch.Tensor, signs: torch.Tensor, k_centroids: torch.Tensor,
                           v_centroids: torch.Tensor, out: torch.Tensor, scale: float | None = None,
                           status: torch.Tensor | None = None) -> torch.Tensor:
    """Allocation-free decode for callers that cannot allocate device memory: the caller
    passes `out`, and the split-K partials go to the library's fixed 16 MiB device array
    (so concurrent calls on different streams race; serialise them)."""
    dev = _need_cuda("tq_paged_decode_static", q, k_pages, v_pages, block_table, seq_lens, signs, k_centroids,
                     v_centroids, out)
    b, hq, d = q.shape
    nb, bs, h, _ = k_pages.shape
    kb, vb = _bits_from_centroids(k_centroids), _bits_from_centroids(v_centroids)
    _need_f32("tq_paged_decode_static", d, signs, k_centroids, v_centroids)
    if out.shape != q.shape or out.dtype not in _DTYPES:
        raise ValueError("tq_paged_decode_static: out must be [B, Hq, D] f32/f16/bf16")
    _need_status("tq_paged_decode_static", status, dev)
    with torch.cuda.device(dev):
        _check(lib().tq_paged_decode_static(_ptr(q), _DTYPES[q.dtype], b, hq, h, d, _ptr(k_pages), kb,
                                            _ptr(v_pages), vb, nb, bs, _ptr(block_table), block_table.shape[1],
                                            _ptr(seq_lens), _ptr(signs), _ptr(k_centroids), _ptr(v_centroids),
                                            float(scale or 0.0), _ptr(out), _DTYPES[out.dtype], _ptr(status),
                                            _stream(dev)))
    return out


# ---------------------------------------------------------------- product-quantised keys

def tq_prod_row_bytes(head_dim: int, bits: int) -> int:
    """Bytes of one product-quantised key row: (bits-1)-bit indices, D sign bits, nu, gamma."""
    n = lib().tq_prod_row_bytes(int(head_dim), int(bits))
    if n < 0:
        raise TQError(TQ_ERR_UNSUPPORTED, f"head_dim {head_dim} / bits {bits} unsupported")
    return int(n)


def tq_build_qjl_matrix(head_dim: int, seed: int, device=None) -> torch.Tensor:
    """The N(0, 1) sketch matrix S, float32 [head_dim, head_dim] (host, or moved to `device`)."""
    out = torch.empty(int(head_dim), int(head_dim), dtype=torch.float32)
    _check(lib().tq_build_qjl_matrix(int(head_dim), int(seed) & ((1 << 64) - 1), out.data_ptr()))
    return out if device is None else out.to(device)


def tq_write_kv_prod(raw: torch.Tensor, pages: torch.Tensor, slots: torch.Tensor, signs: torch.Tensor,
                     mse_centroids: torch.Tensor, qjl_matrix: torch.Tensor, status: torch.Tensor | None = None,
                     check: bool = True) -> torch.Tensor:
    """Product-quantised key rows: encode raw[T, H, D] into pages[NB, bs, H, RBP] at
    bits = log2(len(mse_centroids)) + 1.  Same slot rules and status as tq_write_kv."""
    dev = _need_cuda("tq_write_kv_prod", raw, pages, slots, signs, mse_centroids, qjl_matrix)
    if raw.dim() != 3 or pages.dim() != 4 or slots.dim() != 1 or slots.numel() != raw.shape[0]:
        raise ValueError("tq_write_kv_prod: raw [T, H, D], pages [NB, bs, H, RBP], slots [T] expected")
    if raw.dtype not in _DTYPES or pages.dtype != torch.uint8 or slots.dtype != torch.int64 or \
            qjl_matrix.dtype != torch.float32:
        raise ValueError("tq_write_kv_prod: raw f32/f16/bf16, pages uint8, slots int64, qjl_matrix f32 expected")
    t, h, d = raw.shape
    n = mse_centroids.numel()
    bits = n.bit_length()
    if n < 2 or (1 << (bits - 1)) != n:
        raise ValueError(f"tq_write_kv_prod: mse_centroids must hold 2^(bits-1) values, got {n}")
    if tuple(qjl_matrix.shape) != (d, d):
        raise ValueError(f"tq_write_kv_prod: qjl_matrix must be [{d}, {d}]")
    _need_f32("tq_write_kv_prod", d, signs, mse_centroids)
    if pages.shape[2] != h or pages.shape[3] != tq_prod_row_bytes(d, bits):
        raise ValueError(f"tq_write_kv_prod: pages {tuple(pages.shape)} do not match H={h}, "
                         f"RBP={tq_prod_row_bytes(d, bits)}")
    _need_status("tq_write_kv_prod", status, dev)
    if status is None:
        status = _status_buffer(dev)
    with torch.cuda.device(dev):
        _check(lib().tq_write_kv_prod(_ptr(raw), _DTYPES[raw.dtype], t, h, d, bits, _ptr(slots), _ptr(pages),
                                      pages.shape[0], pages.shape[1], _ptr(signs), _ptr(mse_centroids),
                                      _ptr(qjl_matrix), _ptr(status), _stream(dev)))
    if check:
        raise_for_device_status(status)
    return status


def tq_paged_decode_prod(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                         seq_lens: torch.Tensor, signs: torch.Tensor, k_mse_centroids: torch.Tensor,
                         v_centroids: torch.Tensor, qjl_matrix: torch.Tensor, scale: float | None = None,
                         out: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
                         workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                         check: bool = False) -> torch.Tensor:
    """tq_paged_decode with product-quantised key pages (k_bits = log2(len(k_mse_centroids)) + 1)."""
    dev = _need_cuda("tq_paged_decode_prod", q, k_pages, v_pages, block_table, seq_lens, signs, k_mse_centroids,
                     v_centroids, qjl_matrix)
    if q.dim() != 3 or k_pages.dim() != 4 or v_pages.dim() != 4 or block_table.dim() != 2:
        raise ValueError("tq_paged_decode_prod: q [B, Hq, D], pages [NB, bs, H, RB], block_table [B, maxblk] expected")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32 or q.dtype not in _DTYPES:
        raise ValueError("tq_paged_decode_prod: block_table / seq_lens int32, q f32/f16/bf16 expected")
    b, hq, d = q.shape
    nb, bs, h, _ = k_pages.shape
    n = k_mse_centroids.numel()
    kb = n.bit_length()
    if n < 2 or (1 << (kb - 1)) != n:
        raise ValueError(f"tq_paged_decode_prod: k_mse_centroids must hold 2^(k_bits-1) values, got {n}")
    vb = _bits_from_centroids(v_centroids)
    _need_f32("tq_paged_decode_prod", d, signs, k_mse_centroids, v_centroids, qjl_matrix)
    if k_pages.shape[3] != tq_prod_row_bytes(d, kb) or v_pages.shape[3] != tq_row_bytes(d, vb) or \
            tuple(v_pages.shape[:3]) != (nb, bs, h) or block_table.shape[0] != b or seq_lens.numel() != b or \
            tuple(qjl_matrix.shape) != (d, d):
        raise ValueError("tq_paged_decode_prod: page / table / matrix shapes inconsistent with q and the codebooks")
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((b, hq, d), dtype=out_dtype, device=dev)
    _need_out("tq_paged_decode_prod", out, (b, hq, d), dev)
    _need_status("tq_paged_decode_prod", status, dev)
    maxb = block_table.shape[1]
    need = int(lib().tq_paged_decode_prod_workspace(b, hq, h, d, maxb, bs))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().tq_paged_decode_prod(_ptr(q), _DTYPES[q.dtype], b, hq, h, d, _ptr(k_pages), kb, _ptr(v_pages),
                                          vb, nb, bs, _ptr(block_table), maxb, _ptr(seq_lens), _ptr(signs),
                                          _ptr(k_mse_centroids), _ptr(v_centroids), _ptr(qjl_matrix),
                                          float(scale or 0.0), _ptr(out), _DTYPES[out.dtype], _ptr(workspace),
                                          workspace.numel(), _ptr(status), _stream(dev)))
    if check and status is not None:
        raise_for_device_status(status)
    return out


# ---------------------------------------------------------------- recipe modes

def _recipe_id(recipe) -> int:
    if isinstance(recipe, str):
        if recipe not in RECIPES:
            raise ValueError(f"unknown recipe {recipe!r}")
        return RECIPES[recipe]
    return int(recipe)


def tq_recipe_row_bytes(recipe, head_dim: int) -> int:
    rb = int(lib().tq_recipe_row_bytes(_recipe_id(recipe), int(head_dim)))
    if rb < 0:
        raise ValueError(f"recipe {recipe!r} at head_dim {head_dim} is not supported")
    return rb


def tq_recipe_channel_order(recipe, head_dim: int, high) -> torch.Tensor:
    """Checks the metadata's high groups [H, head_dim / 2] and returns the channel order
    int32 [H, head_dim] (high group, then the rest ascending) on the host."""
    high = torch.as_tensor(high).to(torch.int32).contiguous().cpu()
    if high.dim() != 2 or high.shape[1] * 2 != int(head_dim):
        raise ValueError(f"tq_recipe_channel_order: high groups must be [H, {int(head_dim) // 2}], got "
                         f"{tuple(high.shape)}")
    order = torch.empty(high.shape[0], int(head_dim), dtype=torch.int32)
    _check(lib().tq_recipe_channel_order(_recipe_id(recipe), int(head_dim), high.shape[0], high.data_ptr(),
                                         order.data_ptr()))
    return order


def tq_recipe_calibrate(recipe, samples) -> torch.Tensor:
    """High groups int32 [H, D / 2] from calibration rows samples[N, H, D] (host)."""
    x = torch.as_tensor(samples).to(torch.float32).contiguous().cpu()
    if x.dim() != 3:
        raise ValueError("tq_recipe_calibrate: samples must be [N, H, D]")
    n, h, d = x.shape
    high = torch.empty(h, d // 2, dtype=torch.int32)
    _check(lib().tq_recipe_calibrate(_recipe_id(recipe), d, h, x.data_ptr(), n, high.data_ptr()))
    return high


class RecipeCodec:
    """The shared group codec of a recipe at one head_dim, on a device: the signs of R_d
    (seed 42), the MSE codebooks of both groups and S_d (seed 43), d = head_dim / 2."""

    def __init__(self, recipe, head_dim: int, device=None):
        rid = _recipe_id(recipe)
        bits = {TQ_RECIPE_TURBOQUANT25: (3, 2), TQ_RECIPE_TURBOQUANT35: (4, 3)}.get(rid)
        if bits is None:
            raise ValueError(f"unknown recipe {recipe!r}")
        self.recipe, self.head_dim, self.d, self.bits = rid, int(head_dim), int(head_dim) // 2, bits
        self.row_bytes = tq_recipe_row_bytes(rid, head_dim)
        self.signs = tq_build_rotation(self.d, RECIPE_ROTATION_SEED, device)
        self.mse_high = tq_codebook(self.d, bits[0] - 1, device)[0]
        self.mse_low = tq_codebook(self.d, bits[1] - 1, device)[0]
        self.smat = tq_build_qjl_matrix(self.d, RECIPE_SKETCH_SEED, device)


def _need_order(name: str, order: torch.Tensor, h: int, d: int, device) -> None:
    if order.dtype != torch.int32 or tuple(order.shape) != (h, d) or not order.is_contiguous() or \
            order.device != device:
        raise ValueError(f"{name}: channel order must be contiguous int32 [{h}, {d}] on {device}")


def tq_write_kv_recipe(raw: torch.Tensor, pages: torch.Tensor, slots: torch.Tensor, order: torch.Tensor,
                       codec: RecipeCodec, status: torch.Tensor | None = None, check: bool = True) -> torch.Tensor:
    """Encode raw[T, H, D] into recipe pages[NB, bs, H, RB] (tq_write_kv's slot rules)."""
    dev = _need_cuda("tq_write_kv_recipe", raw, pages, slots, order, codec.signs, codec.smat)
    if raw.dim() != 3 or pages.dim() != 4 or slots.dim() != 1 or slots.numel() != raw.shape[0]:
        raise ValueError("tq_write_kv_recipe: raw [T, H, D], pages [NB, bs, H, RB], slots [T] expected")
    if raw.dtype not in _DTYPES or pages.dtype != torch.uint8 or slots.dtype != torch.int64:
        raise ValueError("tq_write_kv_recipe: raw f32/f16/bf16, pages uint8, slots int64 expected")
    t, h, d = raw.shape
    if d != codec.head_dim or pages.shape[2] != h or pages.shape[3] != codec.row_bytes:
        raise ValueError("tq_write_kv_recipe: raw / pages do not match the codec's head_dim and row bytes")
    _need_order("tq_write_kv_recipe", order, h, d, dev)
    _need_status("tq_write_kv_recipe", status, dev)
    if status is None:
        status = _status_buffer(dev)
    with torch.cuda.device(dev):
        _check(lib().tq_write_kv_recipe(_ptr(raw), _DTYPES[raw.dtype], t, h, d, codec.recipe, _ptr(slots),
                                        _ptr(pages), pages.shape[0], pages.shape[1], _ptr(order), _ptr(codec.signs),
                                        _ptr(codec.mse_high), _ptr(codec.mse_low), _ptr(codec.smat), _ptr(status),
                                        _stream(dev)))
    if check:
        raise_for_device_status(status)
    return status


def tq_paged_decode_recipe(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                           seq_lens: torch.Tensor, order: torch.Tensor, codec: RecipeCodec,
                           scale: float | None = None, out: torch.Tensor | None = None,
                           out_dtype: torch.dtype | None = None, workspace: torch.Tensor | None = None,
                           status: torch.Tensor | None = None, check: bool = False) -> torch.Tensor:
    """tq_paged_decode over recipe K and V pages."""
    dev = _need_cuda("tq_paged_decode_recipe", q, k_pages, v_pages, block_table, seq_lens, order, codec.signs)
    if q.dim() != 3 or k_pages.dim() != 4 or v_pages.dim() != 4 or block_table.dim() != 2:
        raise ValueError("tq_paged_decode_recipe: q [B, Hq, D], pages [NB, bs, H, RB], block_table [B, maxblk] "
                         "expected")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32 or q.dtype not in _DTYPES:
        raise ValueError("tq_paged_decode_recipe: block_table / seq_lens int32, q f32/f16/bf16 expected")
    b, hq, d = q.shape
    nb, bs, h, rb = k_pages.shape
    if d != codec.head_dim or rb != codec.row_bytes or tuple(v_pages.shape) != tuple(k_pages.shape) or \
            block_table.shape[0] != b or seq_lens.numel() != b:
        raise ValueError("tq_paged_decode_recipe: page / table shapes inconsistent with q and the codec")
    _need_order("tq_paged_decode_recipe", order, h, d, dev)
    out_dtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((b, hq, d), dtype=out_dtype, device=dev)
    _need_out("tq_paged_decode_recipe", out, (b, hq, d), dev)
    _need_status("tq_paged_decode_recipe", status, dev)
    maxb = block_table.shape[1]
    need = int(lib().tq_paged_decode_recipe_workspace(b, hq, h, d, maxb, bs))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().tq_paged_decode_recipe(_ptr(q), _DTYPES[q.dtype], b, hq, h, d, _ptr(k_pages), _ptr(v_pages),
                                            codec.recipe, nb, bs, _ptr(block_table), maxb, _ptr(seq_lens),
                                            _ptr(order), _ptr(codec.signs), _ptr(codec.mse_high),
                                            _ptr(codec.mse_low), _ptr(codec.smat), float(scale or 0.0), _ptr(out),
                                            _DTYPES[out.dtype], _ptr(workspace), workspace.numel(), _ptr(status),
                                            _stream(dev)))
    if check and status is not None:
        raise_for_device_status(status)
    return out
