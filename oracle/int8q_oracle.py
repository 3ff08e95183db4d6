"""INT8-query prefill over the packed cache: a plain CPU oracle.

TEST INFRASTRUCTURE ONLY, like ``tq_oracle``: nothing on the product path may import,
call or run this module.  It builds on ``tq_oracle.paged_prefill`` and shares nothing with
the CUDA library.

Sources (TurboQuant documentation pages):
  * "vLLM Usage", Runtime Dispatch: a cache plus the INT8 prefill gate takes the int8
    query path (mixed prefill/decode over the packed cache);
  * "vLLM Reference Audit", File Map: the INT8-Q prefill kernel, described as int8 query
    scale over packed pages (absent from the pages' own repository).

The pages give neither the quantiser nor where the scale lives.  Readings (each listed in
the design notes), the plainest that "int8 query scale" supports:
  * one symmetric scale per (query row, q head): s = amax / 127 with amax = max_j |q_j|;
  * code_j = round-half-to-even(q_j / s), inside [-127, 127]; a zero row has s = 0 and
    codes 0;
  * the quantiser's arithmetic is fp32 (the division amax / 127 and q_j / s each rounded
    once to fp32), so the integer decisions are taken in the precision the kernel takes
    them in;
  * the attention is the packed-cache prefill attention on the dequantised query
    s * code (fp64 from there on, as in ``tq_oracle``).

Pins live in ``tests/test_int8q_oracle_pins.py``.
"""

from __future__ import annotations

import numpy as np

from oracle import tq_oracle as o

QMAX = 127


def quantize_queries_int8(q: np.ndarray):
    """q[..., D] (any float dtype) -> (codes int8[..., D], scales float32[...])."""
    q32 = np.asarray(q, dtype=np.float32)
    amax = np.max(np.abs(q32), axis=-1)
    scale = (amax / np.float32(QMAX)).astype(np.float32)  # one fp32 division per row
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    ratio = (q32 / safe[..., None]).astype(np.float32)   # one fp32 division per element
    codes = np.clip(np.rint(ratio), -QMAX, QMAX)         # ties to even
    codes = np.where(scale[..., None] > 0, codes, 0.0)
    return codes.astype(np.int8), scale


def dequantize_queries(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """s * code in fp64."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def paged_prefill_int8q(codes, scales, q_seq, q_len, k_pages, v_pages, k_bits, v_bits, block_table, signs,
                        k_centroids32, v_centroids32, scale=None):
    """Mixed prefill/decode attention of int8 query rows codes[T, Hq, D] with scales[T, Hq]:
    ``tq_oracle.paged_prefill`` on the dequantised query."""
    return o.paged_prefill(dequantize_queries(codes, scales), q_seq, q_len, k_pages, v_pages, k_bits, v_bits,
                           block_table, signs, k_centroids32, v_centroids32, scale=scale)
