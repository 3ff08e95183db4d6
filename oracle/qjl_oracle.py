"""TurboQuant product-quantised ("QJL residual") key rows: a plain fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY, like ``tq_oracle``: nothing on the product path may import,
call or run this module.  It builds on ``tq_oracle`` (rotation, codebooks, bit packing)
and shares nothing with the CUDA library.

Sources (TurboQuant documentation pages):
  * "vLLM Reference Audit", File Map: the quantizer module holds "MSE and QJL codecs"
    whose data are "indices, norms, signs", with public classes TurboQuantMSE and
    TurboQuantProd.
  * "vLLM Reference Audit", Feature Checklist: "QJL residual" is partial, next action
    "add recipe decode contract".
  * "Architecture", vLLM Runtime Mapping: recipe vector rows pack and unpack "grouped
    MSE+QJL rows" (the grouped recipe layouts are a separate item and not modelled here).

The pages name the codec but give neither its arithmetic nor a row layout.  Readings
(each listed in the design notes), following the product quantiser that TurboQuantProd
names -- an MSE quantiser at b - 1 bits whose residual gets a one-bit quantised
Johnson-Lindenstrauss sketch, so that inner products with a query are unbiased:
  * encode (per row x, fp64): nu = ||x||, u = x / nu, y = R u (the same rotation as the
    MSE rows), idx = nearest centroid of the (b - 1)-bit codebook (ties to the lower
    index), residual r = y - c[idx] (rotated space), gamma = ||r||, sign bits
    z_i = [ (S r)_i >= 0 ] with S a D x D matrix of independent N(0, 1) entries;
  * inner product with a query q (qt = R q): <q, x> ~ nu (<qt, c[idx]> +
    gamma sqrt(pi / 2) / D <S qt, 2 z - 1>), unbiased over the draw of S because
    E[(s . v) sign(s . r)] = sqrt(2 / pi) <v, r> / ||r|| for s ~ N(0, I);
    the reconstruction it corresponds to is nu R^T (c[idx] + gamma sqrt(pi/2)/D S^T (2z-1));
  * S: entry (i, j) is normal number i D + j of a stream seeded with ``seed``: the
    splitmix64 outputs (Steele, Lea & Flood 2014) taken in pairs (z1, z2) give
    u1 = ((z1 >> 11) + 1) 2^-53 in (0, 1] and u2 = (z2 >> 11) 2^-53 in [0, 1), and the
    Box-Muller transform (Box & Muller 1958) gives sqrt(-2 ln u1) cos(2 pi u2) and
    sqrt(-2 ln u1) sin(2 pi u2), in that order;
  * row layout: the (b - 1)-bit MSE indices LSB-first (ceil(D (b-1) / 8) bytes), then the
    D sign bits LSB-first (ceil(D / 8) bytes, bit = 1 for a non-negative projection),
    then nu and gamma as little-endian fp32: RB = ceil(D (b-1) / 8) + ceil(D / 8) + 8;
  * keys only: values keep the plain MSE rows of ``tq_oracle`` (the checklist item is
    about scores).

Parity pins live in ``tests/test_qjl_oracle_pins.py``.
"""

from __future__ import annotations

import math

import numpy as np

from oracle import tq_oracle as o

MASK64 = (1 << 64) - 1
SQRT_HALF_PI = math.sqrt(math.pi / 2.0)


def splitmix64_stream(seed: int, n: int) -> list[int]:
    """The first n outputs of splitmix64 seeded with ``seed`` (as published)."""
    state = seed & MASK64
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        out.append(z ^ (z >> 31))
    return out


def normal_matrix(rows: int, cols: int, seed: int) -> np.ndarray:
    """rows x cols independent N(0, 1) numbers, row-major, from the splitmix64 stream of
    ``seed`` through the Box-Muller transform (see the module notes)."""
    n = rows * cols
    z = splitmix64_stream(seed, 2 * ((n + 1) // 2))
    vals = np.empty(2 * ((n + 1) // 2), dtype=np.float64)
    for k in range(0, len(z), 2):
        u1 = ((z[k] >> 11) + 1) * 2.0 ** -53
        u2 = (z[k + 1] >> 11) * 2.0 ** -53
        rad = math.sqrt(-2.0 * math.log(u1))
        vals[k] = rad * math.cos(2.0 * math.pi * u2)
        vals[k + 1] = rad * math.sin(2.0 * math.pi * u2)
    return vals[:n].reshape(rows, cols)


def prod_row_bytes(head_dim: int, bits: int) -> int:
    """Bytes of one product-quantised key row at ``bits`` bits per coordinate in total."""
    if not 2 <= bits <= 5:
        raise ValueError("bits must be 2..5 (an MSE part of 1..4 bits plus one sign bit)")
    return o.index_bytes(head_dim, bits - 1) + (head_dim + 7) // 8 + 8


def encode_prod(x: np.ndarray, rot: np.ndarray, mse_centroids32: np.ndarray, smat: np.ndarray) -> dict:
    """Encode rows x[N, D]: MSE indices, sign bits, norms and residual norms (fp64 arithmetic).

    Returns a dict with idx[N, D], z[N, D] (0/1), nu[N] and gamma[N] (as stored, fp32),
    and the residual r[N, D] in rotated space (fp64, for the pins)."""
    x = np.asarray(x, dtype=np.float64)
    idx, nu32, _ = o.encode_rows(x, rot, mse_centroids32)
    nu = np.sqrt(np.sum(x * x, axis=1))
    u = np.zeros_like(x)
    nz = nu > 0
    u[nz] = x[nz] / nu[nz, None]
    y = u @ rot.T
    r = y - mse_centroids32.astype(np.float64)[idx]
    gamma = np.sqrt(np.sum(r * r, axis=1))
    z = ((r @ smat.T) >= 0.0).astype(np.int64)
    return dict(idx=idx, z=z, nu=nu32, gamma=gamma.astype(np.float32), residual=r)


def pack_prod_rows(idx: np.ndarray, z: np.ndarray, nu: np.ndarray, gamma: np.ndarray, bits: int) -> np.ndarray:
    """Row bytes: MSE indices ((bits - 1)-bit, LSB-first), sign bits, fp32 nu, fp32 gamma."""
    idx = np.asarray(idx, dtype=np.int64)
    n, d = idx.shape
    mse = o.pack_indices(idx, bits - 1)
    sgn = np.packbits(np.asarray(z, dtype=np.uint8).reshape(n, d), axis=1, bitorder="little")
    norms = np.stack([np.asarray(nu, dtype="<f4"), np.asarray(gamma, dtype="<f4")], axis=1).view(np.uint8)
    return np.concatenate([mse, sgn, norms.reshape(n, 8)], axis=1)


def unpack_prod_rows(rows: np.ndarray, head_dim: int, bits: int):
    """Inverse of pack_prod_rows: (idx[N, D], z[N, D], nu[N] fp32, gamma[N] fp32)."""
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    ib = o.index_bytes(head_dim, bits - 1)
    sb = (head_dim + 7) // 8
    idx = o.unpack_indices(rows[:, :ib], head_dim, bits - 1)
    z = np.unpackbits(rows[:, ib:ib + sb], axis=1, bitorder="little")[:, :head_dim].astype(np.int64)
    tail = np.ascontiguousarray(rows[:, ib + sb:ib + sb + 8]).view("<f4").reshape(n, 2)
    return idx, z, tail[:, 0].copy(), tail[:, 1].copy()


def prod_scores(q: np.ndarray, rows: np.ndarray, head_dim: int, bits: int, rot: np.ndarray,
                mse_centroids32: np.ndarray, smat: np.ndarray) -> np.ndarray:
    """Estimates of <q_a, x_t> for queries q[A, D] and packed rows[T, RB]: out[A, T]."""
    idx, z, nu, gamma = unpack_prod_rows(rows, head_dim, bits)
    c = mse_centroids32.astype(np.float64)
    qt = np.asarray(q, dtype=np.float64) @ rot.T                         # R q
    mse = qt @ c[idx].T                                                   # <R q, c[idx]>
    qjl = (qt @ smat.T) @ (2.0 * z - 1.0).T                               # <S R q, 2z - 1>
    nu64, g64 = nu.astype(np.float64), gamma.astype(np.float64)
    return (mse + qjl * (g64 * SQRT_HALF_PI / head_dim)[None, :]) * nu64[None, :]


def prod_dequant(rows: np.ndarray, head_dim: int, bits: int, rot: np.ndarray, mse_centroids32: np.ndarray,
                 smat: np.ndarray) -> np.ndarray:
    """The reconstruction nu R^T (c[idx] + gamma sqrt(pi/2)/D S^T (2z - 1)) of rows[T, RB]."""
    idx, z, nu, gamma = unpack_prod_rows(rows, head_dim, bits)
    c = mse_centroids32.astype(np.float64)
    rot_space = c[idx] + (gamma.astype(np.float64) * SQRT_HALF_PI / head_dim)[:, None] * ((2.0 * z - 1.0) @ smat)
    return (rot_space @ rot) * nu.astype(np.float64)[:, None]


def paged_decode_prod_keys(q, kprod_pages, v_pages, k_bits, v_bits, block_table, seq_lens, signs,
                           k_mse_centroids32, v_centroids32, smat, scale=None):
    """fp64 attention whose scores come from product-quantised key rows and whose values
    are plain MSE rows: out[b, h] = sum_t softmax_t(scale * est<q_bh, k_t>) vhat_t, with
    the same paging, GQA mapping and length rules as ``tq_oracle.paged_decode``."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    h = kprod_pages.shape[2]
    grp = hq // h
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    rot = o.rotation_matrix(signs)
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    for b in range(bsz):
        n = int(seq_lens[b])
        if n <= 0:
            continue
        for kvh in range(h):
            krows, ok = o._gather_rows(kprod_pages, block_table[b], n, kvh)
            vrows, _ = o._gather_rows(v_pages, block_table[b], n, kvh)
            krows, vrows = krows[ok], vrows[ok]
            if krows.shape[0] == 0:
                continue
            vhat = o.dequant_rows(vrows, d, v_bits, rot, v_centroids32)
            s = scale * prod_scores(q[b, kvh * grp:(kvh + 1) * grp], krows, d, k_bits, rot, k_mse_centroids32, smat)
            p = np.exp(s - np.max(s, axis=1, keepdims=True))
            p /= np.sum(p, axis=1, keepdims=True)
            out[b, kvh * grp:(kvh + 1) * grp] = p @ vhat
    return out
