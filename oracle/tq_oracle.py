"""TurboQuant packed-KV oracle: a plain, slow, fp64 CPU restatement of the packed
row writer and of the paged decode attention that reads those rows.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` use it.  It shares no code with the CUDA library
(``quantized_kv_cache_06_gb300``) and imports nothing from it; the only thing
the two sides share is the seeded input generator, which holds none of the
method's arithmetic.

Sources (TurboQuant documentation pages):
  * "vLLM Usage", section "TQ Byte Layout": a row is ceil(head_dim*bits/8) index
    bytes followed by the fp32 norm in the last four bytes; K and V are stored
    independently.
  * "vLLM Usage", sections "Slot Mapping" and "TQ Packed Page Contract": flat
    slots, negative slots ignored, a slot outside the allocated pages raises;
    the contract call builds an RHT rotation with seed 42 and a codebook from
    (head_dim, bits).
  * "Architecture", section "Cache Storage Objects" (PackedPageCache): page
    tensor shape [num_blocks, block_size, num_kv_heads, row_bytes], uint8.
  * "vLLM Reference Audit", section "Feature Checklist": Lloyd-Max codebooks with
    "exact Beta" tests, RHT rotation, 1..5-bit packing.
  * "Architecture", section "Diagnostic vs Serving Paths": the paged decode reads
    packed pages and reconstructs rows; direct-QK consumes keys compressed; the
    diagnostic dense reconstruction (the "vLLM Reference Audit" file map's
    tq4_decompress readback) is ``dequant_slots``.

Readings where the pages are silent (each one is listed in the design notes):
  * signs of the RHT: the i-th output of splitmix64 (Steele, Lea & Flood 2014)
    seeded with ``seed``; sign = -1 when its top bit is set;
  * rotation R = H_D diag(s) / sqrt(D), H_D the Sylvester-ordered Hadamard matrix
    H[i, j] = (-1)^popcount(i & j) (sign flip first, then the normalised WHT);
  * codebook: Lloyd-Max quantizer of one coordinate of a uniformly random unit
    vector in R^D, density f_D(x) = C_D (1 - x^2)^((D-3)/2) on [-1, 1]
    (x = 2T - 1 with T ~ Beta((D-1)/2, (D-1)/2)); centroids stored in fp32;
  * encode: nu = ||x||_2, u = x / nu (u = 0 when nu = 0), y = R u, index = the
    nearest fp32 centroid, ties to the lower index; stored norm = fp32(nu);
  * bit order: index j occupies stream bits [j*b, (j+1)*b), stream bit k is bit
    (k mod 8) of byte k // 8 (LSB first); the norm is little-endian fp32;
  * decode: scale defaults to 1/sqrt(D); GQA maps q head h to kv head h // G;
    tokens of a block id outside [0, num_blocks) are left out (and flagged);
    a sequence of length 0 gives a zero output.

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import betainc, betaincinv, gammaln

MASK64 = (1 << 64) - 1


class SlotOutOfRange(ValueError):
    """A write slot lies at or beyond num_blocks * block_size ("vLLM Usage", Slot Mapping)."""


# --------------------------------------------------------------------------
# Row geometry ("vLLM Usage", TQ Byte Layout)
# --------------------------------------------------------------------------

def index_bytes(head_dim: int, bits: int) -> int:
    """ceil(head_dim * bits / 8)."""
    return -(-head_dim * bits // 8)


def row_bytes(head_dim: int, bits: int) -> int:
    """Index bytes plus the 4 fp32 norm bytes."""
    return index_bytes(head_dim, bits) + 4


# --------------------------------------------------------------------------
# Rotation ("vLLM Usage", TQ Packed Page Contract: build_rotation(dim, RHT, seed))
# --------------------------------------------------------------------------

def splitmix64_signs(head_dim: int, seed: int) -> np.ndarray:
    """D signs in {-1, +1}: sign i is -1 when the top bit of the i-th splitmix64 output is set.

    splitmix64 as published (Steele, Lea & Flood, OOPSLA 2014; Vigna's reference
    code): state += 0x9E3779B97F4A7C15, then two xor-shift-multiply rounds and a
    final xor-shift of the state.
    """
    state = seed & MASK64
    out = np.empty(head_dim, dtype=np.float64)
    for i in range(head_dim):
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        z = z ^ (z >> 31)
        out[i] = -1.0 if (z >> 63) else 1.0
    return out


def hadamard(head_dim: int) -> np.ndarray:
    """Sylvester-ordered Hadamard matrix from its definition H[i, j] = (-1)^popcount(i & j)."""
    h = np.empty((head_dim, head_dim), dtype=np.float64)
    for i in range(head_dim):
        for j in range(head_dim):
            h[i, j] = -1.0 if bin(i & j).count("1") % 2 else 1.0
    return h


def rotation_matrix(signs: np.ndarray) -> np.ndarray:
    """Dense fp64 R = H_D diag(s) / sqrt(D): sign flip, then normalised Walsh-Hadamard."""
    d = signs.shape[0]
    return hadamard(d) * signs[None, :] / math.sqrt(d)


# --------------------------------------------------------------------------
# Codebook ("vLLM Reference Audit", Feature Checklist: Lloyd-Max, exact Beta tests)
# --------------------------------------------------------------------------

def coord_density_const(head_dim: int) -> float:
    """C_D = Gamma(D/2) / (sqrt(pi) Gamma((D-1)/2)), the normaliser of (1 - x^2)^((D-3)/2)."""
    d = head_dim
    return math.exp(gammaln(d / 2.0) - 0.5 * math.log(math.pi) - gammaln((d - 1) / 2.0))


def coord_density(x, head_dim: int):
    """Density of one coordinate of a uniform random unit vector in R^D."""
    x = np.asarray(x, dtype=np.float64)
    return coord_density_const(head_dim) * np.power(np.clip(1.0 - x * x, 0.0, None), (head_dim - 3) / 2.0)


def coord_cdf(x, head_dim: int):
    """P(X <= x) with X = 2T - 1, T ~ Beta(a, a), a = (D-1)/2 (regularised incomplete beta)."""
    a = (head_dim - 1) / 2.0
    t = (np.clip(np.asarray(x, dtype=np.float64), -1.0, 1.0) + 1.0) / 2.0
    return betainc(a, a, t)


def coord_partial_moment(lo, hi, head_dim: int):
    """Integral of x f_D(x) over [lo, hi], in closed form:
    d/dx [-(1 - x^2)^(p+1) / (2 (p+1))] = x (1 - x^2)^p with p = (D-3)/2."""
    p = (head_dim - 3) / 2.0
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    g = lambda x: np.power(np.clip(1.0 - x * x, 0.0, None), p + 1.0)
    return coord_density_const(head_dim) * (g(lo) - g(hi)) / (2.0 * (p + 1.0))


def lloyd_max(head_dim: int, bits: int, tol: float = 1e-14, max_iter: int = 500000):
    """Lloyd-Max quantizer for f_D with 2^bits levels, in fp64.

    Start from the centroids at the (k + 1/2)/n quantiles; then alternate
    boundaries = midpoints of neighbouring centroids and centroids = conditional
    means of their cells, until no centroid moves by more than ``tol``; finally
    make the result exactly odd-symmetric.  Returns (centroids, boundaries), both
    ascending fp64.
    """
    n = 1 << bits
    a = (head_dim - 1) / 2.0
    c = 2.0 * betaincinv(a, a, (np.arange(n) + 0.5) / n) - 1.0
    for _ in range(max_iter):
        b = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate([[-1.0], b, [1.0]])
        mass = np.diff(coord_cdf(edges, head_dim))
        mom = coord_partial_moment(edges[:-1], edges[1:], head_dim)
        c_new = mom / mass
        moved = np.max(np.abs(c_new - c))
        c = c_new
        if moved < tol:
            break
    else:
        raise RuntimeError("Lloyd-Max iteration did not converge")
    # f_D is even, so the optimum is odd-symmetric; remove the rounding noise of the
    # iteration so that c[k] == -c[n-1-k] exactly and the middle boundary is exactly 0.
    c = 0.5 * (c - c[::-1])
    return c, 0.5 * (c[:-1] + c[1:])


def codebook_f32(head_dim: int, bits: int):
    """(centroids fp32, boundaries fp32): fp64 solution rounded once; boundaries are the
    fp64 midpoints of the fp64 centroids, rounded to fp32."""
    c, b = lloyd_max(head_dim, bits)
    return c.astype(np.float32), b.astype(np.float32)


# --------------------------------------------------------------------------
# Encode + pack ("vLLM Usage", TQ Byte Layout)
# --------------------------------------------------------------------------

def encode_rows(x: np.ndarray, rot: np.ndarray, centroids32: np.ndarray, chunk: int = 8192):
    """Encode rows x[N, D].

    Returns (idx[N, D] int64, norms[N] fp32, margin[N, D] fp64) where margin is the
    distance of the normalised rotated coordinate y/nu to the nearest decision
    point between two fp32 centroids (for counting near-boundary coordinates).
    The index is the brute-force nearest centroid; ties go to the lower index.
    """
    x = np.asarray(x, dtype=np.float64)
    n, d = x.shape
    c = centroids32.astype(np.float64)
    mids = 0.5 * (c[:-1] + c[1:])
    idx = np.empty((n, d), dtype=np.int64)
    margin = np.empty((n, d), dtype=np.float64)
    nu = np.sqrt(np.sum(x * x, axis=1))
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        xs, ns = x[s:e], nu[s:e]
        u = np.zeros_like(xs)
        nz = ns > 0
        u[nz] = xs[nz] / ns[nz, None]
        y = u @ rot.T
        dist = np.abs(y[:, :, None] - c[None, None, :])
        idx[s:e] = np.argmin(dist, axis=2)
        margin[s:e] = np.min(np.abs(y[:, :, None] - mids[None, None, :]), axis=2)
    return idx, nu.astype(np.float32), margin


def pack_indices(idx: np.ndarray, bits: int) -> np.ndarray:
    """LSB-first bit packing of b-bit indices: idx[N, D] -> uint8[N, ceil(D*b/8)]."""
    idx = np.asarray(idx, dtype=np.int64)
    n, d = idx.shape
    planes = (idx[:, :, None] >> np.arange(bits)[None, None, :]) & 1
    stream = planes.reshape(n, d * bits).astype(np.uint8)
    pad = index_bytes(d, bits) * 8 - d * bits
    if pad:
        stream = np.concatenate([stream, np.zeros((n, pad), dtype=np.uint8)], axis=1)
    return np.packbits(stream, axis=1, bitorder="little")


def unpack_indices(packed: np.ndarray, head_dim: int, bits: int) -> np.ndarray:
    """Inverse of pack_indices: uint8[N, >= ceil(D*b/8)] -> int64[N, D]."""
    packed = np.asarray(packed, dtype=np.uint8)
    n = packed.shape[0]
    stream = np.unpackbits(packed[:, : index_bytes(head_dim, bits)], axis=1, bitorder="little")
    planes = stream[:, : head_dim * bits].reshape(n, head_dim, bits).astype(np.int64)
    return np.sum(planes << np.arange(bits)[None, None, :], axis=2)


def make_rows(idx: np.ndarray, norms: np.ndarray, bits: int) -> np.ndarray:
    """Packed index bytes followed by the little-endian fp32 norm."""
    nb = pack_indices(idx, bits)
    normb = np.asarray(norms, dtype="<f4").reshape(-1, 1).view(np.uint8)
    return np.concatenate([nb, normb], axis=1)


def encode_to_rows(x, rot, centroids32, bits):
    """x[N, D] -> (rows uint8[N, row_bytes], margin[N, D])."""
    idx, norms, margin = encode_rows(x, rot, centroids32)
    return make_rows(idx, norms, bits), margin


# --------------------------------------------------------------------------
# Slot scatter ("vLLM Usage", Slot Mapping; "Architecture", PackedPageCache)
# --------------------------------------------------------------------------

def write_kv(raw: np.ndarray, pages: np.ndarray, slots: np.ndarray, signs: np.ndarray,
             centroids32: np.ndarray, bits: int) -> np.ndarray:
    """Return a copy of ``pages`` with the rows of raw[T, H, D] written at their flat slots.

    Row (t, h) lands at pages[slot_t // bs, slot_t % bs, h, :].  Negative slots are
    skipped.  If any slot is >= num_blocks * block_size, SlotOutOfRange is raised and
    nothing is written.  Duplicate non-negative slots: the last token wins here (the
    contract leaves it open).
    """
    t, h, d = raw.shape
    nblk, bs, hp, rb = pages.shape
    assert hp == h and rb == row_bytes(d, bits)
    slots = np.asarray(slots, dtype=np.int64)
    if np.any(slots >= nblk * bs):
        raise SlotOutOfRange("slot outside allocated pages")
    out = pages.copy()
    keep = np.nonzero(slots >= 0)[0]
    if keep.size == 0:
        return out
    rot = rotation_matrix(signs)
    rows, _ = encode_to_rows(raw[keep].reshape(-1, d), rot, centroids32, bits)
    rows = rows.reshape(keep.size, h, rb)
    for i, tok in enumerate(keep):
        s = slots[tok]
        out[s // bs, s % bs] = rows[i]
    return out


# --------------------------------------------------------------------------
# Decode ("Architecture", Diagnostic vs Serving Paths)
# --------------------------------------------------------------------------

def dequant_rows(rows: np.ndarray, head_dim: int, bits: int, rot: np.ndarray,
                 centroids32: np.ndarray) -> np.ndarray:
    """Fully reconstructed rows: nu * R^T c[idx] (fp64)."""
    rows = np.asarray(rows, dtype=np.uint8)
    nb = index_bytes(head_dim, bits)
    idx = unpack_indices(rows[:, :nb], head_dim, bits)
    norms = np.ascontiguousarray(rows[:, nb:nb + 4]).view("<f4").reshape(-1).astype(np.float64)
    rotated = centroids32.astype(np.float64)[idx]
    return norms[:, None] * (rotated @ rot)


def dequant_slots(pages: np.ndarray, slots: np.ndarray, signs: np.ndarray, centroids32: np.ndarray,
                  bits: int) -> np.ndarray:
    """Dense readback of the rows a write put at ``slots`` ("vLLM Reference Audit", file map:
    tq4_decompress, diagnostic readback; "Architecture", Diagnostic vs Serving Paths: dense
    reconstruction from packed bytes).  pages uint8[NB, bs, H, RB]; returns fp64[T, H, D]
    with nu * R^T c[idx] for every slot >= 0 and a zero row for a negative slot.  A slot
    at or beyond NB * bs raises SlotOutOfRange, as for the write."""
    pages = np.asarray(pages, dtype=np.uint8)
    nblk, bs, nh, _ = pages.shape
    d = len(signs)
    slots = np.asarray(slots, dtype=np.int64)
    if np.any(slots >= nblk * bs):
        raise SlotOutOfRange("slot outside the allocated pages")
    rot = rotation_matrix(signs)
    out = np.zeros((len(slots), nh, d), dtype=np.float64)
    keep = np.nonzero(slots >= 0)[0]
    for h in range(nh):
        rows = pages[slots[keep] // bs, slots[keep] % bs, h]
        if len(keep):
            out[keep, h] = dequant_rows(rows, d, bits, rot, centroids32)
    return out


def _gather_rows(pages, block_table_row, seq_len, head):
    bs = pages.shape[1]
    nblk = pages.shape[0]
    t = np.arange(seq_len)
    blk = np.asarray(block_table_row, dtype=np.int64)[t // bs]
    ok = (blk >= 0) & (blk < nblk)
    rows = pages[np.where(ok, blk, 0), t % bs, head]
    return rows, ok


def paged_decode(q, k_pages, v_pages, k_bits, v_bits, block_table, seq_lens, signs,
                 k_centroids32, v_centroids32, scale=None, heads=None, return_flags=False):
    """fp64 softmax attention over fully dequantised rows.

    q[B, Hq, D]; pages [NB, bs, H, RB]; token t of sequence b sits at block
    block_table[b, t // bs], offset t % bs; q head h reads kv head h // (Hq / H).
    ``heads`` optionally restricts the work to a list of (b, q_head) pairs (the
    other outputs stay zero).  Returns out[B, Hq, D] (and a flag telling whether a
    block id outside [0, NB) was met, whose tokens are left out).
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    h = k_pages.shape[2]
    grp = hq // h
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    rot = rotation_matrix(signs)
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    bad_block = False
    wanted = heads if heads is not None else [(b, j) for b in range(bsz) for j in range(hq)]
    by_kv = {}
    for b, j in wanted:
        by_kv.setdefault((b, j // grp), []).append(j)
    for (b, kvh), qheads in sorted(by_kv.items()):
        n = int(seq_lens[b])
        if n <= 0:
            continue
        krows, ok = _gather_rows(k_pages, block_table[b], n, kvh)
        vrows, _ = _gather_rows(v_pages, block_table[b], n, kvh)
        if not np.all(ok):
            bad_block = True
        krows, vrows = krows[ok], vrows[ok]
        if krows.shape[0] == 0:
            continue
        khat = dequant_rows(krows, d, k_bits, rot, k_centroids32)
        vhat = dequant_rows(vrows, d, v_bits, rot, v_centroids32)
        for j in qheads:
            s = scale * (khat @ q[b, j])
            p = np.exp(s - np.max(s))
            p /= np.sum(p)
            out[b, j] = p @ vhat
    return (out, bad_block) if return_flags else out


def paged_prefill(q, q_seq, q_len, k_pages, v_pages, k_bits, v_bits, block_table, signs,
                  k_centroids32, v_centroids32, scale=None, return_flags=False):
    """Mixed prefill/decode attention over the packed cache ("vLLM Usage", Runtime
    Dispatch: cache plus mixed prefill/decode reads the packed cache).

    q[T, Hq, D]: query row i belongs to sequence q_seq[i] and sees the first q_len[i]
    tokens of it (causal: its position + 1); the cache already holds the new tokens.
    Row i is the decode of one query over block_table[q_seq[i]] with length q_len[i], so
    a decode batch is the case of one row per sequence.  Returns out[T, Hq, D] (and the
    bad-block flag of paged_decode).
    """
    q_seq = np.asarray(q_seq, dtype=np.int64)
    q_len = np.asarray(q_len, dtype=np.int64)
    rows_table = np.asarray(block_table)[q_seq]
    return paged_decode(q, k_pages, v_pages, k_bits, v_bits, rows_table, q_len, signs, k_centroids32,
                        v_centroids32, scale=scale, return_flags=return_flags)


def paged_decode_rotated(q, k_pages, v_pages, k_bits, v_bits, block_table, seq_lens, signs,
                         k_centroids32, v_centroids32, scale=None):
    """Same attention in rotated space ("Architecture": direct-QK and packed-V):
    score = scale * nu_k <R q, c_k[idx]>, acc = sum p nu_v c_v[idx_v], o = R^T acc.
    Used only to cross-check paged_decode."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    h = k_pages.shape[2]
    grp = hq // h
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    rot = rotation_matrix(signs)
    ck = k_centroids32.astype(np.float64)
    cv = v_centroids32.astype(np.float64)
    nbk, nbv = index_bytes(d, k_bits), index_bytes(d, v_bits)
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    for b in range(bsz):
        n = int(seq_lens[b])
        if n <= 0:
            continue
        for j in range(hq):
            kvh = j // grp
            krows, ok = _gather_rows(k_pages, block_table[b], n, kvh)
            vrows, _ = _gather_rows(v_pages, block_table[b], n, kvh)
            krows, vrows = krows[ok], vrows[ok]
            kidx = unpack_indices(krows[:, :nbk], d, k_bits)
            vidx = unpack_indices(vrows[:, :nbv], d, v_bits)
            knorm = np.ascontiguousarray(krows[:, nbk:nbk + 4]).view("<f4").reshape(-1).astype(np.float64)
            vnorm = np.ascontiguousarray(vrows[:, nbv:nbv + 4]).view("<f4").reshape(-1).astype(np.float64)
            qrot = rot @ q[b, j]
            s = scale * knorm * (ck[kidx] @ qrot)
            p = np.exp(s - np.max(s))
            p /= np.sum(p)
            acc = (p * vnorm) @ cv[vidx]
            out[b, j] = rot.T @ acc
    return out
