"""Comparison helpers for the GPU-vs-oracle parity tests (test code, not the oracle).

Tolerances:
  * packed index bytes: bit-exact, except coordinates whose normalised rotated value
    lies within 1e-6 of a decision point (measured in the oracle's fp64); those are
    counted and must be fewer than 1e-5 of all compared coordinates.  That is a rate: a
    sample of n < 1e6 coordinates (expected count below 10 at the rate) cannot resolve
    it, so there the count is held to what a process at exactly that rate exceeds with
    probability below 1e-3 (Poisson upper quantile); samples of >= 1e6 coordinates are
    held to 1e-5 n, and the rate itself is measured at scale by
    test_index_flip_rate_at_scale (3.4e7 coordinates per shape);
  * norms: within 1e-6 relative;
  * decode outputs: |gpu - oracle| <= 2e-3 + 2e-3 |oracle| elementwise.
"""

from __future__ import annotations

import math

import numpy as np

from oracle import tq_oracle as o

BAND = 1e-6
MAX_FLIP_FRACTION = 1e-5
NORM_RTOL = 1e-6
DEC_ATOL = 2e-3
DEC_RTOL = 2e-3


class OracleCodec:
    """The oracle's own signs, rotation and codebooks for one head_dim."""

    def __init__(self, head_dim: int, seed: int = 42):
        self.d = head_dim
        self.signs = o.splitmix64_signs(head_dim, seed)
        self.rot = o.rotation_matrix(self.signs)
        self._cb = {}

    def centroids(self, bits: int) -> np.ndarray:
        if bits not in self._cb:
            self._cb[bits] = o.codebook_f32(self.d, bits)[0]
        return self._cb[bits]


def compare_rows(gpu_rows: np.ndarray, raw_rows: np.ndarray, codec: OracleCodec, bits: int) -> dict:
    """gpu_rows uint8[N, RB] written by the GPU for raw rows raw_rows[N, D]."""
    d = codec.d
    idx, norms, margin = o.encode_rows(np.asarray(raw_rows, dtype=np.float64), codec.rot, codec.centroids(bits))
    nb = o.index_bytes(d, bits)
    gidx = o.unpack_indices(gpu_rows[:, :nb], d, bits)
    gnorm = np.ascontiguousarray(gpu_rows[:, nb:nb + 4]).view("<f4").reshape(-1)
    diff = gidx != idx
    flips = int(diff.sum())
    outside_band = int((diff & (margin >= BAND)).sum())
    near = int((margin < BAND).sum())
    rel = np.abs(gnorm.astype(np.float64) - norms) / np.maximum(norms.astype(np.float64), 1e-30)
    rel[norms == 0] = np.abs(gnorm[norms == 0])
    return dict(coords=idx.size, flips=flips, flips_outside_band=outside_band, near_boundary=near,
                max_norm_rel=float(rel.max()) if rel.size else 0.0,
                max_index_step=int(np.abs(gidx - idx).max()) if idx.size else 0)


def allowed_flips(coords: int) -> float:
    """In-band exceptions a sample of `coords` coordinates may hold (see the tolerances)."""
    lam = MAX_FLIP_FRACTION * coords
    if coords >= 1_000_000:
        return lam
    k, term, cdf = 0, math.exp(-lam), math.exp(-lam)
    while 1.0 - cdf >= 1e-3:  # smallest k with P(Poisson(lam) > k) < 1e-3
        k += 1
        term *= lam / k
        cdf += term
    return float(k)


def assert_rows_match(stats: dict) -> None:
    assert stats["flips_outside_band"] == 0, stats
    assert stats["flips"] <= allowed_flips(stats["coords"]), stats
    assert stats["max_index_step"] <= 1, stats
    assert stats["max_norm_rel"] <= NORM_RTOL, stats


def assert_decode_close(gpu: np.ndarray, ref: np.ndarray) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = DEC_ATOL + DEC_RTOL * np.abs(ref)
    worst = float(np.max(err / bound)) if err.size else 0.0
    assert np.all(np.isfinite(gpu))
    assert np.all(err <= bound), f"worst err/bound = {worst:.3f}, max abs err {err.max():.3e}"
    return worst
