"""TurboQuant recipe cache modes turboquant25 / turboquant35: a plain fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY, like ``tq_oracle`` and ``qjl_oracle``: nothing on the product path
may import, call or run this module.  It builds on those two (rotation, codebooks, product
rows) and shares nothing with the CUDA library.

Sources (TurboQuant documentation pages):
  * "vLLM Usage", Cache Dtypes: the recipe names turboquant25 and turboquant35; recipe
    modes require metadata.
  * "vLLM Usage", Metadata Validation Rules: the loader checks the metadata version, a known
    recipe, an integer head size, the layer object shape, sorted unique high-group indices,
    their index range and the high-group count the recipe expects; runtime resolution also
    checks that recipe and head dimension match.
  * "vLLM Usage", Runtime Dispatch: both recipes decode on the recipe_paged path; Page
    Geometry: recipe mode takes recipe row-byte overrides instead of the TQ formula.
  * "Architecture", vLLM Runtime Mapping: the metadata holds group sizes per layer;
    activation calibration selects channels by energy; recipe vector rows pack and unpack
    grouped MSE+QJL rows.
  * "vLLM Reference Audit", File Map: the recipe layout and vector codec (group layout) and
    the recipe update / decode kernels (missing there); Feature Checklist: the
    turboquant25/35 recipe layout is partial, and the QJL residual still lacks its recipe
    decode contract.

The pages name the parts and give none of the numbers.  Readings (each listed in the design
notes), the plainest that the names and the rules above support:
  * the recipe name is the mean bits per channel, 2.5 or 3.5.  Each row splits its D
    channels into a high group and a low group of D/2 channels each, coded at ceil and floor
    of the mean: turboquant25 -> 3 and 2 bits, turboquant35 -> 4 and 3 bits.  So the
    expected high-group count is D/2 for both recipes;
  * the metadata gives, per kv head, the high group as D/2 sorted unique channel indices in
    [0, D).  The low group is the complement, in ascending order;
  * calibration: a channel's energy is the sum of its squares over the calibration rows of
    that kv head.  The high group is the D/2 channels of largest energy (ties to the lower
    channel index), sorted ascending;
  * each group is one product-quantised ("MSE+QJL") vector of dimension d = D/2: at b bits,
    (b-1)-bit MSE indices after the rotation R_d, one sign bit per coordinate of S_d r, then
    nu and gamma (``qjl_oracle``).  R_d is the RHT of dimension d with seed 42 and S_d the
    d x d normal matrix of seed 43.  Both groups, and K and V, share R_d and S_d;
  * row layout: the high-group row, then the low-group row.  At D = 128, turboquant25 rows
    are 32 + 24 = 56 bytes and turboquant35 rows 40 + 32 = 72 bytes;
  * K and V both use the recipe rows.  Scores are the sum over the two groups of the
    product estimates.  Values are the product reconstruction
    nu R_d^T (c[idx] + gamma sqrt(pi/2)/d S_d^T (2z - 1)) of each group, put back at the
    group's channels.

Parity pins live in ``tests/test_recipe_oracle_pins.py``.
"""

from __future__ import annotations

import functools
import math

import numpy as np

from oracle import qjl_oracle as qo
from oracle import tq_oracle as o

# recipe -> (mean bits, high-group bits, low-group bits)
RECIPES = {"turboquant25": (2.5, 3, 2), "turboquant35": (3.5, 4, 3)}
ROTATION_SEED = 42
SKETCH_SEED = 43


def recipe_bits(recipe: str) -> tuple[int, int]:
    """(high-group bits, low-group bits) of a recipe; raises on an unknown name."""
    if recipe not in RECIPES:
        raise ValueError(f"unknown recipe {recipe!r}")
    return RECIPES[recipe][1], RECIPES[recipe][2]


def high_group_count(recipe: str, head_dim: int) -> int:
    """The high-group size the metadata must hold: half the channels."""
    recipe_bits(recipe)
    if head_dim < 4 or head_dim % 2:
        raise ValueError(f"head_dim {head_dim} cannot be split in two groups")
    return head_dim // 2


def recipe_row_bytes(recipe: str, head_dim: int) -> int:
    """Bytes of one recipe row: the high-group product row, then the low-group one."""
    bh, bl = recipe_bits(recipe)
    d = high_group_count(recipe, head_dim)
    return qo.prod_row_bytes(d, bh) + qo.prod_row_bytes(d, bl)


def validate_high_groups(high: np.ndarray, recipe: str, head_dim: int, num_kv_heads: int) -> np.ndarray:
    """Checks the metadata's high-group indices [H, D/2] as the validation rules list them and
    returns them as int64.  Raises ValueError naming the first rule broken."""
    n_hi = high_group_count(recipe, head_dim)
    high = np.asarray(high)
    if high.ndim != 2 or high.shape[0] != num_kv_heads:
        raise ValueError(f"high groups must be [num_kv_heads={num_kv_heads}, n], got {high.shape}")
    if not np.issubdtype(high.dtype, np.integer):
        raise ValueError("high-group indices must be integers")
    if high.shape[1] != n_hi:
        raise ValueError(f"{recipe} at head_dim {head_dim} expects {n_hi} high channels, got {high.shape[1]}")
    if np.any(high < 0) or np.any(high >= head_dim):
        raise ValueError(f"high-group index outside [0, {head_dim})")
    if np.any(np.diff(high, axis=1) <= 0):
        raise ValueError("high-group indices must be sorted and unique")
    return high.astype(np.int64)


def low_groups(high: np.ndarray, head_dim: int) -> np.ndarray:
    """The complement of each kv head's high group, ascending: [H, D - n_hi]."""
    out = []
    for row in np.asarray(high):
        mask = np.ones(head_dim, dtype=bool)
        mask[row] = False
        out.append(np.nonzero(mask)[0])
    return np.asarray(out, dtype=np.int64)


def calibrate_high_groups(samples: np.ndarray, recipe: str) -> np.ndarray:
    """High groups from calibration rows samples[N, H, D]: per kv head, the D/2 channels of
    largest energy sum_t x[t, h, c]^2 (ties to the lower channel), sorted ascending."""
    x = np.asarray(samples, dtype=np.float64)
    _, h, d = x.shape
    n_hi = high_group_count(recipe, d)
    energy = np.sum(x * x, axis=0)  # [H, D]
    out = np.empty((h, n_hi), dtype=np.int64)
    for k in range(h):
        order = sorted(range(d), key=lambda c: (-energy[k, c], c))
        out[k] = np.sort(order[:n_hi])
    return out


@functools.lru_cache(maxsize=None)
def _group_rotation(d: int):
    signs = o.splitmix64_signs(d, ROTATION_SEED)
    return signs, o.rotation_matrix(signs)


@functools.lru_cache(maxsize=None)
def _mse_codebook(d: int, bits: int) -> np.ndarray:
    return o.codebook_f32(d, bits)[0]


class RecipeCodec:
    """The shared group codec of one recipe at one head_dim: R_d, S_d and both codebooks
    (S_d may be given, e.g. to average over sketch draws)."""

    def __init__(self, recipe: str, head_dim: int, smat: np.ndarray | None = None):
        self.recipe = recipe
        self.head_dim = head_dim
        self.d = high_group_count(recipe, head_dim)
        self.bits = recipe_bits(recipe)  # (high, low)
        self.signs, self.rot = _group_rotation(self.d)
        self.smat = qo.normal_matrix(self.d, self.d, SKETCH_SEED) if smat is None else np.asarray(smat, np.float64)
        # MSE codebooks of the groups: b - 1 bits for a group of b bits
        self.mse = tuple(_mse_codebook(self.d, b - 1) for b in self.bits)

    def group_bytes(self) -> tuple[int, int]:
        return qo.prod_row_bytes(self.d, self.bits[0]), qo.prod_row_bytes(self.d, self.bits[1])


def encode_recipe_rows(x: np.ndarray, high: np.ndarray, low: np.ndarray, codec: RecipeCodec) -> np.ndarray:
    """Recipe rows of x[N, D] for one kv head (its channel groups high[d], low[d]): uint8[N, RB]."""
    x = np.asarray(x, dtype=np.float64)
    parts = []
    for g, chans in enumerate((high, low)):
        enc = qo.encode_prod(x[:, chans], codec.rot, codec.mse[g], codec.smat)
        parts.append(qo.pack_prod_rows(enc["idx"], enc["z"], enc["nu"], enc["gamma"], codec.bits[g]))
    return np.concatenate(parts, axis=1)


def _split(rows: np.ndarray, codec: RecipeCodec):
    nh, nl = codec.group_bytes()
    rows = np.asarray(rows, dtype=np.uint8)
    if rows.shape[1] != nh + nl:
        raise ValueError(f"recipe rows must be {nh + nl} bytes, got {rows.shape[1]}")
    return rows[:, :nh], rows[:, nh:]


def recipe_scores(q: np.ndarray, rows: np.ndarray, high: np.ndarray, low: np.ndarray, codec: RecipeCodec) -> np.ndarray:
    """Estimates of <q_a, x_t> for queries q[A, D] and one kv head's rows[T, RB]: the sum of the
    two groups' product estimates on the gathered query channels.  Returns [A, T]."""
    q = np.asarray(q, dtype=np.float64)
    out = 0.0
    for g, (part, chans) in enumerate(zip(_split(rows, codec), (high, low))):
        out = out + qo.prod_scores(q[:, chans], part, codec.d, codec.bits[g], codec.rot, codec.mse[g], codec.smat)
    return out


def recipe_dequant(rows: np.ndarray, high: np.ndarray, low: np.ndarray, codec: RecipeCodec) -> np.ndarray:
    """The reconstruction of rows[T, RB]: each group's product reconstruction put back at its
    channels.  Returns [T, D]."""
    parts = _split(rows, codec)
    out = np.zeros((parts[0].shape[0], codec.head_dim), dtype=np.float64)
    for g, (part, chans) in enumerate(zip(parts, (high, low))):
        out[:, chans] = qo.prod_dequant(part, codec.d, codec.bits[g], codec.rot, codec.mse[g], codec.smat)
    return out


def write_recipe_kv(raw: np.ndarray, pages: np.ndarray, slots: np.ndarray, high: np.ndarray,
                    codec: RecipeCodec) -> np.ndarray:
    """Writes raw[T, H, D] into a copy of pages[NB, bs, H, RB] at the flat slots (negative slots
    skipped; a slot past the pages raises and nothing is written)."""
    raw = np.asarray(raw, dtype=np.float64)
    t, h, d = raw.shape
    nb, bs = pages.shape[:2]
    slots = np.asarray(slots, dtype=np.int64)
    if np.any(slots >= nb * bs):
        raise IndexError("slot out of range")
    high = validate_high_groups(high, codec.recipe, d, h)
    low = low_groups(high, d)
    out = np.array(pages, copy=True)
    keep = np.nonzero(slots >= 0)[0]
    for k in range(h):
        rows = encode_recipe_rows(raw[keep, k], high[k], low[k], codec)
        out[slots[keep] // bs, slots[keep] % bs, k] = rows
    return out


def paged_decode_recipe(q, k_pages, v_pages, block_table, seq_lens, high, codec: RecipeCodec, scale=None):
    """fp64 attention over recipe rows for both K and V: out[b, h] = sum_t softmax_t(scale *
    est<q_bh, k_t>) vhat_t, with the paging, GQA mapping and length rules of
    ``tq_oracle.paged_decode`` (tokens of a block id outside the pages are left out)."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    h = k_pages.shape[2]
    grp = hq // h
    high = validate_high_groups(high, codec.recipe, d, h)
    low = low_groups(high, d)
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    for b in range(bsz):
        n = int(seq_lens[b])
        if n <= 0:
            continue
        for kvh in range(h):
            krows, ok = o._gather_rows(k_pages, block_table[b], n, kvh)
            vrows, _ = o._gather_rows(v_pages, block_table[b], n, kvh)
            krows, vrows = krows[ok], vrows[ok]
            if krows.shape[0] == 0:
                continue
            vhat = recipe_dequant(vrows, high[kvh], low[kvh], codec)
            s = scale * recipe_scores(q[b, kvh * grp:(kvh + 1) * grp], krows, high[kvh], low[kvh], codec)
            p = np.exp(s - np.max(s, axis=1, keepdims=True))
            p /= np.sum(p, axis=1, keepdims=True)
            out[b, kvh * grp:(kvh + 1) * grp] = p @ vhat
    return out
