"""The C-ABI library: it builds for sm_103a, loads, exports every entry point that
include/tq.h declares, and its host-side set-up (row size, RHT signs, Lloyd-Max
codebook, argument checks) agrees with the oracle.  No GPU work is launched here:
every call below returns before enqueuing anything."""

import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT, read_golden_rows
from oracle import tq_oracle as o

HEADER = os.path.join(ROOT, "include", "tq.h")


@pytest.fixture(scope="module")
def tq():
    from quantized_kv_cache_06_gb300 import build

    build.build_library()
    import quantized_kv_cache_06_gb300 as tq

    return tq


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["tq_build_rotation", "tq_codebook", "tq_write_kv", "tq_paged_decode", "tq_paged_decode_workspace",
                 "tq_row_bytes", "tq_last_error"]:
        assert want in names


def test_library_exports_every_declared_symbol(tq):
    lib = ctypes.CDLL(tq.lib()._name)
    for name in declared_functions():
        assert hasattr(lib, name), name
    from quantized_kv_cache_06_gb300 import _lib

    assert set(_lib.SIGNATURES) == set(declared_functions())


def test_row_bytes_matches_pages_table(tq):
    for line in read_golden_rows("row_bytes_d128.txt"):
        d, b, _, rb = map(int, line.split())
        assert tq.tq_row_bytes(d, b) == rb
    for d in (16, 32, 64, 128, 256):
        for b in (2, 3, 4, 5):
            assert tq.tq_row_bytes(d, b) == o.row_bytes(d, b)
    assert tq.lib().tq_row_bytes(48, 4) == -1
    assert tq.lib().tq_row_bytes(8, 4) == -1  # head_dim below 16
    assert tq.lib().tq_row_bytes(128, 6) == -1


@pytest.mark.parametrize("d", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("seed", [0, 42, 2**63 + 5])
def test_rotation_signs_match_oracle(tq, d, seed):
    got = tq.tq_build_rotation(d, seed).numpy()
    assert np.array_equal(got.astype(np.float64), o.splitmix64_signs(d, seed))


@pytest.mark.parametrize("d", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("bits", [2, 3, 4, 5])
def test_codebook_matches_oracle(tq, d, bits):
    c_lib, b_lib = tq.tq_codebook(d, bits)
    c64, _ = o.lloyd_max(d, bits)
    c_or = c64.astype(np.float32)
    c_lib = c_lib.numpy()
    # two independent solvers (incomplete-beta CDF vs Gauss-Legendre quadrature) meet the
    # same fixed point to ~1e-12; after rounding to fp32 at most a rare 1-ulp difference.
    ulp = np.spacing(np.abs(c_or))
    assert np.all(np.abs(c_lib - c_or) <= ulp)
    assert np.mean(c_lib == c_or) > 0.9
    assert np.array_equal(c_lib, -c_lib[::-1])
    mids = (0.5 * (c_lib[:-1].astype(np.float64) + c_lib[1:])).astype(np.float32)
    assert np.array_equal(b_lib.numpy(), mids)
    assert b_lib.numpy()[(1 << bits) // 2 - 1] == 0.0


def test_host_argument_errors(tq):
    lib = tq.lib()
    buf = (ctypes.c_float * 64)()
    assert lib.tq_build_rotation(100, 1, ctypes.addressof(buf)) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_build_rotation(64, 1, None) == tq.TQ_ERR_INVALID_ARG
    assert "NULL" in lib.tq_last_error().decode()
    assert lib.tq_codebook(128, 6, ctypes.addressof(buf), None) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_codebook(128, 0, ctypes.addressof(buf), None) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_codebook(128, 4, ctypes.addressof(buf), None) == tq.TQ_OK
    assert lib.tq_last_error().decode() == ""
    # writer: bad sizes, bad bits, bad head_dim, misalignment -- all rejected on the host, with
    # or without a status word (a NULL one makes a valid call synchronous, not invalid)
    dummy = 1 << 20
    assert lib.tq_write_kv(dummy, 1, -4, 2, 128, 4, dummy, dummy, 4, 16, dummy, dummy, None, None) == \
        tq.TQ_ERR_INVALID_ARG
    assert lib.tq_write_kv(dummy, 1, 4, 2, 128, 6, dummy, dummy, 4, 16, dummy, dummy, None, None) == \
        tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_write_kv(dummy, 1, 4, 2, 128, 6, dummy, dummy, 4, 16, dummy, dummy, dummy, None) == \
        tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_write_kv(dummy, 1, 4, 2, 96, 4, dummy, dummy, 4, 16, dummy, dummy, dummy, None) == \
        tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_write_kv(dummy + 2, 1, 4, 2, 128, 4, dummy, dummy, 4, 16, dummy, dummy, dummy, None) == \
        tq.TQ_ERR_INVALID_ARG  # misaligned raw
    # decode: GQA group not dividing, unsupported group, bad bits
    args = lambda hq, h, kb: (dummy, 1, 2, hq, h, 128, dummy, kb, dummy, 4, 8, 16, dummy, 4, dummy, dummy, dummy,
                              dummy, 0.0, dummy, 1, dummy, 1 << 30, None, None)
    assert lib.tq_paged_decode(*args(12, 8, 4)) == tq.TQ_ERR_INVALID_ARG
    assert lib.tq_paged_decode(*args(48, 3, 4)) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_paged_decode(*args(32, 8, 7)) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_paged_decode_workspace(2, 12, 8, 128, 4, 16) == 0


def test_workspace_queries_cover_every_plan(tq):
    # the queries take no bit widths, so they return the largest workspace over the kernels a
    # call may pick: the prefill query covers the decode query for the same shapes, and both
    # cover at least one split partial (D accumulators + max + sum) per (row, q head)
    lib = tq.lib()
    for r, hq, h, d, maxb, bs in [(64, 32, 8, 128, 512, 16), (1024, 32, 8, 128, 512, 16), (4, 64, 8, 128, 8192, 16),
                                  (16, 32, 8, 256, 256, 16), (5, 8, 8, 64, 3, 5), (3, 4, 4, 32, 2, 16)]:
        dec = lib.tq_paged_decode_workspace(r, hq, h, d, maxb, bs)
        pre = lib.tq_paged_prefill_workspace(r, hq, h, d, maxb, bs)
        assert dec >= r * hq * (d + 2) * 4
        assert pre >= dec
    assert lib.tq_paged_prefill_workspace(2, 12, 8, 128, 4, 16) == 0  # group does not divide


def test_prod_row_bytes_and_sketch_matrix_match_oracle(tq):
    from oracle import qjl_oracle as qo

    for d in (32, 64, 128, 256):
        for b in (2, 3, 4, 5):
            assert tq.tq_prod_row_bytes(d, b) == qo.prod_row_bytes(d, b)
    assert tq.lib().tq_prod_row_bytes(128, 1) == -1
    assert tq.lib().tq_prod_row_bytes(96, 4) == -1
    # the library draws S in fp64 and rounds once: equal to the oracle's S rounded to fp32
    for d, seed in [(64, 43), (128, 7), (32, 2**64 - 1)]:
        got = tq.tq_build_qjl_matrix(d, seed).numpy()
        assert np.array_equal(got, qo.normal_matrix(d, d, seed).astype(np.float32))


def test_prod_host_argument_errors(tq):
    lib = tq.lib()
    dummy = 1 << 20
    assert lib.tq_build_qjl_matrix(64, 1, None) == tq.TQ_ERR_INVALID_ARG
    w = lambda d, b, status: (dummy, 1, 4, 2, d, b, dummy, dummy, 4, 16, dummy, dummy, dummy, status, None)
    assert lib.tq_write_kv_prod(*w(256, 4, dummy)) == tq.TQ_ERR_UNSUPPORTED  # the kernels take D 64 / 128
    assert lib.tq_write_kv_prod(*w(128, 2, dummy)) == tq.TQ_ERR_UNSUPPORTED  # and 3..5 bits
    assert lib.tq_write_kv_prod(*w(128, 2, None)) == tq.TQ_ERR_UNSUPPORTED  # NULL status: checked all the same
    dec = lambda d, kb, vb, ws: (dummy, 1, 2, 32, 8, d, dummy, kb, dummy, vb, 8, 16, dummy, 4, dummy, dummy, dummy,
                                 dummy, dummy, 0.0, dummy, 1, dummy, ws, None, None)
    assert lib.tq_paged_decode_prod(*dec(256, 4, 4, 1 << 30)) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_paged_decode_prod(*dec(128, 6, 4, 1 << 30)) == tq.TQ_ERR_UNSUPPORTED
    assert lib.tq_paged_decode_prod(*dec(128, 4, 4, 16)) == tq.TQ_ERR_INVALID_ARG  # workspace too small
    for r, hq, h, d, maxb, bs in [(64, 32, 8, 128, 512, 16), (5, 8, 8, 64, 3, 5)]:
        # partials per (row, q head) plus the projected query S R q
        assert lib.tq_paged_decode_prod_workspace(r, hq, h, d, maxb, bs) >= r * hq * (2 * d + 2) * 4
    assert lib.tq_paged_decode_prod_workspace(2, 12, 8, 128, 4, 16) == 0


def test_binding_refuses_float_buffers_the_kernels_would_overread(tq):
    # signs, codebooks and the sketch matrix are fp32 arrays of known length on the device side
    import torch

    from quantized_kv_cache_06_gb300 import _lib

    f32 = torch.zeros(128, dtype=torch.float32)
    _lib._need_f32("x", 128, f32, torch.zeros(16), torch.zeros(128, 128))
    with pytest.raises(ValueError, match="float32"):
        _lib._need_f32("x", 128, f32.half(), torch.zeros(16))
    with pytest.raises(ValueError, match="float32"):
        _lib._need_f32("x", 128, f32, torch.zeros(128, 128, dtype=torch.float16))
    with pytest.raises(ValueError, match="head_dim"):
        _lib._need_f32("x", 128, torch.zeros(64), torch.zeros(16))


def test_binding_refuses_outputs_and_status_words_the_kernels_would_overrun(tq):
    import torch

    from quantized_kv_cache_06_gb300 import _lib

    with pytest.raises(ValueError, match="out must be"):
        _lib._need_out("x", torch.zeros(2, 4, 64), (2, 4, 128), torch.device("cpu"))
    with pytest.raises(ValueError, match="out must be"):
        _lib._need_out("x", torch.zeros(2, 4, 128, dtype=torch.int32), (2, 4, 128), torch.device("cpu"))
    _lib._need_status("x", None)
    for bad in (torch.zeros(1, dtype=torch.int64), torch.zeros(0, dtype=torch.int32), torch.zeros(1, dtype=torch.int32)):
        with pytest.raises(ValueError, match="status"):
            _lib._need_status("x", bad)  # wrong dtype, empty, or not on a CUDA device


def test_build_compiles_every_source_file():
    # a translation unit left out of the build list would be missing from the library on a
    # machine that builds from source
    from quantized_kv_cache_06_gb300 import build

    on_disk = {f for f in os.listdir(build.CSRC) if f.endswith((".cu", ".cpp"))}
    assert set(build.SOURCES) == on_disk


def test_wait_limit_hook_round_trips(tq):
    # host-only: the value later decode launches take for their bounded waits
    lib = tq.lib()
    default = lib.tq_set_wait_limit(-1)
    assert default > 0
    assert lib.tq_set_wait_limit(5) == default
    assert lib.tq_set_wait_limit(0) == 5
    assert lib.tq_set_wait_limit(-7) == 0
    assert lib.tq_set_wait_limit(-1) == default
