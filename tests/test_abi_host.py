"""The C-ABI library builds, loads and exports every symbol include/flce.h
declares; host-side argument checks return statuses without touching a GPU."""
import ctypes

import pytest

from chunked_lm_head_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_header_declares_the_expected_entry_points():
    names = set(_lib.header_symbols())
    assert {"flce_forward", "flce_backward", "flce_workspace_bytes", "flce_status_string"} <= names
    assert names == set(_lib.SIGNATURES), names ^ set(_lib.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in _lib.header_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert _lib.flce_status_string(code) == name
    assert _lib.flce_status_string(99) == "FLCE_ERR_UNKNOWN"


def test_workspace_size_is_chunk_bounded(lib):
    # dlogits chunk R x V bf16 dominates; growing N at fixed chunk must not grow it
    # beyond the O(N) forward partials.
    V, H = 151936, 4096
    a = _lib.flce_workspace_bytes(16384, H, V, 4096)
    b = _lib.flce_workspace_bytes(131072, H, V, 4096)
    assert a >= 4096 * V * 2
    assert b - a < 131072 * 8 * 64  # at most O(N) growth (per-row split partials)
    assert b < 131072 * V * 2 / 8  # far below the full bf16 logits
    assert _lib.flce_workspace_bytes(-1, H, V, 256) == 0


def test_forward_rejects_bad_arguments_before_any_launch(lib):
    f = _lib.flce_forward
    nonnull = 16  # any non-null, 16-byte aligned value; never dereferenced on these paths
    # no outputs requested
    assert f(nonnull, nonnull, nonnull, None, 8, 64, 100, 16, -100, None, None, None, None, None, 0, 0) == 1
    # negative sizes
    assert f(nonnull, nonnull, nonnull, None, -1, 64, 100, 16, -100, nonnull, None, None, None, None, 0, 0) == 1
    # null inputs with N > 0
    assert f(None, nonnull, nonnull, None, 8, 64, 100, 16, -100, nonnull, None, None, None, None, 0, 0) == 1
    # H not a multiple of 8
    assert f(nonnull, nonnull, nonnull, None, 8, 60, 100, 16, -100, nonnull, None, None, None, None, 0, 0) == 3
    # misaligned h
    assert f(nonnull + 2, nonnull, nonnull, None, 8, 64, 100, 16, -100, nonnull, None, None, None, None, 0, 0) == 3


def test_backward_rejects_bad_arguments_before_any_launch(lib):
    b = _lib.flce_backward
    p = 16
    # neither dH nor dW requested
    assert b(p, p, p, None, p, 1.0, None, None, 8, 64, 100, 16, -100, None, 0, 0) == 1
    # lse missing
    assert b(p, p, p, None, None, 1.0, p, p, 8, 64, 100, 16, -100, None, 0, 0) == 1
    # H not a multiple of 8
    assert b(p, p, p, None, p, 1.0, p, p, 8, 12, 100, 16, -100, None, 0, 0) == 3
    # V = 0
    assert b(p, p, p, None, p, 1.0, p, p, 8, 64, 0, 16, -100, None, 0, 0) == 1


def test_profile_kinds(lib):
    n = lib.flce_profile_num_kinds()
    names = [lib.flce_profile_kind_name(k).decode() for k in range(n)]
    assert "fwd_logits_lse" in names and "bwd_dW" in names
    assert lib.flce_profile_kind_name(n) is None
