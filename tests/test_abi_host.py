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


def test_forward_ex2_rejects_unknown_flags(lib):
    # checked before any pointer or device access
    assert _lib.flce_forward_ex2(None, None, None, None, 8, 8, 8, 8, -100, None, 2, None, None, None,
                                 None, stream=0) == 1  # FLCE_ERR_INVALID_ARG


def test_grpo_one_call_rejects_bad_objective_arguments(lib):
    # eps_low outside [0, 1), negative beta, beta > 0 without reference
    # log-probs: all refused before any device access
    for eps_low, eps_high, beta in ((1.0, 0.2, 0.0), (0.2, 0.2, -0.1), (0.2, 0.2, 0.5)):
        assert _lib.flce_grpo_forward_backward(None, None, None, 8, None, None, eps_low, eps_high, beta,
                                               8, 8, 8, 8, -100, None, 1.0, None, None, None, None, 8, None,
                                               stream=0) == 1


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert _lib.flce_status_string(code) == name
    assert _lib.flce_status_string(99) == "FLCE_ERR_UNKNOWN"


def test_workspace_size_is_chunk_bounded(lib):
    # the dlogits block (at most round_up(chunk, 128) x V bf16) plus dH partials
    # and gathered rows (together no larger) dominate; growing N at a fixed
    # chunk adds only O(N) bytes (per-row split partials, row indices)
    V, H = 151936, 4096
    for chunk in (256, 4096):
        d_bound = ((chunk + 127) // 128 * 128) * V * 2
        sizes = [_lib.flce_workspace_bytes(n, H, V, chunk) for n in (16384, 131072, 1 << 20)]
        assert sizes[0] >= d_bound // 2
        for n, ws in zip((16384, 131072, 1 << 20), sizes):
            assert ws <= 2 * d_bound + (256 << 20) + 64 * n, (chunk, n, ws)
            assert ws < n * V * 2 * (chunk * 4 / n)  # a fraction of the full bf16 logits


@pytest.mark.parametrize("shape", [(64, 64, 1000, 16), (256, 2048, 248320, 256),
                                   (16384, 4096, 151936, 256), (16384, 4096, 151936, 4096),
                                   (32768, 4096, 128000, 4096), (131072, 2560, 151936, 256),
                                   (3000, 512, 20000, 256), (2000, 256, 30011, 128),
                                   (5, 8, 3, 1), (100000, 8, 7, 100000)])
@pytest.mark.parametrize("workers,cg", [(74, 2), (148, 1), (76, 2), (1, 2)])
def test_backward_plan_covers_the_problem_within_the_chunk_budget(shape, workers, cg):
    N, H, V, chunk = shape
    p = _lib.flce_backward_plan(N, H, V, chunk, workers, cg)
    c = min((chunk + 127) // 128 * 128, (N + 127) // 128 * 128)
    budget = c * ((V + 7) // 8 * 8) * 2
    assert p["dlogits_bytes"] <= budget
    assert p["rows_per_block"] % 128 == 0 and p["rows_per_block"] >= c
    assert p["row_blocks"] == -(-N // p["rows_per_block"])
    assert p["vocab_slabs"] * p["vocab_per_slab"] >= V
    if p["vocab_slabs"] > 1:
        assert p["vocab_per_slab"] % 256 == 0
        assert (p["vocab_slabs"] - 1) * p["vocab_per_slab"] < V  # no empty slab
    else:
        assert p["vocab_per_slab"] == V
    assert 1 <= p["dh_splits"] <= 16
    assert p["workspace_bytes"] <= 2 * budget + 16 * N + (1 << 20)


def test_backward_plan_prefers_row_blocks_over_literal_small_chunks():
    # 131,072 x 2,560 x 151,936 at 256-row chunks: dW is read-modified-written
    # once per row block, so the plan must hold many more than 256 rows
    p = _lib.flce_backward_plan(131072, 2560, 151936, 256, 74, 2)
    assert p["rows_per_block"] >= 1024 and p["vocab_slabs"] > 1
    # a chunk that already holds the whole problem stays one block, one slab
    q = _lib.flce_backward_plan(256, 2048, 248320, 256, 74, 2)
    assert (q["row_blocks"], q["vocab_slabs"]) == (1, 1)


def test_backward_plan_kinds_on_the_workloads(flce_opts):
    """Which backward the workloads run (76 SM pairs): the 16K SFT step one
    slab per 4,096-row block with 256 x 512 dH tiles; the long-context step
    at 256-row chunks pipelined row blocks over two dlogits buffers inside
    the chunk's budget; the single chunk 256 x 256 dH tiles (too few tiles
    for two waves)."""
    p = _lib.flce_backward_plan(16384, 4096, 151936, 4096, 76, 2)
    assert (p["vocab_slabs"], p["dlogits_buffers"], p["dh_wide"]) == (1, 1, 1)
    q = _lib.flce_backward_plan(131072, 2560, 151936, 256, 76, 2)
    assert q["vocab_slabs"] > 1 and q["dlogits_buffers"] == 2 and q["dh_wide"] == 0
    assert q["dlogits_bytes"] <= 256 * 151936 * 2
    r = _lib.flce_backward_plan(256, 2048, 248320, 256, 76, 2)
    assert (r["vocab_slabs"], r["dlogits_buffers"], r["dh_wide"]) == (1, 1, 0)
    # the options turn them off
    flce_opts.set("dh_wide", "0")
    flce_opts.set("pipeline", "0")
    assert _lib.flce_backward_plan(16384, 4096, 151936, 4096, 76, 2)["dh_wide"] == 0
    assert _lib.flce_backward_plan(131072, 2560, 151936, 256, 76, 2)["dlogits_buffers"] == 1


def test_backward_plan_row_override(flce_opts):
    flce_opts.set("bwd_rows", "768")
    flce_opts.set("pipeline", "0")  # one dlogits buffer
    p = _lib.flce_backward_plan(3000, 512, 20000, 256, 74, 2)
    assert (p["rows_per_block"], p["vocab_per_slab"], p["row_blocks"], p["vocab_slabs"]) == (768, 5120, 4, 4)
    assert p["dlogits_buffers"] == 1
    # pipelined row blocks: two buffers of half the budget each
    flce_opts.set("pipeline", "1")
    p = _lib.flce_backward_plan(3000, 512, 20000, 256, 74, 2)
    assert (p["rows_per_block"], p["vocab_per_slab"], p["row_blocks"], p["vocab_slabs"]) == (768, 3072, 4, 7)
    assert p["dlogits_buffers"] == 2 and p["dlogits_bytes"] == 2 * 768 * 3072 * 2 <= 256 * 20000 * 2
    flce_opts.set("bwd_rows", "100000")  # clamped to the problem, then to the budget
    p = _lib.flce_backward_plan(3000, 512, 20000, 256, 74, 2)
    assert p["dlogits_bytes"] <= 256 * 20000 * 2 and p["rows_per_block"] <= 3072


def test_backward_plan_rejects_bad_arguments(lib):
    info = _lib.BackwardPlanInfo()
    assert lib.flce_backward_plan(-1, 64, 100, 16, 74, 2, ctypes.addressof(info)) == 1
    assert lib.flce_backward_plan(10, 64, 0, 16, 74, 2, ctypes.addressof(info)) == 1
    assert lib.flce_backward_plan(10, 64, 100, 16, 74, 2, None) == 1


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


def test_jsd_rejects_beta_outside_the_open_interval_before_any_launch(lib):
    p = 256  # never dereferenced: the beta check comes before any launch
    for beta in (0.0, 1.0, -0.25, 2.0, float("nan")):
        assert _lib.flce_jsd_forward(p, p, 64, p, p, 64, None, None, 8, 100, 16, -100, beta, None,
                                     p, None, None, None, None, None, stream=0) == 1
        assert _lib.flce_jsd_backward(p, p, 64, p, p, 64, None, None, p, p, p, beta, 1.0, p, p, 8, 100,
                                      16, -100, None, stream=0) == 1


def test_a_missing_library_raises_instead_of_falling_back(tmp_path):
    # no CPU path stands in for the CUDA library
    with pytest.raises(FileNotFoundError):
        _lib.load(str(tmp_path / "libflce.so"), build_if_missing=False)


@pytest.mark.parametrize("shape", [(32768, 4096, 4096, 128000, 4096), (1100, 256, 384, 6000, 128),
                                   (900, 192, 256, 2100, 256), (7, 8, 4096, 50, 1)])
def test_distillation_workspace_holds_the_backward_and_both_gathered_heads(lib, shape):
    # the distillation backward compacts rows like the cross-entropy backward
    # and also gathers one row block of the teacher's h ([rows, H_t] bf16)
    N, Hs, Ht, V, chunk = shape
    p = _lib.flce_backward_plan(N, Hs, V, chunk)
    ws = _lib.flce_kd_workspace_bytes(N, Hs, Ht, V, chunk)
    assert ws >= p["workspace_bytes"] + p["rows_per_block"] * Ht * 2


def test_options_round_trip_and_range_checks(lib, flce_opts):
    # every option in the header's enum has a name here, and reads back what was set
    for name in _lib.OPTIONS:
        v = _lib.flce_get_option(name)
        flce_opts.set(name, v)
        assert _lib.flce_get_option(name) == v
    flce_opts.set("cta_group", 1)
    assert _lib.flce_get_option("cta_group") == 1
    flce_opts.set("dh_group", 0)
    assert _lib.flce_get_option("dh_group") == 0
    # out-of-range values and unknown options change nothing
    for name, bad in (("cta_group", 3), ("compact", 2), ("validate", -1), ("fwd_splits", 257),
                      ("dh_splits", 17), ("fwd_block_rows", -2), ("grid_workers", 4097), ("grid_workers", -1)):
        before = _lib.flce_get_option(name)
        assert lib.flce_set_option(_lib.OPTIONS[name], bad) == 1
        assert _lib.flce_get_option(name) == before
    v = ctypes.c_int64(0)
    assert lib.flce_set_option(len(_lib.OPTIONS), 0) == 1
    assert lib.flce_get_option(len(_lib.OPTIONS), ctypes.byref(v)) == 1
    assert lib.flce_get_option(0, None) == 1


def test_options_change_the_plan_without_the_environment(lib, flce_opts, monkeypatch):
    # the environment is read once; later changes to it are not seen
    p0 = _lib.flce_backward_plan(3000, 512, 20000, 256, 74, 2)
    monkeypatch.setenv("FLCE_BWD_ROWS", "768")
    assert _lib.flce_backward_plan(3000, 512, 20000, 256, 74, 2) == p0
    flce_opts.set("bwd_rows", 768)
    assert _lib.flce_backward_plan(3000, 512, 20000, 256, 74, 2)["rows_per_block"] == 768


def test_option_names_follow_the_header_enum():
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    h = open(os.path.join(root, "include", "flce.h")).read()
    body = h[h.index("typedef enum flce_option"):h.index("} flce_option;")]
    names = [n.lower() for n in re.findall(r"FLCE_OPT_([A-Z_]+)[ ,=]", body) if n != "COUNT"]
    assert [k for k, _ in sorted(_lib.OPTIONS.items(), key=lambda kv: kv[1])] == names
