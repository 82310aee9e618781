"""The C-ABI library on a machine without a GPU: it builds for sm_103a, loads,
exports every entry point the header declares, and rejects bad arguments with
status codes before it touches a device (no compute call is made here)."""

import ctypes
import os
import re

import pytest

import latent_projection_top_gb300 as route

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "route.h")


@pytest.fixture(scope="module")
def lib():
    route.build()
    return route.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(route_\w+|latent_\w+|topk16_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_binding_exports():
    fns = header_functions()
    assert "route_prepare" in fns and "latent_router_forward" in fns and "topk16_select" in fns
    assert sorted(route.EXPORTS) == fns


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


@pytest.mark.slow
def test_debug_library_builds_and_exports_every_declared_symbol():
    """The bounds-checked library (-DROUTE_DEBUG) builds from the same sources
    and exports the same entry points."""
    path = route.build(debug=True)
    assert path.endswith("libroute_debug.so")
    dbg = ctypes.CDLL(path)
    for name in header_functions():
        assert hasattr(dbg, name), name


def _prepare(lib, mode, rows):
    h = ctypes.c_void_p(123)
    st = lib.route_prepare(mode, rows, 0, ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("rows", [0, -1, 21, 1000])
def test_decode_envelope_rejected_at_preparation(lib, rows, figures):
    st, h = _prepare(lib, route.DECODE, rows)
    assert st == 1 and h.value is None  # ROUTE_ERR_ROWS, *out cleared
    assert b"1-20" in lib.route_last_error()


def test_the_21_row_rejection_matches_the_pages(lib, figures):
    assert figures["decode_rows_rejected"] == route.DECODE_MAX_ROWS + 1
    st, _ = _prepare(lib, route.DECODE, figures["decode_rows_rejected"])
    assert st == 1


@pytest.mark.parametrize("rows", [0, route.PREFILL_MAX_ROWS + 1])
def test_prefill_envelope(lib, rows):
    st, _ = _prepare(lib, route.PREFILL, rows)
    assert st == 1


def test_bad_mode_and_null_out(lib):
    st, _ = _prepare(lib, 7, 8)
    assert st == 2
    assert lib.route_prepare(route.DECODE, 8, 0, None) == 3


def test_valid_request_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = _prepare(lib, route.DECODE, 8)
    assert st in (5, 8) and h.value is None  # ROUTE_ERR_CUDA / ROUTE_ERR_DEVICE
    assert lib.route_last_error()


def test_calls_with_null_plan(lib):
    null = ctypes.c_void_p(0)
    x = ctypes.c_void_p(0x1000)
    assert lib.latent_router_forward(null, x, x, x, x, x, None) == 3
    assert lib.topk16_select(null, x, x, x, None) == 3
    assert lib.route_step(null, x, x, x, x, x, x, x, None) == 3
    assert lib.route_step_host(null, x, x, x, x, x, x, x, None) == 3
    assert lib.route_step_sumsq(null, x, x, x, x, x, x, x, x, None) == 3
    assert lib.route_set_overlap(null, 1) == 3
    assert lib.route_set_latent_ksplit(null, 1) == 3
    assert lib.route_test_stall(null, 1, 0) == 3
    assert lib.route_device_status(null) == 3
    out = ctypes.c_void_p(0x1000)
    assert lib.route_host_step_create(null, x, x, x, x, x, x, x, None, ctypes.byref(out)) == 3
    assert lib.route_host_step_run(null) == 3
    assert lib.route_host_step_launch(null) == 3
    assert lib.route_host_step_wait(null) == 3
    assert lib.route_host_step_destroy(null) == 0
    assert lib.route_test_poison_scratch(null, None) == 3
    assert lib.route_destroy(null) == 0
    for f in ("route_plan_rows", "route_plan_mode", "route_plan_grid", "route_plan_segments",
              "route_plan_latent_cols", "route_plan_experts"):
        assert getattr(lib, f)(null) == -1
    assert lib.route_shard_step(null, x, x, x, x, x, x, x, None) == 3


def test_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(route, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(route, "_lib", None)
    with pytest.raises(route.RouteError):
        route.lib()


def test_binding_checks_tensors_before_any_call():
    """The binding's marshalling: wrong device, dtype, shape or layout raise
    before any C entry point runs (a stand-in plan object is enough)."""
    import torch

    class FakePlan:
        rows, device, mode = 4, 0, route.DECODE
        handle = None

    p = FakePlan()
    cpu = torch.zeros((4, route.K_HIDDEN), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="must be on cuda:0"):
        route._proj_ptrs(p, cpu, cpu, cpu, cpu, cpu)
    with pytest.raises(TypeError, match="must be a torch.Tensor"):
        route._dev_tensor([1, 2], "hidden", (4, route.K_HIDDEN), route._bf16_types(), 0)
    # host tensors: dtype, shape and contiguity
    h = torch.zeros((4, route.K_HIDDEN), dtype=torch.bfloat16)
    assert route._host_tensor(h, "hidden_host", (4, route.K_HIDDEN), route._bf16_types()).value
    with pytest.raises(TypeError, match="dtype"):
        route._host_tensor(h.float(), "hidden_host", (4, route.K_HIDDEN), route._bf16_types())
    with pytest.raises(ValueError, match="contiguous with shape"):
        route._host_tensor(h[:2], "hidden_host", (4, route.K_HIDDEN), route._bf16_types())
    with pytest.raises(ValueError, match="contiguous with shape"):
        route._host_tensor(torch.zeros((route.K_HIDDEN, 4), dtype=torch.bfloat16).t(),
                           "hidden_host", (4, route.K_HIDDEN), route._bf16_types())
    with pytest.raises(TypeError, match="CPU torch.Tensor"):
        route._host_tensor(None, "hidden_host", (4, route.K_HIDDEN), route._bf16_types())


@pytest.mark.parametrize("W", [0, 3, 5, 6, 9, 17, 32, -2])
def test_shard_counts_outside_the_supported_set_are_rejected(lib, W):
    """A shard count must divide the 896 experts (and so the 3584 latent
    columns) with at least 16 experts a shard, at most 16 shards."""
    h = ctypes.c_void_p(123)
    assert lib.route_prepare_shard(8, 0, 0, W, ctypes.byref(h)) == 7  # ROUTE_ERR_PLAN
    assert h.value is None


def test_supported_shard_counts_divide_both_widths():
    for W in route.SHARD_COUNTS:
        NL, NE = route.shard_columns(W)
        assert NL * W == route.N_LATENT and NE * W == route.N_EXPERTS and NE >= route.TOPK
        assert (NL * 2) % 16 == 0 and (NE * 2) % 16 == 0 and (NE * 4) % 16 == 0  # TMA strides


def test_shard_index_and_rows_checked_before_the_device(lib):
    h = ctypes.c_void_p(123)
    assert lib.route_prepare_shard(8, 0, 8, 8, ctypes.byref(h)) == 7
    assert lib.route_prepare_shard(8, 0, -1, 8, ctypes.byref(h)) == 7
    assert lib.route_prepare_shard(0, 0, 0, 8, ctypes.byref(h)) == 1  # ROUTE_ERR_ROWS
    assert lib.route_prepare_shard(route.PREFILL_MAX_ROWS + 1, 0, 0, 8, ctypes.byref(h)) == 1
    assert lib.route_prepare_shard(8, 0, 0, 8, None) == 3


def test_merge_arguments_checked_before_the_device(lib):
    x = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    assert lib.route_merge_candidates(0, 2, x, x, x, x, None) == 1
    assert lib.route_merge_candidates(route.PREFILL_MAX_ROWS + 1, 2, x, x, x, x, None) == 1
    assert lib.route_merge_candidates(8, 0, x, x, x, x, None) == 7
    assert lib.route_merge_candidates(8, 17, x, x, x, x, None) == 7
    assert lib.route_merge_candidates(8, 2, None, x, x, x, None) == 3
    assert lib.route_merge_candidates(8, 2, x, x, odd, x, None) == 4
