"""The allocation-free decode entry point, route_step_decode_noalloc.

Some callers cannot allocate device memory: code running inside a host
framework that owns all device memory and gives its plug-ins no allocator,
and latency-critical paths that cannot afford cudaMalloc's device-wide
synchronisation.  For them the library offers one decode entry point that
needs no plan and keeps its split-K scratch in a fixed device array.  These
tests call it through the C ABI and check it against route_step on a plan
(which allocates its own scratch), on two calls in a row with different
inputs, so that a second call cannot pass on stale scratch.

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import latent_projection_top_gb300 as route
import synth

DEV = "cuda:0"


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def _outputs(rows):
    lat = torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16, device=DEV)
    lg = torch.empty((rows, route.N_EXPERTS), dtype=torch.float32, device=DEV)
    ids = torch.empty((rows, route.TOPK), dtype=torch.int32, device=DEV)
    w = torch.empty((rows, route.TOPK), dtype=torch.float32, device=DEV)
    lat.view(torch.int16).fill_(0x7FC0)  # NaN poison: every element must be written
    lg.fill_(float("nan"))
    ids.fill_(-1)
    w.fill_(float("nan"))
    return lat, lg, ids, w


def _host(outs):
    lat, lg, ids, w = outs
    return (lat.view(torch.int16).cpu().numpy(), lg.cpu().numpy().view(np.uint32),
            ids.cpu().numpy(), w.cpu().numpy().view(np.uint32))


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_status_query_rejects_a_device_out_of_range():
    """route_noalloc_status checks the device index before any CUDA call."""
    route.build()
    lib = route.lib()
    for dev in (-1, 64, 1000):
        assert lib.route_noalloc_status(dev) == 8  # ROUTE_ERR_DEVICE


def test_rows_beyond_the_fixed_scratch_are_rejected():
    """rows outside 1..20 fail with ROUTE_ERR_ROWS before any device work."""
    route.build()
    lib = route.lib()
    x = ctypes.c_void_p(0x1000)
    for rows in (0, -1, route.DECODE_MAX_ROWS + 1, 1000):
        assert lib.route_step_decode_noalloc(rows, x, x, x, x, x, x, x, None) == 1
        assert b"1-20" in lib.route_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("rows", [8, 20])
def test_noalloc_matches_route_step_on_two_calls(rows):
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    route.build()
    lib = route.lib()
    torch.cuda.set_device(0)
    wk = synth.WORKLOADS["decode_r8"]
    stream = torch.cuda.current_stream(0)
    for call, bank in enumerate((0, 1)):
        hid = _dev(synth.hidden(wk.seed, bank, rows))
        wl, wr = (_dev(w) for w in synth.weight_bank(wk.seed, bank))
        want = _outputs(rows)
        with route.Plan(route.DECODE, rows) as plan:
            route.route_step(plan, hid, wl, wr, *want)
            route.route_device_status(plan)
            plan_grid = plan.grid
        got = _outputs(rows)
        st = lib.route_step_decode_noalloc(rows, _p(hid), _p(wl), _p(wr), *(_p(t) for t in got),
                                           ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, lib.route_last_error().decode()
        torch.cuda.synchronize()
        g = _host(got)
        w = _host(want)
        assert np.all(g[2] >= 0), f"call {call}: ids not written"
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        noalloc_grid = lib.route_noalloc_grid(0)
        if sms <= 160:  # the cap does not bind: the plan's partition exactly
            assert noalloc_grid == plan_grid, (noalloc_grid, plan_grid)
        if plan_grid == noalloc_grid:
            # Same kernels and the same split-K partition: identical bits.
            for name, a, b in zip(("latent", "logits", "ids", "weights"), g, w):
                assert np.array_equal(a, b), f"call {call}: {name} differs"
        else:
            # Another partition: the sums differ only in rounding order.
            lat_g = (g[0].astype(np.uint32) << 16).view(np.float32)
            lat_w = (w[0].astype(np.uint32) << 16).view(np.float32)
            ulp = np.spacing(np.abs(lat_w).astype(np.float32)) * 2 ** 16
            assert np.all(np.abs(lat_g - lat_w) <= ulp)
            lg_g, lg_w = g[1].view(np.float32), w[1].view(np.float32)
            assert np.allclose(lg_g, lg_w, rtol=1e-5, atol=1e-6)
        assert lib.route_noalloc_status(0) == 0, lib.route_last_error().decode()


def test_noalloc_stall_hook_rejects_a_device_out_of_range():
    route.build()
    lib = route.lib()
    for dev in (-1, 64):
        assert lib.route_test_noalloc_stall(dev, 1, 0) == 8  # ROUTE_ERR_DEVICE


@pytest.mark.gpu
def test_noalloc_timeout_is_reported_then_cleared():
    """A wait of route_step_decode_noalloc that runs out (the stall hook) is
    reported by route_noalloc_status, which then clears it; the next call,
    without the hook, matches route_step again."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    route.build()
    lib = route.lib()
    torch.cuda.set_device(0)
    rows = 8
    wk = synth.WORKLOADS["decode_r8"]
    stream = torch.cuda.current_stream(0)
    hid = _dev(synth.hidden(wk.seed, 2, rows))
    wl, wr = (_dev(w) for w in synth.weight_bank(wk.seed, 2))
    args = (_p(hid), _p(wl), _p(wr))
    try:
        assert lib.route_test_noalloc_stall(0, 1, 1_000_000) == 0, lib.route_last_error().decode()
        got = _outputs(rows)
        assert lib.route_step_decode_noalloc(rows, *args, *(_p(t) for t in got),
                                             ctypes.c_void_p(stream.cuda_stream)) == 0
        torch.cuda.synchronize()
        assert lib.route_noalloc_status(0) == route.STATUS_CODES["ROUTE_ERR_DEVICE_TIMEOUT"]
        assert lib.route_noalloc_status(0) == 0  # cleared by the query
    finally:
        assert lib.route_test_noalloc_stall(0, 0, 0) == 0
    want = _outputs(rows)
    with route.Plan(route.DECODE, rows) as plan:
        route.route_step(plan, hid, wl, wr, *want)
        route.route_device_status(plan)
    got = _outputs(rows)
    assert lib.route_step_decode_noalloc(rows, *args, *(_p(t) for t in got),
                                         ctypes.c_void_p(stream.cuda_stream)) == 0
    torch.cuda.synchronize()
    assert lib.route_noalloc_status(0) == 0
    for name, a, b in zip(("latent", "logits", "ids", "weights"), _host(got), _host(want)):
        assert np.array_equal(a, b), f"{name} differs after the stall"
