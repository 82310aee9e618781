"""The latent's per-row sum of squares (route_step_sumsq) against the oracle,
through the C ABI: decode (computed where the split-K sums are finished) and
prefill (computed in the top-16 kernel).  Every other output must equal
route_step's bit for bit, and the statistic must be bitwise reproducible."""

import ctypes

import numpy as np
import pytest
import torch

import latent_projection_top_gb300 as route
import oracle
from gpu_util import DEV, bank, bits_of, outputs, require_gpu, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _ss_step(plan, h, wl, wr):
    lat, lg, ids, w = outputs(plan.rows)
    ss = torch.full((plan.rows,), float("nan"), dtype=torch.float32, device=DEV)
    route.route_step_sumsq(plan, h, wl, wr, lat, lg, ids, w, ss)
    route.route_device_status(plan)
    torch.cuda.synchronize()
    return bits_of(lat), lg.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), ss.cpu().numpy()


def _plain_step(plan, h, wl, wr):
    lat, lg, ids, w = outputs(plan.rows)
    route.route_step(plan, h, wl, wr, lat, lg, ids, w)
    route.route_device_status(plan)
    torch.cuda.synchronize()
    return bits_of(lat), lg.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def _check(got, want, rows):
    lat, lg, ids, w, ss = got
    for name, a, b in zip(("latent", "logits", "ids", "weights"), (lat, lg, ids, w), want):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8)), name
    ref = oracle.latent_sumsq(lat)
    ulps = np.abs(ss.astype(np.float64) - ref) / np.spacing(ref)
    assert ss.shape == (rows,) and np.all(np.isfinite(ss))
    assert ulps.max() <= 1.0, f"sum of squares {ulps.max()} ULP off"
    assert np.mean(ulps == 0) >= 0.99


@pytest.mark.parametrize("mode,workload,rows", [
    (route.DECODE, "decode_r1", 1), (route.DECODE, "decode_r8", 8),
    (route.DECODE, "decode_sweep", 17), (route.DECODE, "decode_sweep", 20),
    (route.PREFILL, "prefill_r1024", 40), (route.PREFILL, "prefill_r1024", 1024)])
def test_sumsq_matches_oracle_and_route_step(mode, workload, rows):
    hid, wl, wr = bank(workload, 0)
    h = to_dev_bf16(np.ascontiguousarray(np.resize(hid, (rows, hid.shape[1]))))
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    with route.Plan(mode, rows) as plan:
        want = _plain_step(plan, h, dwl, dwr)
        first = _ss_step(plan, h, dwl, dwr)
        _check(first, want, rows)
        # three more calls: the per-row arrival counters re-arm every launch
        for _ in range(3):
            again = _ss_step(plan, h, dwl, dwr)
            assert np.array_equal(again[4].view(np.uint32), first[4].view(np.uint32))


def test_sumsq_requires_an_output():
    with route.Plan(route.DECODE, 2) as plan:
        lat, lg, ids, w = outputs(2)
        h = torch.zeros((2, route.K_HIDDEN), dtype=torch.bfloat16, device=DEV)
        W = torch.zeros((route.K_HIDDEN, route.N_LATENT), dtype=torch.bfloat16, device=DEV)
        R = torch.zeros((route.K_HIDDEN, route.N_EXPERTS), dtype=torch.bfloat16, device=DEV)
        lib = route.lib()
        vp = ctypes.c_void_p
        st = lib.route_step_sumsq(plan.handle, vp(h.data_ptr()), vp(W.data_ptr()), vp(R.data_ptr()),
                                  vp(lat.data_ptr()), vp(lg.data_ptr()), vp(ids.data_ptr()),
                                  vp(w.data_ptr()), None, None)
        assert st == 3  # ROUTE_ERR_NULL
