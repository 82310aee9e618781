"""Failure detection without a GPU fault: a wait inside the projection kernel
is made to run out (a copy that is never issued), and the kernel must report
it through the device status word and leave the context usable."""

import numpy as np
import pytest
import torch

import latent_projection_top_gb300 as route
from gpu_util import bank, require_gpu, run_step, to_dev_bf16, outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("mode,rows", [(route.DECODE, 4), (route.PREFILL, 64)])
def test_bounded_wait_expires_reports_and_recovers(mode, rows):
    hid, wl, wr = bank("decode_r8", 0)
    h = to_dev_bf16(np.ascontiguousarray(np.resize(hid, (rows, hid.shape[1]))))
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    with route.Plan(mode, rows) as ref_plan:
        want = run_step(ref_plan, h, dwl, dwr)
    with route.Plan(mode, rows) as plan:
        route.route_test_stall(plan, True, 20_000_000)  # 20 ms bound
        lat, lg, ids, w = outputs(rows)
        route.route_step(plan, h, dwl, dwr, lat, lg, ids, w)
        with pytest.raises(route.RouteError) as err:
            route.route_device_status(plan)
        assert err.value.status == 6  # ROUTE_ERR_DEVICE_TIMEOUT
        route.route_device_status(plan)  # the status word was cleared
        route.route_test_stall(plan, False)
        got = run_step(plan, h, dwl, dwr)
    for a, b in zip(got, want):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
    torch.cuda.synchronize()
