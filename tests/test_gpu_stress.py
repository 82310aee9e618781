"""Robustness under many CUDA-graph replays, at the scale of the stress runs
of the prefill-latent page ("Optionally gather the Kimi3 prefill latent
instead of reducing it", Tests: 2,000 graph replays with a new input bank on
every replay, outputs poisoned inside the graph, staging memory filled with
0xFF).

One graph per weight bank holds: every output filled with 0xFF bytes (NaN /
-1), the plan's scratch filled with 0xFF bytes (route_test_poison_scratch),
then the route step with the latent sum of squares.  Replays cycle the
banks; after each replay every output is compared on the device, bit for
bit, with the eager result of its bank, and the 4 KB canaries on both sides
of every output must stay untouched."""

import numpy as np
import pytest
import torch

import latent_projection_top_gb300 as route
from gpu_util import DEV, bank, require_gpu, to_dev_bf16

pytestmark = pytest.mark.gpu

GUARD = 4096


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _guarded(shape, dtype):
    """An output tensor inside a byte buffer with GUARD canary bytes (0xA5) on
    each side; returns (tensor, buffer, nbytes)."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((GUARD + n + GUARD,), 0xA5, dtype=torch.uint8, device=DEV)
    return buf[GUARD:GUARD + n].view(dtype).view(shape), buf, n


def _shapes(rows):
    return [((rows, route.N_LATENT), torch.bfloat16), ((rows, route.N_EXPERTS), torch.float32),
            ((rows, route.TOPK), torch.int32), ((rows, route.TOPK), torch.float32),
            ((rows,), torch.float32)]


def _stress(mode, rows, inputs, replays):
    """inputs: [(hidden, W_latent, W_router)] device tensors, one per bank."""
    with route.Plan(mode, rows) as plan:
        want = []
        for d in inputs:
            o = [torch.empty(sh, dtype=dt, device=DEV) for sh, dt in _shapes(rows)]
            route.route_step_sumsq(plan, *d, *o)
            want.append(o)
        torch.cuda.synchronize()
        route.route_device_status(plan)
        outs = [[_guarded(sh, dt) for sh, dt in _shapes(rows)] for _ in inputs]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graphs = []
        with torch.cuda.stream(s):
            for d, o in zip(inputs, outs):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    for t, _, _ in o:
                        t.view(torch.uint8).fill_(0xFF)
                    route.route_test_poison_scratch(plan, stream=s)
                    route.route_step_sumsq(plan, *d, *[t for t, _, _ in o], stream=s)
                graphs.append(g)
        torch.cuda.synchronize()
        bad = torch.zeros((), dtype=torch.int64, device=DEV)
        with torch.cuda.stream(s):
            for i in range(replays):
                b = i % len(graphs)
                graphs[b].replay()
                for (t, _, _), r in zip(outs[b], want[b]):
                    bad += torch.ne(t.view(torch.uint8), r.view(torch.uint8)).any().to(torch.int64)
        torch.cuda.synchronize()
        route.route_device_status(plan)
        assert int(bad) == 0, f"{int(bad)} output tensors differed from the eager bits"
        for o in outs:
            for _, buf, n in o:
                assert bool((buf[:GUARD] == 0xA5).all()) and bool((buf[GUARD + n:] == 0xA5).all())


@pytest.mark.parametrize("workload,rows,banks", [("decode_r8", 8, 8), ("decode_sweep", 20, 6)])
def test_decode_2000_replays_new_bank_each(workload, rows, banks):
    inputs = []
    for b in range(banks):
        h, wl, wr = bank(workload, b)
        inputs.append((to_dev_bf16(np.ascontiguousarray(h[:rows])), to_dev_bf16(wl), to_dev_bf16(wr)))
    _stress(route.DECODE, rows, inputs, 2000)


@pytest.mark.parametrize("rows,replays", [(300, 400), (1024, 200)])
def test_prefill_replays_new_bank_each(rows, replays):
    inputs = []
    for b in range(4):
        h, wl, wr = bank("prefill_r3072", b)
        inputs.append((to_dev_bf16(np.ascontiguousarray(h[:rows])), to_dev_bf16(wl), to_dev_bf16(wr)))
    _stress(route.PREFILL, rows, inputs, replays)
