"""Column shards of the route step on one GPU, run one after another, then the
merge of their candidates.

Shard s of W computes latent columns [3584 s / W, ...) and experts
[896 s / W, ...) from the full hidden rows, plus its local top-16; the merge
ranks the W x 16 candidates.  This is the per-rank work of the pages' sharded
layout: each TP rank computes its own latent columns and the results are
gathered ("Optionally gather the Kimi3 prefill latent instead of reducing
it", Description: 448 columns a rank at TP8); the decode gather pairs latent
and router columns a rank (224 and 56 at TP16: "Use two row blocks for
eight-row Kimi paired gathers", body); candidate merge is named by that
page's tests and the first's.

Checks: the shards' latent and logits are bit-identical to the matching
columns of a whole-layer prefill plan (the per-column arithmetic is the
same); every shard's candidates are the oracle's top-16 of that shard's GPU
logits; the merged ids and weights equal the whole plan's and pass G1
against the oracle's top-16 of the concatenated GPU logits; sampled rows pass
G2-G4 against the oracle's float64 sums.  The merge alone is also checked on
candidates with exact ties across shards, NaN, -0/+0 and -inf."""

import numpy as np
import pytest
import torch

import latent_projection_top_gb300 as route
import oracle
from gates import check_topk_exact, record
from gpu_util import DEV, bank, bits_of, oracle_rows, require_gpu, run_step, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run_shards(h_dev, wl, wr, W, rows, ksplit=False):
    """Every shard of W in turn on one GPU, then the merge.  Returns the
    concatenated latent bits and logits, the merged ids and weights and the
    candidates (numpy)."""
    NL, NE = route.shard_columns(W)
    cand_ids = torch.full((W, rows, route.TOPK), -1, dtype=torch.int32, device=DEV)
    cand_lg = torch.full((W, rows, route.TOPK), float("nan"), dtype=torch.float32, device=DEV)
    lats, lgs = [], []
    for s in range(W):
        dwl = to_dev_bf16(np.ascontiguousarray(wl[:, s * NL:(s + 1) * NL]))
        dwr = to_dev_bf16(np.ascontiguousarray(wr[:, s * NE:(s + 1) * NE]))
        lat = torch.empty((rows, NL), dtype=torch.bfloat16, device=DEV)
        lat.view(torch.int16).fill_(0x7FC0)
        lg = torch.full((rows, NE), float("nan"), dtype=torch.float32, device=DEV)
        with route.ShardPlan(rows, s, W) as plan:
            assert (route.lib().route_plan_latent_cols(plan.handle),
                    route.lib().route_plan_experts(plan.handle)) == (NL, NE)
            if ksplit:
                route.route_set_latent_ksplit(plan, True)
            route.route_shard_step(plan, h_dev, dwl, dwr, lat, lg, cand_ids[s], cand_lg[s])
            route.route_device_status(plan)
        lats.append(bits_of(lat))
        lgs.append(lg.cpu().numpy())
    ids = torch.full((rows, route.TOPK), -1, dtype=torch.int32, device=DEV)
    w = torch.full((rows, route.TOPK), float("nan"), dtype=torch.float32, device=DEV)
    route.route_merge_candidates(cand_ids, cand_lg, ids, w)
    torch.cuda.synchronize()
    return (np.concatenate(lats, axis=1), np.concatenate(lgs, axis=1), ids.cpu().numpy(),
            w.cpu().numpy(), cand_ids.cpu().numpy(), cand_lg.cpu().numpy())


def _check_candidates(lg, cids, clg, W):
    """Each shard's candidates: the oracle's top-16 of that shard's GPU
    logits, as global ids, with those logits."""
    NE = route.N_EXPERTS // W
    for s in range(W):
        part = np.ascontiguousarray(lg[:, s * NE:(s + 1) * NE])
        ids_o, _ = oracle.topk(part)
        assert np.array_equal(cids[s], ids_o + s * NE), f"shard {s}: candidates differ"
        got = np.take_along_axis(part, ids_o, axis=1)
        assert np.array_equal(clg[s].view(np.uint32), got.view(np.uint32)), \
            f"shard {s}: candidate logits differ"


def _whole(h_dev, wl, wr, rows, ksplit=False):
    with route.Plan(route.PREFILL, rows) as plan:
        if ksplit:
            route.route_set_latent_ksplit(plan, True)
        return run_step(plan, h_dev, to_dev_bf16(wl), to_dev_bf16(wr))


@pytest.mark.parametrize("W", [2, 4, 7, 8, 14, 16, 1])
def test_shards_then_merge_equal_the_whole_layer_and_the_oracle(W):
    rows = 300  # two 256-row blocks, the second ragged
    hid, wl, wr = bank("prefill_r3072", 0)
    h_bits = np.ascontiguousarray(hid[:rows])
    h_dev = to_dev_bf16(h_bits)
    lat, lg, ids, w, cids, clg = _run_shards(h_dev, wl, wr, W, rows)
    lat0, lg0, ids0, w0 = _whole(h_dev, wl, wr, rows)
    assert np.array_equal(lat, lat0), "shard latent differs from the whole layer's"
    assert np.array_equal(lg.view(np.uint32), lg0.view(np.uint32)), "shard logits differ"
    _check_candidates(lg, cids, clg, W)
    assert np.array_equal(ids, ids0)
    assert np.array_equal(w.view(np.uint32), w0.view(np.uint32))
    ids_o, w_o = oracle.topk(lg)
    s1 = check_topk_exact(ids, w, ids_o, w_o)
    # G2-G4 on sampled rows (every row's latent/logits equal the whole
    # layer's, which the parity tests gate on all rows of other workloads)
    from test_gpu_parity import _prefill_gates
    idx = tuple(int(i) for i in np.sort(np.random.default_rng(77).choice(rows, 24, replace=False)))
    ref = oracle_rows("prefill_r3072", 0, idx)
    _prefill_gates(lat, lg, ids, w, ref, list(idx), f"shard_W{W}_r{rows}")
    record(f"shard_W{W}_merge", **s1)


def _whole_decode(h_dev, wl, wr, rows):
    with route.Plan(route.DECODE, rows) as plan:
        return run_step(plan, h_dev, to_dev_bf16(wl), to_dev_bf16(wr))


@pytest.mark.parametrize("workload,rows,W", [("decode_r8", 8, 8), ("decode_r8", 8, 2),
                                             ("decode_r8", 8, 16), ("decode_r1", 1, 4),
                                             ("decode_sweep", 20, 7), ("decode_r8", 8, 1),
                                             ("decode_sweep", 12, 14), ("decode_sweep", 20, 16)])
def test_decode_size_shards(workload, rows, W):
    """Up to 20 rows a shard streams its weights with the decode path's split
    K (TP8: 448 latent columns and 112 experts a shard; TP16: 224 and 56).
    The shards' latent and logits pass the decode gates against the oracle's
    float64 sums; every shard's candidates are the oracle's top-16 of that
    shard's GPU logits; the merged ids and weights are the oracle's top-16 of
    the concatenated GPU logits (G1) and agree with the oracle's ids end to
    end (G4, differences only on rows built as near ties); the logits agree
    with a whole-layer decode plan's to the decode gate's bound."""
    from gates import check_ids_end_to_end, check_latent, check_logits
    from test_gpu_parity import _near_tie_rows
    hid, wl, wr = bank(workload, 0)
    h_dev = to_dev_bf16(np.ascontiguousarray(hid[:rows]))
    lat, lg, ids, w, cids, clg = _run_shards(h_dev, wl, wr, W, rows)
    ref = oracle_rows(workload, 0, tuple(range(rows)))
    s1 = check_latent(lat, ref["latent"], ref["y_lat"], ref["abs_lat"])
    s2 = check_logits(lg, ref["y_log"], ref["abs_log"], "decode")
    _check_candidates(lg, cids, clg, W)
    ids_o, w_o = oracle.topk(lg)
    s3 = check_topk_exact(ids, w, ids_o, w_o)
    ids_ref, _ = oracle.topk(ref["logits"])
    s4 = check_ids_end_to_end(ids, ids_ref, ref["logits"],
                              swap_rows_allowed=_near_tie_rows(workload, rows))
    lat0, lg0, _, _ = _whole_decode(h_dev, wl, wr, rows)
    assert np.all(np.abs(lg.astype(np.float64) - lg0) <= 2.0 ** -24 * ref["abs_log"])
    record(f"shard_decode_W{W}_{workload}_r{rows}", **s1, **s2, **s3, **s4)


def test_ksplit_latent_on_shards():
    rows = 300
    hid, wl, wr = bank("prefill_r3072", 0)
    h_dev = to_dev_bf16(np.ascontiguousarray(hid[:rows]))
    lat, lg, ids, w, _, _ = _run_shards(h_dev, wl, wr, 4, rows, ksplit=True)
    lat0, lg0, ids0, w0 = _whole(h_dev, wl, wr, rows, ksplit=True)
    assert np.array_equal(lat, lat0), "K-split shard latent differs from the whole layer's"
    assert np.array_equal(lg.view(np.uint32), lg0.view(np.uint32))
    assert np.array_equal(ids, ids0)


def _tie_logits(rows, rng):
    """[rows, 896] FP32 logits with exact ties across shards at the top-16
    boundary, NaN, -0/+0 and -inf entries."""
    lg = rng.standard_normal((rows, route.N_EXPERTS)).astype(np.float32)
    for r in range(rows):
        kind = r % 4
        if kind == 0:  # 20 experts spread over every shard share one top value
            e = rng.choice(route.N_EXPERTS, 20, replace=False)
            lg[r, e] = np.float32(5.0)
        elif kind == 1:  # ties straddling the 16th place, in different shards
            order = np.argsort(-lg[r], kind="stable")
            v = lg[r, order[15]]
            e = rng.choice(route.N_EXPERTS, 6, replace=False)
            lg[r, e] = v
        elif kind == 2:  # NaN, +-0, -inf
            lg[r, rng.choice(route.N_EXPERTS, 30, replace=False)] = np.nan
            lg[r, rng.choice(route.N_EXPERTS, 10, replace=False)] = np.float32(-0.0)
            lg[r, rng.choice(route.N_EXPERTS, 10, replace=False)] = np.float32(0.0)
            lg[r, rng.choice(route.N_EXPERTS, 10, replace=False)] = -np.inf
        else:  # almost every logit NaN: the picks run into the NaNs
            lg[r, :] = np.nan
            lg[r, rng.choice(route.N_EXPERTS, 5, replace=False)] = np.float32(1.5)
    return lg


@pytest.mark.parametrize("W", [2, 7, 8, 16])
def test_merge_kernel_on_ties_nan_and_signed_zero(W):
    rows = 64
    lg = _tie_logits(rows, np.random.default_rng(300 + W))
    NE = route.N_EXPERTS // W
    cids = np.empty((W, rows, route.TOPK), np.int32)
    clg = np.empty((W, rows, route.TOPK), np.float32)
    for s in range(W):
        part = np.ascontiguousarray(lg[:, s * NE:(s + 1) * NE])
        i_s, _ = oracle.topk(part)
        cids[s] = i_s + s * NE
        clg[s] = np.take_along_axis(part, i_s, axis=1)
    ids = torch.full((rows, route.TOPK), -1, dtype=torch.int32, device=DEV)
    w = torch.full((rows, route.TOPK), float("nan"), dtype=torch.float32, device=DEV)
    route.route_merge_candidates(torch.from_numpy(cids).to(DEV), torch.from_numpy(clg).to(DEV),
                                 ids, w)
    torch.cuda.synchronize()
    ids_o, w_o = oracle.topk(lg)
    check_topk_exact(ids.cpu().numpy(), w.cpu().numpy(), ids_o, w_o)


def test_shard_plan_refuses_the_whole_layer_entry_points():
    rows = 8
    with route.ShardPlan(rows, 0, 8) as plan:
        lat = torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16, device=DEV)
        lg = torch.empty((rows, route.N_EXPERTS), dtype=torch.float32, device=DEV)
        ids = torch.empty((rows, route.TOPK), dtype=torch.int32, device=DEV)
        w = torch.empty((rows, route.TOPK), dtype=torch.float32, device=DEV)
        h = torch.zeros((rows, route.K_HIDDEN), dtype=torch.bfloat16, device=DEV)
        wl = torch.zeros((route.K_HIDDEN, route.N_LATENT), dtype=torch.bfloat16, device=DEV)
        wr = torch.zeros((route.K_HIDDEN, route.N_EXPERTS), dtype=torch.bfloat16, device=DEV)
        with pytest.raises(route.RouteError) as ei:  # decode-size shards: full-K latent only
            route.route_set_latent_ksplit(plan, True)
        assert ei.value.status == route.STATUS_CODES["ROUTE_ERR_PLAN"]
        for call in (lambda: route.route_step(plan, h, wl, wr, lat, lg, ids, w),
                     lambda: route.latent_router_forward(plan, h, wl, wr, lat, lg),
                     lambda: route.topk16_select(plan, lg, ids, w)):
            with pytest.raises(route.RouteError) as ei:
                call()
            assert ei.value.status == route.STATUS_CODES["ROUTE_ERR_PLAN"]
    with route.Plan(route.PREFILL, rows) as whole:  # a whole-layer plan runs no shard step
        st = route.lib().route_shard_step(whole.handle, h.data_ptr(), wl.data_ptr(), wr.data_ptr(),
                                          lat.data_ptr(), lg.data_ptr(), ids.data_ptr(),
                                          w.data_ptr(), None)
        assert st == route.STATUS_CODES["ROUTE_ERR_PLAN"]
