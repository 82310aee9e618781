"""Parity of the CUDA route step with the oracle, through the C ABI.

Sizes are chosen so the oracle finishes in seconds while the kernels still
span several tiles and a ragged tail; at the full prefill sizes outputs are
checked on sampled rows that the oracle computes one by one."""

import numpy as np
import pytest
import torch

import latent_projection_top_gb300 as route
import oracle
import synth
from gates import (check_ids_end_to_end, check_latent, check_logits, check_topk_exact, record)
from gpu_util import (DEV, bank, bits_of, oracle_rows, outputs, require_gpu, run_step,
                      to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


# ---------------------------------------------------------------- top-16 (G1)

def _topk_gpu(logits: np.ndarray, mode=route.DECODE):
    R = logits.shape[0]
    with route.Plan(mode, R) as plan:
        lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).to(DEV)
        _, _, ids, w = outputs(R)
        route.topk16_select(plan, lg, ids, w)
        torch.cuda.synchronize()
        return ids.cpu().numpy(), w.cpu().numpy()


def special_rows() -> np.ndarray:
    E = 896
    rng = np.random.default_rng(0)
    rows = [
        -np.arange(E, dtype=np.float32),
        np.arange(E, dtype=np.float32),
        np.full(E, 0.75, np.float32),
        (np.round(rng.standard_normal(E) * 2) / 2).astype(np.float32),   # many ties
        np.where(rng.random(E) < 0.5, -0.0, 0.0).astype(np.float32),   # +-0 only
    ]
    r = -np.arange(E, dtype=np.float32) - 10
    r[:15] = 5.0 + np.arange(15, 0, -1)
    r[[700, 40, 41]] = 1.5                                             # tie at ranks 16/17
    rows.append(r)
    r = rng.standard_normal(E).astype(np.float32)
    r[[3, 600]] = np.inf
    r[[5, 6]] = -np.inf
    r[[7, 800, 801]] = np.nan
    rows.append(r)
    r = np.full(E, np.nan, np.float32)
    r[[3, 7]] = [-np.inf, 2.0]
    rows.append(r)                                                      # mostly NaN
    r = np.full(E, -np.inf, np.float32)
    rows.append(r)                                                      # all -Inf
    r = rng.standard_normal(E).astype(np.float32) * 1e-30              # tiny and subnormal
    r[::7] = np.float32(1e-45)
    rows.append(r)
    r = rng.standard_normal(E).astype(np.float32) * 40                 # sigmoid saturation
    rows.append(r)
    r = np.full(E, -3.0, np.float32)
    r[np.arange(0, E, 31)] = 2.0                                       # equal values per lane stride
    rows.append(r)
    return np.stack(rows)


def test_topk_bit_exact_special_rows():
    logits = special_rows()
    ids, w = _topk_gpu(logits)
    ids_ref, w_ref = oracle.topk(logits)
    check_topk_exact(ids, w, ids_ref, w_ref)


@pytest.mark.parametrize("R,mode", [(20, route.DECODE), (3072, route.PREFILL)])
def test_topk_bit_exact_random(R, mode):
    rng = np.random.default_rng(R)
    logits = (rng.standard_normal((R, 896)) * 2).astype(np.float32)
    # a quarter of the rows get exact duplicates across the 16/17 boundary
    srt = np.sort(logits, axis=1)[:, ::-1]
    for r in range(0, R, 4):
        j = int(np.argwhere(logits[r] == srt[r, 16])[0, 0])
        logits[r, j] = srt[r, 15]
    ids, w = _topk_gpu(logits, mode)
    ids_ref, w_ref = oracle.topk(logits)
    check_topk_exact(ids, w, ids_ref, w_ref)


def test_decode_fused_topk_on_special_logits():
    """The decode step's own top-16 (the block-wide selection in its finish
    kernel, including the fallback for rows with heavy ties) on logits with
    ties, +-0, +-Inf and NaN.  A one-hot hidden row makes the logits equal one
    row of W_router (all other rows zero), so the special values pass through
    the projection unchanged."""
    K, E = route.K_HIDDEN, route.N_EXPERTS
    h = np.zeros((1, K), np.uint16)
    h[0, 0] = 0x3F80  # 1.0
    dh = to_dev_bf16(h)
    dwl = to_dev_bf16(np.zeros((K, route.N_LATENT), np.uint16))
    with route.Plan(route.DECODE, 1) as plan:
        for i, p in enumerate(special_rows()):
            wr = np.zeros((K, E), np.uint16)
            wr[0] = oracle.bf16_rne(p)
            lat, lg, ids, w = run_step(plan, dh, dwl, to_dev_bf16(wr))
            want = (wr[0].astype(np.uint32) << 16).view(np.float32)
            nan = np.isnan(want)
            assert np.array_equal(np.isnan(lg[0]), nan), f"pattern {i}: NaN positions"
            assert np.array_equal(lg[0][~nan], want[~nan]), f"pattern {i}: logits"
            assert not lat.any(), f"pattern {i}: latent of a zero W_latent"
            ids_o, w_o = oracle.topk(lg)
            check_topk_exact(ids, w, ids_o, w_o)


# ------------------------------------------------------------ decode (G1-G5)

DECODE_CASES = [("decode_r1", 1), ("decode_r8", 8), ("decode_sweep", 9), ("decode_sweep", 12),
                ("decode_sweep", 16), ("decode_sweep", 20)]


def _near_tie_rows(workload, rows):
    """Rows built as near ties at ranks 16/17 (the only rows where the GPU's
    ids may differ from the oracle's)."""
    wk = synth.WORKLOADS[workload]
    return [r for r in range(rows) if wk.near_tie and r % 4 == 3]


def _decode_parity(workload, b, rows, check_unfused=False):
    hid, wl, wr = bank(workload, b)
    ref = oracle_rows(workload, b, tuple(range(max(synth.WORKLOADS[workload].rows))))
    h = to_dev_bf16(hid[:rows])
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    with route.Plan(route.DECODE, rows) as plan:
        lat, lg, ids, w = run_step(plan, h, dwl, dwr, fused=True)
        if check_unfused:
            unfused = run_step(plan, h, dwl, dwr, fused=False)
    sl = slice(0, rows)
    s1 = check_latent(lat, ref["latent"][sl], ref["y_lat"][sl], ref["abs_lat"][sl])
    s2 = check_logits(lg, ref["y_log"][sl], ref["abs_log"][sl], "decode")
    # the fused top-16 equals the oracle's top-16 on the same (GPU) logits
    ids_o, w_o = oracle.topk(lg)
    s3 = check_topk_exact(ids, w, ids_o, w_o)
    # end to end against the oracle's own logits
    ids_ref, _ = oracle.topk(ref["logits"][sl])
    s4 = check_ids_end_to_end(ids, ids_ref, ref["logits"][sl], _near_tie_rows(workload, rows))
    record(f"decode_{workload}_b{b}_r{rows}", **s1, **s2, **s3, **s4)
    if check_unfused:  # the unfused path computes the same bits
        lat2, lg2, ids2, w2 = unfused
        assert np.array_equal(lat, lat2) and np.array_equal(lg.view(np.uint32), lg2.view(np.uint32))
        assert np.array_equal(ids, ids2) and np.array_equal(w.view(np.uint32), w2.view(np.uint32))
    return s4


@pytest.mark.parametrize("workload,rows", DECODE_CASES)
def test_decode_route_step_parity(workload, rows):
    _decode_parity(workload, 0, rows, check_unfused=True)


@pytest.mark.parametrize("workload,b,rows", [("decode_r8", b, 8) for b in range(1, 8)] +
                         [("decode_sweep", b, r) for b in range(1, 6) for r in (16, 20)])
def test_decode_parity_every_bank(workload, b, rows):
    """Every weight bank of the 8-row workload and of the 9..20-row sweep (16
    rows run the 16-row tile, 20 rows the 32-row one) against the oracle."""
    _decode_parity(workload, b, rows)


def test_decode_batch_invariance_and_determinism():
    hid, wl, wr = bank("decode_sweep", 1)
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    results = {}
    for rows in (20, 1, 8, 16, 17):
        with route.Plan(route.DECODE, rows) as plan:
            results[rows] = run_step(plan, to_dev_bf16(hid[:rows]), dwl, dwr)
            again = run_step(plan, to_dev_bf16(hid[:rows]), dwl, dwr)
            for a, b in zip(results[rows], again):
                assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
    full = results[20]
    for rows in (1, 8, 16, 17):
        for a, b in zip(results[rows], full):
            assert np.array_equal(np.asarray(a).view(np.uint8),
                                  np.asarray(b)[:rows].view(np.uint8)), f"rows={rows}"


@pytest.mark.parametrize("mode,rows,workload", [(route.DECODE, 8, "decode_r8"),
                                                (route.PREFILL, 300, "prefill_r1024")])
@pytest.mark.parametrize("overlap", [False, True])
def test_bank_cycling_under_graph_replay(mode, rows, workload, overlap):
    """Banks cycled inside one captured CUDA graph give the eager bits, also
    when consecutive steps overlap (hidden is not written by route calls):
    decode, and prefill (whose GEMM then reads hidden under the previous
    step's top-16 and writes only after it)."""
    banks = [bank(workload, b) for b in range(3)]
    dev = [(to_dev_bf16(h[:rows]), to_dev_bf16(wl), to_dev_bf16(wr)) for h, wl, wr in banks]
    with route.Plan(mode, rows) as plan:
        eager = [run_step(plan, *d) for d in dev]
        route.route_set_overlap(plan, overlap)
        outs = [outputs(rows) for _ in dev]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for d, o in zip(dev, outs):
                    route.route_step(plan, *d, *o, stream=s)
        for _ in range(20):
            for o in outs:
                o[0].view(torch.int16).fill_(0x7FC0)
                o[1].fill_(float("nan"))
                o[2].fill_(-1)
            g.replay()
        torch.cuda.synchronize()
        route.route_device_status(plan)
        for o, e in zip(outs, eager):
            assert np.array_equal(bits_of(o[0]), e[0])
            assert np.array_equal(o[1].cpu().numpy().view(np.uint32), e[1].view(np.uint32))
            assert np.array_equal(o[2].cpu().numpy(), e[2])
            assert np.array_equal(o[3].cpu().numpy().view(np.uint32), e[3].view(np.uint32))


def _guarded(shape, dtype, guard=4096):
    """An output tensor inside a byte buffer with `guard` canary bytes (0xA5)
    on each side; returns (tensor, buffer, nbytes)."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((guard + n + guard,), 0xA5, dtype=torch.uint8, device=DEV)
    return buf[guard:guard + n].view(dtype).view(shape), buf, n


@pytest.mark.parametrize("rows", [8, 20])
def test_decode_replays_poisoned_scratch_and_canaries(rows):
    """Robustness under replay: every step's split-K scratch is filled with
    0xFF bytes before it runs (inside the captured graph), outputs are
    poisoned before every replay, the bank changes every step, and each of
    200 replays must give the eager bits (compared on the device) without
    touching 4 KB of canary bytes on either side of every output."""
    banks = [bank("decode_sweep", b) for b in range(3)]
    dev = [(to_dev_bf16(np.resize(h, (rows, h.shape[1]))), to_dev_bf16(wl), to_dev_bf16(wr))
           for h, wl, wr in banks]
    with route.Plan(route.DECODE, rows) as plan:
        want = []
        for d in dev:
            lat, lg, ids, w = outputs(rows)
            ss = torch.empty((rows,), dtype=torch.float32, device=DEV)
            route.route_step_sumsq(plan, *d, lat, lg, ids, w, ss)
            want.append((lat, lg, ids, w, ss))
        torch.cuda.synchronize()
        shapes = [((rows, route.N_LATENT), torch.bfloat16), ((rows, route.N_EXPERTS), torch.float32),
                  ((rows, route.TOPK), torch.int32), ((rows, route.TOPK), torch.float32),
                  ((rows,), torch.float32)]
        outs = [[_guarded(sh, dt) for sh, dt in shapes] for _ in dev]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for d, o in zip(dev, outs):
                    route.route_test_poison_scratch(plan, stream=s)
                    route.route_step_sumsq(plan, *d, *[t for t, _, _ in o], stream=s)
        torch.cuda.synchronize()
        bad = 0
        for _ in range(200):
            for o in outs:
                for t, _, _ in o:
                    t.view(torch.uint8).fill_(0xFF)  # NaN / -1 everywhere
            g.replay()
            for o, ref in zip(outs, want):
                for (t, _, _), r in zip(o, ref):
                    bad += int(not torch.equal(t.view(torch.uint8), r.view(torch.uint8)))
        torch.cuda.synchronize()
        route.route_device_status(plan)
        assert bad == 0, f"{bad} output tensors differed from the eager bits"
        for o in outs:
            for _, buf, n in o:
                assert bool((buf[:4096] == 0xA5).all()) and bool((buf[4096 + n:] == 0xA5).all())


# ------------------------------------------------------------------- prefill

@pytest.mark.parametrize("rows,sample", [(1, None), (40, None), (256, (0, 100, 255)),
                                         (300, (0, 255, 256, 299))])
def test_prefill_ragged_parity(rows, sample):
    hid, wl, wr = bank("prefill_r1024", 0)
    idx = tuple(range(rows)) if sample is None else sample
    ref = oracle_rows("prefill_r1024", 0, idx)
    with route.Plan(route.PREFILL, rows) as plan:
        lat, lg, ids, w = run_step(plan, to_dev_bf16(hid[:rows]), to_dev_bf16(wl), to_dev_bf16(wr))
    sel = list(idx)
    s1 = check_latent(lat[sel], ref["latent"], ref["y_lat"], ref["abs_lat"])
    s2 = check_logits(lg[sel], ref["y_log"], ref["abs_log"], "prefill")
    ids_o, w_o = oracle.topk(lg)
    s3 = check_topk_exact(ids, w, ids_o, w_o)
    ids_ref, _ = oracle.topk(ref["logits"])
    s4 = check_ids_end_to_end(ids[sel], ids_ref, ref["logits"], y64=ref["y_log"], logits_out=lg[sel])
    record(f"prefill_ragged_r{rows}", **s1, **s2, **s3, **s4)


def test_prefill_1024_cancel_group_sampled():
    """Rows d < 448 see cancelling K-slice partials on latent column d."""
    hid, wl, wr = bank("prefill_r1024", 0)
    idx = (0, 1, 2, 63, 127, 128, 255, 300, 447, 448, 511, 640, 767, 896, 1000, 1023)
    ref = oracle_rows("prefill_r1024", 0, idx)
    with route.Plan(route.PREFILL, 1024) as plan:
        lat, lg, ids, w = run_step(plan, to_dev_bf16(hid), to_dev_bf16(wl), to_dev_bf16(wr))
    sel = list(idx)
    s1 = check_latent(lat[sel], ref["latent"], ref["y_lat"], ref["abs_lat"])
    s2 = check_logits(lg[sel], ref["y_log"], ref["abs_log"], "prefill")
    ids_o, w_o = oracle.topk(lg)
    s3 = check_topk_exact(ids, w, ids_o, w_o)
    ids_ref, _ = oracle.topk(ref["logits"])
    s4 = check_ids_end_to_end(ids[sel], ids_ref, ref["logits"], y64=ref["y_log"], logits_out=lg[sel])
    record("prefill_r1024_cancel_sampled", **s1, **s2, **s3, **s4)
    # the cancel-group columns of the sampled rows d < 448, on their own
    cols = [(i, d) for i, d in enumerate(idx) if d < 448]
    out = np.array([lat[d, d] for _, d in cols], np.uint16)
    refc = np.array([ref["latent"][i, d] for i, d in cols], np.uint16)
    yc = np.array([ref["y_lat"][i, d] for i, d in cols])
    ac = np.array([ref["abs_lat"][i, d] for i, d in cols])
    record("prefill_r1024_cancel_columns", **check_latent(out, refc, yc, ac, rms_bar=False))


def _prefill_gates(lat, lg, ids, w, ref, sel, case):
    s1 = check_latent(lat[sel], ref["latent"], ref["y_lat"], ref["abs_lat"])
    s2 = check_logits(lg[sel], ref["y_log"], ref["abs_log"], "prefill")
    ids_o, w_o = oracle.topk(lg[sel])
    s3 = check_topk_exact(ids[sel], w[sel], ids_o, w_o)
    ids_ref, _ = oracle.topk(ref["logits"])
    s4 = check_ids_end_to_end(ids[sel], ids_ref, ref["logits"], y64=ref["y_log"],
                              logits_out=lg[sel])
    record(case, **s1, **s2, **s3, **s4)


def test_prefill_1024_every_row():
    """All 1024 rows of the cancel-group workload against the oracle (G2-G4);
    the oracle runs on row blocks in parallel (see gpu_util.oracle_block)."""
    hid, wl, wr = bank("prefill_r1024", 0)
    ref = oracle_rows("prefill_r1024", 0, tuple(range(1024)))
    with route.Plan(route.PREFILL, 1024) as plan:
        lat, lg, ids, w = run_step(plan, to_dev_bf16(hid), to_dev_bf16(wl), to_dev_bf16(wr))
    _prefill_gates(lat, lg, ids, w, ref, list(range(1024)), "prefill_r1024_all")


@pytest.mark.parametrize("b", [1, 2, 45, 91])
def test_prefill_3072_other_banks_sampled(b):
    """64 seeded rows of a 3072-row chunk on weight banks other than 0 (the
    workload has 92, one per MoE layer) against the oracle (G2-G4)."""
    hid, wl, wr = bank("prefill_r3072", b)
    idx = tuple(int(i) for i in np.sort(np.random.default_rng(1000 + b).choice(3072, 64, replace=False)))
    ref = oracle_rows("prefill_r3072", b, idx)
    with route.Plan(route.PREFILL, 3072) as plan:
        lat, lg, ids, w = run_step(plan, to_dev_bf16(hid), to_dev_bf16(wl), to_dev_bf16(wr))
    _prefill_gates(lat, lg, ids, w, ref, list(idx), f"prefill_r3072_b{b}_s64")


def test_prefill_3072_sampled_and_deterministic():
    hid, wl, wr = bank("prefill_r3072", 0)
    rng = np.random.default_rng(1000)
    idx = tuple(sorted(set((0, 1, 255, 256, 1000, 1535, 2047, 2048, 2900, 3071)) |
                       set(int(i) for i in rng.choice(3072, 54, replace=False))))
    ref = oracle_rows("prefill_r3072", 0, idx)
    dh, dwl, dwr = to_dev_bf16(hid), to_dev_bf16(wl), to_dev_bf16(wr)
    with route.Plan(route.PREFILL, 3072) as plan:
        a = run_step(plan, dh, dwl, dwr)
        b = run_step(plan, dh, dwl, dwr)
    for x, y in zip(a, b):
        assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))
    lat, lg, ids, w = a
    _prefill_gates(lat, lg, ids, w, ref, list(idx), "prefill_r3072_b0_s64")
    ids_o, w_o = oracle.topk(lg)
    check_topk_exact(ids, w, ids_o, w_o)


def test_prefill_8192_rows_sampled_and_position_independent():
    """A chunk well past the pages' largest (8192 rows, 7.6 waves of CTA-pair
    tiles): the 3072-row bank repeated, so rows r and r + 3072 hold the same
    hidden values and must give the same bits wherever they sit."""
    hid, wl, wr = bank("prefill_r3072", 0)
    big = np.ascontiguousarray(np.concatenate([hid, hid, hid[:2048]]))
    rows = big.shape[0]
    base = (0, 255, 1000, 2047, 3071)
    ref = oracle_rows("prefill_r3072", 0, base)
    with route.Plan(route.PREFILL, rows) as plan:
        lat, lg, ids, w = run_step(plan, to_dev_bf16(big), to_dev_bf16(wl), to_dev_bf16(wr))
    for off in (0, 3072, 6144):
        sel = [b + off for b in base if b + off < rows]
        k = len(sel)
        check_latent(lat[sel], ref["latent"][:k], ref["y_lat"][:k], ref["abs_lat"][:k])
        check_logits(lg[sel], ref["y_log"][:k], ref["abs_log"][:k], "prefill")
    for r in (0, 1000, 2047):
        for off in (3072, 6144):
            assert np.array_equal(lat[r], lat[r + off]) and np.array_equal(
                lg[r].view(np.uint32), lg[r + off].view(np.uint32))
    ids_o, w_o = oracle.topk(lg[:64])
    check_topk_exact(ids[:64], w[:64], ids_o, w_o)


@pytest.mark.parametrize("mode,rows", [(route.DECODE, 8), (route.DECODE, 20), (route.PREFILL, 40)])
def test_router_column_permutation_permutes_ids(mode, rows):
    """Pin P7 on the GPU: with W_router's columns permuted, logit column e is
    bit for bit the plain run's column perm[e] (every output is summed over
    the same K slices in the same order wherever its column sits), so
    perm[ids] are the plain run's ids and the weights are the same bits."""
    hid, wl, wr = bank("decode_r8" if mode == route.DECODE else "prefill_r1024", 0)
    hid = np.ascontiguousarray(np.resize(hid, (rows, hid.shape[1])))
    perm = np.random.default_rng(7).permutation(route.N_EXPERTS)
    dh, dwl = to_dev_bf16(hid), to_dev_bf16(wl)
    with route.Plan(mode, rows) as plan:
        lat_a, lg_a, ids_a, w_a = run_step(plan, dh, dwl, to_dev_bf16(wr))
        lat_b, lg_b, ids_b, w_b = run_step(plan, dh, dwl, to_dev_bf16(wr[:, perm]))
    assert np.array_equal(lat_a, lat_b)  # the latent does not see the router's columns
    assert np.array_equal(lg_b.view(np.uint32), lg_a[:, perm].view(np.uint32))
    assert np.array_equal(perm[ids_b], ids_a)
    assert np.array_equal(w_b.view(np.uint32), w_a.view(np.uint32))


# ------------------------------------------------------- host entry / errors

@pytest.mark.parametrize("mode,rows", [(route.DECODE, 8), (route.DECODE, 20), (route.PREFILL, 40)])
@pytest.mark.parametrize("pinned", [True, False])
def test_route_step_host_matches_device(mode, rows, pinned):
    """Page-locked buffers take the direct path for decode (staging kernel in,
    results written straight to host memory); pageable ones the copy path."""
    hid, wl, wr = bank("decode_r8" if mode == route.DECODE else "prefill_r1024", 0)
    hid = np.ascontiguousarray(np.resize(hid, (rows, hid.shape[1])))
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    with route.Plan(mode, rows) as plan:
        dev = run_step(plan, to_dev_bf16(hid), dwl, dwr)
        h_host = pin(torch.from_numpy(hid.view(np.int16).copy()).view(torch.bfloat16))
        lat = pin(torch.full((rows, route.N_LATENT), float("nan"), dtype=torch.bfloat16))
        lg = pin(torch.full((rows, route.N_EXPERTS), float("nan"), dtype=torch.float32))
        ids = pin(torch.full((rows, route.TOPK), -1, dtype=torch.int32))
        w = pin(torch.full((rows, route.TOPK), float("nan"), dtype=torch.float32))
        for _ in range(2):  # twice: the staging buffer is reused
            route.route_step_host(plan, h_host, dwl, dwr, lat, lg, ids, w)
        route.route_device_status(plan)
    assert np.array_equal(lat.view(torch.int16).numpy().view(np.uint16), dev[0])
    assert np.array_equal(lg.numpy().view(np.uint32), dev[1].view(np.uint32))
    assert np.array_equal(ids.numpy(), dev[2])
    assert np.array_equal(w.numpy().view(np.uint32), dev[3].view(np.uint32))


@pytest.mark.parametrize("rows", [1, 8, 20])
def test_host_step_reuses_buffers(rows):
    """HostStep: checked once and captured as a graph, then each call runs the
    copy-free host path on the same buffers -- new hidden rows written into
    hidden_host give that step's results; once the plan is closed a call is
    refused, not run."""
    _, wl, wr = bank("decode_r8", 0)
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    h0 = np.ascontiguousarray(np.resize(bank("decode_r8", 0)[0], (rows, route.K_HIDDEN)))
    h1 = np.ascontiguousarray(np.resize(bank("decode_r8", 1)[0], (rows, route.K_HIDDEN)))
    with route.Plan(route.DECODE, rows) as plan:
        want = [run_step(plan, to_dev_bf16(h), dwl, dwr) for h in (h0, h1)]
        h_host = torch.empty((rows, route.K_HIDDEN), dtype=torch.bfloat16).pin_memory()
        lat = torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16).pin_memory()
        lg = torch.empty((rows, route.N_EXPERTS), dtype=torch.float32).pin_memory()
        ids = torch.empty((rows, route.TOPK), dtype=torch.int32).pin_memory()
        w = torch.empty((rows, route.TOPK), dtype=torch.float32).pin_memory()
        step = route.HostStep(plan, h_host, dwl, dwr, lat, lg, ids, w)
        assert step.graph  # decode, page-locked: the captured graph
        for h, dev in zip((h0, h1, h0), want + want[:1]):
            h_host.copy_(torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16))
            step()
            assert np.array_equal(lat.view(torch.int16).numpy().view(np.uint16), dev[0])
            assert np.array_equal(lg.numpy().view(np.uint32), dev[1].view(np.uint32))
            assert np.array_equal(ids.numpy(), dev[2])
            assert np.array_equal(w.numpy().view(np.uint32), dev[3].view(np.uint32))
        route.route_device_status(plan)
    with pytest.raises(route.RouteError):
        step()  # the plan released the step's graph
    step.close()
    with pytest.raises(route.RouteError):
        step()


@pytest.mark.parametrize("mode,workload,rows", [(route.DECODE, "decode_r8", 8),
                                               (route.PREFILL, "prefill_r1024", 300)])
def test_step_object_equals_route_step(mode, workload, rows):
    """Step: the tensors checked once, each call one C call on the same
    buffers; new hidden values written in place give that call's results."""
    _, wl, wr = bank(workload, 0)
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    hs = [to_dev_bf16(np.ascontiguousarray(np.resize(bank(workload, b)[0], (rows, route.K_HIDDEN))))
          for b in (0, 1)]
    with route.Plan(mode, rows) as plan:
        want = [run_step(plan, h, dwl, dwr) for h in hs]
        h = torch.empty_like(hs[0])
        lat, lg, ids, w = outputs(rows)
        step = route.Step(plan, h, dwl, dwr, lat, lg, ids, w)
        for b in (0, 1, 0):
            h.copy_(hs[b])
            step()
            torch.cuda.synchronize()
            got = (bits_of(lat), lg.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy())
            for x, y in zip(got, want[b]):
                assert np.array_equal(np.asarray(x).view(np.uint8), np.asarray(y).view(np.uint8))
        route.route_device_status(plan)
    with pytest.raises(route.RouteError):
        step()  # the plan is closed


def test_host_step_results_visible_on_return_many_steps():
    """route_host_step_run returns on the step's completion word, not on the
    stream: 400 steps alternating two inputs, each step's results checked in
    the host buffers right after the call returns."""
    rows = 8
    _, wl, wr = bank("decode_r8", 0)
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    hs = [np.ascontiguousarray(np.resize(bank("decode_r8", b)[0], (rows, route.K_HIDDEN)))
          for b in (0, 1)]
    with route.Plan(route.DECODE, rows) as plan:
        want = [run_step(plan, to_dev_bf16(h), dwl, dwr) for h in hs]
        h_host = [torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
                  for h in hs]
        buf = torch.empty((rows, route.K_HIDDEN), dtype=torch.bfloat16).pin_memory()
        lat = torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16).pin_memory()
        lg = torch.empty((rows, route.N_EXPERTS), dtype=torch.float32).pin_memory()
        ids = torch.empty((rows, route.TOPK), dtype=torch.int32).pin_memory()
        w = torch.empty((rows, route.TOPK), dtype=torch.float32).pin_memory()
        step = route.HostStep(plan, buf, dwl, dwr, lat, lg, ids, w)
        assert step.graph
        for i in range(400):
            b = i % 2
            buf.copy_(h_host[b])
            lat.view(torch.int16).fill_(-1)
            ids.fill_(-1)
            step()
            assert np.array_equal(ids.numpy(), want[b][2]), f"step {i}"
            assert np.array_equal(w.numpy().view(np.uint32), want[b][3].view(np.uint32)), f"step {i}"
            assert np.array_equal(lat.view(torch.int16).numpy().view(np.uint16), want[b][0]), \
                f"step {i}"
        route.route_device_status(plan)
        step.close()


@pytest.mark.parametrize("depth,rows", [(2, 8), (3, 8), (3, 20), (2, 1)])
def test_host_steps_in_flight_on_one_plan(depth, rows):
    """`depth` HostSteps of one plan on one stream, pipelined: step A is
    launched, then B (and C) are filled and launched before A is waited for,
    and so on for 300 steps over five inputs (so that a step's next input
    differs from its last); each wait is followed by a check of that step's
    host buffers against route_step's bits for its input.  Also: a wait with
    nothing in flight returns at once; after two launches and one wait the
    next launch and wait give that launch's results; a graph call of B behind
    a direct launch of A gives both steps' results.  At 20 rows the staging
    kernel publishes from seven CTAs and the stream kernel takes 32-row MMAs."""
    _, wl, wr = bank("decode_r8", 0)
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    hs = [np.ascontiguousarray(np.resize(bank("decode_r8", b)[0], (rows, route.K_HIDDEN)))
          for b in range(5)]
    s = torch.cuda.Stream()

    def host_bufs():
        return (torch.empty((rows, route.K_HIDDEN), dtype=torch.bfloat16).pin_memory(),
                torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16).pin_memory(),
                torch.empty((rows, route.N_EXPERTS), dtype=torch.float32).pin_memory(),
                torch.empty((rows, route.TOPK), dtype=torch.int32).pin_memory(),
                torch.empty((rows, route.TOPK), dtype=torch.float32).pin_memory())

    def check(b, got, i):
        h, lat, lg, ids, w = got
        assert np.array_equal(ids.numpy(), want[b][2]), f"step {i}"
        assert np.array_equal(w.numpy().view(np.uint32), want[b][3].view(np.uint32)), f"step {i}"
        assert np.array_equal(lg.numpy().view(np.uint32), want[b][1].view(np.uint32)), f"step {i}"
        assert np.array_equal(lat.view(torch.int16).numpy().view(np.uint16), want[b][0]), \
            f"step {i}"

    with route.Plan(route.DECODE, rows) as plan:
        want = [run_step(plan, to_dev_bf16(h), dwl, dwr) for h in hs]
        src = [torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16) for h in hs]
        bufs = [host_bufs() for _ in range(depth)]
        steps = [route.HostStep(plan, b[0], dwl, dwr, *b[1:], stream=s) for b in bufs]
        assert all(st.graph for st in steps)
        steps[0].wait()  # nothing in flight

        def fill_and_launch(j, i):
            h, lat, lg, ids, w = bufs[j]
            h.copy_(src[i % 5])
            lat.view(torch.int16).fill_(-1)
            lg.fill_(float("nan"))
            ids.fill_(-1)
            w.fill_(float("nan"))
            steps[j].launch()

        n = 300
        for i in range(depth - 1):
            fill_and_launch(i, i)
        for i in range(n):
            if i + depth - 1 < n:
                fill_and_launch((i + depth - 1) % depth, i + depth - 1)
            steps[i % depth].wait()
            check(i % 5, bufs[i % depth], i)
        # two launches, one wait: the second launch's input
        bufs[0][0].copy_(src[1])
        steps[0].launch()
        steps[0].wait()
        bufs[0][0].copy_(src[2])
        bufs[0][3].fill_(-1)
        steps[0].launch()
        steps[0].launch()
        steps[0].wait()
        check(2, bufs[0], n)
        fill_and_launch(0, 3)  # the counts stay in step: the next wait is this launch's
        steps[0].wait()
        check(3, bufs[0], n + 1)
        # a direct launch of A, then B as one graph call, then A's wait
        fill_and_launch(0, 1)
        bufs[1][0].copy_(src[2])
        bufs[1][3].fill_(-1)
        steps[1]()
        check(2, bufs[1], n + 2)
        steps[0].wait()
        check(1, bufs[0], n + 3)
        route.route_device_status(plan)
        for st in steps:
            st.close()


def test_host_step_keeps_the_ksplit_setting_of_its_creation():
    """A HostStep created while the plan computes the K-split latent keeps
    that arithmetic after the plan is switched back, in both launch forms
    (the graph call and the direct launch), and a step created afterwards
    gives the full-K bits: each equal to route_step's under the same setting."""
    rows = 8
    _, wl, wr = bank("decode_r8", 0)
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    h = np.ascontiguousarray(np.resize(bank("decode_r8", 2)[0], (rows, route.K_HIDDEN)))
    dh = to_dev_bf16(h)

    def host_bufs():
        return (torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).pin_memory(),
                torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16).pin_memory(),
                torch.empty((rows, route.N_EXPERTS), dtype=torch.float32).pin_memory(),
                torch.empty((rows, route.TOPK), dtype=torch.int32).pin_memory(),
                torch.empty((rows, route.TOPK), dtype=torch.float32).pin_memory())

    def same(bufs, want):
        return (np.array_equal(bufs[1].view(torch.int16).numpy().view(np.uint16), want[0]) and
                np.array_equal(bufs[2].numpy().view(np.uint32), want[1].view(np.uint32)) and
                np.array_equal(bufs[3].numpy(), want[2]) and
                np.array_equal(bufs[4].numpy().view(np.uint32), want[3].view(np.uint32)))

    with route.Plan(route.DECODE, rows) as plan:
        full = run_step(plan, dh, dwl, dwr)
        route.route_set_latent_ksplit(plan, True)
        ks = run_step(plan, dh, dwl, dwr)
        assert not np.array_equal(full[0], ks[0])  # the two arithmetics differ here
        ba = host_bufs()
        a = route.HostStep(plan, ba[0], dwl, dwr, *ba[1:])
        route.route_set_latent_ksplit(plan, False)
        bb = host_bufs()
        b = route.HostStep(plan, bb[0], dwl, dwr, *bb[1:])
        a()
        assert same(ba, ks)
        ba[1].view(torch.int16).fill_(-1)
        a.launch()
        a.wait()
        assert same(ba, ks)
        b.launch()
        b.wait()
        assert same(bb, full)
        b()
        assert same(bb, full)
        route.route_device_status(plan)
        a.close()
        b.close()


def test_host_steps_on_two_streams_are_not_in_flight_together():
    """Two HostSteps of one plan created with different streams would share the
    plan's scratch unordered: while one has a launch in flight the other's
    launch and call are refused (nothing launched), and once it is waited for
    the other runs and gives route_step's bits."""
    rows = 8
    _, wl, wr = bank("decode_r8", 0)
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    h = np.ascontiguousarray(np.resize(bank("decode_r8", 3)[0], (rows, route.K_HIDDEN)))
    with route.Plan(route.DECODE, rows) as plan:
        want = run_step(plan, to_dev_bf16(h), dwl, dwr)

        def make(stream):
            bufs = (torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).pin_memory(),
                    torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16).pin_memory(),
                    torch.empty((rows, route.N_EXPERTS), dtype=torch.float32).pin_memory(),
                    torch.empty((rows, route.TOPK), dtype=torch.int32).pin_memory(),
                    torch.empty((rows, route.TOPK), dtype=torch.float32).pin_memory())
            return bufs, route.HostStep(plan, bufs[0], dwl, dwr, *bufs[1:], stream=stream)

        sa = torch.cuda.Stream()
        (ba, a), (bb, b) = make(sa), make(torch.cuda.Stream())
        assert a.graph and b.graph
        with torch.cuda.stream(sa):
            torch.cuda._sleep(20_000_000)  # A's launch stays in flight behind ~10 ms of spin
        a.launch()
        with pytest.raises(route.RouteError) as e1:
            b.launch()
        with pytest.raises(route.RouteError) as e2:
            b()
        assert e1.value.status == e2.value.status == 7  # ROUTE_ERR_PLAN
        a.wait()
        b.launch()
        b.wait()
        for bufs in (ba, bb):
            assert np.array_equal(bufs[1].view(torch.int16).numpy().view(np.uint16), want[0])
            assert np.array_equal(bufs[3].numpy(), want[2])
            assert np.array_equal(bufs[4].numpy().view(np.uint32), want[3].view(np.uint32))
        route.route_device_status(plan)
        a.close()
        b.close()


@pytest.mark.parametrize("mode,rows,pinned", [(route.DECODE, 8, False), (route.PREFILL, 40, True)])
def test_host_step_without_graph_runs_route_step_host(mode, rows, pinned):
    """Pageable buffers, or a prefill plan: HostStep calls route_step_host."""
    hid, wl, wr = bank("decode_r8" if mode == route.DECODE else "prefill_r1024", 0)
    hid = np.ascontiguousarray(np.resize(hid, (rows, hid.shape[1])))
    dwl, dwr = to_dev_bf16(wl), to_dev_bf16(wr)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    with route.Plan(mode, rows) as plan:
        dev = run_step(plan, to_dev_bf16(hid), dwl, dwr)
        h_host = pin(torch.from_numpy(hid.view(np.int16).copy()).view(torch.bfloat16))
        lat = pin(torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16))
        lg = pin(torch.empty((rows, route.N_EXPERTS), dtype=torch.float32))
        ids = pin(torch.empty((rows, route.TOPK), dtype=torch.int32))
        w = pin(torch.empty((rows, route.TOPK), dtype=torch.float32))
        step = route.HostStep(plan, h_host, dwl, dwr, lat, lg, ids, w)
        assert not step.graph
        step()
        route.route_device_status(plan)
    assert np.array_equal(lat.view(torch.int16).numpy().view(np.uint16), dev[0])
    assert np.array_equal(lg.numpy().view(np.uint32), dev[1].view(np.uint32))
    assert np.array_equal(ids.numpy(), dev[2])
    assert np.array_equal(w.numpy().view(np.uint32), dev[3].view(np.uint32))


def test_gpu_argument_errors():
    lib = route.lib()
    import ctypes
    with route.Plan(route.DECODE, 4) as plan:
        buf = torch.zeros(1 << 22, dtype=torch.uint8, device=DEV)
        base = buf.data_ptr()
        ok = ctypes.c_void_p(base)
        odd = ctypes.c_void_p(base + 2)
        assert lib.latent_router_forward(plan.handle, odd, ok, ok, ok, ok, None) == 4
        assert lib.topk16_select(plan.handle, ok, odd, ok, None) == 4
        assert lib.latent_router_forward(plan.handle, None, ok, ok, ok, ok, None) == 3
    with pytest.raises(route.RouteError):
        route.Plan(route.DECODE, 4, device=torch.cuda.device_count())
    # shape and dtype are checked by the binding before the C call
    with route.Plan(route.DECODE, 2) as plan:
        lat, lg, ids, w = outputs(2)
        bad = torch.zeros((3, route.K_HIDDEN), dtype=torch.bfloat16, device=DEV)
        with pytest.raises(ValueError):
            route.latent_router_forward(plan, bad, bad, bad, lat, lg)
