"""Pins for the oracle: each test checks the oracle against something other
than itself -- exact rational arithmetic, library conversions, closed forms,
hand-computed rows, brute force and invariants -- so that a dropped term, a
wrong sign or index, a transposed operand or a wrong rounding fails one."""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth


def torch_bf16_bits(x) -> np.ndarray:
    """Library FP32 -> BF16 (round to nearest even) as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_f32(u32) -> np.ndarray:
    return np.asarray(u32, dtype=np.uint32).view(np.float32)


def ulp32(x: float) -> float:
    x = abs(np.float32(x))
    return float(np.spacing(x))


# --------------------------------------------------------------------------
# rounding primitives


def test_bf16_rne_matches_library_on_ties_and_edges():
    rng = np.random.default_rng(7)
    upper = rng.integers(0, 1 << 16, size=4000, dtype=np.uint32)
    lower = np.concatenate([
        np.full(1000, 0x8000, np.uint32),                 # exact ties
        np.full(1000, 0x7FFF, np.uint32),                 # just below a tie
        np.full(1000, 0x8001, np.uint32),                 # just above a tie
        rng.integers(0, 1 << 16, size=1000, dtype=np.uint32),
    ])
    pats = (upper << 16) | lower
    extra = np.array([0x00000000, 0x80000000, 0x7F7FFFFF, 0x7F7F8000, 0xFF7F8000,
                      0x7F800000, 0xFF800000, 0x00008000, 0x00018000, 0x00400000,
                      0x3F808000, 0x3F818000], np.uint32)
    pats = np.concatenate([pats, extra])
    x = bits_f32(pats)
    finite = ~np.isnan(x)
    got = oracle.bf16_rne(x[finite])
    want = torch_bf16_bits(x[finite])
    assert np.array_equal(got, want)
    nan_in = bits_f32(np.array([0x7FC00000, 0xFFC00001, 0x7F800001, 0x7FFFFFFF], np.uint32))
    back = (oracle.bf16_rne(nan_in).astype(np.uint32) << 16).view(np.float32)
    assert np.isnan(back).all()


def test_fp32_rne_matches_library():
    rng = np.random.default_rng(3)
    vals = rng.standard_normal(2000) * np.exp2(rng.integers(-30, 30, 2000))
    for v in vals:
        assert oracle.fp32_rne(v) == float(np.float32(v))
    # a double exactly halfway between two floats rounds to the even one
    one_plus_half_ulp = 1.0 + 2.0 ** -24
    assert oracle.fp32_rne(one_plus_half_ulp) == 1.0
    three_half = 1.0 + 3 * 2.0 ** -24
    assert oracle.fp32_rne(three_half) == float(np.float32(1.0 + 2 * 2.0 ** -23))


# --------------------------------------------------------------------------
# the projection (pins P1-P3 and the accuracy statements)


@pytest.mark.parametrize("K", [1, 4, 64, 257])
def test_dot_against_exact_rationals(K):
    """P1: brute force against exact rational sums on tiny shapes."""
    R, N = 3, 8
    h = synth.normal_bf16(11, K, 0, (R, K), 1.0)
    W = synth.normal_bf16(11, K, 1, (K, N), 1.0 / math.sqrt(K))
    hv = oracle.bf16_to_f64(h)
    Wv = oracle.bf16_to_f64(W)
    latent, logits, y_lat, _ = oracle.latent_router(h, W, W)
    exact_hits = 0
    for r in range(R):
        for n in range(N):
            terms = [Fraction(hv[r, k]) * Fraction(Wv[k, n]) for k in range(K)]
            exact = sum(terms, Fraction(0))
            bound = K * 2.0 ** -53 * float(sum(abs(t) for t in terms))
            assert abs(Fraction(y_lat[r, n]) - exact) <= Fraction(bound)
            if Fraction(float(exact)) == exact:
                exact_hits += 1
                assert y_lat[r, n] == float(exact)
                f32 = np.float32(float(exact))
                assert logits[r, n] == f32
                assert latent[r, n] == torch_bf16_bits(np.array([f32]))[0]
    assert exact_hits >= R * N - 2


def test_one_hot_rows_full_size():
    """P2: h = 2^j e_k picks row k of both weights, scaled exactly."""
    wl, wr = synth.weight_bank(5, 0)
    K = wl.shape[0]
    cases = [(0, 0), (4321, 3), (K - 1, -5)]
    h = np.zeros((len(cases), K), np.uint16)
    for i, (k, j) in enumerate(cases):
        h[i, k] = torch_bf16_bits(np.array([2.0 ** j]))[0]
    latent, logits, _, _ = oracle.latent_router(h, wl, wr)
    for i, (k, j) in enumerate(cases):
        want_l = torch_bf16_bits(oracle.bf16_to_f64(wl[k]).astype(np.float32) * np.float32(2.0 ** j))
        assert np.array_equal(latent[i], want_l)
        want_r = (oracle.bf16_to_f64(wr[k]) * 2.0 ** j).astype(np.float32)
        assert np.array_equal(logits[i], want_r)


def test_small_integer_rows_exact():
    """P3: integer operands give exact integer sums (library int64 matmul)."""
    rng = np.random.default_rng(5)
    R, K, N = 4, 64, 16
    hi = rng.integers(-4, 5, size=(R, K))
    wi = rng.integers(-4, 5, size=(K, N))
    h = torch_bf16_bits(hi.astype(np.float32))
    W = torch_bf16_bits(wi.astype(np.float32))
    latent, logits, y, _ = oracle.latent_router(h, W, W)
    exact = hi @ wi
    assert np.array_equal(y, exact.astype(np.float64))
    assert np.array_equal(logits, exact.astype(np.float32))
    assert np.array_equal(latent, torch_bf16_bits(exact.astype(np.float32)))


def test_hand_computed_row():
    """A row small enough to do by hand.

    h = [1, 2, -3], W = [[1, 0.5], [2, 1], [-1, 4]]:
    y0 = 1*1 + 2*2 + (-3)*(-1) = 8 ; y1 = 0.5 + 2 - 12 = -9.5.
    BF16 keeps both exactly; a third column 1/3-ish value tests rounding:
    W[:,2] = [0.333984375, 0, 0] (BF16 of 1/3) -> y2 = 0.333984375 exactly."""
    h = torch_bf16_bits(np.array([[1.0, 2.0, -3.0]]))
    W = torch_bf16_bits(np.array([[1.0, 0.5, 1 / 3], [2.0, 1.0, 0.0], [-1.0, 4.0, 0.0]]))
    latent, logits, y, _ = oracle.latent_router(h, W, W)
    assert list(y[0]) == [8.0, -9.5, 0.333984375]
    assert list(logits[0]) == [8.0, -9.5, 0.333984375]
    assert list(latent[0]) == [0x4100, 0xC118, 0x3EAB]


def test_transposed_operand_would_fail():
    """A non-square weight with distinct rows and columns: swapping the roles of
    k and n (a transposed operand) cannot give this result."""
    h = torch_bf16_bits(np.array([[1.0, 0.0]]))
    W = torch_bf16_bits(np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]]))
    _, logits, _, _ = oracle.latent_router(h, W, W)
    assert list(logits[0]) == [1.0, 2.0, 3.0]


def test_dot_within_double_bound_of_library_matmul():
    """The float64 sums agree with numpy's float64 matmul (a different
    summation order) within the float64 error bound of either."""
    wl, wr = synth.weight_bank(1, 0)
    h = synth.hidden(1, 0, 2)
    y = oracle.dot64(h, wr)
    hv = oracle.bf16_to_f64(h)
    wv = oracle.bf16_to_f64(wr)
    ref = hv @ wv
    bound = 2 * 7168 * 2.0 ** -53 * (np.abs(hv) @ np.abs(wv))
    assert np.all(np.abs(y - ref) <= bound)


@pytest.mark.slow
def test_full_k_more_accurate_than_k_split(figures):
    """P8/P9: the one-rounding full-K latent is closer to float64 than the
    general path's eight BF16-rounded K-slice partials, and its error is the
    BF16 rounding alone (relative RMS between 1e-3 and the 2e-3 bar)."""
    wl, _ = synth.weight_bank(1, 0)
    h = synth.hidden(1, 0, 3)
    y = oracle.dot64(h, wl)
    full = oracle.latent_router(h, wl, wl[:, :8])[0]
    split = oracle.latent_ksplit(h, wl, figures["k_slices_general_path"])

    def rel_rms(bits):
        d = oracle.bf16_to_f64(bits) - y
        return math.sqrt(float((d * d).sum() / (y * y).sum()))

    r_full, r_split = rel_rms(full), rel_rms(split)
    assert 1e-3 < r_full < 2e-3
    assert r_split > 1.2 * r_full


@pytest.mark.slow
def test_cancel_group_full_k_error_much_smaller():
    """On cancelling partial sums the K-split error dwarfs the full-K error
    (the pages report 0.025x); here checked for direction and a 5x margin."""
    w = synth.WORKLOADS["prefill_r1024"]
    hid = w.hidden(0, 4)
    wl, _ = synth.weight_bank(w.seed, 0)
    wl = np.ascontiguousarray(wl[:, :448])
    synth.apply_cancel_group(wl, hid)
    y = oracle.dot64(hid, wl)
    full = oracle.latent_router(hid, wl, wl[:, :8])[0]
    split = oracle.latent_ksplit(hid, wl, 8)
    idx = np.arange(4)  # columns n with n mod rows == r see cancellation on row r
    cols = [np.arange(r, 448, 4) for r in idx]
    e_full = np.concatenate([oracle.bf16_to_f64(full[r, c]) - y[r, c] for r, c in zip(idx, cols)])
    e_split = np.concatenate([oracle.bf16_to_f64(split[r, c]) - y[r, c] for r, c in zip(idx, cols)])
    assert np.sqrt((e_split ** 2).mean()) > 5 * np.sqrt((e_full ** 2).mean())


# --------------------------------------------------------------------------
# top-16 and routing weights (pins P4-P7)


def brute_topk(row, k):
    """k passes of 'largest value, lowest id on equal values, NaN last'."""
    taken = set()
    out = []
    for _ in range(k):
        best = None
        for e, v in enumerate(row):
            if e in taken:
                continue
            if best is None:
                best = e
                continue
            bv = row[best]
            if math.isnan(bv) and not math.isnan(v):
                best = e
            elif not math.isnan(bv) and not math.isnan(v) and v > bv:
                best = e
        taken.add(best)
        out.append(best)
    return out


def test_topk_special_cases(figures):
    k = figures["top_k"]
    E = 896
    ids, w = oracle.topk(-np.arange(E, dtype=np.float32)[None, :])
    assert list(ids[0]) == list(range(k))
    ids, _ = oracle.topk(np.arange(E, dtype=np.float32)[None, :])
    assert list(ids[0]) == list(range(E - 1, E - 1 - k, -1))
    ids, w = oracle.topk(np.full((1, E), 0.75, np.float32))
    assert list(ids[0]) == list(range(k))
    assert np.all(np.abs(w[0] - 1 / 16) <= figures["weight_ulp_bound"] * ulp32(1 / 16))
    # +0 / -0 are equal values: ties go to the lower id
    row = np.full(E, -1.0, np.float32)
    row[[5, 9, 100, 300]] = [-0.0, 0.0, -0.0, 0.0]
    ids, _ = oracle.topk(row[None, :])
    assert list(ids[0][:4]) == [5, 9, 100, 300]
    # exact duplicates straddling ranks 16/17 keep the lower id
    row = -np.arange(E, dtype=np.float32) - 10
    row[:15] = 5.0 + np.arange(15, 0, -1)
    row[[700, 40, 41]] = 1.5
    ids, _ = oracle.topk(row[None, :])
    assert ids[0][15] == 40
    # NaN ranks below every number, -Inf included
    row = -np.arange(E, dtype=np.float32)
    row[0] = np.nan
    row[1] = -np.inf
    ids, _ = oracle.topk(row[None, :])
    assert list(ids[0]) == list(range(2, 18))
    row = np.full(E, np.nan, np.float32)
    row[[3, 7]] = [-np.inf, 2.0]
    ids, w = oracle.topk(row[None, :])
    assert list(ids[0][:3]) == [7, 3, 0] and np.isnan(w[0]).all()


@pytest.mark.parametrize("E,k", [(20, 5), (896, 16)])
def test_topk_matches_brute_force(E, k):
    """P5: many exact ties (values quantised to a coarse grid) and +-0."""
    rng = np.random.default_rng(E)
    logits = (np.round(rng.standard_normal((40, E)) * 4) / 4).astype(np.float32)
    logits[logits == 0] = np.where(rng.random((logits == 0).sum()) < 0.5, -0.0, 0.0)
    ids, _ = oracle.topk(logits, k)
    for r in range(logits.shape[0]):
        assert list(ids[r]) == brute_topk([float(v) for v in logits[r]], k)


def test_weight_closed_forms(figures):
    """P6: sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4, sigmoid(0) = 1/2; with
    all 16 of 16 experts picked the weights are s_i / sum(s)."""
    ln3 = np.float32(math.log(3.0))
    row = np.zeros(16, np.float32)
    row[0], row[1] = ln3, -ln3
    ids, w = oracle.topk(row[None, :], 16)
    by_id = dict(zip(ids[0].tolist(), w[0].tolist()))
    tol = 2
    assert abs(by_id[0] - 3 / 32) <= tol * ulp32(3 / 32)
    assert abs(by_id[1] - 1 / 32) <= tol * ulp32(1 / 32)
    for e in range(2, 16):
        assert abs(by_id[e] - 1 / 16) <= tol * ulp32(1 / 16)
    # symmetry: s(x) + s(-x) = 1, so paired weights sum to 1/8
    rng = np.random.default_rng(2)
    x = rng.uniform(0.1, 6.0, 8).astype(np.float32)
    row = np.concatenate([x, -x])
    ids, w = oracle.topk(row[None, :], 16)
    by_id = dict(zip(ids[0].tolist(), w[0].tolist()))
    for i in range(8):
        assert abs(by_id[i] + by_id[i + 8] - 0.125) <= 4 * ulp32(0.125)
    # the larger logit gets the larger weight; weights sum to 1
    logits = rng.standard_normal((50, 896)).astype(np.float32) * 2
    ids, w = oracle.topk(logits)
    assert np.all(np.diff(w, axis=1) <= 0)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 16 * ulp32(1.0))


def test_topk_permutation_invariance():
    """P7: relabelling experts relabels the picks and keeps the weights."""
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((30, 896)).astype(np.float32)
    perm = rng.permutation(896)
    inv = np.argsort(perm)
    ids, w = oracle.topk(logits)
    ids_p, w_p = oracle.topk(logits[:, perm])
    assert np.array_equal(ids_p, inv[ids])
    assert np.array_equal(w_p, w)


# --------------------------------------------------------------------------
# latent sum of squares ("Optionally gather the Kimi3 prefill latent instead
# of reducing it", Reviewer Notes: an FP32 sum of squares per row for the
# latent norm)

def _f32_nearest_even(q: Fraction) -> np.float32:
    """The FP32 value nearest to the rational q, ties to the even significand
    (exact: candidates around a double approximation, compared as rationals)."""
    c = np.float32(float(q))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = min(cands, key=lambda x: (abs(Fraction(float(x)) - q),
                                     int(np.asarray(x).view(np.uint32)) & 1))
    return np.float32(best)


def test_sumsq_closed_forms():
    N = oracle.N_LATENT
    rows = np.stack([
        np.ones(N, np.float32),
        np.full(N, 2.0, np.float32),
        np.where(np.arange(N) % 2 == 0, 1.5, -1.5).astype(np.float32),
        np.zeros(N, np.float32),
        np.where(np.arange(N) == 7, -3.0, 0.0).astype(np.float32),
    ])
    got = oracle.latent_sumsq(torch_bf16_bits(rows))
    assert got.tolist() == [N, 4.0 * N, 2.25 * N, 0.0, 9.0]


def test_sumsq_rounds_once():
    # 1.0 followed by 3583 values of 2^-12 (squares 2^-24, half an FP32 ulp
    # of 1): a running FP32 sum never moves off 1.0; the exact sum does.
    N = oracle.N_LATENT
    row = np.full((1, N), 2.0 ** -12, np.float32)
    row[0, 0] = 1.0
    got = oracle.latent_sumsq(torch_bf16_bits(row))[0]
    want = _f32_nearest_even(1 + Fraction(N - 1, 2 ** 24))
    assert got == want and got > np.float32(1.0)


@pytest.mark.parametrize("N", [1, 31, 257, 3584])
def test_sumsq_against_exact_rationals(N):
    rng = np.random.default_rng(N)
    vals = (rng.standard_normal((4, N)) * np.exp2(rng.integers(-20, 20, (4, N)))).astype(np.float32)
    bits = torch_bf16_bits(vals)
    got = oracle.latent_sumsq(bits)
    v = bits.astype(np.uint32) << 16
    for r in range(4):
        exact = sum(Fraction(float(x)) ** 2 for x in v[r].view(np.float32))
        assert got[r] == _f32_nearest_even(exact), r


def test_ksplit_hand_computed_slice_boundary():
    """K-split latent on a hand-computed row: slice 0 (k < 896) holds the
    partial 1 + 2^-8 + 2^-10, slice 1 (896 <= k < 1792) the partial -2^-9.
    General path: bf16(1 + 2^-8 + 2^-10) = 1 + 2^-7, plus -2^-9 gives
    1 + 2^-8 + 2^-9, which rounds to 1 + 2^-7.  Full K: the exact sum
    1 + 2^-8 - 2^-10 rounds to 1.  Slices of another width, or partials not
    rounded to BF16, give 1."""
    K, N = 7168, 2
    h = np.zeros((1, K), np.float32)
    h[0, [893, 894, 895, 896]] = 1.0
    W = np.zeros((K, N), np.float32)
    W[893, 0], W[894, 0], W[895, 0], W[896, 0] = 1.0, 2.0 ** -8, 2.0 ** -10, -(2.0 ** -9)
    W[895, 1] = 3.0  # column 1: one product, same in both paths
    hb, Wb = torch_bf16_bits(h), torch_bf16_bits(W)
    split = oracle.bf16_to_f64(oracle.latent_ksplit(hb, Wb, 8))
    full, _, _, _ = oracle.latent_router(hb, Wb, np.zeros((K, 896), np.uint16))
    full = oracle.bf16_to_f64(full)
    assert split[0, 0] == 1.0 + 2.0 ** -7
    assert full[0, 0] == 1.0
    assert split[0, 1] == full[0, 1] == 3.0
