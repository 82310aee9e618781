"""The seeded input generator: determinism, independence from the thread
split, prefix stability and the stated distributions."""

import ctypes
import math

import numpy as np

import synth


def test_same_seed_same_bytes_and_streams_differ():
    a = synth.normal_bf16(1, 0, 1, (64, 448), synth.W_SIGMA)
    b = synth.normal_bf16(1, 0, 1, (64, 448), synth.W_SIGMA)
    c = synth.normal_bf16(1, 1, 1, (64, 448), synth.W_SIGMA)
    d = synth.normal_bf16(2, 0, 1, (64, 448), synth.W_SIGMA)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_thread_split_does_not_change_values():
    lib = synth._load()
    key = synth.stream_key(3, 2, 1)
    n = 300_001
    outs = []
    for threads in (1, 3, 8):
        out = np.empty(n, np.uint16)
        lib.synth_normal_bf16(key, n, 1.0, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                              threads)
        outs.append(out)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_hidden_prefix_rows_are_stable():
    h20 = synth.hidden(2, 1, 20)
    h9 = synth.hidden(2, 1, 9)
    assert np.array_equal(h20[:9], h9)
    r20 = synth.hidden(3, 0, 20, rms_rows=True)
    r5 = synth.hidden(3, 0, 5, rms_rows=True)
    assert np.array_equal(r20[:5], r5)


def _vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_distributions():
    z = synth.normal_f64(0, 0, 9, (400_000,))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs(((z ** 4).mean()) - 3.0) < 0.05  # normal kurtosis
    wl, wr = synth.weight_bank(0, 0)
    for w in (wl, wr):
        v = _vals(w)
        assert abs(v.std() - 1 / math.sqrt(7168)) < 2e-4
    h = _vals(synth.hidden(3, 0, 16, rms_rows=True))
    rms = np.sqrt((h * h).mean(axis=1))
    assert np.all(np.abs(rms - 1.0) < 5e-3)


def test_cancel_group_sets_alternating_signs():
    w = synth.WORKLOADS["prefill_r1024"]
    hid = w.hidden(0, 4)
    wl, _ = synth.weight_bank(w.seed, 0)
    orig = wl.copy()
    synth.apply_cancel_group(wl, hid, ncols=8, slice_k=896)
    assert np.array_equal(wl[:, 8:], orig[:, 8:])
    assert np.array_equal(wl & 0x7FFF, orig & 0x7FFF)
    hv = _vals(hid)
    wv = _vals(wl)
    for n in range(8):
        d = n % 4
        parts = [(hv[d, s * 896:(s + 1) * 896] * wv[s * 896:(s + 1) * 896, n]).sum()
                 for s in range(8)]
        signs = np.sign(parts)
        assert list(signs) == [1, -1, 1, -1, 1, -1, 1, -1]
