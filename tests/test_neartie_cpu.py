"""The near-tie construction used by the 9..20-row sweep: it lands the gap
between ranks 16 and 17 inside the stated FP32-ULP window, keeps both experts
at ranks 16/17, and the oracle then picks per its tie rule."""

import numpy as np

import neartie
import oracle
import synth
from gates import ulp_f32


def test_near_tie_rows_land_in_their_window():
    wk = synth.WORKLOADS["decode_sweep"]
    hid = wk.hidden(0, 20)
    _, wr = synth.weight_bank(wk.seed, 0)
    h2, done = neartie.inject(hid, wr)
    assert [d[0] for d in done] == [3, 7, 11, 15, 19]
    untouched = [r for r in range(20) if r % 4 != 3]
    assert np.array_equal(h2[untouched], hid[untouched])
    y = oracle.dot64(h2, wr)
    for i, (r, a, b, gap) in enumerate(done):
        g = (y[r, a] - y[r, b]) / float(ulp_f32(y[r, a]))
        assert (0 < g <= 1) if i % 2 == 0 else (1 < g <= 2)
        order = np.lexsort((np.arange(896), -y[r]))
        assert order[15] == a and order[16] == b
        # in FP32 the two logits are within 2 ULP; the oracle ranks them by
        # value, then by the lower id
        lg = y[r].astype(np.float32)
        assert abs(float(lg[a]) - float(lg[b])) <= 2 * float(ulp_f32(lg[a]))
        ids, _ = oracle.topk(lg[None, :])
        if lg[a] == lg[b]:
            assert ids[0][15] == min(a, b)
        else:
            assert ids[0][15] == a
