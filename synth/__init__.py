"""Seeded synthetic inputs for the MoE route step.

The pages measure on real Kimi K3.1 weights and serving traffic, which are not
available here; these seeded inputs stand in for them at the pages' shapes
(K = 7168 hidden, 3584 latent columns, 896 experts).  The module holds no part
of the route step's arithmetic: it only draws numbers (``synth.c``) and
arranges them into BF16 bit arrays (``uint16``) that both the oracle and the
CUDA library read.

Workload recipes (one per named workload):

* ``decode_r1``   rows 1, hidden ~ N(0,1), W ~ N(0, 1/7168), seed 0, 1 bank
* ``decode_r8``   rows 8, same distributions, seed 1, 8 banks
* ``decode_sweep`` rows 9/12/16/20, seed 2, 6 banks (near-tie rows are
  injected by the parity tests with the oracle's help)
* ``prefill_r1024`` rows 1024, hidden rows N(0,1) scaled to unit RMS, seed 3,
  1 bank, latent columns 0..447 given cancelling partial sums
* ``prefill_r3072`` rows 3072, as above without the cancel group, seed 4,
  92 banks (one per MoE layer)
"""

from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

K_HIDDEN = 7168
N_LATENT = 3584
N_EXPERTS = 896
W_SIGMA = 1.0 / math.sqrt(K_HIDDEN)

T_HIDDEN, T_LATENT, T_ROUTER = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64 = ctypes.c_uint64
            lib.synth_stream_key.argtypes = [u64, u64, u64]
            lib.synth_stream_key.restype = u64
            lib.synth_draw.argtypes = [u64, u64]
            lib.synth_draw.restype = u64
            lib.synth_normal_bf16.argtypes = [u64, u64, ctypes.c_double,
                                              ctypes.POINTER(ctypes.c_uint16), ctypes.c_int]
            lib.synth_normal_f64.argtypes = [u64, u64, ctypes.c_double,
                                             ctypes.POINTER(ctypes.c_double), ctypes.c_int]
            lib.synth_hidden_rms_bf16.argtypes = [u64, ctypes.c_int, ctypes.c_int,
                                                  ctypes.POINTER(ctypes.c_uint16), ctypes.c_int]
            lib.synth_cancel_group.argtypes = [ctypes.POINTER(ctypes.c_uint16), ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_uint16), ctypes.c_int,
                                               ctypes.c_int]
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _u16p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def stream_key(seed: int, bank: int, tensor: int) -> int:
    return int(_load().synth_stream_key(seed, bank, tensor))


def draw(key: int, i: int) -> int:
    return int(_load().synth_draw(key, i))


def normal_bf16(seed: int, bank: int, tensor: int, shape, sigma: float = 1.0) -> np.ndarray:
    """BF16 bits of sigma * N(0,1), element i of the (seed, bank, tensor) stream
    at flat index i of ``shape``."""
    out = np.empty(shape, np.uint16)
    _load().synth_normal_bf16(stream_key(seed, bank, tensor), out.size, float(sigma),
                              _u16p(out), _threads())
    return out


def normal_f64(seed: int, bank: int, tensor: int, shape, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, np.float64)
    _load().synth_normal_f64(stream_key(seed, bank, tensor), out.size, float(sigma),
                             out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), _threads())
    return out


def hidden(seed: int, bank: int, rows: int, rms_rows: bool = False) -> np.ndarray:
    """Hidden rows [rows, 7168] (BF16 bits).  A prefix of rows is the same for
    any ``rows``."""
    if rms_rows:
        out = np.empty((rows, K_HIDDEN), np.uint16)
        _load().synth_hidden_rms_bf16(stream_key(seed, bank, T_HIDDEN), rows, K_HIDDEN,
                                      _u16p(out), _threads())
        return out
    return normal_bf16(seed, bank, T_HIDDEN, (rows, K_HIDDEN), 1.0)


def weight_bank(seed: int, bank: int):
    """(W_latent [7168, 3584], W_router [7168, 896]) BF16 bits ~ N(0, 1/7168)."""
    wl = normal_bf16(seed, bank, T_LATENT, (K_HIDDEN, N_LATENT), W_SIGMA)
    wr = normal_bf16(seed, bank, T_ROUTER, (K_HIDDEN, N_EXPERTS), W_SIGMA)
    return wl, wr


def apply_cancel_group(W_latent: np.ndarray, hidden_bits: np.ndarray, ncols: int = 448,
                       slice_k: int = 896) -> None:
    """In place: columns < ncols get alternating-sign K-slices matched to the
    signs of hidden row (n mod rows), so that row's slice partials are large
    and cancel (448 columns = one TP8 rank's share of the latent; 896 = one of
    eight K-slices of the general path)."""
    W = W_latent
    assert W.flags.c_contiguous and W.dtype == np.uint16
    h = np.ascontiguousarray(hidden_bits)
    K, N = W.shape
    _load().synth_cancel_group(_u16p(W), K, N, ncols, _u16p(h), h.shape[0], slice_k)


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "decode" or "prefill"
    rows: tuple          # row counts covered by the workload
    seed: int
    banks: int
    rms_rows: bool
    cancel_group: bool
    near_tie: bool

    def hidden(self, bank: int, rows: int) -> np.ndarray:
        return hidden(self.seed, bank, rows, self.rms_rows)

    def bank(self, bank: int, hidden_bits: np.ndarray | None = None):
        wl, wr = weight_bank(self.seed, bank)
        if self.cancel_group:
            if hidden_bits is None:
                hidden_bits = self.hidden(bank, max(self.rows))
            apply_cancel_group(wl, hidden_bits)
        return wl, wr


WORKLOADS = {
    "decode_r1": Workload("decode_r1", "decode", (1,), 0, 1, False, False, False),
    "decode_r8": Workload("decode_r8", "decode", (8,), 1, 8, False, False, False),
    "decode_sweep": Workload("decode_sweep", "decode", (9, 12, 16, 20), 2, 6, False, False, True),
    "prefill_r1024": Workload("prefill_r1024", "prefill", (1024,), 3, 1, True, True, False),
    "prefill_r3072": Workload("prefill_r3072", "prefill", (3072,), 4, 92, True, False, False),
}
