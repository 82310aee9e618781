"""Route-step oracle (TEST INFRASTRUCTURE ONLY).

A plain single-threaded C definition of the MoE route step, in float64 where
the pages leave the precision open, wrapped with ctypes.  Only the tests, the
smoke check and the benchmark's CPU-baseline leg may import this package; the
product library never calls it and shares no code with it.

What each function follows (page title, section):

* ``latent_router`` -- "Optionally gather the Kimi3 prefill latent instead of
  reducing it", Description, Numerics and Compile bullets: one FP32-accumulated
  full-K dot product per latent value, rounded once to BF16 (K = 7168, 3584
  latent columns); "Use two row blocks for eight-row Kimi paired gathers",
  body: FP32 router logits over 56 x 16 = 896 experts.
* ``latent_ksplit`` -- the first page's commit body: the general path's BF16
  partials, FP32 sum and second BF16 rounding.
* ``topk`` -- "Kimi K3.1 recipe: route 9..20 decode rows through the pushed
  pair gather and standalone top-16", commit message: the standalone top-16
  and its routing weights.
* ``latent_sumsq`` -- the first page's Reviewer Notes: the FP32 sum of squares
  per row that the latent norm needs.

Readings where the pages are silent are stated in ``route_oracle.c``.
Every function is pinned by tests in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "route_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

K_HIDDEN = 7168
N_LATENT = 3584
N_EXPERTS = 896
TOPK = 16

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``route_oracle.c`` with gcc into ``oracle/_build/liboracle.so``.

    ``-ffp-contract=off`` keeps every multiply and add separately rounded on
    both x86-64 and aarch64 (no fused multiply-add contraction)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int32)
            c_int = ctypes.c_int
            lib.oracle_dot64.argtypes = [u16p, u16p, c_int, c_int, c_int, f64p]
            lib.oracle_latent_router.argtypes = [u16p, u16p, u16p, c_int, c_int, c_int,
                                                 c_int, u16p, f32p, f64p, f64p]
            lib.oracle_latent_ksplit.argtypes = [u16p, u16p, c_int, c_int, c_int, c_int, u16p]
            lib.oracle_topk.argtypes = [f32p, c_int, c_int, c_int, i32p, f32p]
            lib.oracle_latent_sumsq.argtypes = [u16p, c_int, c_int, f32p]
            lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_fp32_rne.argtypes = [ctypes.c_double]
            lib.oracle_fp32_rne.restype = ctypes.c_float
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("BF16 operands are passed as uint16 bit patterns")
    return a


def dot64(h_bits, W_bits) -> np.ndarray:
    """float64 ``h @ W`` summed k-ascending, for BF16 bit arrays [R,K], [K,N]."""
    h = _bits(h_bits)
    W = _bits(W_bits)
    R, K = h.shape
    K2, N = W.shape
    assert K == K2
    y = np.empty((R, N), np.float64)
    _load().oracle_dot64(_ptr(h, ctypes.c_uint16), _ptr(W, ctypes.c_uint16), R, K, N,
                         _ptr(y, ctypes.c_double))
    return y


def latent_router(h_bits, Wl_bits, Wr_bits):
    """The route projection of one layer.

    Returns ``(latent_bits uint16 [R,NL], logits float32 [R,NR],
    y_lat float64 [R,NL], y_log float64 [R,NR])``."""
    h = _bits(h_bits)
    Wl = _bits(Wl_bits)
    Wr = _bits(Wr_bits)
    R, K = h.shape
    NL = Wl.shape[1]
    NR = Wr.shape[1]
    assert Wl.shape[0] == K and Wr.shape[0] == K
    latent = np.empty((R, NL), np.uint16)
    logits = np.empty((R, NR), np.float32)
    y_lat = np.empty((R, NL), np.float64)
    y_log = np.empty((R, NR), np.float64)
    _load().oracle_latent_router(
        _ptr(h, ctypes.c_uint16), _ptr(Wl, ctypes.c_uint16), _ptr(Wr, ctypes.c_uint16),
        R, K, NL, NR, _ptr(latent, ctypes.c_uint16), _ptr(logits, ctypes.c_float),
        _ptr(y_lat, ctypes.c_double), _ptr(y_log, ctypes.c_double))
    return latent, logits, y_lat, y_log


def latent_ksplit(h_bits, W_bits, shards: int = 8) -> np.ndarray:
    """General-path latent: ``shards`` BF16-rounded K-slice partials, FP32 sum,
    BF16 again.  Returns uint16 bits [R, N]."""
    h = _bits(h_bits)
    W = _bits(W_bits)
    R, K = h.shape
    N = W.shape[1]
    if K % shards:
        raise ValueError("K must divide into equal shards")
    out = np.empty((R, N), np.uint16)
    _load().oracle_latent_ksplit(_ptr(h, ctypes.c_uint16), _ptr(W, ctypes.c_uint16),
                                 R, K, N, shards, _ptr(out, ctypes.c_uint16))
    return out


def topk(logits, k: int = TOPK):
    """Top-k ids (rank order, lower id on equal logits) and routing weights."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    R, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("k out of range")
    ids = np.empty((R, k), np.int32)
    w = np.empty((R, k), np.float32)
    _load().oracle_topk(_ptr(lg, ctypes.c_float), R, E, k, _ptr(ids, ctypes.c_int32),
                        _ptr(w, ctypes.c_float))
    return ids, w


def latent_sumsq(latent_bits) -> np.ndarray:
    """Per-row sum of squares of BF16 latent values [R, N]: float64 sum,
    rounded once to FP32.  Returns float32 [R]."""
    lat = _bits(latent_bits)
    R, N = lat.shape
    out = np.empty(R, np.float32)
    _load().oracle_latent_sumsq(_ptr(lat, ctypes.c_uint16), R, N, _ptr(out, ctypes.c_float))
    return out


def bf16_rne(x) -> np.ndarray:
    """Element-wise FP32 -> BF16 bits with the oracle's rounding."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    flat_in = x.reshape(-1)
    flat_out = out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.oracle_bf16_rne(float(flat_in[i]))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def fp32_rne(x: float) -> float:
    return float(_load().oracle_fp32_rne(float(x)))
