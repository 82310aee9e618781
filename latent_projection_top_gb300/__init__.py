"""Python binding of the route library (``libroute``, C ABI in ``include/route.h``).

Argument marshalling only: tensors are checked for dtype, shape, layout and
device, then their pointers and the CUDA stream are passed to the C entry
points of the same names.  Every step of the route computation runs in the
library's CUDA kernels; there is no Python or CPU fallback, and importing the
package fails loudly if the library has not been built (``build()``).

The route step of one MoE layer (see ``include/route.h``):

* ``latent_router_forward`` -- latent down projection (BF16, one FP32 full-K
  sum rounded once) and FP32 router logits;
* ``topk16_select`` -- standalone top-16 with sigmoid-renormalised weights;
* ``route_step`` -- both (for decode plans, a weight-stream kernel and a kernel
  that finishes the split-K sums and runs the top-16);
* ``Step`` -- ``route_step`` on fixed device tensors, checked once (each call
  is one C call: for eager loops whose host time would otherwise exceed a
  decode step's device time);
* ``route_step_sumsq`` -- ``route_step`` plus each latent row's sum of squares;
* ``route_step_host`` -- ``route_step`` with host tensors (transfers included);
  ``HostStep`` -- the same on fixed buffers, checked once and (decode,
  page-locked buffers) captured as a CUDA graph, for serving loops;
* ``route_set_overlap``, ``route_set_latent_ksplit`` -- plan options;
* ``ShardPlan``, ``route_shard_step``, ``route_merge_candidates`` -- one column
  shard of the step (its latent columns, its experts and its local top-16)
  and the merge of the shards' candidates into the final top-16;
  ``gather_candidates`` is the exchange between them (torch.distributed), and
  ``gather_latent_logits`` the paired gather of the shards' latent and logit
  columns into the whole layer's.
"""

from __future__ import annotations

import ctypes
import os

K_HIDDEN = 7168
N_LATENT = 3584
N_EXPERTS = 896
TOPK = 16
DECODE_MAX_ROWS = 20
PREFILL_MAX_ROWS = 65536

DECODE = 0
PREFILL = 1

ROUTE_OK = 0
STATUS_NAMES = {
    0: "ROUTE_OK", 1: "ROUTE_ERR_ROWS", 2: "ROUTE_ERR_MODE", 3: "ROUTE_ERR_NULL",
    4: "ROUTE_ERR_ALIGN", 5: "ROUTE_ERR_CUDA", 6: "ROUTE_ERR_DEVICE_TIMEOUT",
    7: "ROUTE_ERR_PLAN", 8: "ROUTE_ERR_DEVICE", 9: "ROUTE_ERR_DEVICE_BOUNDS",
}
STATUS_CODES = {name: code for code, name in STATUS_NAMES.items()}

_HERE = os.path.dirname(os.path.abspath(__file__))
RELEASE_LIB_PATH = os.path.join(_HERE, "_build", "libroute.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "_build", "debug", "libroute_debug.so")
# ROUTE_DEBUG_LIB=1 selects the checked library (every computed global index
# of the kernels bounds-checked; see builder.py), e.g. for a test process.
LIB_PATH = DEBUG_LIB_PATH if os.environ.get("ROUTE_DEBUG_LIB") == "1" else RELEASE_LIB_PATH

# Every symbol the header declares (checked by the CPU tests).
EXPORTS = (
    "route_prepare", "route_destroy", "latent_router_forward", "topk16_select", "route_step",
    "route_step_host", "route_device_status", "route_plan_rows", "route_plan_mode",
    "route_plan_grid", "route_plan_segments", "route_last_error", "route_test_stall",
    "route_set_overlap", "route_step_decode_noalloc", "route_step_sumsq",
    "route_set_latent_ksplit", "route_host_step_create", "route_host_step_run",
    "route_host_step_launch", "route_host_step_wait", "route_host_step_destroy", "route_test_poison_scratch", "route_noalloc_status",
    "route_noalloc_grid", "route_prepare_shard", "route_shard_step", "route_merge_candidates",
    "route_plan_latent_cols", "route_plan_experts", "route_test_noalloc_stall",
)
SHARD_COUNTS = (1, 2, 4, 7, 8, 14, 16)


class RouteError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


_lib = None


def build(force: bool = False, debug: bool = False, both: bool = False) -> str:
    """Compile the route library (see builder.py): the release one, the checked
    one (debug=True), or both (both=True)."""
    from . import builder as _b
    return _b.build(force=force, debug=debug or LIB_PATH == DEBUG_LIB_PATH, both=both)


def lib() -> ctypes.CDLL:
    """The loaded ``libroute.so``; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RouteError(5, f"{LIB_PATH} is missing: the CUDA library must be built "
                                "(latent_projection_top_gb300.build())")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        L.route_prepare.argtypes = [i32, i32, i32, ctypes.POINTER(vp)]
        L.route_destroy.argtypes = [vp]
        L.latent_router_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp]
        L.topk16_select.argtypes = [vp, vp, vp, vp, vp]
        L.route_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.route_step_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.route_step_sumsq.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.route_device_status.argtypes = [vp]
        L.route_step_decode_noalloc.argtypes = [i32, vp, vp, vp, vp, vp, vp, vp, vp]
        L.route_step_decode_noalloc.restype = i32
        L.route_set_overlap.argtypes = [vp, i32]
        L.route_set_overlap.restype = i32
        L.route_set_latent_ksplit.argtypes = [vp, i32]
        L.route_set_latent_ksplit.restype = i32
        L.route_test_stall.argtypes = [vp, i32, ctypes.c_uint64]
        L.route_test_stall.restype = i32
        L.route_host_step_create.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(vp)]
        L.route_host_step_run.argtypes = [vp]
        L.route_host_step_launch.argtypes = [vp]
        L.route_host_step_wait.argtypes = [vp]
        L.route_host_step_destroy.argtypes = [vp]
        L.route_test_poison_scratch.argtypes = [vp, vp]
        L.route_noalloc_status.argtypes = [i32]
        L.route_noalloc_status.restype = i32
        L.route_noalloc_grid.argtypes = [i32]
        L.route_noalloc_grid.restype = i32
        L.route_prepare_shard.argtypes = [i32, i32, i32, i32, ctypes.POINTER(vp)]
        L.route_prepare_shard.restype = i32
        L.route_shard_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.route_shard_step.restype = i32
        L.route_merge_candidates.argtypes = [i32, i32, vp, vp, vp, vp, vp]
        L.route_merge_candidates.restype = i32
        L.route_test_noalloc_stall.argtypes = [i32, i32, ctypes.c_uint64]
        L.route_test_noalloc_stall.restype = i32
        for f in ("route_host_step_create", "route_host_step_run", "route_host_step_launch",
                  "route_host_step_wait", "route_host_step_destroy", "route_test_poison_scratch"):
            getattr(L, f).restype = i32
        for f in ("route_plan_rows", "route_plan_mode", "route_plan_grid", "route_plan_segments",
                  "route_plan_latent_cols", "route_plan_experts"):
            getattr(L, f).argtypes = [vp]
            getattr(L, f).restype = i32
        L.route_last_error.argtypes = []
        L.route_last_error.restype = ctypes.c_char_p
        for f in ("route_prepare", "route_destroy", "latent_router_forward", "topk16_select",
                  "route_step", "route_step_host", "route_step_sumsq", "route_device_status"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != ROUTE_OK:
        msg = lib().route_last_error().decode(errors="replace")
        raise RouteError(status, msg)


class Plan:
    """A prepared route plan (``route_prepare``): mode, rows, device, launch
    geometry and the plan's scratch memory.  Use as a context manager or call
    ``close()``."""

    def __init__(self, mode: int, rows: int, device: int = 0):
        h = ctypes.c_void_p()
        _check(lib().route_prepare(int(mode), int(rows), int(device), ctypes.byref(h)))
        self._h = h
        self.mode = int(mode)
        self.rows = int(rows)
        self.device = int(device)

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None or not self._h.value:
            raise RouteError(7, "plan is closed")
        return self._h

    @property
    def grid(self) -> int:
        return lib().route_plan_grid(self.handle)

    @property
    def segments(self) -> int:
        return lib().route_plan_segments(self.handle)

    def close(self) -> None:
        if self._h is not None and self._h.value:
            lib().route_destroy(self._h)
            # a HostStep made on this plan shares the handle object: it now
            # passes NULL and gets ROUTE_ERR_NULL instead of a freed plan
            self._h.value = None
        self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def route_prepare(mode: int, rows: int, device: int = 0) -> Plan:
    return Plan(mode, rows, device)


def shard_columns(num_shards: int) -> tuple[int, int]:
    """(latent columns, experts) of each of `num_shards` column shards."""
    return N_LATENT // num_shards, N_EXPERTS // num_shards


class ShardPlan(Plan):
    """A plan for column shard `shard` of `num_shards` (``route_prepare_shard``):
    latent columns [NL shard, NL (shard + 1)) and experts [NE shard, NE (shard
    + 1)), NL, NE = ``shard_columns(num_shards)``."""

    def __init__(self, rows: int, shard: int, num_shards: int, device: int = 0):
        h = ctypes.c_void_p()
        _check(lib().route_prepare_shard(int(rows), int(device), int(shard), int(num_shards),
                                         ctypes.byref(h)))
        self._h = h
        # up to 20 rows the decode weight stream, else the prefill GEMM
        self.mode = DECODE if int(rows) <= DECODE_MAX_ROWS else PREFILL
        self.rows = int(rows)
        self.device = int(device)
        self.shard = int(shard)
        self.num_shards = int(num_shards)
        self.n_latent, self.n_experts = shard_columns(num_shards)


# ---- marshalling helpers ---------------------------------------------------

def _torch():
    import torch
    return torch


def _dev_tensor(t, name, shape, dtypes, device):
    # the common case in one expression (this runs on every call)
    try:
        if (t.is_cuda and t.get_device() == device and t.dtype in dtypes and t.shape == shape
                and t.is_contiguous()):
            return ctypes.c_void_p(t.data_ptr())
    except AttributeError:
        pass
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda" or t.device.index != device:
        raise ValueError(f"{name} must be on cuda:{device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}; expected {tuple(shape)}")
    raise ValueError(f"{name} must be contiguous")


def _host_tensor(t, name, shape, dtypes):
    try:
        if t.is_cpu and t.dtype in dtypes and t.shape == shape and t.is_contiguous():
            return ctypes.c_void_p(t.data_ptr())
    except AttributeError:
        pass
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a CPU torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    raise ValueError(f"{name} must be contiguous with shape {tuple(shape)}")


_BF16_TYPES = None


def _bf16_types():
    global _BF16_TYPES
    if _BF16_TYPES is None:
        torch = _torch()
        _BF16_TYPES = (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") \
            else (torch.bfloat16, torch.int16)
    return _BF16_TYPES


def _stream(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _proj_ptrs(plan, hidden, W_latent, W_router, latent, logits):
    torch = _torch()
    R, d = plan.rows, plan.device
    bf = _bf16_types()
    return (_dev_tensor(hidden, "hidden", (R, K_HIDDEN), bf, d),
            _dev_tensor(W_latent, "W_latent", (K_HIDDEN, N_LATENT), bf, d),
            _dev_tensor(W_router, "W_router", (K_HIDDEN, N_EXPERTS), bf, d),
            _dev_tensor(latent, "latent", (R, N_LATENT), bf, d),
            _dev_tensor(logits, "logits", (R, N_EXPERTS), (torch.float32,), d))


def _topk_ptrs(plan, ids, weights):
    torch = _torch()
    R, d = plan.rows, plan.device
    return (_dev_tensor(ids, "ids", (R, TOPK), (torch.int32,), d),
            _dev_tensor(weights, "weights", (R, TOPK), (torch.float32,), d))


# ---- the C entry points ------------------------------------------------------

def latent_router_forward(plan: Plan, hidden, W_latent, W_router, latent, logits,
                          stream=None) -> None:
    p = _proj_ptrs(plan, hidden, W_latent, W_router, latent, logits)
    _check(lib().latent_router_forward(plan.handle, *p, _stream(stream, plan.device)))


def topk16_select(plan: Plan, logits, ids, weights, stream=None) -> None:
    torch = _torch()
    lg = _dev_tensor(logits, "logits", (plan.rows, N_EXPERTS), (torch.float32,), plan.device)
    i, w = _topk_ptrs(plan, ids, weights)
    _check(lib().topk16_select(plan.handle, lg, i, w, _stream(stream, plan.device)))


def route_step(plan: Plan, hidden, W_latent, W_router, latent, logits, ids, weights,
               stream=None) -> None:
    p = _proj_ptrs(plan, hidden, W_latent, W_router, latent, logits)
    i, w = _topk_ptrs(plan, ids, weights)
    _check(lib().route_step(plan.handle, *p, i, w, _stream(stream, plan.device)))


def route_step_sumsq(plan: Plan, hidden, W_latent, W_router, latent, logits, ids, weights,
                     latent_sumsq, stream=None) -> None:
    """route_step that also writes each latent row's sum of squares (FP32 [rows])."""
    torch = _torch()
    p = _proj_ptrs(plan, hidden, W_latent, W_router, latent, logits)
    i, w = _topk_ptrs(plan, ids, weights)
    ss = _dev_tensor(latent_sumsq, "latent_sumsq", (plan.rows,), (torch.float32,), plan.device)
    _check(lib().route_step_sumsq(plan.handle, *p, i, w, ss, _stream(stream, plan.device)))


def route_shard_step(plan: ShardPlan, hidden, W_latent_shard, W_router_shard, latent_shard,
                     logits_shard, cand_ids, cand_logits, stream=None) -> None:
    """One column shard: its latent columns, its logits and its local top-16
    (global expert ids and their logits)."""
    torch = _torch()
    R, d, NL, NE = plan.rows, plan.device, plan.n_latent, plan.n_experts
    bf = _bf16_types()
    p = (_dev_tensor(hidden, "hidden", (R, K_HIDDEN), bf, d),
         _dev_tensor(W_latent_shard, "W_latent_shard", (K_HIDDEN, NL), bf, d),
         _dev_tensor(W_router_shard, "W_router_shard", (K_HIDDEN, NE), bf, d),
         _dev_tensor(latent_shard, "latent_shard", (R, NL), bf, d),
         _dev_tensor(logits_shard, "logits_shard", (R, NE), (torch.float32,), d),
         _dev_tensor(cand_ids, "cand_ids", (R, TOPK), (torch.int32,), d),
         _dev_tensor(cand_logits, "cand_logits", (R, TOPK), (torch.float32,), d))
    _check(lib().route_shard_step(plan.handle, *p, _stream(stream, d)))


def route_merge_candidates(cand_ids, cand_logits, ids, weights, stream=None) -> None:
    """The top-16 and weights of each row from the shards' candidates
    ([num_shards, rows, 16] ids and logits, shard after shard)."""
    torch = _torch()
    if not isinstance(cand_ids, torch.Tensor) or cand_ids.dim() != 3:
        raise ValueError("cand_ids must be a [num_shards, rows, 16] tensor")
    W, R = int(cand_ids.shape[0]), int(cand_ids.shape[1])
    d = cand_ids.device.index if cand_ids.is_cuda else -1
    p = (_dev_tensor(cand_ids, "cand_ids", (W, R, TOPK), (torch.int32,), d),
         _dev_tensor(cand_logits, "cand_logits", (W, R, TOPK), (torch.float32,), d),
         _dev_tensor(ids, "ids", (R, TOPK), (torch.int32,), d),
         _dev_tensor(weights, "weights", (R, TOPK), (torch.float32,), d))
    with torch.cuda.device(d):
        _check(lib().route_merge_candidates(R, W, *p, _stream(stream, d)))


def gather_candidates(cand_ids, cand_logits, group=None):
    """The exchange step of a column-sharded route step, one shard per rank:
    every rank's [rows, 16] candidate ids and logits all-gathered into the
    [num_shards, rows, 16] layout ``route_merge_candidates`` reads (the block
    of group rank r at index r).  Needs an initialised torch.distributed
    group; device tensors need a GPU backend (NCCL)."""
    torch = _torch()
    import torch.distributed as dist
    W = dist.get_world_size(group)
    out = []
    for t in (cand_ids, cand_logits):
        t = t.contiguous()
        g = torch.empty((W,) + tuple(t.shape), dtype=t.dtype, device=t.device)
        dist.all_gather(list(g.unbind(0)), t, group=group)
        out.append(g)
    return out[0], out[1]


def gather_latent_logits(latent_shard, logits_shard, group=None):
    """The paired gather of a column-sharded step, one shard per rank: every
    rank's [rows, 3584/W] BF16 latent columns and [rows, 896/W] FP32 logit
    columns travel together in one all-gather (one message per rank, the two
    blocks side by side as bytes) and come back as the whole layer's
    [rows, 3584] latent and [rows, 896] logits, shard s at columns s * n ..
    (s + 1) * n.  Layout plumbing around the collective; needs an initialised
    torch.distributed group (NCCL for device tensors)."""
    torch = _torch()
    import torch.distributed as dist
    W = dist.get_world_size(group)
    lat, lg = latent_shard.contiguous(), logits_shard.contiguous()
    R, NL = lat.shape
    NE = lg.shape[1]
    if lg.shape[0] != R or lat.dtype != torch.bfloat16 or lg.dtype != torch.float32:
        raise ValueError("latent_shard [rows, n] BF16 and logits_shard [rows, m] FP32 expected")
    mine = torch.cat([lat.view(torch.uint8), lg.view(torch.uint8)], dim=1)  # [R, 2 NL + 4 NE]
    g = torch.empty((W,) + tuple(mine.shape), dtype=torch.uint8, device=mine.device)
    dist.all_gather(list(g.unbind(0)), mine, group=group)
    latent = g[:, :, :2 * NL].contiguous().view(torch.bfloat16)        # [W, R, NL]
    logits = g[:, :, 2 * NL:].contiguous().view(torch.float32)        # [W, R, NE]
    return (latent.permute(1, 0, 2).reshape(R, W * NL),
            logits.permute(1, 0, 2).reshape(R, W * NE))


def _host_step_args(plan, hidden_host, W_latent, W_router, latent_host, logits_host, ids_host,
                    weights_host):
    torch = _torch()
    R, d = plan.rows, plan.device
    bf = _bf16_types()
    return (_host_tensor(hidden_host, "hidden_host", (R, K_HIDDEN), bf),
            _dev_tensor(W_latent, "W_latent", (K_HIDDEN, N_LATENT), bf, d),
            _dev_tensor(W_router, "W_router", (K_HIDDEN, N_EXPERTS), bf, d),
            _host_tensor(latent_host, "latent_host", (R, N_LATENT), bf),
            _host_tensor(logits_host, "logits_host", (R, N_EXPERTS), (torch.float32,)),
            _host_tensor(ids_host, "ids_host", (R, TOPK), (torch.int32,)),
            _host_tensor(weights_host, "weights_host", (R, TOPK), (torch.float32,)))


def route_step_host(plan: Plan, hidden_host, W_latent, W_router, latent_host, logits_host,
                    ids_host, weights_host, stream=None) -> None:
    args = _host_step_args(plan, hidden_host, W_latent, W_router, latent_host, logits_host,
                           ids_host, weights_host)
    _check(lib().route_step_host(plan.handle, *args, _stream(stream, plan.device)))


class Step:
    """``route_step`` on fixed device tensors, checked once.

    For an eager loop that runs the step on the same buffers every time (new
    values written into ``hidden``, results read from the outputs): the
    tensors are validated and their pointers marshalled here, so each call
    is one C call (the library reuses its tensor maps for unchanged
    addresses).  The object keeps references to the tensors and the plan;
    the caller must not resize them.  Once the plan is closed a call raises.
    """

    def __init__(self, plan: Plan, hidden, W_latent, W_router, latent, logits, ids, weights,
                 stream=None):
        p = _proj_ptrs(plan, hidden, W_latent, W_router, latent, logits)
        i, w = _topk_ptrs(plan, ids, weights)
        self._keep = (plan, hidden, W_latent, W_router, latent, logits, ids, weights, stream)
        self._args = (plan.handle,) + tuple(p) + (i, w, _stream(stream, plan.device))
        self._fn = lib().route_step

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != ROUTE_OK:
            _check(st)


class HostStep:
    """``route_step_host`` on fixed buffers, checked once.

    For a serving loop that refills the same page-locked ``hidden_host`` and
    reads the same result buffers every step: the tensors are validated and
    their pointers marshalled here, and for a decode plan with page-locked
    buffers the step is prepared once as a captured graph
    (``route_host_step_create``), so each call is one graph launch and a wait
    (``route_host_step_run``).  Otherwise each call goes straight to
    ``route_step_host``.  The object keeps references to the tensors and the
    plan; the caller must not resize them.  ``close()`` (or the plan's)
    releases the graph.

    ``launch()`` and ``wait()`` split a call in two
    (``route_host_step_launch`` / ``route_host_step_wait``) so that two
    steps of one plan, created on the same stream, can be in flight together:
    launch B, wait A, refill A, launch A, wait B, ...  ``launch()`` enqueues
    the step's kernels directly, chained to the step before it on the
    stream, so that its weights stream in, and its published rows are read,
    under that step's tail.  Between a step's launch and its wait its hidden buffer is not
    written and its results are not read.  Without a graph, ``launch()``
    runs the whole step and ``wait()`` returns at once.
    """

    def __init__(self, plan: Plan, hidden_host, W_latent, W_router, latent_host, logits_host,
                 ids_host, weights_host, stream=None):
        self._keep = (plan, hidden_host, W_latent, W_router, latent_host, logits_host, ids_host,
                      weights_host, stream)
        self._args = (plan.handle,) + _host_step_args(
            plan, hidden_host, W_latent, W_router, latent_host, logits_host, ids_host,
            weights_host) + (_stream(stream, plan.device),)
        L = lib()
        self._step = None
        h = ctypes.c_void_p()
        st = L.route_host_step_create(*self._args, ctypes.byref(h))
        if st == ROUTE_OK:
            self._step = h
            self._fn, self._call_args = L.route_host_step_run, (h,)
        elif st == STATUS_CODES["ROUTE_ERR_PLAN"]:  # not the copy-free decode path
            self._fn, self._call_args = L.route_step_host, self._args
        else:
            _check(st)

    @property
    def graph(self) -> bool:
        """True when calls launch the captured graph."""
        return self._step is not None

    def __call__(self) -> None:
        if self._fn is None:
            raise RouteError(STATUS_CODES["ROUTE_ERR_NULL"], "host step is closed")
        st = self._fn(*self._call_args)
        if st != ROUTE_OK:
            _check(st)

    def launch(self) -> None:
        if self._step is None:
            self()
            return
        st = lib().route_host_step_launch(self._step)
        if st != ROUTE_OK:
            _check(st)

    def wait(self) -> None:
        if self._step is None:
            if self._fn is None:
                raise RouteError(STATUS_CODES["ROUTE_ERR_NULL"], "host step is closed")
            return
        st = lib().route_host_step_wait(self._step)
        if st != ROUTE_OK:
            _check(st)

    def close(self) -> None:
        if self._step is not None:
            lib().route_host_step_destroy(self._step)
            self._step = None
        self._fn = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def route_set_overlap(plan: Plan, enable: bool) -> None:
    """Let the decode weight stream overlap the previous route step's tail; only
    when `hidden` is not written by the route call just before (include/route.h)."""
    _check(lib().route_set_overlap(plan.handle, int(bool(enable))))


def route_set_latent_ksplit(plan: Plan, enable: bool) -> None:
    """Decode latent with the general path's K-split arithmetic (eight BF16-rounded
    K-slice partials, FP32 sum, BF16 again); see include/route.h."""
    _check(lib().route_set_latent_ksplit(plan.handle, int(bool(enable))))


def route_test_stall(plan: Plan, enable: bool, timeout_ns: int = 1_000_000) -> None:
    """Test hook: make the plan's projection kernel wait for a copy that never
    comes, so that its bounded wait expires (see include/route.h)."""
    _check(lib().route_test_stall(plan.handle, int(bool(enable)), int(timeout_ns)))


def route_test_poison_scratch(plan: Plan, stream=None) -> None:
    """Test hook: fill the plan's split-K scratch with 0xFF bytes (include/route.h)."""
    _check(lib().route_test_poison_scratch(plan.handle, _stream(stream, plan.device)))


def route_device_status(plan: Plan) -> None:
    """Synchronise and raise RouteError if a kernel of this plan gave up waiting."""
    _check(lib().route_device_status(plan.handle))
