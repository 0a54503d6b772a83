"""Python binding of the C ABI in include/cm.h (argument marshalling only).

Every step of the decomposed collective matmul runs in the CUDA library
(_build/libcm.so); this module only turns torch tensors into device pointers
and the current CUDA stream into a cudaStream_t.  It raises if the library is
missing -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libcm.so")
# the bounds-checked build of the same library (CM_DEBUG_BOUNDS)
DEBUG_LIB_PATH = os.path.join(PKG, "_build_debug", "libcm_debug.so")

CM_OK, CM_ERR_INVALID_ARG, CM_ERR_SHAPE, CM_ERR_ALIGNMENT = 0, 1, 2, 3
CM_ERR_UNSUPPORTED, CM_ERR_CUDA, CM_ERR_TIMEOUT, CM_ERR_WORKSPACE = 4, 5, 6, 7
CM_ERR_BOUNDS = 8
CM_RING_UNI, CM_RING_BIDI, CM_RING_NONE = 0, 1, 2
CM_BF16, CM_F32 = 0, 1
CM_W_KN, CM_W_NK = 0, 1
CM_OP_AG_GEMM, CM_OP_GEMM_RS = 0, 1
CM_OPT_TIMEOUT_NS, CM_OPT_SERIAL_STEPS, CM_OPT_GRID, CM_OPT_SKIP_SIGNAL, CM_OPT_KERNEL = 0, 1, 2, 3, 4
CM_OPT_STATIC_TILES, CM_OPT_TILE_GROUP, CM_OPT_L2_HINTS, CM_OPT_L2_PROMOTION, CM_OPT_ROW_BAND = 5, 6, 7, 8, 9
CM_OPT_BULK_OVERLAP = 10
CM_OPT_RS_PRELOAD = 11
CM_OPT_RS_IN_PLACE = 12
CM_OPT_TASK_ORDER = 13
CM_OPT_RS_EPILOGUE = 14
CM_OPT_DEBUG_FLAG_OFFSET = 15
CM_OPT_RS_COL_SLABS = 16
CM_OPT_RS_BUCKET_HINT = 17
CM_MAX_RANKS, CM_MAX_CHUNKS = 16, 8

DIRECTIONS = {"uni": CM_RING_UNI, "bidi": CM_RING_BIDI, "none": CM_RING_NONE}
LAYOUTS = {"kn": CM_W_KN, "nk": CM_W_NK}

# Every symbol include/cm.h declares.
EXPORTS = ["cm_plan", "cm_plan_destroy", "cm_plan_steps", "cm_plan_step", "cm_plan_tasks",
           "cm_ag_gemm_workspace_size", "cm_gemm_rs_workspace_size", "cm_ag_gemm", "cm_gemm_rs",
           "cm_check_status", "cm_status_string", "cm_plan_set_option", "cm_version",
           "cm_ag_gemm_noalloc", "cm_ag_gemm_noalloc_check_status", "cm_cost_estimate", "cm_plan_choose",
           "cm_gemm_rs_pipelined_workspace_size", "cm_gemm_rs_pipelined",
           "cm_backward_pair_workspace_size", "cm_backward_pair",
           "cm_cannon_workspace_size", "cm_cannon_gemm", "cm_einsum_cost", "cm_plan_choose_einsum"]
CM_NOALLOC_SCRATCH_BYTES = 64 << 20


class cm_rates(ctypes.Structure):
    """Per-rank peak rates for the cost model (see cm_cost_estimate)."""
    _fields_ = [("gemm_tflops", ctypes.c_double), ("ring_gbs", ctypes.c_double), ("coll_gbs", ctypes.c_double),
                ("hop_us", ctypes.c_double), ("mem_gbs", ctypes.c_double)]


class cm_task(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int16), ("a_slab", ctypes.c_int16), ("a_src", ctypes.c_int16),
                ("out_idx", ctypes.c_int16), ("out_buf", ctypes.c_int16),
                ("in_buf", ctypes.c_int16 * 2), ("fwd_slot", ctypes.c_int16 * 2),
                ("wait_in", ctypes.c_int16 * 2), ("wait_free", ctypes.c_int16 * 2),
                ("sig_fwd", ctypes.c_int16 * 2), ("sig_done", ctypes.c_int16),
                ("step", ctypes.c_int16), ("stream", ctypes.c_int16), ("tile_group", ctypes.c_int16)]


class CMError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def load():
    """Load the in-tree library (built by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    i32, i64, p, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    lib.cm_plan.argtypes = [i32, i32, i32, ctypes.POINTER(p)]
    lib.cm_plan.restype = i32
    lib.cm_plan_destroy.argtypes = [p]
    lib.cm_plan_destroy.restype = i32
    lib.cm_plan_steps.argtypes = [p, i32]
    lib.cm_plan_steps.restype = i32
    lib.cm_plan_step.argtypes = [p, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                 ctypes.POINTER(i32)]
    lib.cm_plan_step.restype = i32
    lib.cm_plan_tasks.argtypes = [p, i32, p, i32]
    lib.cm_plan_tasks.restype = i32
    lib.cm_ag_gemm_workspace_size.argtypes = [p, i64, i64]
    lib.cm_ag_gemm_workspace_size.restype = sz
    lib.cm_gemm_rs_workspace_size.argtypes = [p, i64, i64]
    lib.cm_gemm_rs_workspace_size.restype = sz
    lib.cm_ag_gemm.argtypes = [p, p, p, i32, p, i32, i64, i64, i64, p, sz, p]
    lib.cm_ag_gemm.restype = i32
    lib.cm_gemm_rs.argtypes = [p, p, p, i32, p, i32, i64, i64, i64, p, sz, p]
    lib.cm_gemm_rs.restype = i32
    lib.cm_check_status.argtypes = [p, p, ctypes.POINTER(i32)]
    lib.cm_check_status.restype = i32
    lib.cm_status_string.argtypes = [i32]
    lib.cm_status_string.restype = ctypes.c_char_p
    lib.cm_plan_set_option.argtypes = [p, i32, i64]
    lib.cm_plan_set_option.restype = i32
    lib.cm_version.argtypes = []
    lib.cm_version.restype = ctypes.c_char_p
    lib.cm_ag_gemm_noalloc.argtypes = [p, p, p, i32, p, i32, i64, i64, i64, p]
    lib.cm_ag_gemm_noalloc.restype = i32
    lib.cm_ag_gemm_noalloc_check_status.argtypes = [p, ctypes.POINTER(i32)]
    lib.cm_ag_gemm_noalloc_check_status.restype = i32
    lib.cm_gemm_rs_pipelined_workspace_size.argtypes = [p, i64, i64]
    lib.cm_gemm_rs_pipelined_workspace_size.restype = sz
    lib.cm_gemm_rs_pipelined.argtypes = [p, p, p, i32, p, i32, i64, i64, i64, p, sz, p]
    lib.cm_gemm_rs_pipelined.restype = i32
    lib.cm_backward_pair_workspace_size.argtypes = [p, i64, i64, i64]
    lib.cm_backward_pair_workspace_size.restype = sz
    lib.cm_backward_pair.argtypes = [p, p, p, p, p, i32, p, i32, i64, i64, i64, p, sz, p]
    lib.cm_backward_pair.restype = i32
    lib.cm_cannon_workspace_size.argtypes = [p, i64, i64, i64]
    lib.cm_cannon_workspace_size.restype = sz
    lib.cm_cannon_gemm.argtypes = [p, p, p, i32, p, i32, i64, i64, i64, p, sz, p]
    lib.cm_cannon_gemm.restype = i32
    rp = ctypes.POINTER(cm_rates)
    lib.cm_cost_estimate.argtypes = [i32, i32, i32, i32, i64, i64, i64, rp, ctypes.POINTER(ctypes.c_double)]
    lib.cm_cost_estimate.restype = i32
    lib.cm_plan_choose.argtypes = [i32, i32, i64, i64, i64, rp, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                   ctypes.POINTER(ctypes.c_double)]
    lib.cm_plan_choose.restype = i32
    lib.cm_einsum_cost.argtypes = [i32, i32, i32, i32, i64, i64, i64, rp, ctypes.POINTER(ctypes.c_double)]
    lib.cm_einsum_cost.restype = i32
    lib.cm_plan_choose_einsum.argtypes = [i32, i64, i64, i64, rp, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                          ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_double)]
    lib.cm_plan_choose_einsum.restype = i32
    _lib = lib
    return lib


def bounds_checked():
    """A second binding of this module, to the bounds-checked build of the
    library (every computed flag, slot, row and buffer index checked in the
    kernels; an index outside its buffer is reported as CM_ERR_BOUNDS)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(__name__ + "_bounds_checked", os.path.abspath(__file__))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.LIB_PATH = DEBUG_LIB_PATH
    mod.load()
    return mod


def status_string(status: int) -> str:
    return load().cm_status_string(int(status)).decode()


def _check(status, what):
    if status != CM_OK:
        raise CMError(status, what)


class Plan:
    """Owns a cm_plan_t (cm_plan / cm_plan_destroy)."""

    def __init__(self, n_ranks: int, chunks: int = 1, direction: str = "uni"):
        lib = load()
        h = ctypes.c_void_p()
        _check(lib.cm_plan(int(n_ranks), int(chunks), DIRECTIONS[direction], ctypes.byref(h)), "cm_plan")
        self.handle = h
        self.N, self.chunks, self.direction = int(n_ranks), int(chunks), direction

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            _lib.cm_plan_destroy(h)
            self.handle = None

    def steps(self, op: int) -> int:
        return load().cm_plan_steps(self.handle, int(op))

    def step(self, op: int, rank: int, step: int, stream: int = 0):
        o, s, d = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(load().cm_plan_step(self.handle, int(op), rank, step, stream,
                                   ctypes.byref(o), ctypes.byref(s), ctypes.byref(d)), "cm_plan_step")
        return o.value, s.value, d.value

    def tasks(self, op: int):
        lib = load()
        n = lib.cm_plan_tasks(self.handle, int(op), None, 0)
        arr = (cm_task * max(n, 1))()
        lib.cm_plan_tasks(self.handle, int(op), ctypes.cast(arr, ctypes.c_void_p), n)
        return [arr[i] for i in range(n)]

    def set_option(self, option: int, value: int):
        _check(load().cm_plan_set_option(self.handle, int(option), int(value)), "cm_plan_set_option")

    def ag_workspace_size(self, m: int, K: int) -> int:
        return int(load().cm_ag_gemm_workspace_size(self.handle, int(m), int(K)))

    def cannon_workspace_size(self, bm: int, bk: int, bn: int) -> int:
        return load().cm_cannon_workspace_size(self.handle, bm, bk, bn)

    def backward_pair_workspace_size(self, m: int, K: int, n: int) -> int:
        return load().cm_backward_pair_workspace_size(self.handle, m, K, n)

    def rs_pipelined_workspace_size(self, M: int, n: int) -> int:
        return load().cm_gemm_rs_pipelined_workspace_size(self.handle, M, n)

    def rs_workspace_size(self, M: int, n: int) -> int:
        return int(load().cm_gemm_rs_workspace_size(self.handle, int(M), int(n)))


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _ydtype(y):
    import torch
    if y.dtype == torch.bfloat16:
        return CM_BF16
    if y.dtype == torch.float32:
        return CM_F32
    raise TypeError("y must be bf16 or fp32")


def cm_ag_gemm(plan: Plan, x, w, y, ws, w_layout: str = "nk", stream=None):
    """Decomposed AllGather->GEMM: x [N][m][K], w per rank, y [N][N*m][n]."""
    N, m, K = x.shape
    n = w.shape[1] if w_layout == "nk" else w.shape[2]
    st = load().cm_ag_gemm(plan.handle, _ptr(x), _ptr(w), LAYOUTS[w_layout], _ptr(y), _ydtype(y),
                           m, K, n, _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream))
    _check(st, "cm_ag_gemm")


def cm_ag_gemm_noalloc(plan: Plan, x, w, y, w_layout: str = "nk", stream=None):
    """cm_ag_gemm without a workspace: for callers that cannot allocate device
    memory; the library's fixed scratch array (CM_NOALLOC_SCRATCH_BYTES) is
    used instead, shared by every call (calls must not overlap on the GPU)."""
    N, m, K = x.shape
    n = w.shape[1] if w_layout == "nk" else w.shape[2]
    st = load().cm_ag_gemm_noalloc(plan.handle, _ptr(x), _ptr(w), LAYOUTS[w_layout], _ptr(y), _ydtype(y),
                                   m, K, n, _stream_ptr(stream))
    _check(st, "cm_ag_gemm_noalloc")


def cm_ag_gemm_noalloc_check_status(stream=None):
    """Synchronise and return (status, info[4]) of the last cm_ag_gemm_noalloc call."""
    info = (ctypes.c_int * 4)()
    st = load().cm_ag_gemm_noalloc_check_status(_stream_ptr(stream), info)
    return st, list(info)


def cm_gemm_rs(plan: Plan, x, w, y, ws, w_layout: str = "nk", stream=None):
    """Decomposed GEMM->ReduceScatter: x [N][M][k], w per rank, y [N][M/N][n]."""
    N, M, k = x.shape
    n = w.shape[1] if w_layout == "nk" else w.shape[2]
    st = load().cm_gemm_rs(plan.handle, _ptr(x), _ptr(w), LAYOUTS[w_layout], _ptr(y), _ydtype(y),
                           M, k, n, _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream))
    _check(st, "cm_gemm_rs")


def cm_gemm_rs_pipelined(plan: Plan, x, w, y, ws, w_layout: str = "nk", stream=None):
    """GEMM->ReduceScatter with pipeline chunks: x [N][M][k], w per rank, y [N][M/N][n]."""
    N, M, k = x.shape
    n = w.shape[1] if w_layout == "nk" else w.shape[2]
    st = load().cm_gemm_rs_pipelined(plan.handle, _ptr(x), _ptr(w), LAYOUTS[w_layout], _ptr(y), _ydtype(y),
                                     M, k, n, _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream))
    _check(st, "cm_gemm_rs_pipelined")


def cm_backward_pair(plan: Plan, x, w, dy, dx, dw, ws, stream=None):
    """Backward pair of the column-parallel layer: dx [N][m][K] = GEMM-RS of dy_r @ W_r,
    dw [N][n][K] = dy_r^T @ concat_j(x_j) (its AllGather overlapped with the GEMM-RS)."""
    N, m, K = x.shape
    n = w.shape[1]
    st = load().cm_backward_pair(plan.handle, _ptr(x), _ptr(w), _ptr(dy), _ptr(dx), _ydtype(dx), _ptr(dw),
                                 _ydtype(dw), m, K, n, _ptr(ws), ws.numel() * ws.element_size(),
                                 _stream_ptr(stream))
    _check(st, "cm_backward_pair")


def cm_cannon_gemm(plan: Plan, a, b, c, ws, b_layout: str = "nk", stream=None):
    """Cannon-style 2-D rotation: a [q*q][bm][bk], b blocks, c [q*q][bm][bn]."""
    P, bm, bk = a.shape
    bn = b.shape[1] if b_layout == "nk" else b.shape[2]
    st = load().cm_cannon_gemm(plan.handle, _ptr(a), _ptr(b), LAYOUTS[b_layout], _ptr(c), _ydtype(c), bm, bk, bn,
                               _ptr(ws), ws.numel() * ws.element_size(), _stream_ptr(stream))
    _check(st, "cm_cannon_gemm")


def cm_check_status(ws, stream=None):
    """Synchronise and return (status, info[4]) of the last call that used ws."""
    info = (ctypes.c_int * 4)()
    st = load().cm_check_status(_ptr(ws), _stream_ptr(stream), info)
    return st, list(info)


def _rates(rates):
    if isinstance(rates, cm_rates):
        return rates
    return cm_rates(*(float(rates[k]) for k in ("gemm_tflops", "ring_gbs", "coll_gbs", "hop_us", "mem_gbs")))


def cost_estimate(n_ranks, chunks, direction, op, rows, K, n, rates) -> float:
    """Predicted time (us) of one candidate; direction "none" = native collective + GEMM."""
    us = ctypes.c_double()
    r = _rates(rates)
    _check(load().cm_cost_estimate(n_ranks, chunks, DIRECTIONS[direction], op, rows, K, n, ctypes.byref(r),
                                   ctypes.byref(us)), "cm_cost_estimate")
    return us.value


def plan_choose(n_ranks, op, rows, K, n, rates, max_chunks=CM_MAX_CHUNKS):
    """The cost model's pick: (chunks, direction name, predicted us); "none" = decline."""
    c, d, us = ctypes.c_int(), ctypes.c_int(), ctypes.c_double()
    r = _rates(rates)
    _check(load().cm_plan_choose(n_ranks, op, rows, K, n, ctypes.byref(r), max_chunks, ctypes.byref(c),
                                 ctypes.byref(d), ctypes.byref(us)), "cm_plan_choose")
    name = {v: k for k, v in DIRECTIONS.items()}[d.value]
    return c.value, name, us.value


def einsum_cost(n_ranks, chunks, direction, decompose, m, K, n, rates) -> float:
    """Predicted time (us) of one way to run an Einsum that offers both
    collectives: decompose = "ag", "rs" or "none" (both native)."""
    which = {"ag": CM_OP_AG_GEMM, "rs": CM_OP_GEMM_RS, "none": -1}[decompose]
    us = ctypes.c_double()
    r = _rates(rates)
    _check(load().cm_einsum_cost(n_ranks, chunks, DIRECTIONS[direction], which, m, K, n, ctypes.byref(r),
                                 ctypes.byref(us)), "cm_einsum_cost")
    return us.value


def plan_choose_einsum(n_ranks, m, K, n, rates, max_chunks=CM_MAX_CHUNKS):
    """Which collective of such an Einsum to decompose: ("ag" | "rs" | "none", chunks, direction, us)."""
    w, c, d, us = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_double()
    r = _rates(rates)
    _check(load().cm_plan_choose_einsum(n_ranks, m, K, n, ctypes.byref(r), max_chunks, ctypes.byref(w),
                                        ctypes.byref(c), ctypes.byref(d), ctypes.byref(us)), "cm_plan_choose_einsum")
    name = {CM_OP_AG_GEMM: "ag", CM_OP_GEMM_RS: "rs", -1: "none"}[w.value]
    return name, c.value, {v: k for k, v in DIRECTIONS.items()}[d.value], us.value


def version() -> str:
    return load().cm_version().decode()
