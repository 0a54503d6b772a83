"""fp64 CPU oracle for the decomposed collective matmul.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA path and imports nothing from it; inputs reach
it as raw bf16 bit patterns (numpy uint16) from the shared seeded generator.

Contents
--------
* ``cm_oracle.c`` (built here into ``_build/liboracle.so`` with gcc/OpenMP):
  the plain definitions, see its header.
    - AllGather->GEMM:   Y_r = concat_j(X_j) @ W_r
    - GEMM->ReduceScatter: Y_o = (sum_r X_r @ W_r)[rows of bucket o]
    - weight gradient of the column-parallel layer (the backward pair's
      wgrad): dW_r = dY_r^T @ concat_j(X_j); its data gradient is the
      GEMM->ReduceScatter above with W_r read as [n][K]
* ``ring.py``: a rank-by-rank simulation of the ring schedules the pages
  describe (shards / accumulating buckets handed to a neighbour each step),
  in fp64, with its own schedule derived from the pages -- a second,
  independent path that checks the schedule rather than the arithmetic --
  and of Cannon-style 2-D rotation on a q x q grid (A blocks move left, B
  blocks move up), whose definition is the plain GEMM of the assembled
  blocks.

Parity pins (what each function is checked against, in ``tests/``) are listed
in the test files; every function here has at least one pin.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

W_LAYOUTS = {"kn": 0, "nk": 1}

_lib = None


def build(force: bool = False) -> str:
    """Compile cm_oracle.c into _build/liboracle.so (gcc, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        # -ffp-contract=off: every `s += a*b` rounds the product and the sum
        # separately, identically on x86 and Arm.
        cmd = ["gcc", "-O3", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.cm_oracle_gemm.argtypes = [i64, i64, i64, p, p, i32, p]
        lib.cm_oracle_ag_gemm.argtypes = [i32, i64, i64, i64, p, p, i32, p]
        lib.cm_oracle_ag_gemm_rows.argtypes = [i32, i64, i64, i64, p, p, i32, i64, p, p, p]
        lib.cm_oracle_gemm_rs.argtypes = [i32, i64, i64, i64, p, p, i32, p]
        lib.cm_oracle_gemm_rs_rows.argtypes = [i32, i64, i64, i64, p, p, i32, i64, p, p, p]
        lib.cm_oracle_wgrad.argtypes = [i32, i64, i64, i64, p, p, p]
        lib.cm_oracle_wgrad_rows.argtypes = [i32, i64, i64, i64, p, p, i64, p, p, p]
        lib.cm_oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy uint16)")
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def threads() -> int:
    """Number of OpenMP threads the oracle runs on."""
    return int(_load().cm_oracle_threads())


def bf16_to_f64(bits) -> np.ndarray:
    """Exact decode of bf16 bit patterns (uint16) to float64."""
    b = _bits(bits)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm(a_bits, w_bits, w_layout: str = "kn") -> np.ndarray:
    """Plain C = A @ W in fp64; A [M][K], W [K][n] ("kn") or [n][K] ("nk")."""
    a, w = _bits(a_bits), _bits(w_bits)
    M, K = a.shape
    n = w.shape[1] if w_layout == "kn" else w.shape[0]
    assert (w.shape[0] if w_layout == "kn" else w.shape[1]) == K
    c = np.empty((M, n), dtype=np.float64)
    _load().cm_oracle_gemm(M, K, n, _ptr(a), _ptr(w), W_LAYOUTS[w_layout], _ptr(c))
    return c


def _ag_dims(x, w, w_layout):
    N, m, K = x.shape
    n = w.shape[2] if w_layout == "kn" else w.shape[1]
    assert w.shape[0] == N and (w.shape[1] if w_layout == "kn" else w.shape[2]) == K
    return N, m, K, n


def ag_gemm(x_bits, w_bits, w_layout: str = "nk") -> np.ndarray:
    """AllGather->GEMM definition: y[r] = concat_j(x[j]) @ W_r, y [N][N*m][n] fp64."""
    x, w = _bits(x_bits), _bits(w_bits)
    N, m, K, n = _ag_dims(x, w, w_layout)
    y = np.empty((N, N * m, n), dtype=np.float64)
    _load().cm_oracle_ag_gemm(N, m, K, n, _ptr(x), _ptr(w), W_LAYOUTS[w_layout], _ptr(y))
    return y


def ag_gemm_rows(x_bits, w_bits, ranks, rows, w_layout: str = "nk") -> np.ndarray:
    """Sampled rows of the AllGather->GEMM definition: out[t] = y[ranks[t]][rows[t]]."""
    x, w = _bits(x_bits), _bits(w_bits)
    N, m, K, n = _ag_dims(x, w, w_layout)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert ranks.shape == rows.shape and ranks.ndim == 1
    assert ((0 <= ranks) & (ranks < N)).all() and ((0 <= rows) & (rows < N * m)).all()
    out = np.empty((len(rows), n), dtype=np.float64)
    _load().cm_oracle_ag_gemm_rows(N, m, K, n, _ptr(x), _ptr(w), W_LAYOUTS[w_layout],
                                   len(rows), _ptr(ranks), _ptr(rows), _ptr(out))
    return out


def _wgrad_dims(x, dy):
    N, m, K = x.shape
    assert dy.shape[0] == N and dy.shape[1] == N * m
    return N, m, K, dy.shape[2]


def wgrad(x_bits, dy_bits) -> np.ndarray:
    """Weight gradient of the column-parallel layer: dW[r][i][k] = sum_t dY_r[t][i] * X_all[t][k],
    x [N][m][K], dy [N][N*m][n] -> [N][n][K] fp64."""
    x, dy = _bits(x_bits), _bits(dy_bits)
    N, m, K, n = _wgrad_dims(x, dy)
    out = np.empty((N, n, K), dtype=np.float64)
    _load().cm_oracle_wgrad(N, m, K, n, _ptr(x), _ptr(dy), _ptr(out))
    return out


def wgrad_rows(x_bits, dy_bits, ranks, rows) -> np.ndarray:
    """Sampled rows of the weight gradient: out[s] = dW[ranks[s]][rows[s]]."""
    x, dy = _bits(x_bits), _bits(dy_bits)
    N, m, K, n = _wgrad_dims(x, dy)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert ranks.shape == rows.shape and ranks.ndim == 1
    assert ((0 <= ranks) & (ranks < N)).all() and ((0 <= rows) & (rows < n)).all()
    out = np.empty((len(rows), K), dtype=np.float64)
    _load().cm_oracle_wgrad_rows(N, m, K, n, _ptr(x), _ptr(dy), len(rows), _ptr(ranks), _ptr(rows), _ptr(out))
    return out


def _rs_dims(x, w, w_layout):
    N, M, k = x.shape
    n = w.shape[2] if w_layout == "kn" else w.shape[1]
    assert w.shape[0] == N and (w.shape[1] if w_layout == "kn" else w.shape[2]) == k
    assert M % N == 0
    return N, M, k, n


def gemm_rs(x_bits, w_bits, w_layout: str = "nk") -> np.ndarray:
    """GEMM->ReduceScatter definition: y[o] = (sum_r x[r] @ W_r)[o*M/N:(o+1)*M/N]."""
    x, w = _bits(x_bits), _bits(w_bits)
    N, M, k, n = _rs_dims(x, w, w_layout)
    y = np.empty((N, M // N, n), dtype=np.float64)
    _load().cm_oracle_gemm_rs(N, M, k, n, _ptr(x), _ptr(w), W_LAYOUTS[w_layout], _ptr(y))
    return y


def gemm_rs_rows(x_bits, w_bits, owners, rows, w_layout: str = "nk") -> np.ndarray:
    """Sampled rows of the GEMM->ReduceScatter definition: out[t] = y[owners[t]][rows[t]]."""
    x, w = _bits(x_bits), _bits(w_bits)
    N, M, k, n = _rs_dims(x, w, w_layout)
    owners = np.ascontiguousarray(owners, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert owners.shape == rows.shape and owners.ndim == 1
    assert ((0 <= owners) & (owners < N)).all() and ((0 <= rows) & (rows < M // N)).all()
    out = np.empty((len(rows), n), dtype=np.float64)
    _load().cm_oracle_gemm_rs_rows(N, M, k, n, _ptr(x), _ptr(w), W_LAYOUTS[w_layout],
                                   len(rows), _ptr(owners), _ptr(rows), _ptr(out))
    return out


def normwise_max_rel_err(y, ref) -> float:
    """max|y - ref| / max|ref| over one output tensor (the parity metric)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(y - ref))) if ref.size else 0.0
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
