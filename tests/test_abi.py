"""The C ABI library loads on a machine without a GPU, exports every symbol
include/cm.h declares, and rejects bad arguments before any device work."""

import ctypes
import os
import re

import pytest

import __graft_entry__
from collective_matmul_decomposition_gb300 import cm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return cm.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "cm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cm_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(cm.EXPORTS) == names


def test_version_and_status_strings(lib):
    assert "sm_103a" in cm.version()
    for s in range(8):
        assert cm.status_string(s)


def test_plan_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.cm_plan(0, 1, 0, ctypes.byref(h)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_plan(17, 1, 0, ctypes.byref(h)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_plan(4, 0, 0, ctypes.byref(h)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_plan(4, 9, 0, ctypes.byref(h)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_plan(4, 1, 7, ctypes.byref(h)) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_plan(4, 1, 0, None) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_plan_destroy(None) == cm.CM_OK
    p = cm.Plan(4, 2, "bidi")
    with pytest.raises(cm.CMError):
        p.step(cm.CM_OP_AG_GEMM, 4, 0, 0)
    with pytest.raises(cm.CMError):
        p.set_option(cm.CM_OPT_TIMEOUT_NS, 0)
    for opt, bad in ((cm.CM_OPT_L2_HINTS, -1), (cm.CM_OPT_L2_HINTS, 256),
                     (cm.CM_OPT_L2_PROMOTION, -1), (cm.CM_OPT_L2_PROMOTION, 4),
                     (cm.CM_OPT_ROW_BAND, -1), (cm.CM_OPT_ROW_BAND, 4097),
                     (cm.CM_OPT_RS_PRELOAD, -1), (cm.CM_OPT_RS_PRELOAD, 4),
                     (cm.CM_OPT_KERNEL, -1), (cm.CM_OPT_KERNEL, 3),
                     (cm.CM_OPT_RS_EPILOGUE, -1), (cm.CM_OPT_RS_EPILOGUE, 4),
                     (cm.CM_OPT_RS_COL_SLABS, -1), (cm.CM_OPT_RS_COL_SLABS, 65),
                     (cm.CM_OPT_RS_BUCKET_HINT, -1), (cm.CM_OPT_RS_BUCKET_HINT, 4),
                     (cm.CM_OPT_TASK_ORDER, -1), (cm.CM_OPT_TASK_ORDER, 3)):
        with pytest.raises(cm.CMError):
            p.set_option(opt, bad)
    for v in (0, 1, 2, 3):
        p.set_option(cm.CM_OPT_RS_PRELOAD, v)
    p.set_option(cm.CM_OPT_L2_HINTS, 0x21)
    p.set_option(cm.CM_OPT_L2_PROMOTION, 0)


def test_steps_counts(lib):
    for N in range(1, 17):
        assert cm.Plan(N, 1, "uni").steps(cm.CM_OP_AG_GEMM) == N
        assert cm.Plan(N, 1, "uni").steps(cm.CM_OP_GEMM_RS) == N
        assert cm.Plan(N, 1, "bidi").steps(cm.CM_OP_AG_GEMM) == (N - 1 + 1) // 2 + 1
        assert cm.Plan(N, 1, "none").steps(cm.CM_OP_GEMM_RS) == 1


def test_workspace_sizes(lib):
    p = cm.Plan(8, 1, "uni")
    m, K = 1024, 8192
    assert p.ag_workspace_size(m, K) >= 2 * 8 * m * K * 2
    # RS, automatic: 268 MB of buckets do not fit L2, so per-step buffers
    # (one per rank and step); 64 MB do, so in place (one per bucket)
    assert p.rs_workspace_size(8192, 8192) >= 8 * 8 * 1024 * 8192 * 4
    assert 8 * 512 * 4096 * 4 <= p.rs_workspace_size(4096, 4096) < 9 * 512 * 4096 * 4
    p.set_option(cm.CM_OPT_RS_IN_PLACE, 1)     # in place: one [M/N][n] fp32 buffer per bucket
    assert 8 * 1024 * 8192 * 4 <= p.rs_workspace_size(8192, 8192) < 9 * 1024 * 8192 * 4
    p.set_option(cm.CM_OPT_RS_IN_PLACE, 0)     # one per (rank, step)
    assert p.rs_workspace_size(4096, 4096) >= 8 * 8 * 512 * 4096 * 4
    with pytest.raises(cm.CMError):
        p.set_option(cm.CM_OPT_RS_IN_PLACE, 3)
    b = cm.Plan(8, 1, "bidi")
    assert b.ag_workspace_size(m, K) >= 4 * 8 * m * K * 2
    assert cm.Plan(8, 1, "none").ag_workspace_size(m, K) < 1 << 20
    assert cm.Plan(1, 1, "uni").ag_workspace_size(m, K) < 1 << 20
    assert lib.cm_ag_gemm_workspace_size(None, 1, 1) == 0


def test_rs_bucket_mode_boundary(lib):
    """The automatic bucket mode keeps buckets in place up to 128 MiB of
    buckets per ring stream (M*n*4 bytes) and gives every hop its own buffer
    above that; the workspace size follows the mode the call will take."""
    N, n = 8, 8192
    p = cm.Plan(N, 1, "uni")
    at = 4096                      # 4096 * 8192 * 4 B = 128 MiB exactly: in place
    above = at + N                 # one more row per bucket: per-step buffers
    assert at * n * 4 == 128 << 20
    one_set = at * n * 4
    assert one_set <= p.rs_workspace_size(at, n) < one_set + (8 << 20)
    steps = p.steps(cm.CM_OP_GEMM_RS)
    assert p.rs_workspace_size(above, n) >= steps * above * n * 4
    p.set_option(cm.CM_OPT_RS_IN_PLACE, 1)
    assert p.rs_workspace_size(above, n) < above * n * 4 + (8 << 20)
    p.set_option(cm.CM_OPT_RS_IN_PLACE, 0)
    assert p.rs_workspace_size(at, n) >= steps * one_set
    # two-way rings: one bucket set per ring stream, the rule per stream
    b = cm.Plan(N, 1, "bidi")
    assert 2 * one_set <= b.rs_workspace_size(at, n) < 2 * one_set + (8 << 20)


def test_compute_calls_reject_bad_arguments_without_device_work(lib):
    p = cm.Plan(2, 2, "uni")
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: every check fails first
    ws = p.ag_workspace_size(64, 256)
    # null pointers
    assert lib.cm_ag_gemm(p.handle, None, fake, 1, fake, 0, 64, 256, 512, fake, ws, None) == cm.CM_ERR_INVALID_ARG
    # K not a multiple of 8
    assert lib.cm_ag_gemm(p.handle, fake, fake, 1, fake, 0, 64, 250, 512, fake, ws, None) == cm.CM_ERR_ALIGNMENT
    # m not divisible by chunks
    assert lib.cm_ag_gemm(p.handle, fake, fake, 1, fake, 0, 63, 256, 512, fake, ws, None) == cm.CM_ERR_SHAPE
    # workspace too small
    assert lib.cm_ag_gemm(p.handle, fake, fake, 1, fake, 0, 64, 256, 512, fake, 16, None) == cm.CM_ERR_WORKSPACE
    # misaligned pointer
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert lib.cm_ag_gemm(p.handle, odd, fake, 1, fake, 0, 64, 256, 512, fake, ws, None) == cm.CM_ERR_ALIGNMENT
    # RS: M not divisible by N
    wsr = p.rs_workspace_size(128, 512)
    assert lib.cm_gemm_rs(p.handle, fake, fake, 1, fake, 0, 127, 128, 512, fake, wsr, None) == cm.CM_ERR_SHAPE
    # RS: bucket rows not divisible by chunks
    assert lib.cm_gemm_rs(p.handle, fake, fake, 1, fake, 0, 6, 128, 512, fake, wsr, None) == cm.CM_ERR_SHAPE
    # bad enums
    assert lib.cm_gemm_rs(p.handle, fake, fake, 5, fake, 0, 128, 128, 512, fake, wsr, None) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_gemm_rs(p.handle, fake, fake, 1, fake, 9, 128, 128, 512, fake, wsr, None) == cm.CM_ERR_INVALID_ARG
    assert lib.cm_check_status(None, None, None) == cm.CM_ERR_INVALID_ARG


def test_empty_shapes_are_rejected(lib):
    """Empty problems (a zero size) are shape errors, returned before any
    device work; their workspace size is 0."""
    p = cm.Plan(2, 1, "uni")
    fake = ctypes.c_void_p(1 << 20)
    ws = p.ag_workspace_size(64, 256)
    for m, K, n in ((0, 256, 512), (64, 0, 512), (64, 256, 0)):
        assert lib.cm_ag_gemm(p.handle, fake, fake, 1, fake, 0, m, K, n, fake, ws, None) == cm.CM_ERR_SHAPE
    wsr = p.rs_workspace_size(128, 512)
    for M, k, n in ((0, 128, 512), (128, 0, 512), (128, 128, 0)):
        assert lib.cm_gemm_rs(p.handle, fake, fake, 1, fake, 0, M, k, n, fake, wsr, None) == cm.CM_ERR_SHAPE
    assert p.ag_workspace_size(0, 256) == 0
    assert p.rs_workspace_size(0, 512) == 0


def test_no_oracle_in_product_path():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "collective_matmul_decomposition_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "cm_oracle" not in text, f


def test_no_multicast_load_in_the_kernels():
    """No TMA load of the library is a cluster-multicast load: every operand
    tile is loaded into the loading CTA's own shared memory.  (The tcgen05
    commit that arrives on both CTAs' barriers is not a load.)"""
    csrc = os.path.join(ROOT, "collective_matmul_decomposition_gb300", "csrc")
    for f in os.listdir(csrc):
        for line in open(os.path.join(csrc, f)):
            if "multicast::cluster" in line:
                assert "cp.async" not in line and "tcgen05.commit" in line, (f, line)


def test_bounds_checked_build_loads_and_only_it_takes_the_planted_offset(lib):
    """The bounds-checked build exports the same symbols; only it accepts
    CM_OPT_DEBUG_FLAG_OFFSET (a testing aid for its checks)."""
    dbg = cm.bounds_checked()
    for name in _declared():
        assert hasattr(dbg.load(), name), name
    assert "bounds-checked" in dbg.version()
    p = cm.Plan(4, 1, "uni")
    with pytest.raises(cm.CMError):
        p.set_option(cm.CM_OPT_DEBUG_FLAG_OFFSET, 8)
    q = dbg.Plan(4, 1, "uni")
    q.set_option(dbg.CM_OPT_DEBUG_FLAG_OFFSET, 8)
    base = {t.sig_done for t in cm.Plan(4, 1, "uni").tasks(cm.CM_OP_GEMM_RS)}
    moved = {t.sig_done for t in q.tasks(dbg.CM_OP_GEMM_RS)}
    assert moved == {s + 8 for s in base}
    assert cm.status_string(cm.CM_ERR_BOUNDS)
