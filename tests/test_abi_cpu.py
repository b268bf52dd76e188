"""CPU-side checks of the C ABI: the library builds and loads, exports every
function include/varlen_ssm.h declares, sizes its workspaces sanely, and
rejects bad arguments on the host (before touching the GPU)."""
import os
import re

import pytest

from selective_ssm_packed_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "varlen_ssm.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([a-z][A-Za-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for need in ("varlen_position_indices", "varlen_conv1d_fwd", "varlen_conv1d_bwd",
                 "varlen_selective_scan_fwd", "varlen_selective_scan_bwd"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows the signature of each
    assert set(declared_functions()) <= set(binding.SIGNATURES)


def test_workspace_queries(lib):
    assert binding.scan_fwd_workspace_size(32768, 4096, 16) > 0
    small = binding.scan_bwd_workspace_size(16, 8, 4)
    big = binding.scan_bwd_workspace_size(32768, 4096, 16)
    assert 0 < small < big
    assert lib.varlen_selective_scan_chunk_states_size(33, 8, 4) == 4 * 2 * 8 * 4
    assert binding.conv1d_fwd_workspace_size(0, 8, 4) > 0
    assert binding.conv1d_bwd_workspace_size(16, 8, 5) == 0
    assert binding.scan_fwd_workspace_size(-1, 8, 4) == 0


def test_strerror_and_status_codes(lib):
    for code in binding.ERR:
        assert binding.strerror(code)
    assert binding.status_code(0) == 0
    assert binding.status_code(1) == -16
    assert binding.status_code(2) == -17
    assert binding.status_code(4) == -17          # a tile-copy wait ran out
    assert binding.status_code(8) == -18          # a non-finite output (VSSM_DBG_CHECK_FINITE)
    assert binding.status_code(16) == -19         # a device index check (checked build)
    assert binding.status_code(1 | 8 | 16) == -16  # malformed input outranks what follows from it
    assert lib.vssm_checks_build() == 0           # the ordinary build


def test_checked_build_compiles_and_reports_itself():
    """The VSSM_CHECKS=1 variant builds beside the ordinary library (nvcc
    cross-compiles here) and says which build it is."""
    import ctypes
    path = build.build(checks=True)
    assert path == build.CHECKS_LIB_PATH != build.LIB_PATH
    L = ctypes.CDLL(path)
    assert L.vssm_checks_build() == 1


def _conv_fwd(lib, **kw):
    a = dict(x=16, weight=16, bias=None, cu=16, pos=None, S=1, T=16, D=8, W=4, silu=1, dt=0,
             u=16, x_init=None, x_last=None, ws=16, wsb=1 << 20, st=None)
    a.update(kw)
    return lib.varlen_conv1d_fwd(a["x"], a["weight"], a["bias"], a["cu"], a["pos"], a["S"], a["T"],
                                 a["D"], a["W"], a["silu"], a["dt"], a["u"], a["x_init"], a["x_last"],
                                 a["ws"], a["wsb"], a["st"])


def test_host_validation_rejects_bad_arguments(lib):
    # pointers are never dereferenced: validation fails before any CUDA call
    assert _conv_fwd(lib, dt=7) == -2
    assert _conv_fwd(lib, W=5) == -6
    assert _conv_fwd(lib, D=0) == -1
    assert _conv_fwd(lib, D=6) == -3            # 6 * 4 bytes is not a multiple of 16
    assert _conv_fwd(lib, dt=1, D=4) == -3       # 4 * 2 bytes
    assert _conv_fwd(lib, x=8) == -3             # misaligned pointer
    assert _conv_fwd(lib, x_init=8) == -3        # misaligned tail array
    assert _conv_fwd(lib, cu=None) == -1
    assert _conv_fwd(lib, wsb=16) == -4
    assert "workspace" in binding.last_error()
    assert _conv_fwd(lib, ws=None) == -4
    assert _conv_fwd(lib, T=-1) == -1
    scan = lib.varlen_selective_scan_fwd
    args = [16, 16, 16, 16, 16, None, None, None, 1, 0.0, 0, 16, None, 1, 16, 8, 3, 0, 16, None, None, None,
            None, 16, 1 << 30, None]
    assert scan(*args) == -6                     # N = 3
    args[16] = 4
    args[17] = 1
    assert scan(*args) == -3                     # N * 2 bytes = 8
    args[17] = 0
    args[19] = 8
    assert scan(*args) == -3                     # misaligned y
    args[19] = None
    args[21] = 8
    assert scan(*args) == -3                     # misaligned initial_states
    args[21] = None
    args[13] = 0
    args[21] = 16
    assert scan(*args) == -1                     # initial states for 16 tokens but no sequence
    args[13] = 1
    args[21] = None
    args[23] = None
    assert scan(*args) == -4


def test_debug_knobs(lib):
    assert lib.vssm_debug_set(99, 0) == -1
    assert lib.vssm_debug_set(binding.VSSM_DBG_WAIT_NS, 0) == -1
    assert lib.vssm_debug_set(binding.VSSM_DBG_WAIT_NS, 10**9) == 0
    assert lib.vssm_debug_set(binding.VSSM_DBG_DROP_FLAG, -1) == 0
    assert lib.vssm_debug_set(binding.VSSM_DBG_DELAY_NS, 0) == -1
    assert lib.vssm_debug_set(binding.VSSM_DBG_DELAY_NS, 10**8) == -1
    assert lib.vssm_debug_set(binding.VSSM_DBG_DELAY_NS, 200_000) == 0
    assert lib.vssm_debug_set(binding.VSSM_DBG_DELAY_ITEM, -1) == 0
    assert lib.vssm_debug_set(binding.VSSM_DBG_FORCE_COPY_TIMEOUT, -1) == 0
    assert lib.vssm_debug_set(binding.VSSM_DBG_CHECK_FINITE, 2) == -1
    assert lib.vssm_debug_set(binding.VSSM_DBG_CHECK_FINITE, 0) == 0
    assert lib.vssm_debug_set(binding.VSSM_DBG_KERNEL_EVENTS, 3) == -1
    assert lib.vssm_debug_set(binding.VSSM_DBG_KERNEL_EVENTS, 0) == 0
    assert binding.kernel_time("scan_bwd") == (0.0, 0)  # nothing recorded
    import ctypes
    ms, n = ctypes.c_double(), ctypes.c_int64()
    assert lib.vssm_kernel_time(9, ctypes.byref(ms), ctypes.byref(n)) == -1
