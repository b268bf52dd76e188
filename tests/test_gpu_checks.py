"""Failure detection on the GPU, without a GPU fault: the optional
non-finite check of the outputs (VSSM_DBG_CHECK_FINITE) and the checked
build of the library (VSSM_CHECKS=1).  Both report through the call's
status word; nothing traps."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import selective_ssm_packed_gb300 as vs
from selective_ssm_packed_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_ssm_packed_gb300 import build
    build.build()
    binding.lib()


def _dv(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


@pytest.fixture
def finite_check():
    binding.debug_set(binding.VSSM_DBG_CHECK_FINITE, 1)
    try:
        yield
    finally:
        binding.debug_set(binding.VSSM_DBG_CHECK_FINITE, 0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_nonfinite_outputs_are_reported_when_the_check_is_on(finite_check, dtype):
    """A NaN in one input value reaches the outputs of the scan's forward
    call, and an infinity in x those of the conv call; the knob makes each
    call report VSSM_ERR_NONFINITE.  Clean inputs stay clean, and with the
    knob off the same bad inputs go unreported."""
    lengths = [200, 1, 77, 300]
    D, N, W = 64, 16, 4
    cu_np = workloads.cu_seqlens_from_lengths(lengths)
    T = int(cu_np[-1])
    r = workloads.draw_values(T, D, N, W, 61, scan_input=True, params="general")
    cu = torch.from_numpy(cu_np).cuda()
    pos = vs.varlen_position_indices(cu, T)
    io = lambda k: _dv(r[k]).to(dtype)  # noqa: E731
    args = dict(delta_raw=io("delta_raw"), A=_dv(r["A"]), B=io("B"), C=io("C"), Dskip=_dv(r["Dskip"]),
                z=io("z"), dt_bias=_dv(r["dt_bias"]))
    ws = torch.empty(binding.scan_bwd_workspace_size(T, D, N), dtype=torch.uint8, device="cuda")
    wsc = torch.empty(binding.conv1d_fwd_workspace_size(T, D, W), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(binding.conv1d_bwd_workspace_size(T, D, W), dtype=torch.uint8, device="cuda")
    u, x = io("u"), io("x")
    w, b = _dv(r["conv_w"]), _dv(r["conv_b"])

    # clean inputs: every call's status stays clean with the check on
    out, states, y = vs.varlen_selective_scan_fwd(u, **args, cu_seqlens=cu, position_indices=pos, y=True,
                                                  workspace=ws)
    assert binding.read_status(ws) == 0
    g = vs.varlen_selective_scan_bwd(u, **args, dout=io("dout"), cu_seqlens=cu, chunk_states=states,
                                     position_indices=pos, y=y, workspace=ws)
    assert binding.read_status(ws) == 0
    vs.varlen_conv1d_fwd(x, w, b, cu, pos, workspace=wsc)
    assert binding.read_status(wsc) == 0
    vs.varlen_conv1d_bwd(x, w, b, g["du"], cu, pos, workspace=wsb)
    assert binding.read_status(wsb) == 0

    # one bad value: a NaN in u (token 250, channel 5), an infinity in x
    u_bad = u.clone()
    u_bad[250, 5] = float("nan")
    vs.varlen_selective_scan_fwd(u_bad, **args, cu_seqlens=cu, position_indices=pos, workspace=ws)
    assert binding.read_status(ws) == -18
    dout_bad = io("dout").clone()
    dout_bad[T - 1, D - 1] = float("nan")
    vs.varlen_selective_scan_bwd(u, **args, dout=dout_bad, cu_seqlens=cu, chunk_states=states,
                                 position_indices=pos, workspace=ws)
    assert binding.read_status(ws) == -18
    x_bad = x.clone()
    x_bad[0, 0] = float("inf")
    vs.varlen_conv1d_fwd(x_bad, w, b, cu, pos, workspace=wsc)
    assert binding.read_status(wsc) == -18

    # the knob off: nothing checks, nothing is reported
    binding.debug_set(binding.VSSM_DBG_CHECK_FINITE, 0)
    vs.varlen_selective_scan_fwd(u_bad, **args, cu_seqlens=cu, position_indices=pos, workspace=ws)
    assert binding.read_status(ws) == 0


def test_position_indices_are_trusted_by_the_ordinary_build():
    """The ordinary build does not check caller-supplied position indices
    (the checked build does; see the next test)."""
    assert binding.lib().vssm_checks_build() == 0
    lengths = [100, 60]
    D, N = 32, 8
    cu_np = workloads.cu_seqlens_from_lengths(lengths)
    T = int(cu_np[-1])
    r = workloads.draw_values(T, D, N, 4, 62, scan_input=True, params="general")
    cu = torch.from_numpy(cu_np).cuda()
    bad = vs.varlen_position_indices(cu, T).clone()
    bad[130] += 1
    ws = torch.empty(binding.scan_fwd_workspace_size(T, D, N), dtype=torch.uint8, device="cuda")
    vs.varlen_selective_scan_fwd(_dv(r["u"]), _dv(r["delta_raw"]), _dv(r["A"]), _dv(r["B"]), _dv(r["C"]),
                                 None, None, None, cu, position_indices=bad, workspace=ws)
    assert binding.read_status(ws) == 0


def test_checked_build_gives_the_same_results_and_reports_bad_position_indices():
    """The VSSM_CHECKS=1 build, in a child process: conv and scan forward and
    backward with sequence states and conv tails match the oracle with a
    clean status word, and position indices that disagree with cu_seqlens
    are reported as VSSM_ERR_BAD_CU_SEQLENS."""
    env = dict(os.environ, VSSM_CHECKS="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_build_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout[-3000:] + r.stderr[-3000:]


def test_kernel_event_timing_counts_each_main_kernel():
    """VSSM_DBG_KERNEL_EVENTS: each call records one event pair around its
    main kernel; vssm_kernel_time returns the launches and their time, then
    forgets them; with the knob off nothing is recorded."""
    lengths = [300, 1, 77]
    D, N, W = 64, 16, 4
    cu_np = workloads.cu_seqlens_from_lengths(lengths)
    T = int(cu_np[-1])
    r = workloads.draw_values(T, D, N, W, 63, scan_input=True, params="general")
    cu = torch.from_numpy(cu_np).cuda()
    pos = vs.varlen_position_indices(cu, T)
    bf = lambda k: _dv(r[k]).to(torch.bfloat16)  # noqa: E731
    args = dict(delta_raw=bf("delta_raw"), A=_dv(r["A"]), B=bf("B"), C=bf("C"), Dskip=_dv(r["Dskip"]),
                z=bf("z"), dt_bias=_dv(r["dt_bias"]))
    try:
        binding.debug_set(binding.VSSM_DBG_KERNEL_EVENTS, 1)
        for _ in range(3):
            out, states = vs.varlen_selective_scan_fwd(bf("u"), **args, cu_seqlens=cu, position_indices=pos)
        vs.varlen_selective_scan_bwd(bf("u"), **args, dout=bf("dout"), cu_seqlens=cu, chunk_states=states,
                                     position_indices=pos)
        vs.varlen_conv1d_fwd(bf("x"), _dv(r["conv_w"]), _dv(r["conv_b"]), cu, pos)
        ms, n = binding.kernel_time("scan_fwd")
        assert n == 3 and ms > 0.0
        ms, n = binding.kernel_time("scan_bwd")
        assert n == 1 and ms > 0.0
        ms, n = binding.kernel_time("conv_fwd")
        assert n == 1 and ms > 0.0
        assert binding.kernel_time("scan_fwd") == (0.0, 0)  # read and forgotten
        assert binding.kernel_time("conv_bwd") == (0.0, 0)  # never launched
    finally:
        binding.debug_set(binding.VSSM_DBG_KERNEL_EVENTS, 0)
    vs.varlen_selective_scan_fwd(bf("u"), **args, cu_seqlens=cu, position_indices=pos)
    torch.cuda.synchronize()
    assert binding.kernel_time("scan_fwd") == (0.0, 0)
