"""The allocation-free forward scan, varlen_selective_scan_fwd_noalloc.

Callers that cannot allocate device memory where they run the scan (inside an
allocator's own callbacks, under a runtime that reserved the whole device up
front, or on a hot path where allocation is forbidden) use this entry point:
it keeps its look-back scratch in a fixed array built into the library instead
of a caller-supplied workspace.  This test calls it through the C ABI and
checks it against the ordinary entry point on calls in a row (different
shapes, so whatever one call leaves in the shared scratch must not leak into
the next).  Both entry points run the same kernel on the same inputs, so their
results must agree bit for bit; each result is also checked against the CPU
oracle.  The calls cover the library building the position indices itself
and the caller passing them, per-sequence initial and final states, and a call
without a status word (errors then land in the scratch's own header).  An
oversized problem must be refused up front.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import selective_ssm_packed_gb300 as vs
from selective_ssm_packed_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-4, "bf16": 1e-2}
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def lib():
    from selective_ssm_packed_gb300 import build
    build.build()
    return binding.lib()


def _case(lengths, D, N, dtype, seed):
    cu = workloads.cu_seqlens_from_lengths(lengths)
    T = int(cu[-1])
    r = workloads.rounded(workloads.draw_values(T, D, N, 4, seed, backward=False, params="general"), dtype)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dt)  # noqa: E731
    t = {k: dev(r[k], TDT[dtype]) for k in ("u", "delta_raw", "z", "B", "C")}
    t.update({k: dev(r[k], torch.float32) for k in ("A", "Dskip", "dt_bias")})
    t["cu"] = torch.from_numpy(cu).cuda()
    return T, t, r, cu


def _p(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _noalloc(lib, t, T, D, N, dtype, out, states, status, pos=None, y=None, h0=None, fin=None):
    return lib.varlen_selective_scan_fwd_noalloc(
        _p(t["u"]), _p(t["delta_raw"]), _p(t["A"]), _p(t["B"]), _p(t["C"]), _p(t["Dskip"]), _p(t["z"]),
        _p(t["dt_bias"]), 1, 0.0, 0, _p(t["cu"]), _p(pos), t["cu"].numel() - 1, T, D, N,
        binding.VSSM_F32 if dtype == "f32" else binding.VSSM_BF16, _p(out), _p(y), _p(states), _p(h0), _p(fin),
        _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(name, got, ref, tol):
    got, ref = got.double().cpu(), ref.double().cpu()
    assert torch.isfinite(got).all(), name
    err = (got - ref).abs().max().item()
    scale = ref.abs().max().item()
    assert err <= tol * max(scale, 1e-30), f"{name}: {err:.3e} > {tol} * {scale:.3e}"


def _check_against_oracle(r, cu, out, y, fin, dtype, h0=None):
    """The no-alloc results against the double-precision CPU oracle."""
    args = [r["u"], r["delta_raw"], r["A"], r["B"], r["C"], r["Dskip"], r["z"], r["dt_bias"]]
    if h0 is None:
        out_ref = oracle.scan_fwd_threaded(*args, cu)
    else:
        out_ref, fin_ref = oracle.scan_fwd(*args, cu, h_init=h0, return_last_state=True)
        _close("final_states vs oracle", fin, torch.from_numpy(fin_ref), TOL[dtype])
    _close("out vs oracle", out, torch.from_numpy(out_ref), TOL[dtype])
    if y is not None:  # the output before the gate: the oracle's output with no gate
        if h0 is None:
            y_ref = oracle.scan_fwd_threaded(*args[:6], None, args[7], cu)
        else:
            y_ref = oracle.scan_fwd(*args[:6], None, args[7], cu, h_init=h0)
        _close("y vs oracle", y, torch.from_numpy(y_ref), TOL[dtype])


# Calls in a row on one process's shared scratch: a larger problem, a smaller
# one with a different N and dtype, then one with sequence states and the
# caller's position indices and no status word.
CALLS = [
    dict(lengths=[700, 1, 33, 2000, 129, 1], D=256, N=16, dtype="bf16", seed=41),
    dict(lengths=[5, 300, 1, 90], D=72, N=8, dtype="f32", seed=42),
    dict(lengths=[128, 1, 0, 95, 300, 33], D=64, N=16, dtype="f32", seed=44, states=True, own_pos=True,
         no_status=True),
]


def test_noalloc_forward_matches_the_workspace_entry_point_on_calls_in_a_row(lib):
    for c in CALLS:
        D, N, dtype = c["D"], c["N"], c["dtype"]
        T, t, r, cu = _case(c["lengths"], D, N, dtype, c["seed"])
        S = len(c["lengths"])
        h0 = None
        if c.get("states"):
            h0 = np.random.default_rng(c["seed"] + 1).standard_normal((S, D, N)).astype(np.float32)
        h0_t = torch.from_numpy(h0).cuda() if h0 is not None else None
        pos = vs.varlen_position_indices(t["cu"], T) if c.get("own_pos") else None
        ref = vs.varlen_selective_scan_fwd(
            t["u"], t["delta_raw"], t["A"], t["B"], t["C"], t["Dskip"], t["z"], t["dt_bias"], t["cu"],
            position_indices=pos, y=True, initial_states=h0_t, final_states=h0 is not None)
        ref_out, ref_states, ref_y = ref[0], ref[1], ref[2]
        out = torch.full_like(t["u"], float("nan"))
        y = torch.full_like(t["u"], float("nan"))
        states = torch.full_like(ref_states, float("nan"))
        fin = torch.full((S, D, N), float("nan"), device="cuda") if h0 is not None else None
        status = None if c.get("no_status") else torch.full((1,), 7, dtype=torch.int32, device="cuda")
        rc = _noalloc(lib, t, T, D, N, dtype, out, states, status, pos=pos, y=y, h0=h0_t, fin=fin)
        assert rc == 0, binding.last_error()
        torch.cuda.synchronize()
        if status is not None:
            assert binding.status_code(int(status.item())) == 0
        # the same kernel on the same inputs: identical results
        assert torch.equal(out, ref_out), "out differs from the workspace entry point"
        assert torch.equal(y, ref_y), "y differs from the workspace entry point"
        assert torch.equal(states, ref_states), "chunk_states differ from the workspace entry point"
        if fin is not None:
            assert torch.equal(fin, ref[3]), "final_states differ from the workspace entry point"
        _check_against_oracle(r, cu, out, y, fin, dtype, h0=h0)


def test_noalloc_refuses_a_problem_larger_than_its_scratch(lib):
    T, t, _, _ = _case([64], 64, 16, "bf16", 43)
    out = torch.empty_like(t["u"])
    # claims 16384 tokens at D = 4096; refused on the host before any launch
    rc = lib.varlen_selective_scan_fwd_noalloc(
        _p(t["u"]), _p(t["delta_raw"]), _p(t["A"]), _p(t["B"]), _p(t["C"]), None, None, None, 1, 0.0, 0,
        _p(t["cu"]), None, 1, 16384, 4096, 16, binding.VSSM_BF16, _p(out), None, None, None, None, None,
        None)
    assert rc == -4
    msg = binding.last_error()
    assert "scratch" in msg and str(64 << 20) in msg


def test_noalloc_reports_a_lookback_wait_that_runs_out(lib):
    """The test knobs of vssm_debug_set apply to this entry point too: a work
    item that never publishes its look-back state makes the next one's wait
    run out (after 1 ms); the call completes and its status word reports the
    timeout, and the next call is clean and equals the workspace entry point
    bit for bit."""
    T, t, r, cu = _case([1024], 32, 16, "f32", 45)
    out = torch.empty_like(t["u"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        binding.debug_set(binding.VSSM_DBG_WAIT_NS, 1_000_000)
        binding.debug_set(binding.VSSM_DBG_DROP_FLAG, 3)
        assert _noalloc(lib, t, T, 32, 16, "f32", out, None, status) == 0, binding.last_error()
        torch.cuda.synchronize()
        assert binding.status_code(int(status.item())) == -17
    finally:
        binding.debug_set(binding.VSSM_DBG_DROP_FLAG, -1)
        binding.debug_set(binding.VSSM_DBG_WAIT_NS, 1_000_000_000)
    assert _noalloc(lib, t, T, 32, 16, "f32", out, None, status) == 0, binding.last_error()
    torch.cuda.synchronize()
    assert binding.status_code(int(status.item())) == 0
    ref = vs.varlen_selective_scan_fwd(t["u"], t["delta_raw"], t["A"], t["B"], t["C"], t["Dskip"], t["z"],
                                       t["dt_bias"], t["cu"], chunk_states=False)
    assert torch.equal(out, ref[0])
