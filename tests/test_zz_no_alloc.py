"""The allocation-free forward scan, varlen_selective_scan_fwd_noalloc.

Callers that cannot allocate device memory where they run the scan (inside an
allocator's own callbacks, under a runtime that reserved the whole device up
front, or on a hot path where allocation is forbidden) use this entry point:
it keeps its look-back scratch in a fixed array built into the library instead
of a caller-supplied workspace.  This test calls it through the C ABI and
checks it against the ordinary entry point on two calls in a row (different
shapes, so whatever the first call leaves in the shared scratch must not leak
into the second), then checks that an oversized problem is refused up front.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

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
    r = workloads.rounded(workloads.draw_values(T, D, N, 4, seed, backward=False), dtype)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dt)  # noqa: E731
    t = {k: dev(r[k], TDT[dtype]) for k in ("u", "delta_raw", "z", "B", "C")}
    t.update({k: dev(r[k], torch.float32) for k in ("A", "Dskip", "dt_bias")})
    t["cu"] = torch.from_numpy(cu).cuda()
    return T, t


def _p(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _noalloc(lib, t, T, D, N, dtype, out, states, status, pos=None, y=None):
    return lib.varlen_selective_scan_fwd_noalloc(
        _p(t["u"]), _p(t["delta_raw"]), _p(t["A"]), _p(t["B"]), _p(t["C"]), _p(t["Dskip"]), _p(t["z"]),
        _p(t["dt_bias"]), 1, 0.0, 0, _p(t["cu"]), _p(pos), t["cu"].numel() - 1, T, D, N,
        binding.VSSM_F32 if dtype == "f32" else binding.VSSM_BF16, _p(out), _p(y), _p(states), None, None,
        _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(name, got, ref, tol):
    got, ref = got.double().cpu(), ref.double().cpu()
    assert torch.isfinite(got).all(), name
    err = (got - ref).abs().max().item()
    scale = ref.abs().max().item()
    assert err <= tol * max(scale, 1e-30), f"{name}: {err:.3e} > {tol} * {scale:.3e}"


def test_noalloc_forward_matches_the_workspace_entry_point_on_two_calls(lib):
    cases = [([700, 1, 33, 2000, 129, 1], 256, 16, "bf16", 41),   # first call: larger
             ([5, 300, 1, 90], 72, 8, "f32", 42)]                  # second call: smaller
    for lengths, D, N, dtype, seed in cases:
        T, t = _case(lengths, D, N, dtype, seed)
        ref_out, ref_states, ref_y = vs.varlen_selective_scan_fwd(
            t["u"], t["delta_raw"], t["A"], t["B"], t["C"], t["Dskip"], t["z"], t["dt_bias"], t["cu"], y=True)
        out = torch.full_like(t["u"], float("nan"))
        y = torch.full_like(t["u"], float("nan"))
        states = torch.full_like(ref_states, float("nan"))
        status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
        rc = _noalloc(lib, t, T, D, N, dtype, out, states, status, y=y)
        assert rc == 0, binding.last_error()
        torch.cuda.synchronize()
        assert binding.status_code(int(status.item())) == 0
        _close("out", out, ref_out, TOL[dtype])
        _close("y", y, ref_y, TOL[dtype])
        _close("chunk_states", states, ref_states, TOL[dtype])


def test_noalloc_refuses_a_problem_larger_than_its_scratch(lib):
    T, t = _case([64], 64, 16, "bf16", 43)
    out = torch.empty_like(t["u"])
    # claims 16384 tokens at D = 4096; refused on the host before any launch
    rc = lib.varlen_selective_scan_fwd_noalloc(
        _p(t["u"]), _p(t["delta_raw"]), _p(t["A"]), _p(t["B"]), _p(t["C"]), None, None, None, 1, 0.0, 0,
        _p(t["cu"]), None, 1, 16384, 4096, 16, binding.VSSM_BF16, _p(out), None, None, None, None, None,
        None)
    assert rc == -4
    msg = binding.last_error()
    assert "scratch" in msg and str(64 << 20) in msg
