"""Runs in a child process with VSSM_CHECKS=1 (test_gpu_checks.py starts it):
the checked build of the library must give the ordinary results on good
inputs, with a clean status word, and report position indices that
disagree with cu_seqlens as VSSM_ERR_BAD_CU_SEQLENS.  Prints OK at the end.

A child of its own because a process loads one build of the library: the
binding picks the checked one from the environment."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
import selective_ssm_packed_gb300 as vs  # noqa: E402
from selective_ssm_packed_gb300 import binding, build, workloads  # noqa: E402


def close(name, got, ref, tol=2e-4):
    got = got.double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), name
    err = float(np.max(np.abs(got - ref)))
    scale = float(np.max(np.abs(ref)))
    assert err <= tol * max(scale, 1e-30), f"{name}: {err:.3e} > {tol} * {scale:.3e}"


def main():
    assert os.environ.get("VSSM_CHECKS") == "1"
    build.build(checks=True)
    oracle.build()
    assert binding.library_path() == build.CHECKS_LIB_PATH
    assert binding.lib().vssm_checks_build() == 1

    # conv (with tails) -> scan (with sequence states) forward and backward:
    # every state row the kernels index is checked, and all must pass
    lengths = [128, 32, 1, 0, 95, 2, 300, 64]
    D, N, W = 64, 16, 4
    cu_np = workloads.cu_seqlens_from_lengths(lengths)
    T, S = int(cu_np[-1]), len(lengths)
    r = workloads.draw_values(T, D, N, W, 51, scan_input=False, params="general")
    rng = np.random.default_rng(52)
    h0, dfin = rng.standard_normal((2, S, D, N)).astype(np.float32)
    xi, dxl = rng.standard_normal((2, S, D, W - 1)).astype(np.float32)
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()  # noqa: E731
    cu = dv(cu_np).to(torch.int32)
    pos = vs.varlen_position_indices(cu, T)
    ws = torch.empty(binding.scan_bwd_workspace_size(T, D, N), dtype=torch.uint8, device="cuda")
    wsc = torch.empty(binding.conv1d_fwd_workspace_size(T, D, W), dtype=torch.uint8, device="cuda")

    x = dv(r["x"])
    u, _ = vs.varlen_conv1d_fwd(x, dv(r["conv_w"]), dv(r["conv_b"]), cu, pos, workspace=wsc,
                                x_init=dv(xi), x_last=True)
    assert binding.read_status(wsc) == 0
    args = dict(u=u, delta_raw=dv(r["delta_raw"]), A=dv(r["A"]), B=dv(r["B"]), C=dv(r["C"]),
                Dskip=dv(r["Dskip"]), z=dv(r["z"]), dt_bias=dv(r["dt_bias"]))
    out, states, fin = vs.varlen_selective_scan_fwd(**args, cu_seqlens=cu, position_indices=pos, workspace=ws,
                                                    initial_states=dv(h0), final_states=True)
    assert binding.read_status(ws) == 0
    g = vs.varlen_selective_scan_bwd(**args, dout=dv(r["dout"]), cu_seqlens=cu, chunk_states=states,
                                     position_indices=pos, workspace=ws, initial_states=dv(h0),
                                     d_final_states=dv(dfin), d_initial_states=True)
    assert binding.read_status(ws) == 0
    wsb = torch.empty(max(binding.conv1d_bwd_workspace_size(T, D, W), 256), dtype=torch.uint8, device="cuda")
    dx, dw, db, dxi = vs.varlen_conv1d_bwd(x, dv(r["conv_w"]), dv(r["conv_b"]), g["du"], cu, pos,
                                           workspace=wsb, x_init=dv(xi), dx_last=dv(dxl), dx_init=True)
    assert binding.read_status(wsb) == 0
    torch.cuda.synchronize()

    u_ref = oracle.conv1d_fwd(r["x"], r["conv_w"], r["conv_b"], cu_np, x_init=xi)
    close("u", u, u_ref)
    sargs = [u.double().cpu().numpy(), r["delta_raw"], r["A"], r["B"], r["C"], r["Dskip"], r["z"], r["dt_bias"]]
    out_ref, fin_ref = oracle.scan_fwd(*sargs, cu_np, h_init=h0, return_last_state=True)
    close("out", out, out_ref)
    close("final_states", fin, fin_ref)
    ref = oracle.scan_bwd_threaded(*sargs, r["dout"], cu_np, h_init=h0, dh_last=dfin)
    for k in ("du", "ddelta_raw", "dz", "dA", "dB", "dC", "dDskip", "d_dt_bias"):
        close(k, g[k], ref[k])
    close("d_initial_states", g["d_initial_states"], ref["dh_init"])
    cref = oracle.conv1d_bwd(r["x"], r["conv_w"], r["conv_b"], g["du"].double().cpu().numpy(), cu_np,
                             x_init=xi, dx_last=dxl, return_dx_init=True)
    for name, got, want in zip(("dx", "dweight", "dbias", "dx_init"), (dx, dw, db, dxi), cref):
        close(name, got, want)

    # position indices off by one inside the second sequence: the ordinary
    # build trusts them, the checked build reports them
    bad = pos.clone()
    bad[130] += 1
    vs.varlen_selective_scan_fwd(**args, cu_seqlens=cu, position_indices=bad, workspace=ws)
    assert binding.read_status(ws) == -16, binding.read_status(ws)
    # and the next call with good indices is clean again
    vs.varlen_selective_scan_fwd(**args, cu_seqlens=cu, position_indices=pos, workspace=ws)
    assert binding.read_status(ws) == 0
    print("OK")


if __name__ == "__main__":
    main()
