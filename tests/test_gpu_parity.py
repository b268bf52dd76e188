"""GPU parity: every C-ABI call against the CPU oracle on the same seeded inputs.

Tolerances (per output tensor, from the scan's arithmetic: fp32 state and
accumulation, MUFU ex2 with ~2^-22 relative error, bf16 rounding once at the
store):  fp32 I/O  max|gpu - ref| <= 2e-4 * max|ref|;  bf16 I/O  <= 1e-2 *
max|ref|.  Integer outputs (position indices, status codes) are compared
exactly, and the packing invariants (a sequence's outputs do not depend on its
neighbours; repeated runs agree) bit for bit.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import selective_ssm_packed_gb300 as vs
from selective_ssm_packed_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = {"f32": 2e-4, "bf16": 1e-2}
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_ssm_packed_gb300 import build
    build.build()
    oracle.build()
    binding.lib()


def dev(a, dtype="f32"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(TDT[dtype])


def f32(a):
    return dev(a, "f32")


def host(t):
    return t.double().cpu().numpy()


def assert_close(name, got, ref, tol):
    got = host(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = float(np.max(np.abs(got - ref)))
    scale = float(np.max(np.abs(ref)))
    assert err <= tol * max(scale, 1e-30), f"{name}: max|err| {err:.3e} > {tol:g} * max|ref| {scale:.3e}"


def rand_case(lengths, D, N, dtype, seed, W=4, params="general"):
    """A seeded case; by default A and Dskip are drawn as a learned layer holds
    them (A = -U(0.05, 4) per entry, Dskip ~ N(0, 1)), so no kernel can lean on
    the S4D-real initialisation A = -(n + 1)."""
    cu = workloads.cu_seqlens_from_lengths(lengths)
    T = int(cu[-1])
    r = workloads.rounded(workloads.draw_values(T, D, N, W, seed, scan_input=False, params=params), dtype)
    return cu, T, r


def run_chain(cu_np, T, r, dtype, with_bwd=True, z=True, skip=True, bias=True, softplus=True, use_y=False):
    """conv fwd -> scan fwd (-> scan bwd -> conv bwd) through the C ABI.  use_y:
    the forward also writes its pre-gate output and the backward takes it (the
    bench step's configuration)."""
    cu = torch.from_numpy(cu_np).cuda()
    pos = vs.varlen_position_indices(cu, T)
    x = dev(r["x"], dtype)
    u = vs.varlen_conv1d_fwd(x, f32(r["conv_w"]), f32(r["conv_b"]), cu, pos)
    args = dict(u=u, delta_raw=dev(r["delta_raw"], dtype), A=f32(r["A"]), B=dev(r["B"], dtype),
                C=dev(r["C"], dtype), Dskip=f32(r["Dskip"]) if skip else None,
                z=dev(r["z"], dtype) if z else None, dt_bias=f32(r["dt_bias"]) if bias else None)
    y = None
    if use_y:
        out, states, y = vs.varlen_selective_scan_fwd(**args, cu_seqlens=cu, position_indices=pos,
                                                      delta_softplus=softplus, y=True)
    else:
        out, states = vs.varlen_selective_scan_fwd(**args, cu_seqlens=cu, position_indices=pos,
                                                   delta_softplus=softplus)
    res = dict(pos=pos, u=u, out=out, states=states)
    if y is not None:
        res["y"] = y
    if with_bwd:
        g = vs.varlen_selective_scan_bwd(**args, dout=dev(r["dout"], dtype), cu_seqlens=cu,
                                         chunk_states=states, position_indices=pos,
                                         delta_softplus=softplus, y=y)
        dx, dw, db = vs.varlen_conv1d_bwd(x, f32(r["conv_w"]), f32(r["conv_b"]), g["du"], cu, pos)
        res.update(g)
        res.update(dx=dx, dweight=dw, dbias=db)
    torch.cuda.synchronize()
    return res


def check_chain(cu_np, r, res, dtype, with_bwd=True, z=True, skip=True, bias=True, softplus=True,
                channels=None):
    """Compare a run_chain result with the oracle, optionally on a channel subset
    (every channel is an independent computation, so a column subset of the
    inputs gives exactly those columns of every per-channel output)."""
    tol = TOL[dtype]
    idx = np.arange(r["A"].shape[0]) if channels is None else np.asarray(channels)
    col = lambda a: a[:, idx]  # noqa: E731
    u_gpu = host(res["u"])
    assert_close("u", col(u_gpu),
                 oracle.conv1d_fwd_threaded(col(r["x"]), r["conv_w"][idx], r["conv_b"][idx], cu_np), tol)
    sargs = [col(u_gpu), col(r["delta_raw"]), r["A"][idx], r["B"], r["C"],
             r["Dskip"][idx] if skip else None, col(r["z"]) if z else None,
             r["dt_bias"][idx] if bias else None]
    assert_close("out", col(host(res["out"])),
                 oracle.scan_fwd_threaded(*sargs, cu_np, delta_softplus=softplus), tol)
    if "y" in res:  # the output before the gate: the oracle's output with no gate
        assert_close("y", col(host(res["y"])),
                     oracle.scan_fwd_threaded(*sargs[:6], None, sargs[7], cu_np, delta_softplus=softplus), tol)
    if not with_bwd:
        return
    g = oracle.scan_bwd_threaded(*sargs, col(r["dout"]), cu_np, delta_softplus=softplus)
    for k in ("du", "ddelta_raw", "dz"):
        if g[k] is not None:
            assert_close(k, col(host(res[k])), g[k], tol)
    assert_close("dA", host(res["dA"])[idx], g["dA"], tol)
    if skip:
        assert_close("dDskip", host(res["dDskip"])[idx], g["dDskip"], tol)
    if bias:
        assert_close("d_dt_bias", host(res["d_dt_bias"])[idx], g["d_dt_bias"], tol)
    if channels is None:
        assert_close("dB", res["dB"], g["dB"], tol)
        assert_close("dC", res["dC"], g["dC"], tol)
    dx, dw, db = oracle.conv1d_bwd_threaded(col(r["x"]), r["conv_w"][idx], r["conv_b"][idx],
                                            col(host(res["du"])), cu_np)
    assert_close("dx", col(host(res["dx"])), dx, tol)
    assert_close("dweight", host(res["dweight"])[idx], dw, tol)
    assert_close("dbias", host(res["dbias"])[idx], db, tol)


# ------------------------------------------------------------------ position indices

def test_position_indices_golden_example():
    with open(os.path.join(GOLDEN, "position_indices_4_2_3_7.txt")) as f:
        rows = [list(map(int, ln.split())) for ln in f if ln.strip() and not ln.startswith("#")]
    cu = torch.tensor(rows[1], dtype=torch.int32, device="cuda")
    pos = vs.varlen_position_indices(cu, 16)
    assert pos.cpu().tolist() == rows[2]


def test_position_indices_random_with_empty_sequences():
    rng = np.random.default_rng(3)
    lengths = [int(v) for v in rng.integers(0, 300, size=2000)]
    lengths[5:15] = [0] * 10
    cu_np = workloads.cu_seqlens_from_lengths(lengths)
    T = int(cu_np[-1])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = vs.varlen_position_indices(torch.from_numpy(cu_np).cuda(), T, status=status)
    assert np.array_equal(pos.cpu().numpy(), oracle.position_indices(cu_np))
    assert binding.status_code(int(status.item())) == 0


@pytest.mark.parametrize("cu", [[1, 4, 6], [0, 4, 3, 6], [0, 2, 5]])
def test_position_indices_reports_malformed_cu_seqlens(cu):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    vs.varlen_position_indices(torch.tensor(cu, dtype=torch.int32, device="cuda"), 6, status=status)
    assert binding.status_code(int(status.item())) == -16


def test_malformed_cu_seqlens_reach_the_call_status():
    # the scan call builds its own position indices and reports through the workspace
    cu = torch.tensor([0, 5, 3, 16], dtype=torch.int32, device="cuda")
    T, D, N = 16, 8, 4
    u = torch.randn(T, D, device="cuda")
    ws = torch.empty(binding.scan_fwd_workspace_size(T, D, N), dtype=torch.uint8, device="cuda")
    vs.varlen_selective_scan_fwd(u, u, -torch.ones(D, N, device="cuda"), torch.randn(T, N, device="cuda"),
                                 torch.randn(T, N, device="cuda"), None, None, None, cu, workspace=ws)
    assert binding.read_status(ws) == -16


# ------------------------------------------------------------------ small exact-parity cases

def test_tiny_worked_example_fwd_bwd():
    w = workloads.make("tiny")
    r = workloads.rounded(w, "f32")
    res = run_chain(w["cu_seqlens"], w["T"], r, "f32")
    assert res["pos"].cpu().tolist() == [0, 1, 2, 3, 0, 1, 0, 1, 2, 0, 1, 2, 3, 4, 5, 6]
    check_chain(w["cu_seqlens"], r, res, "f32")


CASES = [
    # lengths, D, N, dtype (D = 104 and 320 leave a partial 64-channel tile; D = 48
    # is narrower than one; 256 and 320 span several tiles)
    ([1, 1, 2, 3, 700, 1, 40, 129, 5], 40, 4, "f32"),
    ([300, 0, 1, 257, 0, 0, 33, 128, 2], 72, 8, "f32"),
    ([1000, 31, 1, 64, 200], 48, 16, "f32"),
    ([513, 1, 7, 90, 300, 1], 64, 8, "bf16"),
    ([129, 1, 1, 1, 640, 77], 104, 16, "bf16"),
    ([700, 3, 1, 290, 33, 1000], 256, 16, "bf16"),
    ([5, 640, 1, 2, 380], 320, 16, "f32"),
]


@pytest.mark.parametrize("lengths,D,N,dtype", CASES)
def test_ragged_packs_fwd_bwd(lengths, D, N, dtype):
    cu, T, r = rand_case(lengths, D, N, dtype, seed=sum(lengths) + D + N)
    res = run_chain(cu, T, r, dtype)
    check_chain(cu, r, res, dtype)


@pytest.mark.parametrize("lengths,D,N,dtype", [([300, 1, 2, 257, 40], 72, 8, "f32"),
                                               ([129, 1, 640, 77, 3], 104, 16, "bf16")])
def test_backward_reads_the_forward_pre_gate_output(lengths, D, N, dtype):
    """The forward call's optional y output is the pre-gate output (the oracle's
    output with no gate); the backward call that takes it computes dz from it
    and leaves every other gradient bitwise unchanged."""
    cu_np, T, r = rand_case(lengths, D, N, dtype, seed=sum(lengths) + 7)
    cu = torch.from_numpy(cu_np).cuda()
    pos = vs.varlen_position_indices(cu, T)
    u = dev(r["x"], dtype)  # any (T, D) input serves as the scan's u here
    args = dict(u=u, delta_raw=dev(r["delta_raw"], dtype), A=f32(r["A"]), B=dev(r["B"], dtype),
                C=dev(r["C"], dtype), Dskip=f32(r["Dskip"]), z=dev(r["z"], dtype), dt_bias=f32(r["dt_bias"]))
    out, states, y = vs.varlen_selective_scan_fwd(**args, cu_seqlens=cu, position_indices=pos, y=True)
    dout = dev(r["dout"], dtype)
    g_re = vs.varlen_selective_scan_bwd(**args, dout=dout, cu_seqlens=cu, chunk_states=states,
                                        position_indices=pos)
    g_y = vs.varlen_selective_scan_bwd(**args, dout=dout, cu_seqlens=cu, chunk_states=states,
                                       position_indices=pos, y=y)
    torch.cuda.synchronize()
    sargs = [host(u), r["delta_raw"], r["A"], r["B"], r["C"], r["Dskip"], r["z"], r["dt_bias"]]
    y_ref = oracle.scan_fwd_threaded(*sargs[:6], None, sargs[7], cu_np)
    assert_close("y", y, y_ref, TOL[dtype])
    g = oracle.scan_bwd_threaded(*sargs, host(dout), cu_np)
    assert_close("dz (from y)", g_y["dz"], g["dz"], TOL[dtype])
    for k in ("du", "ddelta_raw", "dA", "dB", "dC", "dDskip", "d_dt_bias"):
        assert torch.equal(g_y[k], g_re[k]), k


@pytest.mark.parametrize("N,dtype", [(8, "f32"), (8, "bf16"), (16, "f32"), (16, "bf16")])
def test_gate_floor_and_a_log_variants(N, dtype):
    """GateFloor (out = y (SiLU(z) + delta)) and the A_log parameterisation
    (A = -exp(A_log); the backward returns dA_log = dA * A) against the oracle."""
    cu_np, T, r = rand_case([300, 1, 2, 257, 0, 40], 72, N, dtype, seed=29)
    a_log = np.random.default_rng(30).uniform(-1.0, 1.5, size=r["A"].shape).astype(np.float32)
    A_ref = -np.exp(a_log.astype(np.float64))
    floor = 0.05
    cu = torch.from_numpy(cu_np).cuda()
    pos = vs.varlen_position_indices(cu, T)
    u = dev(r["x"], dtype)
    args = dict(u=u, delta_raw=dev(r["delta_raw"], dtype), A=f32(a_log), B=dev(r["B"], dtype),
                C=dev(r["C"], dtype), Dskip=f32(r["Dskip"]), z=dev(r["z"], dtype), dt_bias=f32(r["dt_bias"]))
    out, states, y = vs.varlen_selective_scan_fwd(**args, cu_seqlens=cu, position_indices=pos, y=True,
                                                  gate_floor=floor, a_log=True)
    dout = dev(r["dout"], dtype)
    g = vs.varlen_selective_scan_bwd(**args, dout=dout, cu_seqlens=cu, chunk_states=states,
                                     position_indices=pos, y=y, gate_floor=floor, a_log=True)
    torch.cuda.synchronize()
    sargs = [host(u), r["delta_raw"], A_ref, r["B"], r["C"], r["Dskip"], r["z"], r["dt_bias"]]
    tol = TOL[dtype]
    assert_close("out", out, oracle.scan_fwd_threaded(*sargs, cu_np, gate_floor=floor), tol)
    assert_close("y", y, oracle.scan_fwd_threaded(*sargs[:6], None, sargs[7], cu_np), tol)
    ref = oracle.scan_bwd_threaded(*sargs, host(dout), cu_np, gate_floor=floor)
    ref["dA"] = ref["dA"] * A_ref  # dA_log by the chain rule
    for k in ("du", "ddelta_raw", "dz", "dA", "dB", "dC", "dDskip", "d_dt_bias"):
        assert_close(k, g[k], ref[k], tol)


@pytest.mark.parametrize("lengths,D,N,W,dtype,silu,bias", [
    ([1, 1, 2, 3, 700, 1, 40, 129, 5], 40, 4, 4, "f32", True, True),
    ([129, 1, 1, 1, 640, 77], 104, 16, 4, "bf16", True, True),
    ([300, 0, 1, 257, 33, 2], 72, 8, 2, "f32", True, False),
    ([5, 90, 1, 200], 64, 16, 1, "f32", False, True),
    ([700, 3, 1, 290, 33, 1000], 256, 16, 3, "bf16", True, True),
])
def test_fused_conv_scan_forward_equals_the_two_calls(lengths, D, N, W, dtype, silu, bias):
    """varlen_conv1d_scan_fwd computes u on chip in the conv call's arithmetic
    and order, rounded as its store rounds: u, out, y, the saved states and the
    final states equal those of conv1d_fwd followed by selective_scan_fwd bit
    for bit, and match the oracle's conv1d -> selective scan."""
    cu_np, T, r = rand_case(lengths, D, N, dtype, seed=sum(lengths) + 3 * W, W=W)
    S = len(lengths)
    cu = torch.from_numpy(cu_np).cuda()
    pos = vs.varlen_position_indices(cu, T)
    x = dev(r["x"], dtype)
    cw, cb = f32(r["conv_w"]), (f32(r["conv_b"]) if bias else None)
    h0 = f32(np.random.default_rng(7).standard_normal((S, D, N)))
    sargs = dict(delta_raw=dev(r["delta_raw"], dtype), A=f32(r["A"]), B=dev(r["B"], dtype),
                 C=dev(r["C"], dtype), Dskip=f32(r["Dskip"]), z=dev(r["z"], dtype), dt_bias=f32(r["dt_bias"]))
    u_ref = vs.varlen_conv1d_fwd(x, cw, cb, cu, pos, apply_silu=silu)
    ref = vs.varlen_selective_scan_fwd(u_ref, **sargs, cu_seqlens=cu, position_indices=pos, y=True,
                                       initial_states=h0, final_states=True)
    got = vs.varlen_conv1d_scan_fwd(x, cw, cb, **sargs, cu_seqlens=cu, position_indices=pos, apply_silu=silu,
                                    y=True, initial_states=h0, final_states=True)
    torch.cuda.synchronize()
    assert torch.equal(got[0], u_ref), "u"
    for name, g, e in zip(("out", "chunk_states", "y", "final_states"), got[1:], ref):
        assert torch.equal(g, e), name
    # and against the oracle: conv1d, the u the device holds, selective scan
    u_o = oracle.conv1d_fwd(r["x"], r["conv_w"], r["conv_b"] if bias else np.zeros(D, np.float32), cu_np,
                            apply_silu=silu)
    assert_close("u", got[0], u_o, TOL[dtype])
    out_o = oracle.scan_fwd(host(got[0]), r["delta_raw"], r["A"], r["B"], r["C"], r["Dskip"], r["z"],
                            r["dt_bias"], cu_np, h_init=host(h0))
    assert_close("out", got[1], out_o, TOL[dtype])


@pytest.mark.parametrize("D,N,dtype", [(72, 8, "f32"), (104, 16, "bf16")])
def test_sequence_states_fwd_bwd(D, N, dtype):
    """Per-sequence initial states in, final states out, and their gradients
    (the article's future work: cut sequences pass their state on).  The
    lengths put sequence ends on the forward's 128-token and the backward's
    32-token chunk edges, and include length-1 and empty sequences."""
    lengths = [128, 32, 1, 0, 95, 2, 300, 64]
    cu_np, T, r = rand_case(lengths, D, N, dtype, seed=31)
    S = len(lengths)
    rng = np.random.default_rng(32)
    h0 = rng.standard_normal((S, D, N)).astype(np.float32)
    dfin = rng.standard_normal((S, D, N)).astype(np.float32)
    cu = torch.from_numpy(cu_np).cuda()
    pos = vs.varlen_position_indices(cu, T)
    u = dev(r["x"], dtype)
    args = dict(u=u, delta_raw=dev(r["delta_raw"], dtype), A=f32(r["A"]), B=dev(r["B"], dtype),
                C=dev(r["C"], dtype), Dskip=f32(r["Dskip"]), z=dev(r["z"], dtype), dt_bias=f32(r["dt_bias"]))
    h0_t, dfin_t = f32(h0), f32(dfin)
    out, states, y, fin = vs.varlen_selective_scan_fwd(**args, cu_seqlens=cu, position_indices=pos, y=True,
                                                       initial_states=h0_t, final_states=True)
    dout = dev(r["dout"], dtype)
    g = vs.varlen_selective_scan_bwd(**args, dout=dout, cu_seqlens=cu, chunk_states=states,
                                     position_indices=pos, y=y, initial_states=h0_t,
                                     d_final_states=dfin_t, d_initial_states=True)
    torch.cuda.synchronize()
    sargs = [host(u), r["delta_raw"], r["A"], r["B"], r["C"], r["Dskip"], r["z"], r["dt_bias"]]
    tol = TOL[dtype]
    out_ref, fin_ref = oracle.scan_fwd(*sargs, cu_np, h_init=h0, return_last_state=True)
    assert_close("out", out, out_ref, tol)
    assert_close("final_states", fin, fin_ref, tol)
    assert np.array_equal(host(fin)[3], h0[3].astype(np.float64))  # the empty sequence
    ref = oracle.scan_bwd_threaded(*sargs, host(dout), cu_np, h_init=h0, dh_last=dfin)
    for k in ("du", "ddelta_raw", "dz", "dA", "dB", "dC", "dDskip", "d_dt_bias"):
        assert_close(k, g[k], ref[k], tol)
    assert_close("d_initial_states", g["d_initial_states"], ref["dh_init"], tol)
    assert np.array_equal(host(g["d_initial_states"])[3], dfin[3].astype(np.float64))


def test_a_cut_sequence_passes_its_state_on_gpu():
    """One 900-token sequence run whole, and run as two parts (the first 400
    tokens, then the rest from the first part's final state, the first part's
    backward taking the second part's starting-state gradient): the same
    outputs and gradients."""
    L, L1, D, N = 900, 400, 64, 16
    cu_np, T, r = rand_case([L], D, N, "f32", seed=33)
    cu = torch.from_numpy(cu_np).cuda()
    f = lambda k, sl=slice(None): f32(r[k][sl])  # noqa: E731
    def call(sl, n, h0=None, dfin=None):
        c = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        args = dict(u=f("x", sl), delta_raw=f("delta_raw", sl), A=f("A"), B=f("B", sl), C=f("C", sl),
                    Dskip=f("Dskip"), z=f("z", sl), dt_bias=f("dt_bias"))
        out, st, fin = vs.varlen_selective_scan_fwd(**args, cu_seqlens=c, initial_states=h0, final_states=True)
        g = vs.varlen_selective_scan_bwd(**args, dout=f("dout", sl), cu_seqlens=c, chunk_states=st,
                                         initial_states=h0, d_final_states=dfin, d_initial_states=True)
        return out, fin, g
    out_w, _, g_w = call(slice(None), L)
    out_2, fin_2, g_2 = None, None, None
    out_1, fin_1, _ = call(slice(0, L1), L1)
    out_2, _, g_2 = call(slice(L1, L), L - L1, h0=fin_1)
    _, _, g_1 = call(slice(0, L1), L1, dfin=g_2["d_initial_states"])
    torch.cuda.synchronize()
    tol = TOL["f32"]
    assert_close("out", torch.cat([out_1, out_2]), host(out_w), tol)
    for k in ("du", "ddelta_raw", "dz", "dB", "dC"):
        assert_close(k, torch.cat([g_1[k], g_2[k]]), host(g_w[k]), tol)
    for k in ("dA", "dDskip", "d_dt_bias"):
        assert_close(k, g_1[k] + g_2[k], host(g_w[k]), tol)
    assert_close("d_initial_states", g_1["d_initial_states"], host(g_w["d_initial_states"]), tol)


@pytest.mark.parametrize("W,dtype", [(4, "f32"), (4, "bf16"), (2, "f32")])
def test_conv_tails_fwd_bwd(W, dtype):
    """Conv tails of cut sequences: x_init read by the taps that reach before
    a sequence's start, x_last out, and their gradients.  Lengths shorter
    than W-1, an empty sequence, and starts just before, on and just after the
    192-token tile edges (190, 192, 193; 384, 386, 387), with a ragged last
    tile."""
    lengths = [190, 2, 1, 0, 191, 2, 1, 130, 40]
    D = 136
    cu_np, T, r = rand_case(lengths, D, 4, dtype, seed=34, W=W)
    S = len(lengths)
    rng = np.random.default_rng(35)
    x0 = rng.standard_normal((S, D, W - 1)).astype(np.float32)
    dxl = rng.standard_normal((S, D, W - 1)).astype(np.float32)
    if dtype == "bf16":  # tail values are inputs like x: give them bf16-exact values
        x0 = torch.from_numpy(x0).to(torch.bfloat16).float().numpy()
    cu = torch.from_numpy(cu_np).cuda()
    x = dev(r["x"], dtype)
    w, b = f32(r["conv_w"]), f32(r["conv_b"])
    u, xl = vs.varlen_conv1d_fwd(x, w, b, cu, x_init=f32(x0), x_last=True)
    g = dev(r["dout"], dtype)
    dx, dw, db, dxi = vs.varlen_conv1d_bwd(x, w, b, g, cu, x_init=f32(x0), dx_last=f32(dxl), dx_init=True)
    torch.cuda.synchronize()
    tol = TOL[dtype]
    u_ref, xl_ref = oracle.conv1d_fwd(r["x"], r["conv_w"], r["conv_b"], cu_np, x_init=x0, return_last=True)
    assert_close("u", u, u_ref, tol)
    assert np.array_equal(host(xl), xl_ref)  # plain copies of inputs
    ref = oracle.conv1d_bwd(r["x"], r["conv_w"], r["conv_b"], host(g), cu_np, x_init=x0, dx_last=dxl,
                            return_dx_init=True)
    for name, got, want in zip(("dx", "dweight", "dbias", "dx_init"), (dx, dw, db, dxi), ref):
        assert_close(name, got, want, tol)


def test_a_cut_sequence_passes_its_conv_tail_on_gpu():
    L, L1, D = 700, 333, 96
    cu_np, T, r = rand_case([L], D, 4, "f32", seed=36)
    w, b = f32(r["conv_w"]), f32(r["conv_b"])
    one = lambda n: torch.tensor([0, n], dtype=torch.int32, device="cuda")  # noqa: E731
    x, g = f32(r["x"]), f32(r["dout"])
    u_w = vs.varlen_conv1d_fwd(x, w, b, one(L))
    dx_w, dw_w, db_w = vs.varlen_conv1d_bwd(x, w, b, g, one(L))
    u_1, xl_1 = vs.varlen_conv1d_fwd(x[:L1].contiguous(), w, b, one(L1), x_last=True)
    u_2 = vs.varlen_conv1d_fwd(x[L1:].contiguous(), w, b, one(L - L1), x_init=xl_1)
    dx_2, dw_2, db_2, dxi_2 = vs.varlen_conv1d_bwd(x[L1:].contiguous(), w, b, g[L1:].contiguous(), one(L - L1),
                                                   x_init=xl_1, dx_init=True)
    dx_1, dw_1, db_1 = vs.varlen_conv1d_bwd(x[:L1].contiguous(), w, b, g[:L1].contiguous(), one(L1),
                                            dx_last=dxi_2)
    torch.cuda.synchronize()
    tol = TOL["f32"]
    assert_close("u", torch.cat([u_1, u_2]), host(u_w), tol)
    assert_close("dx", torch.cat([dx_1, dx_2]), host(dx_w), tol)
    assert_close("dweight", dw_1 + dw_2, host(dw_w), tol)
    assert_close("dbias", db_1 + db_2, host(db_w), tol)


@pytest.mark.parametrize("flags", [dict(z=False), dict(skip=False), dict(bias=False),
                                   dict(softplus=False), dict(z=False, skip=False, bias=False)])
def test_optional_inputs(flags):
    cu, T, r = rand_case([100, 3, 260, 1], 40, 8, "f32", seed=11)
    if flags.get("softplus") is False:
        # without softplus the step is delta_raw + dt_bias itself: keep it positive
        # (a negative step makes exp(delta A) grow and the state overflow fp32)
        r["delta_raw"] = np.abs(r["delta_raw"]) * np.float32(0.1)
        r["dt_bias"] = np.full_like(r["dt_bias"], 0.01)
    res = run_chain(cu, T, r, "f32", **flags)
    check_chain(cu, r, res, "f32", **flags)


@pytest.mark.parametrize("W", [1, 2, 3])
def test_conv_widths(W):
    cu, T, r = rand_case([5, 1, 2, 90, 3], 24, 4, "f32", seed=W, W=W)
    cu_t = torch.from_numpy(cu).cuda()
    x = f32(r["x"])
    u = vs.varlen_conv1d_fwd(x, f32(r["conv_w"]), f32(r["conv_b"]), cu_t)
    du = f32(r["dout"])
    dx, dw, db = vs.varlen_conv1d_bwd(x, f32(r["conv_w"]), f32(r["conv_b"]), du, cu_t)
    assert_close("u", u, oracle.conv1d_fwd(r["x"], r["conv_w"], r["conv_b"], cu), 2e-4)
    rdx, rdw, rdb = oracle.conv1d_bwd(r["x"], r["conv_w"], r["conv_b"], r["dout"], cu)
    assert_close("dx", dx, rdx, 2e-4)
    assert_close("dweight", dw, rdw, 2e-4)
    assert_close("dbias", db, rdb, 2e-4)


def test_zero_tokens_is_a_noop_that_zeroes_parameter_grads():
    D, N = 8, 4
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    e = torch.empty(0, D, device="cuda")
    eb = torch.empty(0, N, device="cuda")
    A = -torch.ones(D, N, device="cuda")
    out, st = vs.varlen_selective_scan_fwd(e, e, A, eb, eb, torch.ones(D, device="cuda"), e,
                                           torch.zeros(D, device="cuda"), cu)
    g = vs.varlen_selective_scan_bwd(e, e, A, eb, eb, torch.ones(D, device="cuda"), e,
                                     torch.zeros(D, device="cuda"), e, cu, st,
                                     grads=dict(dA=torch.full((D, N), 7.0, device="cuda"),
                                                dDskip=torch.full((D,), 7.0, device="cuda"),
                                                d_dt_bias=torch.full((D,), 7.0, device="cuda")))
    torch.cuda.synchronize()
    assert torch.count_nonzero(g["dA"]) == 0 and torch.count_nonzero(g["dDskip"]) == 0
    assert torch.count_nonzero(g["d_dt_bias"]) == 0


# ------------------------------------------------------------------ packing invariants on the GPU

def _per_token_outputs(res):
    return {k: res[k].clone() for k in ("u", "out", "du", "ddelta_raw", "dz", "dB", "dC", "dx")}


def test_sequences_do_not_interact_bitwise():
    lengths = [300, 1, 129, 4, 600, 2]
    cu, T, r = rand_case(lengths, 64, 16, "bf16", seed=21)
    base = _per_token_outputs(run_chain(cu, T, r, "bf16"))
    victim = 2
    r2 = {k: v.copy() for k, v in r.items()}
    sl = slice(int(cu[victim]), int(cu[victim + 1]))
    for k in ("x", "delta_raw", "z", "B", "C", "dout"):
        r2[k][sl] = workloads.round_to(r2[k][sl] * -1.5 + 0.25, "bf16")
    pert = _per_token_outputs(run_chain(cu, T, r2, "bf16"))
    for k in base:
        for s in range(len(lengths)):
            a, b = int(cu[s]), int(cu[s + 1])
            same = torch.equal(base[k][a:b], pert[k][a:b])
            assert same == (s != victim), (k, s)


def test_repeated_runs_are_bitwise_identical():
    cu, T, r = rand_case([2000, 1, 3, 1500, 600], 256, 16, "bf16", seed=5)
    first = run_chain(cu, T, r, "bf16")
    keys = ("u", "out", "du", "ddelta_raw", "dz", "dA", "dB", "dC", "dDskip", "d_dt_bias", "dx",
            "dweight", "dbias", "states")
    ref = {k: first[k].clone() for k in keys}
    for _ in range(4):
        again = run_chain(cu, T, r, "bf16")
        for k in keys:
            assert torch.equal(again[k], ref[k]), k


def test_right_padded_layout_matches_packed_on_real_tokens():
    lengths = [700, 1, 5, 300, 1100]
    cu, T, r = rand_case(lengths, 64, 16, "f32", seed=8)
    packed = run_chain(cu, T, r, "f32")
    cu_pad, idx = workloads.padded_layout(lengths)
    Tp = int(cu_pad[-1])
    rp = dict(r)
    rng = np.random.default_rng(99)
    for k in ("x", "delta_raw", "z", "B", "C", "dout"):
        arr = rng.standard_normal((Tp,) + r[k].shape[1:]).astype(np.float32) * 3
        arr[idx] = r[k]
        if k == "dout":
            arr[np.setdiff1d(np.arange(Tp), idx)] = 0.0   # padding carries no loss
        rp[k] = workloads.round_to(arr, "f32")
    padded = run_chain(cu_pad, Tp, rp, "f32")
    ii = torch.from_numpy(idx).cuda()
    assert torch.equal(padded["u"][ii], packed["u"])          # conv is per token: exact
    for k in ("out", "du", "ddelta_raw", "dz", "dB", "dC", "dx"):
        assert_close(k, padded[k][ii], host(packed[k]), 2e-4)
    for k in ("dA", "dDskip", "d_dt_bias", "dweight", "dbias"):
        assert_close(k, padded[k], host(packed[k]), 2e-4)


# ------------------------------------------------------------------ failure reporting

@pytest.mark.parametrize("N,dtype", [(8, "f32"), (16, "f32"), (16, "bf16")])
def test_lookback_wait_timeout_is_reported_not_hung(N, dtype):
    """A work item that never publishes its flag makes the next one's wait run
    out (after 1 ms); the call still completes and reports the timeout (each
    forward and backward kernel: bf16 with N = 16 runs the channel-pair
    forward)."""
    cu_np = np.array([0, 1024], dtype=np.int32)
    T, D = 1024, 32
    rng = np.random.default_rng(1)
    u = dev(rng.standard_normal((T, D)), dtype)
    B = dev(rng.standard_normal((T, N)), dtype)
    A = -torch.ones(D, N, device="cuda")
    cu = torch.from_numpy(cu_np).cuda()
    ws = torch.empty(binding.scan_fwd_workspace_size(T, D, N), dtype=torch.uint8, device="cuda")
    try:
        binding.debug_set(binding.VSSM_DBG_WAIT_NS, 1_000_000)
        binding.debug_set(binding.VSSM_DBG_DROP_FLAG, 3)
        vs.varlen_selective_scan_fwd(u, u, A, B, B, None, None, None, cu, workspace=ws)
        assert binding.read_status(ws) == -17
        wsb = torch.empty(binding.scan_bwd_workspace_size(T, D, N), dtype=torch.uint8, device="cuda")
        binding.debug_set(binding.VSSM_DBG_DROP_FLAG, -1)
        out, st = vs.varlen_selective_scan_fwd(u, u, A, B, B, None, None, None, cu)
        binding.debug_set(binding.VSSM_DBG_DROP_FLAG, 5)
        vs.varlen_selective_scan_bwd(u, u, A, B, B, None, None, None, u, cu, st, workspace=wsb)
        assert binding.read_status(wsb) == -17
    finally:
        binding.debug_set(binding.VSSM_DBG_DROP_FLAG, -1)
        binding.debug_set(binding.VSSM_DBG_WAIT_NS, 1_000_000_000)
    # and the context is still healthy
    vs.varlen_selective_scan_fwd(u, u, A, B, B, None, None, None, cu, workspace=ws)
    assert binding.read_status(ws) == 0


def test_conv_copy_timeout_is_reported_in_the_call_status():
    """The conv calls report a tile-copy wait that runs out in their status
    word.  The test knob makes one CTA treat its wait as timed out once its
    copy has landed (no copy fails); the call completes, vssm_read_status
    returns VSSM_ERR_LOOKBACK_TIMEOUT, and the next call is clean and right."""
    cu_np, T, r = rand_case([300, 1, 40, 700], 64, 4, "f32", seed=45)
    cu = torch.from_numpy(cu_np).cuda()
    pos = vs.varlen_position_indices(cu, T)
    x, w, b = f32(r["x"]), f32(r["conv_w"]), f32(r["conv_b"])
    D, W = 64, 4
    wsf = torch.empty(binding.conv1d_fwd_workspace_size(T, D, W), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(binding.conv1d_bwd_workspace_size(T, D, W), dtype=torch.uint8, device="cuda")
    try:
        binding.debug_set(binding.VSSM_DBG_FORCE_COPY_TIMEOUT, 1)
        u = vs.varlen_conv1d_fwd(x, w, b, cu, pos, workspace=wsf)
        assert binding.read_status(wsf) == -17
        vs.varlen_conv1d_bwd(x, w, b, u, cu, pos, workspace=wsb)
        assert binding.read_status(wsb) == -17
    finally:
        binding.debug_set(binding.VSSM_DBG_FORCE_COPY_TIMEOUT, -1)
    u = vs.varlen_conv1d_fwd(x, w, b, cu, pos, workspace=wsf)
    assert binding.read_status(wsf) == 0
    du = f32(r["dout"])
    dx, dw, db = vs.varlen_conv1d_bwd(x, w, b, du, cu, pos, workspace=wsb)
    assert binding.read_status(wsb) == 0
    assert_close("u", u, oracle.conv1d_fwd(r["x"], r["conv_w"], r["conv_b"], cu_np), TOL["f32"])
    ref = oracle.conv1d_bwd(r["x"], r["conv_w"], r["conv_b"], r["dout"], cu_np)
    for name, got, want in zip(("dx", "dweight", "dbias"), (dx, dw, db), ref):
        assert_close(name, got, want, TOL["f32"])


def test_lookback_walk_past_aggregates_is_bitwise_identical():
    """One work item sleeps before it stores its inclusive state, so the items
    after it on the same chain publish their aggregates and later items walk
    back past them to the delayed one and re-evaluate forward.  The results
    must equal, bit for bit, those of a run where every item finds its
    neighbour's inclusive state, and match the oracle."""
    lengths = [700, 1, 1100]  # long chains: few chunks hold a sequence start
    D, N = 32, 16             # one channel tile: every chunk is on the same chain
    cu_np, T, r = rand_case(lengths, D, N, "f32", seed=41)
    base = run_chain(cu_np, T, r, "f32")
    try:
        binding.debug_set(binding.VSSM_DBG_DELAY_NS, 300_000)
        # forward ticket 2 = chunk 2 of 15 (tokens 256..383); backward ticket 9 =
        # chunk 47 of 57, the backward counting from the top (tokens 1504..1535);
        # neither holds a sequence start (those are at tokens 700 and 701)
        binding.debug_set(binding.VSSM_DBG_DELAY_ITEM, 2)
        fwd_delayed = run_chain(cu_np, T, r, "f32", with_bwd=False)
        # and the walk did go past aggregates: some warp published one (the
        # workspace holds a 256-byte header, then the int32 look-back flags)
        ws = torch.empty(binding.scan_fwd_workspace_size(T, D, N), dtype=torch.uint8, device="cuda")
        vs.varlen_selective_scan_fwd(fwd_delayed["u"], f32(r["delta_raw"]), f32(r["A"]), f32(r["B"]), f32(r["C"]),
                                     f32(r["Dskip"]), f32(r["z"]), f32(r["dt_bias"]), torch.from_numpy(cu_np).cuda(),
                                     workspace=ws)
        n_chunks = (T + 127) // 128
        flags = ws[256:256 + 4 * n_chunks * 32].view(torch.int32)
        assert int((flags == 1).sum()) > 0
        binding.debug_set(binding.VSSM_DBG_DELAY_ITEM, 9)
        bwd_delayed = run_chain(cu_np, T, r, "f32")
    finally:
        binding.debug_set(binding.VSSM_DBG_DELAY_ITEM, -1)
    for k in ("u", "out", "states"):
        assert torch.equal(fwd_delayed[k], base[k]), k
    for k in base:
        if isinstance(base[k], torch.Tensor):
            assert torch.equal(bwd_delayed[k], base[k]), k
    check_chain(cu_np, r, bwd_delayed, "f32")


# ------------------------------------------------------------------ the named workloads

def test_workload_m130m_forward_full_parity():
    w = workloads.make("m130m", backward=False, scan_input=False)
    r = workloads.rounded(w, "f32")
    res = run_chain(w["cu_seqlens"], w["T"], r, "f32", with_bwd=False)
    check_chain(w["cu_seqlens"], r, res, "f32", with_bwd=False)


def _big_case(name):
    w = workloads.make(name, backward=True, scan_input=False)
    r = workloads.rounded(w, "bf16")
    for k in workloads.ACTIVATIONS:
        w.pop(k, None)
    return w, r


def _sampled_checks(w, r, res, seq_pick):
    cu = w["cu_seqlens"]
    D = r["A"].shape[0]
    rng = np.random.default_rng(7)
    chans = np.unique(np.concatenate([np.arange(0, 8), np.arange(D - 8, D), rng.choice(D, 32, replace=False)]))
    check_chain(cu, r, res, "bf16", channels=chans)
    # dB / dC sum over every channel: check whole sequences, run alone through the oracle
    u_gpu = res["u"]
    for s in seq_pick:
        a, b = int(cu[s]), int(cu[s + 1])
        sl = slice(a, b)
        one = np.array([0, b - a], dtype=np.int32)
        g = oracle.scan_bwd_threaded(host(u_gpu[a:b]), r["delta_raw"][sl], r["A"], r["B"][sl], r["C"][sl],
                                     r["Dskip"], r["z"][sl], r["dt_bias"], r["dout"][sl], one)
        assert_close(f"dB[seq {s}]", res["dB"][a:b], g["dB"], 1e-2)
        assert_close(f"dC[seq {s}]", res["dC"][a:b], g["dC"], 1e-2)


def test_workload_m14b_forward_sampled_parity():
    """The Mamba-1.4B forward-only configuration (its own seed): conv and scan
    forward at full size, every output of 48 channels against the oracle."""
    w = workloads.make("m14b_fwd", backward=False, scan_input=False)
    r = workloads.rounded(w, "bf16")
    for k in workloads.ACTIVATIONS:
        w.pop(k, None)
    res = run_chain(w["cu_seqlens"], w["T"], r, "bf16", with_bwd=False)
    D = r["A"].shape[0]
    rng = np.random.default_rng(11)
    chans = np.unique(np.concatenate([np.arange(0, 8), np.arange(D - 8, D), rng.choice(D, 32, replace=False)]))
    check_chain(w["cu_seqlens"], r, res, "bf16", with_bwd=False, channels=chans)


def test_workload_m14b_fwd_bwd_sampled_parity():
    w, r = _big_case("m14b")
    res = run_chain(w["cu_seqlens"], w["T"], r, "bf16", use_y=True)  # as the bench step runs
    lengths = np.diff(w["cu_seqlens"])
    picks = [int(np.argmax(lengths)), int(np.argmin(lengths)), len(lengths) // 2]
    _sampled_checks(w, r, res, picks)


def test_workload_longtail_fwd_bwd_sampled_parity():
    w, r = _big_case("longtail")
    res = run_chain(w["cu_seqlens"], w["T"], r, "bf16", use_y=True)
    lengths = np.diff(w["cu_seqlens"])
    picks = [int(np.argmax(lengths)), int(np.argmin(lengths)), int(np.argmax(lengths < 9))]
    _sampled_checks(w, r, res, picks)
