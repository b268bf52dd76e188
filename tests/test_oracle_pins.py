"""Pins for the CPU oracle (CPU only, no GPU).

Each test checks the oracle against something other than itself: the
article's worked packing example, library routines (np.convolve,
torch conv1d, np.cumsum, np.logaddexp, scipy's expit), closed forms,
a brute-force unrolled sum, finite differences, and the packing invariants
the article asks for (a packed sequence behaves exactly as if run alone).
"""
import os

import numpy as np
import pytest
import scipy.special

import oracle
from selective_ssm_packed_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_pack(rng, lengths, D, N, W=4):
    cu = workloads.cu_seqlens_from_lengths(lengths)
    T = int(cu[-1])
    v = dict(
        cu=cu, T=T,
        x=rng.standard_normal((T, D)), u=rng.standard_normal((T, D)),
        dr=0.5 * rng.standard_normal((T, D)), z=rng.standard_normal((T, D)),
        B=rng.standard_normal((T, N)), C=rng.standard_normal((T, N)),
        A=-rng.uniform(0.2, 3.0, size=(D, N)), Dskip=rng.standard_normal(D),
        dt_bias=rng.uniform(-4.0, -1.0, size=D),
        w=rng.uniform(-0.5, 0.5, size=(D, W)), b=rng.uniform(-0.5, 0.5, size=D),
        dout=rng.standard_normal((T, D)),
    )
    return v


def _silu(x):
    return x * scipy.special.expit(x)


def _scan(v, **kw):
    return oracle.scan_fwd(v["u"], v["dr"], v["A"], v["B"], v["C"], v["Dskip"], v["z"],
                           v["dt_bias"], v["cu"], **kw)


def _scan_bwd(v, **kw):
    return oracle.scan_bwd(v["u"], v["dr"], v["A"], v["B"], v["C"], v["Dskip"], v["z"],
                           v["dt_bias"], v["dout"], v["cu"], **kw)


# ---------------------------------------------------------------- position indices

def test_position_indices_golden_example():
    with open(os.path.join(GOLDEN, "position_indices_4_2_3_7.txt")) as f:
        rows = [list(map(int, ln.split())) for ln in f if ln.strip() and not ln.startswith("#")]
    lengths, cu, pos = rows
    assert list(workloads.cu_seqlens_from_lengths(lengths)) == cu
    assert list(oracle.position_indices(np.array(cu, dtype=np.int32))) == pos


def test_position_indices_brute_force():
    rng = _rng(5)
    for trial in range(20):
        lengths = list(rng.integers(0, 9, size=int(rng.integers(1, 12))))
        cu = workloads.cu_seqlens_from_lengths(lengths)
        T = int(cu[-1])
        expect = []
        for t in range(T):
            s = 0
            while not (cu[s] <= t < cu[s + 1]):
                s += 1
            expect.append(t - int(cu[s]))
        assert list(oracle.position_indices(cu)) == expect


@pytest.mark.parametrize("cu", [[1, 4, 6], [0, 4, 3, 6], [0, 2, 5]])
def test_position_indices_rejects_malformed(cu):
    cu = np.array(cu, dtype=np.int32)
    T = 6
    with pytest.raises(oracle.OracleError):
        oracle.position_indices(cu, total_tokens=T)


# ---------------------------------------------------------------- conv1d forward

def test_conv_fwd_equals_np_convolve_per_sequence():
    rng = _rng(1)
    v = _rand_pack(rng, [4, 2, 3, 7, 1, 5], D=5, N=2, W=4)
    u = oracle.conv1d_fwd(v["x"], v["w"], v["b"], v["cu"], apply_silu=True)
    cu = v["cu"]
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        for d in range(5):
            pre = np.convolve(v["x"][a:e, d], v["w"][d, ::-1])[: e - a] + v["b"][d]
            np.testing.assert_allclose(u[a:e, d], _silu(pre), rtol=1e-13, atol=1e-13)


def test_conv_fwd_equals_torch_depthwise_conv1d():
    torch = pytest.importorskip("torch")
    rng = _rng(2)
    D, W, L = 6, 4, 11
    x = rng.standard_normal((L, D))
    w = rng.uniform(-0.5, 0.5, size=(D, W))
    b = rng.uniform(-0.5, 0.5, size=D)
    cu = np.array([0, L], dtype=np.int32)
    ref = torch.nn.functional.conv1d(torch.from_numpy(x.T[None]), torch.from_numpy(w[:, None, :]),
                                     torch.from_numpy(b), padding=W - 1, groups=D)[0, :, :L].T
    np.testing.assert_allclose(oracle.conv1d_fwd(x, w, b, cu, apply_silu=False), ref.numpy(),
                               rtol=1e-13, atol=1e-13)


def test_conv_width_one_is_pointwise():
    rng = _rng(3)
    v = _rand_pack(rng, [3, 5], D=4, N=2, W=1)
    u = oracle.conv1d_fwd(v["x"], v["w"], v["b"], v["cu"], apply_silu=True)
    np.testing.assert_allclose(u, _silu(v["b"] + v["w"][:, 0] * v["x"]), rtol=1e-14, atol=1e-14)


def test_conv_taps_never_cross_a_start_token():
    rng = _rng(4)
    lengths = [4, 2, 3, 7]
    v = _rand_pack(rng, lengths, D=3, N=2)
    cu = v["cu"]
    base = oracle.conv1d_fwd(v["x"], v["w"], v["b"], cu)
    for i in range(len(lengths)):
        x2 = v["x"].copy()
        x2[cu[i]:cu[i + 1]] += rng.standard_normal((lengths[i], 3)) * 10
        pert = oracle.conv1d_fwd(x2, v["w"], v["b"], cu)
        for j in range(len(lengths)):
            if j != i:
                assert np.array_equal(base[cu[j]:cu[j + 1]], pert[cu[j]:cu[j + 1]])
        assert not np.array_equal(base[cu[i]:cu[i + 1]], pert[cu[i]:cu[i + 1]])


def test_conv_packed_equals_alone_and_right_padded():
    rng = _rng(6)
    lengths = [5, 1, 9, 3]
    v = _rand_pack(rng, lengths, D=4, N=2)
    cu = v["cu"]
    packed = oracle.conv1d_fwd(v["x"], v["w"], v["b"], cu)
    for i, L in enumerate(lengths):
        alone = oracle.conv1d_fwd(v["x"][cu[i]:cu[i + 1]], v["w"], v["b"], np.array([0, L], np.int32))
        assert np.array_equal(alone, packed[cu[i]:cu[i + 1]])
    # right-padded rows of length 10: real tokens first, junk padding after
    rows = workloads.cu_seqlens_from_lengths([10] * len(lengths))
    xp = rng.standard_normal((10 * len(lengths), 4)) * 100
    for i, L in enumerate(lengths):
        xp[10 * i:10 * i + L] = v["x"][cu[i]:cu[i + 1]]
    padded = oracle.conv1d_fwd(xp, v["w"], v["b"], rows)
    for i, L in enumerate(lengths):
        assert np.array_equal(padded[10 * i:10 * i + L], packed[cu[i]:cu[i + 1]])


# ---------------------------------------------------------------- conv1d backward

def test_conv_bwd_is_the_adjoint_of_the_linear_conv():
    rng = _rng(7)
    v = _rand_pack(rng, [6, 3, 1, 8], D=5, N=2)
    g = rng.standard_normal(v["x"].shape)
    y = oracle.conv1d_fwd(v["x"], v["w"], None, v["cu"], apply_silu=False)
    dx, dw, db = oracle.conv1d_bwd(v["x"], v["w"], None, g, v["cu"], apply_silu=False)
    lhs = float(np.sum(y * g))
    assert abs(lhs - float(np.sum(v["x"] * dx))) <= 1e-12 * max(1.0, abs(lhs))
    # the weight gradient is the adjoint in w: <conv_w(x), g> = <w, dw>
    assert abs(lhs - float(np.sum(v["w"] * dw))) <= 1e-12 * max(1.0, abs(lhs))


def _fd_check(f, params, grads, eps=1e-6, tol=1e-6):
    """Central finite differences of scalar f over every entry of params[k]."""
    for k, arr in params.items():
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + eps
            fp = f()
            arr[idx] = old - eps
            fm = f()
            arr[idx] = old
            fd[idx] = (fp - fm) / (2 * eps)
        an = grads[k]
        scale = max(np.max(np.abs(an)), 1e-12)
        err = np.max(np.abs(fd - an)) / scale
        assert err <= tol, f"{k}: relative error {err:.3e}"


def test_conv_bwd_finite_differences():
    rng = _rng(8)
    v = _rand_pack(rng, [4, 2, 3, 7], D=3, N=2)
    g = rng.standard_normal(v["x"].shape)
    dx, dw, db = oracle.conv1d_bwd(v["x"], v["w"], v["b"], g, v["cu"], apply_silu=True)

    def f():
        return float(np.sum(oracle.conv1d_fwd(v["x"], v["w"], v["b"], v["cu"], apply_silu=True) * g))

    _fd_check(f, {"x": v["x"], "w": v["w"], "b": v["b"]}, {"x": dx, "w": dw, "b": db})


# ---------------------------------------------------------------- selective scan forward

def test_scan_closed_form_single_state_constant_step():
    """N=1, constant step delta, constant B and u inside each sequence:
    h after k+1 tokens = delta*B*u * (1 - alpha^(k+1)) / (1 - alpha)."""
    rng = _rng(9)
    lengths = [5, 1, 12, 7]
    cu = workloads.cu_seqlens_from_lengths(lengths)
    T, D = int(cu[-1]), 3
    delta = 0.37
    A = -rng.uniform(0.5, 2.0, size=(D, 1))
    Bs = rng.standard_normal(len(lengths))
    us = rng.standard_normal((len(lengths), D))
    B = np.repeat(Bs, lengths)[:, None]
    u = np.repeat(us, lengths, axis=0)
    out = oracle.scan_fwd(u, np.full((T, D), delta), A, B, np.ones((T, 1)), None, None, None, cu,
                          delta_softplus=False)
    for s, L in enumerate(lengths):
        k = np.arange(L)[:, None]
        alpha = np.exp(delta * A[:, 0])[None, :]
        h = delta * Bs[s] * us[s][None, :] * (1 - alpha ** (k + 1)) / (1 - alpha)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], h, rtol=1e-12, atol=1e-14)


def test_scan_brute_force_unrolled_sum():
    """h_t[n] = sum_{s<=t in seq} exp(A_n * sum_{r=s+1..t} delta_r) delta_s B_s[n] u_s."""
    rng = _rng(10)
    v = _rand_pack(rng, [4, 2, 3, 7], D=5, N=3)
    out = _scan(v)
    cu = v["cu"]
    delta = np.logaddexp(0.0, v["dr"] + v["dt_bias"][None, :])
    ref = np.zeros_like(out)
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        for t in range(a, e):
            for d in range(5):
                y = 0.0
                for n in range(3):
                    h = 0.0
                    for j in range(a, t + 1):
                        decay = np.exp(v["A"][d, n] * np.sum(delta[j + 1:t + 1, d]))
                        h += decay * delta[j, d] * v["B"][j, n] * v["u"][j, d]
                    y += v["C"][t, n] * h
                y += v["Dskip"][d] * v["u"][t, d]
                ref[t, d] = y * _silu(v["z"][t, d])
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_scan_zero_A_is_a_segmented_prefix_sum():
    rng = _rng(11)
    v = _rand_pack(rng, [6, 1, 4, 9], D=4, N=3)
    v["A"] = np.zeros_like(v["A"])
    out = oracle.scan_fwd(v["u"], v["dr"], v["A"], v["B"], v["C"], None, None, None, v["cu"],
                          delta_softplus=False)
    cu = v["cu"]
    ref = np.zeros_like(out)
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        bu = v["dr"][a:e, :, None] * v["B"][a:e, None, :] * v["u"][a:e, :, None]   # (L, D, N)
        h = np.cumsum(bu, axis=0)
        ref[a:e] = np.einsum("tdn,tn->td", h, v["C"][a:e])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_scan_zero_B_leaves_the_gated_skip_term():
    rng = _rng(12)
    v = _rand_pack(rng, [3, 8], D=4, N=2)
    v["B"] = np.zeros_like(v["B"])
    out = _scan(v)
    np.testing.assert_allclose(out, v["Dskip"][None, :] * v["u"] * _silu(v["z"]), rtol=1e-14, atol=1e-15)


def test_scan_step_is_softplus_of_raw_plus_bias():
    """A=0, B=C=u=1, N=1, no skip/gate: out_t - out_{t-1} is the step delta_t."""
    rng = _rng(13)
    lengths = [7, 5]
    cu = workloads.cu_seqlens_from_lengths(lengths)
    T, D = 12, 3
    dr = rng.standard_normal((T, D)) * 4
    bias = rng.uniform(-3, 3, size=D)
    out = oracle.scan_fwd(np.ones((T, D)), dr, np.zeros((D, 1)), np.ones((T, 1)), np.ones((T, 1)),
                          None, None, bias, cu, delta_softplus=True)
    for s in range(2):
        a, e = int(cu[s]), int(cu[s + 1])
        steps = np.diff(np.vstack([np.zeros((1, D)), out[a:e]]), axis=0)
        np.testing.assert_allclose(steps, np.logaddexp(0.0, dr[a:e] + bias), rtol=1e-12, atol=1e-14)


def test_scan_packed_equals_alone_right_padded_and_isolated():
    rng = _rng(14)
    lengths = [4, 2, 3, 7]
    v = _rand_pack(rng, lengths, D=4, N=3)
    cu = v["cu"]
    packed = _scan(v)
    for i, L in enumerate(lengths):
        sl = slice(int(cu[i]), int(cu[i + 1]))
        alone = oracle.scan_fwd(v["u"][sl], v["dr"][sl], v["A"], v["B"][sl], v["C"][sl], v["Dskip"],
                                v["z"][sl], v["dt_bias"], np.array([0, L], np.int32))
        assert np.array_equal(alone, packed[sl])
    rows = workloads.cu_seqlens_from_lengths([8] * 4)
    pad = {k: (rng.standard_normal((32,) + v[k].shape[1:]) * 50 if k in ("u", "dr", "z", "B", "C") else v[k])
           for k in ("u", "dr", "z", "B", "C", "A", "Dskip", "dt_bias")}
    for i, L in enumerate(lengths):
        for k in ("u", "dr", "z", "B", "C"):
            pad[k][8 * i:8 * i + L] = v[k][cu[i]:cu[i + 1]]
    pad["cu"] = rows
    padded = _scan(pad)
    for i, L in enumerate(lengths):
        assert np.array_equal(padded[8 * i:8 * i + L], packed[cu[i]:cu[i + 1]])
    for i in range(4):
        w = {k: (val.copy() if isinstance(val, np.ndarray) else val) for k, val in v.items()}
        sl = slice(int(cu[i]), int(cu[i + 1]))
        for k in ("u", "dr", "z", "B", "C"):
            w[k][sl] += 3.0
        pert = _scan(w)
        for j in range(4):
            if j != i:
                assert np.array_equal(pert[cu[j]:cu[j + 1]], packed[cu[j]:cu[j + 1]])


# ---------------------------------------------------------------- selective scan backward

def test_scan_bwd_finite_differences_every_input():
    rng = _rng(15)
    v = _rand_pack(rng, [4, 2, 3, 7], D=8, N=4)
    g = _scan_bwd(v)

    def f():
        return float(np.sum(_scan(v) * v["dout"]))

    _fd_check(f, {"u": v["u"], "dr": v["dr"], "A": v["A"], "B": v["B"], "C": v["C"],
                  "Dskip": v["Dskip"], "z": v["z"], "dt_bias": v["dt_bias"]},
              {"u": g["du"], "dr": g["ddelta_raw"], "A": g["dA"], "B": g["dB"], "C": g["dC"],
               "Dskip": g["dDskip"], "z": g["dz"], "dt_bias": g["d_dt_bias"]})


def test_scan_bwd_finite_differences_without_softplus_gate_or_skip():
    rng = _rng(16)
    v = _rand_pack(rng, [5, 1, 6], D=3, N=2)
    v["dr"] = np.abs(v["dr"]) * 0.3
    g = oracle.scan_bwd(v["u"], v["dr"], v["A"], v["B"], v["C"], None, None, None, v["dout"], v["cu"],
                        delta_softplus=False)

    def f():
        return float(np.sum(oracle.scan_fwd(v["u"], v["dr"], v["A"], v["B"], v["C"], None, None, None,
                                             v["cu"], delta_softplus=False) * v["dout"]))

    _fd_check(f, {"u": v["u"], "dr": v["dr"], "A": v["A"], "B": v["B"], "C": v["C"]},
              {"u": g["du"], "dr": g["ddelta_raw"], "A": g["dA"], "B": g["dB"], "C": g["dC"]})


def test_scan_bwd_skip_gradient_closed_form():
    rng = _rng(17)
    v = _rand_pack(rng, [4, 2, 3, 7], D=6, N=3)
    g = _scan_bwd(v)
    np.testing.assert_allclose(g["dDskip"], np.sum(v["dout"] * _silu(v["z"]) * v["u"], axis=0),
                               rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(g["d_dt_bias"], np.sum(g["ddelta_raw"], axis=0), rtol=1e-13, atol=1e-13)


def test_scan_bwd_pack_grads_are_sums_of_sequence_grads():
    rng = _rng(18)
    lengths = [4, 2, 3, 7]
    v = _rand_pack(rng, lengths, D=5, N=3)
    cu = v["cu"]
    gp = _scan_bwd(v)
    acc = {k: np.zeros_like(gp[k]) for k in ("dA", "dDskip", "d_dt_bias")}
    for i, L in enumerate(lengths):
        sl = slice(int(cu[i]), int(cu[i + 1]))
        gs = oracle.scan_bwd(v["u"][sl], v["dr"][sl], v["A"], v["B"][sl], v["C"][sl], v["Dskip"],
                             v["z"][sl], v["dt_bias"], v["dout"][sl], np.array([0, L], np.int32))
        for k in ("du", "ddelta_raw", "dz", "dB", "dC"):
            assert np.array_equal(gs[k], gp[k][sl])
        for k in acc:
            acc[k] += gs[k]
    for k in acc:
        np.testing.assert_allclose(gp[k], acc[k], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- gate floor, sequence states, A_log

def test_scan_gate_floor_adds_floor_times_the_ungated_output():
    # out = y (SiLU(z) + delta) = y SiLU(z) + delta y: linear in the floor
    rng = _rng(40)
    v = _rand_pack(rng, [4, 2, 3, 7], D=6, N=3)
    base = _scan(v)
    ungated = oracle.scan_fwd(v["u"], v["dr"], v["A"], v["B"], v["C"], v["Dskip"], None, v["dt_bias"], v["cu"])
    np.testing.assert_allclose(_scan(v, gate_floor=0.05), base + 0.05 * ungated, rtol=1e-12, atol=1e-12)


def test_scan_bwd_gate_floor_equals_the_ungated_run_on_gated_dout():
    # with the gate fixed, the scan sees dy = dout (SiLU(z) + delta); dz does not depend on delta
    rng = _rng(41)
    v = _rand_pack(rng, [4, 2, 3, 7], D=5, N=3)
    g = _scan_bwd(v, gate_floor=0.07)
    g0 = _scan_bwd(v)
    ref = oracle.scan_bwd(v["u"], v["dr"], v["A"], v["B"], v["C"], v["Dskip"], None, v["dt_bias"],
                          v["dout"] * (_silu(v["z"]) + 0.07), v["cu"])
    for k in ("du", "ddelta_raw", "dA", "dB", "dC", "dDskip", "d_dt_bias"):
        np.testing.assert_allclose(g[k], ref[k], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(g["dz"], g0["dz"])


def test_scan_bwd_finite_differences_with_gate_floor_initial_and_final_states():
    # loss = sum(out * dout) + sum(h_last * dh_last), so that both states enter it
    rng = _rng(42)
    v = _rand_pack(rng, [4, 2, 3, 7], D=3, N=2)
    S = 4
    h0 = rng.standard_normal((S, 3, 2))
    dhl = rng.standard_normal((S, 3, 2))
    g = _scan_bwd(v, gate_floor=0.03, h_init=h0, dh_last=dhl)

    def f():
        out, hl = _scan(v, gate_floor=0.03, h_init=h0, return_last_state=True)
        return float(np.sum(out * v["dout"]) + np.sum(hl * dhl))

    _fd_check(f, {"u": v["u"], "dr": v["dr"], "A": v["A"], "B": v["B"], "C": v["C"],
                  "Dskip": v["Dskip"], "z": v["z"], "dt_bias": v["dt_bias"], "h0": h0},
              {"u": g["du"], "dr": g["ddelta_raw"], "A": g["dA"], "B": g["dB"], "C": g["dC"],
               "Dskip": g["dDskip"], "z": g["dz"], "dt_bias": g["d_dt_bias"], "h0": g["dh_init"]})


def test_a_cut_sequence_that_passes_its_state_equals_the_whole_sequence():
    # the article's future work: a long sequence cut into two parts that pass
    # the state on gives the whole sequence's outputs and gradients
    rng = _rng(43)
    L, L1 = 37, 16
    v = _rand_pack(rng, [L], D=4, N=3)
    whole = _scan(v)
    gw = _scan_bwd(v)
    one = lambda n: np.array([0, n], np.int32)  # noqa: E731
    p1 = {k: (v[k][:L1] if isinstance(v[k], np.ndarray) and v[k].shape[:1] == (L,) else v[k]) for k in v}
    p2 = {k: (v[k][L1:] if isinstance(v[k], np.ndarray) and v[k].shape[:1] == (L,) else v[k]) for k in v}
    p1["cu"], p2["cu"] = one(L1), one(L - L1)
    out1, h1 = _scan(p1, return_last_state=True)
    out2 = _scan(p2, h_init=h1)
    np.testing.assert_allclose(np.concatenate([out1, out2]), whole, rtol=1e-12, atol=1e-12)
    g2 = _scan_bwd(p2, h_init=h1)
    g1 = _scan_bwd(p1, dh_last=g2["dh_init"])
    for k in ("du", "ddelta_raw", "dz"):
        np.testing.assert_allclose(np.concatenate([g1[k], g2[k]]), gw[k], rtol=1e-11, atol=1e-11)
    for k in ("dB", "dC"):
        np.testing.assert_allclose(np.concatenate([g1[k], g2[k]]), gw[k], rtol=1e-11, atol=1e-11)
    for k in ("dA", "dDskip", "d_dt_bias"):
        np.testing.assert_allclose(g1[k] + g2[k], gw[k], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(g1["dh_init"], gw["dh_init"], rtol=1e-11, atol=1e-11)


def test_an_empty_sequence_passes_its_state_and_gradient_through():
    rng = _rng(44)
    v = _rand_pack(rng, [3, 0, 4], D=2, N=2)
    h0 = rng.standard_normal((3, 2, 2))
    dhl = rng.standard_normal((3, 2, 2))
    _, hl = _scan(v, h_init=h0, return_last_state=True)
    np.testing.assert_array_equal(hl[1], h0[1])
    g = _scan_bwd(v, h_init=h0, dh_last=dhl)
    np.testing.assert_array_equal(g["dh_init"][1], dhl[1])


def test_a_log_gradient_is_dA_times_A():
    # A = -exp(A_log): finite differences in A_log against the chain rule dA * A
    rng = _rng(45)
    v = _rand_pack(rng, [4, 2, 3, 7], D=3, N=2)
    a_log = rng.uniform(-1.0, 1.0, size=(3, 2))
    v["A"] = -np.exp(a_log)
    g = _scan_bwd(v)

    def f():
        w = dict(v, A=-np.exp(a_log))
        return float(np.sum(_scan(w) * v["dout"]))

    _fd_check(f, {"a_log": a_log}, {"a_log": g["dA"] * v["A"]})


# ---------------------------------------------------------------- conv tails (the conv half of a cut sequence)

def test_conv_bwd_finite_differences_with_tails():
    # loss = sum(u * g) + sum(x_last * dx_last); the pack has a sequence shorter than W-1,
    # so its x_last reaches back into its own tail values
    rng = _rng(46)
    v = _rand_pack(rng, [4, 2, 3, 7], D=3, N=2)
    W = v["w"].shape[1]
    x0 = rng.standard_normal((4, 3, W - 1))
    dxl = rng.standard_normal((4, 3, W - 1))
    g = rng.standard_normal(v["x"].shape)
    dx, dw, db, dxi = oracle.conv1d_bwd(v["x"], v["w"], v["b"], g, v["cu"], x_init=x0, dx_last=dxl,
                                        return_dx_init=True)

    def f():
        u, xl = oracle.conv1d_fwd(v["x"], v["w"], v["b"], v["cu"], x_init=x0, return_last=True)
        return float(np.sum(u * g) + np.sum(xl * dxl))

    _fd_check(f, {"x": v["x"], "w": v["w"], "b": v["b"], "x0": x0},
              {"x": dx, "w": dw, "b": db, "x0": dxi})


def test_a_cut_sequence_that_passes_its_conv_tail_equals_the_whole_sequence():
    rng = _rng(47)
    L, L1 = 23, 9
    v = _rand_pack(rng, [L], D=4, N=2)
    one = lambda n: np.array([0, n], np.int32)  # noqa: E731
    g = rng.standard_normal(v["x"].shape)
    uw = oracle.conv1d_fwd(v["x"], v["w"], v["b"], v["cu"])
    dxw, dww, dbw = oracle.conv1d_bwd(v["x"], v["w"], v["b"], g, v["cu"])
    u1, xl1 = oracle.conv1d_fwd(v["x"][:L1], v["w"], v["b"], one(L1), return_last=True)
    u2 = oracle.conv1d_fwd(v["x"][L1:], v["w"], v["b"], one(L - L1), x_init=xl1)
    np.testing.assert_allclose(np.concatenate([u1, u2]), uw, rtol=1e-13, atol=1e-13)
    dx2, dw2, db2, dxi2 = oracle.conv1d_bwd(v["x"][L1:], v["w"], v["b"], g[L1:], one(L - L1), x_init=xl1,
                                            return_dx_init=True)
    dx1, dw1, db1 = oracle.conv1d_bwd(v["x"][:L1], v["w"], v["b"], g[:L1], one(L1), dx_last=dxi2)
    np.testing.assert_allclose(np.concatenate([dx1, dx2]), dxw, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw1 + dw2, dww, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db1 + db2, dbw, rtol=1e-12, atol=1e-12)


def test_an_empty_sequence_passes_its_conv_tail_and_gradient_through():
    rng = _rng(48)
    v = _rand_pack(rng, [3, 0, 4], D=2, N=2)
    W = v["w"].shape[1]
    x0 = rng.standard_normal((3, 2, W - 1))
    dxl = rng.standard_normal((3, 2, W - 1))
    _, xl = oracle.conv1d_fwd(v["x"], v["w"], v["b"], v["cu"], x_init=x0, return_last=True)
    np.testing.assert_array_equal(xl[1], x0[1])
    *_, dxi = oracle.conv1d_bwd(v["x"], v["w"], v["b"], v["dout"], v["cu"], x_init=x0, dx_last=dxl,
                                return_dx_init=True)
    np.testing.assert_array_equal(dxi[1], dxl[1])


# ---------------------------------------------------------------- threaded helpers

def test_threaded_helpers_match_single_call():
    rng = _rng(19)
    v = _rand_pack(rng, [30, 17, 1, 50], D=37, N=4)
    np.testing.assert_array_equal(
        oracle.scan_fwd_threaded(v["u"], v["dr"], v["A"], v["B"], v["C"], v["Dskip"], v["z"],
                                 v["dt_bias"], v["cu"], threads=3), _scan(v))
    a = oracle.scan_bwd_threaded(v["u"], v["dr"], v["A"], v["B"], v["C"], v["Dskip"], v["z"],
                                 v["dt_bias"], v["dout"], v["cu"], threads=3)
    b = _scan_bwd(v)
    for k in b:
        np.testing.assert_allclose(a[k], b[k], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(oracle.conv1d_fwd_threaded(v["x"], v["w"], v["b"], v["cu"], threads=3),
                                  oracle.conv1d_fwd(v["x"], v["w"], v["b"], v["cu"]))
    for p, q in zip(oracle.conv1d_bwd_threaded(v["x"], v["w"], v["b"], v["dout"], v["cu"], threads=3),
                    oracle.conv1d_bwd(v["x"], v["w"], v["b"], v["dout"], v["cu"])):
        np.testing.assert_array_equal(p, q)


# ---------------------------------------------------------------- sequence packing

def test_packing_worked_example():
    # by hand: sequential seals after 5 (4 does not fit) and after 4+3 (4 does
    # not fit): 3 packs, 8 of 24 tokens padding; local greedy sorts 5,4,4,3 and
    # fills 5+3 and 4+4
    lengths, size = [5, 4, 3, 4], 8
    seq = oracle.pack_sequential(lengths, size)
    assert seq == [[0], [1, 2], [3]]
    assert oracle.padding_rate(lengths, seq, size) == pytest.approx(8 / 24)
    gr = oracle.pack_local_greedy(lengths, size, window=4)
    assert gr == [[0, 2], [1, 3]]
    assert oracle.padding_rate(lengths, gr, size) == 0.0


@pytest.mark.parametrize("window", [1, 7, 100, 10000])
def test_packing_invariants(window):
    rng = _rng(49)
    size = 4096
    lengths = [int(v) for v in np.clip(np.exp(rng.normal(np.log(800), 1.0, 3000)), 1, size)]
    lengths[10:15] = [0] * 5
    total = sum(lengths)
    for packs in (oracle.pack_sequential(lengths, size), oracle.pack_local_greedy(lengths, size, window)):
        flat = [i for p in packs for i in p]
        assert sorted(flat) == list(range(len(lengths)))           # every sequence once
        assert all(sum(lengths[i] for i in p) <= size for p in packs)
        assert len(packs) >= -(-total // size)                      # capacity lower bound
    assert [i for p in oracle.pack_sequential(lengths, size) for i in p] == list(range(len(lengths)))
    if window >= len(lengths):  # first fit decreasing over everything: within 11/9 of the bound, + 1
        assert len(oracle.pack_local_greedy(lengths, size, window)) <= 11 / 9 * -(-total // size) + 1
