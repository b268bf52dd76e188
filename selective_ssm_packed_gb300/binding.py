"""Thin ctypes binding of libvarlen_ssm.so (argument marshalling only).

Each function carries the name of the C entry point it calls (see
include/varlen_ssm.h for the definitions, layouts and error behaviour).  It
checks that the torch tensors it is handed are contiguous CUDA tensors of the
right dtype, allocates outputs and workspaces the caller did not pass (with
torch, i.e. the caching allocator), passes raw device pointers and torch's
current stream, and raises VssmError on a non-zero status.  All arithmetic
happens in the library's CUDA kernels; if the library is missing, every call
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

VSSM_F32, VSSM_BF16 = 0, 1
VSSM_STATE_CHUNK = 32
VSSM_DBG_DROP_FLAG, VSSM_DBG_WAIT_NS, VSSM_DBG_DELAY_ITEM, VSSM_DBG_DELAY_NS = 1, 2, 3, 4
VSSM_DBG_FORCE_COPY_TIMEOUT, VSSM_DBG_CHECK_FINITE, VSSM_DBG_KERNEL_EVENTS = 5, 6, 7
# the call kinds vssm_kernel_time reports
KERNEL_KINDS = {"conv_fwd": 0, "scan_fwd": 1, "scan_bwd": 2, "conv_bwd": 3}
ERR = {0: "VSSM_OK", -1: "VSSM_ERR_ARG", -2: "VSSM_ERR_DTYPE", -3: "VSSM_ERR_ALIGN",
       -4: "VSSM_ERR_WORKSPACE", -5: "VSSM_ERR_CUDA", -6: "VSSM_ERR_UNSUPPORTED",
       -16: "VSSM_ERR_BAD_CU_SEQLENS", -17: "VSSM_ERR_LOOKBACK_TIMEOUT", -18: "VSSM_ERR_NONFINITE",
       -19: "VSSM_ERR_DEVICE_CHECK"}

_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t

# name -> (restype, argtypes)
SIGNATURES = {
    "varlen_position_indices": (ctypes.c_int, [_vp, _i32, _i64, _vp, _vp, _vp]),
    "vssm_status_code": (ctypes.c_int, [_i32]),
    "varlen_conv1d_fwd_workspace_size": (_sz, [_i64, _i32, _i32]),
    "varlen_conv1d_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                                         ctypes.c_int, _vp, _vp, _vp, _vp, _sz, _vp]),
    "varlen_conv1d_bwd_workspace_size": (_sz, [_i64, _i32, _i32]),
    "varlen_conv1d_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                                         ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "varlen_selective_scan_fwd_workspace_size": (_sz, [_i64, _i32, _i32]),
    "varlen_selective_scan_chunk_states_size": (_sz, [_i64, _i32, _i32]),
    "varlen_selective_scan_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                                 ctypes.c_float, _i32,
                                                 _vp, _vp, _i32, _i64, _i32, _i32, ctypes.c_int,
                                                 _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "varlen_conv1d_scan_fwd": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                              _i32, ctypes.c_float, _i32,
                                              _vp, _vp, _i32, _i64, _i32, _i32, ctypes.c_int,
                                              _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "varlen_selective_scan_bwd_workspace_size": (_sz, [_i64, _i32, _i32]),
    "varlen_selective_scan_bwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                                 ctypes.c_float, _i32, _vp,
                                                 _vp, _vp, _i32, _i64, _i32, _i32, ctypes.c_int, _vp,
                                                 _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                                 _vp, _vp, _sz, _vp]),
    "varlen_selective_scan_fwd_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                                         ctypes.c_float, _i32,
                                                         _vp, _vp, _i32, _i64, _i32, _i32, ctypes.c_int,
                                                         _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "varlen_pack_sequences": (ctypes.c_int, [_vp, _i32, _i32, _i32, _i32, _vp, _vp,
                                             ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_double)]),
    "vssm_read_status": (ctypes.c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_int)]),
    "vssm_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "vssm_last_error": (ctypes.c_char_p, []),
    "vssm_checks_build": (ctypes.c_int, []),
    "vssm_kernel_time": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_int64)]),
    "vssm_debug_set": (ctypes.c_int, [ctypes.c_int, _i64]),
}

_lib = None


class VssmError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {ERR.get(code, code)} ({code}): {last_error()}")


def library_path() -> str:
    """The library this process loads: the checked build when VSSM_CHECKS=1
    is set in the environment, else the ordinary one."""
    return _build.lib_path()


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first with "
                               "selective_ssm_packed_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().vssm_last_error().decode()


def strerror(code: int) -> str:
    return lib().vssm_strerror(code).decode()


def debug_set(knob: int, value: int) -> None:
    _check(lib().vssm_debug_set(knob, value), "vssm_debug_set")


def _check(rc, what):
    if rc != 0:
        raise VssmError(rc, what)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return VSSM_F32
    if t.dtype == torch.bfloat16:
        return VSSM_BF16
    raise TypeError(f"I/O tensors must be float32 or bfloat16, got {t.dtype}")


def _ptr(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr() or None


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ws(workspace, nbytes, device):
    if workspace is None:
        return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace too small: {workspace.numel()} < {nbytes} bytes")
    return workspace


def read_status(workspace: torch.Tensor, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(lib().vssm_read_status(_ptr(workspace, "workspace"), _stream(stream), ctypes.byref(st)),
           "vssm_read_status")
    return st.value


def kernel_time(kind: str):
    """(total ms, launches) of one kind of call's main kernel since the last
    read, from the events VSSM_DBG_KERNEL_EVENTS records."""
    ms, n = ctypes.c_double(0.0), ctypes.c_int64(0)
    _check(lib().vssm_kernel_time(KERNEL_KINDS[kind], ctypes.byref(ms), ctypes.byref(n)), "vssm_kernel_time")
    return ms.value, n.value


def status_code(word: int) -> int:
    return lib().vssm_status_code(int(word))


# ------------------------------------------------------------------ position indices
def varlen_position_indices(cu_seqlens, total_tokens, out=None, status=None, stream=None):
    cu = cu_seqlens
    _ptr(cu, "cu_seqlens", torch.int32)
    T = int(total_tokens)
    if out is None:
        out = torch.empty(T, dtype=torch.int32, device=cu.device)
    _check(lib().varlen_position_indices(_ptr(cu, "cu_seqlens"), cu.numel() - 1, T,
                                         _ptr(out, "out", torch.int32),
                                         _ptr(status, "status", torch.int32), _stream(stream)),
           "varlen_position_indices")
    return out


# ------------------------------------------------------------------ conv1d
def conv1d_fwd_workspace_size(T, D, W):
    return lib().varlen_conv1d_fwd_workspace_size(int(T), int(D), int(W))


def conv1d_bwd_workspace_size(T, D, W):
    return lib().varlen_conv1d_bwd_workspace_size(int(T), int(D), int(W))


def varlen_conv1d_fwd(x, weight, bias, cu_seqlens, position_indices=None, apply_silu=True,
                      out=None, workspace=None, stream=None, x_init=None, x_last=None):
    """Returns u, or (u, x_last) when x_last is asked for (True allocates,
    a tensor is filled).  x_init: (S, D, W-1) f32 inputs before each sequence
    (a cut sequence's previous part's x_last); None: the plain early stop."""
    T, D = x.shape
    W = weight.shape[1]
    out = torch.empty_like(x) if out is None else out
    want_last = x_last is not None and x_last is not False
    if x_last is True:
        x_last = torch.empty((cu_seqlens.numel() - 1, D, W - 1), dtype=torch.float32, device=x.device)
    elif x_last is False:
        x_last = None
    ws = _ws(workspace, conv1d_fwd_workspace_size(T, D, W), x.device)
    _check(lib().varlen_conv1d_fwd(
        _ptr(x, "x"), _ptr(weight, "weight", torch.float32), _ptr(bias, "bias", torch.float32),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32), _ptr(position_indices, "position_indices", torch.int32),
        cu_seqlens.numel() - 1, T, D, W, int(bool(apply_silu)), _dt(x), _ptr(out, "out", x.dtype),
        _ptr(x_init, "x_init", torch.float32), _ptr(x_last, "x_last", torch.float32),
        _ptr(ws, "workspace"), ws.numel(), _stream(stream)), "varlen_conv1d_fwd")
    return (out, x_last) if want_last else out


def varlen_conv1d_bwd(x, weight, bias, du, cu_seqlens, position_indices=None, apply_silu=True,
                      dx=None, dweight=None, dbias=None, workspace=None, stream=None, x_init=None,
                      dx_last=None, dx_init=None):
    """Returns (dx, dweight, dbias), and dx_init last when it is asked for
    (True allocates, a tensor is filled).  x_init: the forward call's;
    dx_last: (S, D, W-1) gradient reaching each sequence's x_last."""
    T, D = x.shape
    W = weight.shape[1]
    dx = torch.empty_like(x) if dx is None else dx
    dweight = torch.empty_like(weight) if dweight is None else dweight
    if dbias is None and bias is not None:
        dbias = torch.empty_like(bias)
    want_init = dx_init is not None and dx_init is not False
    if dx_init is True:
        dx_init = torch.empty((cu_seqlens.numel() - 1, D, W - 1), dtype=torch.float32, device=x.device)
    elif dx_init is False:
        dx_init = None
    ws = _ws(workspace, conv1d_bwd_workspace_size(T, D, W), x.device)
    _check(lib().varlen_conv1d_bwd(
        _ptr(x, "x"), _ptr(weight, "weight", torch.float32), _ptr(bias, "bias", torch.float32),
        _ptr(du, "du", x.dtype), _ptr(cu_seqlens, "cu_seqlens", torch.int32),
        _ptr(position_indices, "position_indices", torch.int32), cu_seqlens.numel() - 1, T, D, W,
        int(bool(apply_silu)), _dt(x), _ptr(dx, "dx", x.dtype), _ptr(dweight, "dweight", torch.float32),
        _ptr(dbias, "dbias", torch.float32), _ptr(x_init, "x_init", torch.float32),
        _ptr(dx_last, "dx_last", torch.float32), _ptr(dx_init, "dx_init", torch.float32),
        _ptr(ws, "workspace"), ws.numel(), _stream(stream)),
        "varlen_conv1d_bwd")
    return (dx, dweight, dbias, dx_init) if want_init else (dx, dweight, dbias)


# ------------------------------------------------------------------ selective scan
def scan_fwd_workspace_size(T, D, N):
    return lib().varlen_selective_scan_fwd_workspace_size(int(T), int(D), int(N))


def scan_bwd_workspace_size(T, D, N):
    return lib().varlen_selective_scan_bwd_workspace_size(int(T), int(D), int(N))


def chunk_states_shape(T, D, N):
    return ((int(T) + VSSM_STATE_CHUNK - 1) // VSSM_STATE_CHUNK, int(N), int(D))


def varlen_selective_scan_fwd(u, delta_raw, A, B, C, Dskip, z, dt_bias, cu_seqlens,
                              position_indices=None, delta_softplus=True, out=None,
                              chunk_states=True, workspace=None, stream=None, y=None, gate_floor=0.0,
                              a_log=False, initial_states=None, final_states=None):
    """Returns (out, chunk_states), or (out, chunk_states, y) when y is asked
    for.  chunk_states=True allocates the saved-state array the backward call
    needs, False/None skips it, a tensor is filled.  y (the output before the
    gate, which the backward call can take for dz): None/False skips it, True
    allocates it, a tensor is filled.  gate_floor: the GateFloor gate
    SiLU(z) + gate_floor; a_log: A holds A_log (A = -exp(A_log)).
    initial_states: (S, D, N) f32 state each sequence starts from (None: zero).
    final_states: None skips them, True allocates, a tensor is filled; when
    asked for they come last in the returned tuple."""
    T, D = u.shape
    N = A.shape[1]
    out = torch.empty_like(u) if out is None else out
    want_y = y is not None and y is not False
    if y is True:
        y = torch.empty_like(u)
    elif y is False:
        y = None
    S = cu_seqlens.numel() - 1
    want_final = final_states is not None and final_states is not False
    if final_states is True:
        final_states = torch.empty((S, D, N), dtype=torch.float32, device=u.device)
    elif final_states is False:
        final_states = None
    if chunk_states is True:
        chunk_states = torch.empty(chunk_states_shape(T, D, N), dtype=torch.float32, device=u.device)
    elif chunk_states is False:
        chunk_states = None
    ws = _ws(workspace, scan_fwd_workspace_size(T, D, N), u.device)
    dt = u.dtype
    _check(lib().varlen_selective_scan_fwd(
        _ptr(u, "u"), _ptr(delta_raw, "delta_raw", dt), _ptr(A, "A", torch.float32),
        _ptr(B, "B", dt), _ptr(C, "C", dt), _ptr(Dskip, "Dskip", torch.float32), _ptr(z, "z", dt),
        _ptr(dt_bias, "dt_bias", torch.float32), int(bool(delta_softplus)), float(gate_floor),
        int(bool(a_log)),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32), _ptr(position_indices, "position_indices", torch.int32),
        cu_seqlens.numel() - 1, T, D, N, _dt(u), _ptr(out, "out", dt), _ptr(y, "y", dt),
        _ptr(chunk_states, "chunk_states", torch.float32),
        _ptr(initial_states, "initial_states", torch.float32), _ptr(final_states, "final_states", torch.float32),
        _ptr(ws, "workspace"), ws.numel(), _stream(stream)), "varlen_selective_scan_fwd")
    res = (out, chunk_states) + ((y,) if want_y else ()) + ((final_states,) if want_final else ())
    return res


def varlen_conv1d_scan_fwd(x, conv_weight, conv_bias, delta_raw, A, B, C, Dskip, z, dt_bias, cu_seqlens,
                           position_indices=None, apply_silu=True, delta_softplus=True, u=True, out=None,
                           chunk_states=True, workspace=None, stream=None, y=None, gate_floor=0.0,
                           a_log=False, initial_states=None, final_states=None):
    """The conv1d forward and the selective-scan forward in one call (u computed
    on chip; results equal the two calls' bit for bit).  Returns (u, out,
    chunk_states) plus y and final_states when asked for, as
    varlen_selective_scan_fwd; u: True allocates the conv output (the backward
    needs it), None/False skips writing it, a tensor is filled."""
    T, D = x.shape
    N = A.shape[1]
    W = conv_weight.shape[1]
    out = torch.empty_like(x) if out is None else out
    if u is True:
        u = torch.empty_like(x)
    elif u is False:
        u = None
    want_y = y is not None and y is not False
    if y is True:
        y = torch.empty_like(x)
    elif y is False:
        y = None
    S = cu_seqlens.numel() - 1
    want_final = final_states is not None and final_states is not False
    if final_states is True:
        final_states = torch.empty((S, D, N), dtype=torch.float32, device=x.device)
    elif final_states is False:
        final_states = None
    if chunk_states is True:
        chunk_states = torch.empty(chunk_states_shape(T, D, N), dtype=torch.float32, device=x.device)
    elif chunk_states is False:
        chunk_states = None
    ws = _ws(workspace, scan_fwd_workspace_size(T, D, N), x.device)
    dt = x.dtype
    _check(lib().varlen_conv1d_scan_fwd(
        _ptr(x, "x"), _ptr(conv_weight, "conv_weight", torch.float32), _ptr(conv_bias, "conv_bias", torch.float32),
        W, int(bool(apply_silu)), _ptr(delta_raw, "delta_raw", dt), _ptr(A, "A", torch.float32),
        _ptr(B, "B", dt), _ptr(C, "C", dt), _ptr(Dskip, "Dskip", torch.float32), _ptr(z, "z", dt),
        _ptr(dt_bias, "dt_bias", torch.float32), int(bool(delta_softplus)), float(gate_floor), int(bool(a_log)),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32), _ptr(position_indices, "position_indices", torch.int32),
        cu_seqlens.numel() - 1, T, D, N, _dt(x), _ptr(u, "u", dt), _ptr(out, "out", dt), _ptr(y, "y", dt),
        _ptr(chunk_states, "chunk_states", torch.float32),
        _ptr(initial_states, "initial_states", torch.float32), _ptr(final_states, "final_states", torch.float32),
        _ptr(ws, "workspace"), ws.numel(), _stream(stream)), "varlen_conv1d_scan_fwd")
    return (u, out, chunk_states) + ((y,) if want_y else ()) + ((final_states,) if want_final else ())


def varlen_selective_scan_bwd(u, delta_raw, A, B, C, Dskip, z, dt_bias, dout, cu_seqlens,
                              chunk_states, position_indices=None, delta_softplus=True,
                              grads=None, workspace=None, stream=None, y=None, gate_floor=0.0,
                              a_log=False, initial_states=None, d_final_states=None,
                              d_initial_states=None):
    """Returns dict du, ddelta_raw, dA, dB, dC, dDskip, dz, d_dt_bias.  y: the
    forward call's pre-gate output (optional; dz then reads it instead of
    recomputing it).  gate_floor, a_log: as in the forward call; with a_log
    the dA entry holds dA_log = dA * A.  initial_states: the forward call's;
    d_final_states: (S, D, N) gradient reaching each sequence's final state;
    d_initial_states: True allocates (or a tensor to fill) the gradient
    reaching each sequence's starting state, returned as "d_initial_states"."""
    T, D = u.shape
    N = A.shape[1]
    dt = u.dtype
    g = dict(grads or {})
    # outputs the caller did not pass are allocated here (only those)
    make = {"du": lambda: torch.empty_like(u), "ddelta_raw": lambda: torch.empty_like(u),
            "dA": lambda: torch.empty_like(A),
            "dB": lambda: torch.empty((T, N), dtype=torch.float32, device=u.device),
            "dC": lambda: torch.empty((T, N), dtype=torch.float32, device=u.device),
            "dDskip": lambda: torch.empty_like(Dskip) if Dskip is not None else None,
            "dz": lambda: torch.empty_like(z) if z is not None else None,
            "d_dt_bias": lambda: torch.empty_like(dt_bias) if dt_bias is not None else None}
    for k, f in make.items():
        if k not in g:
            g[k] = f()
    if d_initial_states is True:
        d_initial_states = torch.empty((cu_seqlens.numel() - 1, D, N), dtype=torch.float32, device=u.device)
    elif d_initial_states is False:
        d_initial_states = None
    g["d_initial_states"] = d_initial_states
    ws = _ws(workspace, scan_bwd_workspace_size(T, D, N), u.device)
    _check(lib().varlen_selective_scan_bwd(
        _ptr(u, "u"), _ptr(delta_raw, "delta_raw", dt), _ptr(A, "A", torch.float32),
        _ptr(B, "B", dt), _ptr(C, "C", dt), _ptr(Dskip, "Dskip", torch.float32), _ptr(z, "z", dt),
        _ptr(dt_bias, "dt_bias", torch.float32), int(bool(delta_softplus)), float(gate_floor),
        int(bool(a_log)), _ptr(dout, "dout", dt),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32), _ptr(position_indices, "position_indices", torch.int32),
        cu_seqlens.numel() - 1, T, D, N, _dt(u), _ptr(chunk_states, "chunk_states", torch.float32),
        _ptr(y, "y", dt), _ptr(initial_states, "initial_states", torch.float32),
        _ptr(d_final_states, "d_final_states", torch.float32),
        _ptr(d_initial_states, "d_initial_states", torch.float32), _ptr(g["du"], "du", dt), _ptr(g["ddelta_raw"], "ddelta_raw", dt),
        _ptr(g["dA"], "dA", torch.float32), _ptr(g["dB"], "dB", torch.float32),
        _ptr(g["dC"], "dC", torch.float32), _ptr(g["dDskip"], "dDskip", torch.float32),
        _ptr(g["dz"], "dz", dt), _ptr(g["d_dt_bias"], "d_dt_bias", torch.float32),
        _ptr(ws, "workspace"), ws.numel(), _stream(stream)), "varlen_selective_scan_bwd")
    return g


# ------------------------------------------------------------------ packing (host)
PACK_METHODS = {"sequential": 0, "local_greedy": 1}


def pack_sequences(lengths, pack_size, method="local_greedy", window=1000):
    """Packs sequences of the given lengths into packs of at most pack_size
    tokens (host work, no GPU).  Returns (packs, padding_rate): packs is a
    list of int32 arrays of sequence indices, in pack order."""
    import numpy as np
    L = np.ascontiguousarray(lengths, dtype=np.int32)
    n = int(L.size)
    order = np.empty(max(n, 1), dtype=np.int32)
    offs = np.empty(n + 1, dtype=np.int32)
    npk, pad = ctypes.c_int32(0), ctypes.c_double(0.0)
    _check(lib().varlen_pack_sequences(L.ctypes.data if n else None, n, int(pack_size), PACK_METHODS[method],
                                       int(window), order.ctypes.data, offs.ctypes.data, ctypes.byref(npk),
                                       ctypes.byref(pad)), "varlen_pack_sequences")
    return [order[offs[p]:offs[p + 1]].copy() for p in range(npk.value)], pad.value
