"""CPU oracle for the packed Mamba-1 conv1d + selective scan -- TEST INFRASTRUCTURE.

This package wraps ``varlen_ssm_oracle.c`` (plain C, double precision, one
sequence at a time).  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import it.  The product path
(``selective_ssm_packed_gb300``) never does: it shares no code, header, table
or helper with this file.

Arrays are numpy float64 (values) and int32 (``cu_seqlens``), laid out as in
the C file's header comment.  ``d_range`` picks a channel range; the
``*_threaded`` helpers split the channel axis into blocks run on a thread
pool (the C calls release the GIL) and add the per-block dB/dC partials in
block order, so the result does not depend on the thread count.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "varlen_ssm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libvarlen_ssm_oracle.so")

_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE double throughout)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
             _SRC, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_position_indices.argtypes = [_ip, ctypes.c_int32, ctypes.c_int64, _ip]
            lib.oracle_conv1d_fwd.argtypes = [_dp, _dp, _dp, _ip, ctypes.c_int32, ctypes.c_int64,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, _dp, _dp, _dp]
            lib.oracle_conv1d_bwd.argtypes = [_dp, _dp, _dp, _dp, _ip, ctypes.c_int32, ctypes.c_int64,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, _dp, _dp, _dp, _dp, _dp, _dp]
            lib.oracle_scan_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int32,
                                            ctypes.c_double, _dp,
                                            _ip, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _dp, _dp]
            lib.oracle_scan_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int32,
                                            ctypes.c_double, _dp, _dp,
                                            _dp, _ip, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
            for name in ("oracle_position_indices", "oracle_conv1d_fwd", "oracle_conv1d_bwd",
                         "oracle_scan_fwd", "oracle_scan_bwd"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    if a is None:
        return None
    if a.dtype == np.int32:
        return a.ctypes.data_as(_ip)
    return a.ctypes.data_as(_dp)


def _cu(cu):
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    return cu, int(cu.shape[0] - 1), int(cu[-1]) if cu.shape[0] else 0


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc} (malformed cu_seqlens?)")


def position_indices(cu_seqlens, total_tokens=None):
    cu, S, T = _cu(cu_seqlens)
    if total_tokens is not None:
        T = int(total_tokens)
    pos = np.empty(T, dtype=np.int32)
    _check(_load().oracle_position_indices(_p(cu), S, T, _p(pos)), "position_indices")
    return pos


def conv1d_fwd(x, weight, bias, cu_seqlens, apply_silu=True, d_range=None, x_init=None,
               return_last=False):
    """u (T, D); with return_last, also each sequence's last W-1 inputs (S, D, W-1).
    x_init (S, D, W-1): the W-1 inputs before each sequence (zero when None)."""
    x, w, b, x_init = _f64(x), _f64(weight), _f64(bias), _f64(x_init)
    cu, S, T = _cu(cu_seqlens)
    D, W = w.shape
    d0, d1 = d_range if d_range is not None else (0, D)
    u = np.zeros((T, D), dtype=np.float64)
    xl = np.zeros((S, D, W - 1), dtype=np.float64) if return_last else None
    _check(_load().oracle_conv1d_fwd(_p(x), _p(w), _p(b), _p(cu), S, T, D, W, int(apply_silu),
                                     d0, d1, _p(x_init), _p(u), _p(xl)), "conv1d_fwd")
    return (u, xl) if return_last else u


def conv1d_bwd(x, weight, bias, du, cu_seqlens, apply_silu=True, d_range=None, x_init=None,
               dx_last=None, return_dx_init=False):
    """(dx, dweight, dbias), and dx_init (S, D, W-1) last with return_dx_init.
    dx_last (S, D, W-1): the gradient reaching each sequence's last W-1 inputs
    from outside (zero when None)."""
    x, w, b, du = _f64(x), _f64(weight), _f64(bias), _f64(du)
    x_init, dx_last = _f64(x_init), _f64(dx_last)
    cu, S, T = _cu(cu_seqlens)
    D, W = w.shape
    d0, d1 = d_range if d_range is not None else (0, D)
    dx = np.zeros((T, D), dtype=np.float64)
    dw = np.zeros((D, W), dtype=np.float64)
    db = np.zeros(D, dtype=np.float64)
    dxi = np.zeros((S, D, W - 1), dtype=np.float64) if return_dx_init else None
    _check(_load().oracle_conv1d_bwd(_p(x), _p(w), _p(b), _p(du), _p(cu), S, T, D, W,
                                     int(apply_silu), d0, d1, _p(x_init), _p(dx_last), _p(dx), _p(dw),
                                     _p(db), _p(dxi)), "conv1d_bwd")
    return (dx, dw, db, dxi) if return_dx_init else (dx, dw, db)


def scan_fwd(u, delta_raw, A, B, C, Dskip, z, dt_bias, cu_seqlens, delta_softplus=True,
             d_range=None, return_last_state=False, gate_floor=0.0, h_init=None):
    """out (T, D); with return_last_state, also the state after each sequence's
    last token (S, D, N).  h_init (S, D, N): each sequence's starting state
    (zero when None); gate_floor: the GateFloor bias on the gate."""
    u, dr, A, B, C = _f64(u), _f64(delta_raw), _f64(A), _f64(B), _f64(C)
    Dskip, z, dt_bias, h_init = _f64(Dskip), _f64(z), _f64(dt_bias), _f64(h_init)
    cu, S, T = _cu(cu_seqlens)
    D, N = A.shape
    d0, d1 = d_range if d_range is not None else (0, D)
    out = np.zeros((T, D), dtype=np.float64)
    hl = np.zeros((S, D, N), dtype=np.float64) if return_last_state else None
    _check(_load().oracle_scan_fwd(_p(u), _p(dr), _p(A), _p(B), _p(C), _p(Dskip), _p(z),
                                   _p(dt_bias), int(delta_softplus), float(gate_floor), _p(h_init),
                                   _p(cu), S, T, D, N, d0, d1, _p(out), _p(hl)), "scan_fwd")
    return (out, hl) if return_last_state else out


def scan_bwd(u, delta_raw, A, B, C, Dskip, z, dt_bias, dout, cu_seqlens, delta_softplus=True,
             d_range=None, gate_floor=0.0, h_init=None, dh_last=None):
    """Returns dict du, ddelta_raw, dA, dB, dC, dDskip, dz, d_dt_bias and
    dh_init (the gradient reaching each sequence's starting state, (S, D, N)),
    float64.  dh_last (S, D, N): the gradient reaching each sequence's final
    state from outside (zero when None)."""
    u, dr, A, B, C = _f64(u), _f64(delta_raw), _f64(A), _f64(B), _f64(C)
    Dskip, z, dt_bias, dout = _f64(Dskip), _f64(z), _f64(dt_bias), _f64(dout)
    h_init, dh_last = _f64(h_init), _f64(dh_last)
    cu, S, T = _cu(cu_seqlens)
    D, N = A.shape
    d0, d1 = d_range if d_range is not None else (0, D)
    g = {
        "du": np.zeros((T, D)), "ddelta_raw": np.zeros((T, D)), "dA": np.zeros((D, N)),
        "dB": np.zeros((T, N)), "dC": np.zeros((T, N)),
        "dDskip": np.zeros(D) if Dskip is not None else None,
        "dz": np.zeros((T, D)) if z is not None else None,
        "d_dt_bias": np.zeros(D) if dt_bias is not None else None,
        "dh_init": np.zeros((S, D, N)),
    }
    _check(_load().oracle_scan_bwd(_p(u), _p(dr), _p(A), _p(B), _p(C), _p(Dskip), _p(z),
                                   _p(dt_bias), int(delta_softplus), float(gate_floor), _p(h_init),
                                   _p(dh_last), _p(dout), _p(cu), S, T, D, N,
                                   d0, d1, _p(g["du"]), _p(g["ddelta_raw"]), _p(g["dA"]),
                                   _p(g["dB"]), _p(g["dC"]), _p(g["dDskip"]), _p(g["dz"]),
                                   _p(g["d_dt_bias"]), _p(g["dh_init"])), "scan_bwd")
    return g


def _blocks(d0, d1, nblocks):
    nblocks = max(1, min(nblocks, d1 - d0))
    edges = np.linspace(d0, d1, nblocks + 1).round().astype(int)
    return [(int(edges[i]), int(edges[i + 1])) for i in range(nblocks) if edges[i + 1] > edges[i]]


def default_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def scan_fwd_threaded(u, delta_raw, A, B, C, Dskip, z, dt_bias, cu_seqlens, delta_softplus=True,
                      channels=None, threads=None, gate_floor=0.0, h_init=None):
    """Forward scan over a channel range (default all) split across threads."""
    D = np.asarray(A).shape[0]
    d0, d1 = channels if channels is not None else (0, D)
    threads = threads or default_threads()
    args = [_f64(a) for a in (u, delta_raw, A, B, C, Dskip, z, dt_bias)]
    h_init = _f64(h_init)
    outs = []
    with ThreadPoolExecutor(threads) as ex:
        futs = [ex.submit(scan_fwd, *args, cu_seqlens, delta_softplus, blk, False, gate_floor, h_init)
                for blk in _blocks(d0, d1, threads * 2)]
        for blk, f in zip(_blocks(d0, d1, threads * 2), futs):
            outs.append((blk, f.result()))
    T = args[0].shape[0]
    out = np.zeros((T, D))
    for (b0, b1), o in outs:
        out[:, b0:b1] = o[:, b0:b1]
    return out


def scan_bwd_threaded(u, delta_raw, A, B, C, Dskip, z, dt_bias, dout, cu_seqlens,
                      delta_softplus=True, channels=None, threads=None, gate_floor=0.0, h_init=None,
                      dh_last=None):
    """Backward scan over a channel range split across threads; dB/dC are the
    sum over that range, added block by block in channel order."""
    D = np.asarray(A).shape[0]
    d0, d1 = channels if channels is not None else (0, D)
    threads = threads or default_threads()
    args = [_f64(a) for a in (u, delta_raw, A, B, C, Dskip, z, dt_bias, dout)]
    h_init, dh_last = _f64(h_init), _f64(dh_last)
    blocks = _blocks(d0, d1, threads * 2)
    with ThreadPoolExecutor(threads) as ex:
        futs = [ex.submit(scan_bwd, *args, cu_seqlens, delta_softplus, blk, gate_floor, h_init, dh_last)
                for blk in blocks]
        parts = [f.result() for f in futs]
    res = {k: (None if v is None else np.zeros_like(v)) for k, v in parts[0].items()}
    for (b0, b1), g in zip(blocks, parts):
        for k in ("du", "ddelta_raw", "dz"):
            if g[k] is not None:
                res[k][:, b0:b1] = g[k][:, b0:b1]
        for k in ("dA", "dDskip", "d_dt_bias"):
            if g[k] is not None:
                res[k][b0:b1] = g[k][b0:b1]
        res["dh_init"][:, b0:b1] = g["dh_init"][:, b0:b1]
        res["dB"] += g["dB"]
        res["dC"] += g["dC"]
    return res


def conv1d_fwd_threaded(x, weight, bias, cu_seqlens, apply_silu=True, channels=None, threads=None):
    D = np.asarray(weight).shape[0]
    d0, d1 = channels if channels is not None else (0, D)
    threads = threads or default_threads()
    x, w, b = _f64(x), _f64(weight), _f64(bias)
    blocks = _blocks(d0, d1, threads * 2)
    with ThreadPoolExecutor(threads) as ex:
        futs = [ex.submit(conv1d_fwd, x, w, b, cu_seqlens, apply_silu, blk) for blk in blocks]
        parts = [f.result() for f in futs]
    u = np.zeros_like(x)
    for (b0, b1), o in zip(blocks, parts):
        u[:, b0:b1] = o[:, b0:b1]
    return u


def conv1d_bwd_threaded(x, weight, bias, du, cu_seqlens, apply_silu=True, channels=None,
                        threads=None):
    D = np.asarray(weight).shape[0]
    d0, d1 = channels if channels is not None else (0, D)
    threads = threads or default_threads()
    x, w, b, du = _f64(x), _f64(weight), _f64(bias), _f64(du)
    blocks = _blocks(d0, d1, threads * 2)
    with ThreadPoolExecutor(threads) as ex:
        futs = [ex.submit(conv1d_bwd, x, w, b, du, cu_seqlens, apply_silu, blk) for blk in blocks]
        parts = [f.result() for f in futs]
    dx = np.zeros_like(x)
    dw = np.zeros_like(w)
    db = np.zeros(w.shape[0])
    for (b0, b1), (pdx, pdw, pdb) in zip(blocks, parts):
        dx[:, b0:b1] = pdx[:, b0:b1]
        dw[b0:b1] = pdw[b0:b1]
        db[b0:b1] = pdb[b0:b1]
    return dx, dw, db


# ---------------------------------------------------------------- sequence packing
# The article's section 结论与讨论: its pack method takes sequences in arrival
# order and seals a pack when the next sequence does not fit (19.1 % padding
# on its pretraining data); a local greedy method first sorts a portion of the
# pending sequences and then packs greedily (down to 0.46 %).  Both written
# out as plain loops; every pack holds at most pack_size tokens.

def pack_sequential(lengths, pack_size):
    """Packs as lists of sequence indices, in arrival order."""
    packs, cur, used = [], [], 0
    for i, n in enumerate(lengths):
        if n > pack_size:
            raise ValueError("a sequence is longer than a pack")
        if cur and used + n > pack_size:
            packs.append(cur)
            cur, used = [], 0
        cur.append(i)
        used += n
    if cur:
        packs.append(cur)
    return packs


def pack_local_greedy(lengths, pack_size, window):
    """The pending sequences are taken `window` at a time; each window is
    sorted by length, longest first (ties in arrival order), and every
    sequence goes into the first of the window's packs with room for it, or
    opens a new one (first fit, decreasing).  A window's packs are sealed
    before the next window starts."""
    packs = []
    for w0 in range(0, len(lengths), window):
        idx = list(range(w0, min(w0 + window, len(lengths))))
        idx.sort(key=lambda i: (-lengths[i], i))
        open_packs, room = [], []
        for i in idx:
            n = lengths[i]
            if n > pack_size:
                raise ValueError("a sequence is longer than a pack")
            for p in range(len(open_packs)):
                if room[p] >= n:
                    open_packs[p].append(i)
                    room[p] -= n
                    break
            else:
                open_packs.append([i])
                room.append(pack_size - n)
        packs.extend(open_packs)
    return packs


def padding_rate(lengths, packs, pack_size):
    """Padded tokens over pack capacity."""
    if not packs:
        return 0.0
    used = sum(lengths[i] for p in packs for i in p)
    return 1.0 - used / (len(packs) * pack_size)
