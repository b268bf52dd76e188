"""Seeded synthetic workloads for the packed Mamba-1 conv1d + selective scan.

This module only draws inputs: sequence lengths, packs, and parameter /
activation values.  It holds none of the operators' arithmetic, so the CUDA
path and the CPU oracle can both be fed from it without sharing any of the
method's code.  Every draw uses numpy's PCG64 generator with a stated seed.

Workloads (the shapes follow the Mamba-1 layer sizes used for packed
pre-training in the article "Shanghai AI Lab: packed variable-length Mamba
training", section "实验结果": d_model 2048 -> d_inner 4096, pack length
4096; no dataset is available, so lengths are drawn from the stated
log-normal mixes instead of a real corpus):

  tiny       lengths [4,2,3,7] (T=16), D=8,    N=4,  fp32, seed 0, fwd+bwd
  m130m      one 4096-token pack, lengths LogN(ln 300, 1) clipped [16,2048],
             D=1536, N=16, fp32, seed 1, fwd
  m14b_fwd   8 packs x 4096, LogN(ln 800, 1) clipped [32,4096],
             D=4096, N=16, bf16, seed 2, fwd
  m14b       as m14b_fwd, seed 3, fwd+bwd
  m14b_small the first 2 packs of m14b (8192 tokens), for profiler captures
  longtail   2 packs x 65536, each: 2000 lengths U{1..8}, one 32768-token
             sequence, LogN(ln 800, 1) bulk filling the rest; order shuffled;
             D=4096, N=16, bf16, seed 4, fwd+bwd

Values: x (conv input), u (scan input when the scan is run alone), z, B, C,
dout ~ N(0, 1); delta_raw ~ N(0, 0.5^2); dt_bias = inverse-softplus of
dt ~ logU[1e-3, 1e-1] per channel; A[d, n] = -(n + 1); Dskip = 1; conv
weight and bias ~ U(-1/sqrt(W), 1/sqrt(W)).  With params="general" (the
parity cases) A and Dskip are drawn instead, as a learned layer holds them:
A[d, n] = -U(0.05, 4) per entry and Dskip ~ N(0, 1), from a generator of
their own, so every other value is the same as with the default.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BUCKETS = (512, 1024, 2048, 4096, 8192)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    D: int
    N: int
    W: int
    dtype: str  # "f32" or "bf16"
    seed: int
    backward: bool
    description: str


WORKLOADS = {
    "tiny": Workload("tiny", 8, 4, 4, "f32", 0, True,
                     "4 sequences [4,2,3,7] packed into 16 tokens, D=8, N=4, fp32"),
    "m130m": Workload("m130m", 1536, 16, 4, "f32", 1, False,
                      "Mamba-130M layer: 1 pack of 4096 tokens, lengths LogN(median 300), D=1536, N=16, fp32"),
    "m14b_fwd": Workload("m14b_fwd", 4096, 16, 4, "bf16", 2, False,
                         "Mamba-1.4B layer: 8 packs x 4096 tokens, lengths LogN(median 800), D=4096, N=16, bf16"),
    "m14b": Workload("m14b", 4096, 16, 4, "bf16", 3, True,
                     "Mamba-1.4B layer: 8 packs x 4096 tokens, lengths LogN(median 800), D=4096, N=16, bf16, fwd+bwd"),
    "m14b_small": Workload("m14b_small", 4096, 16, 4, "bf16", 3, True,
                           "Mamba-1.4B layer, 2 packs x 4096 tokens (profiling size), D=4096, N=16, bf16, fwd+bwd"),
    "longtail": Workload("longtail", 4096, 16, 4, "bf16", 4, True,
                         "long tail: 2 packs x 65536 tokens (2000 short, one 32768, LogN bulk), D=4096, N=16, bf16, fwd+bwd"),
}


def _lognormal_fill(rng, pack_len, median, lo, hi, sigma=1.0):
    """Draw clipped log-normal lengths until the pack is full; the last one is
    truncated so the pack holds exactly pack_len tokens."""
    lengths = []
    total = 0
    while total < pack_len:
        L = int(round(math.exp(rng.normal(math.log(median), sigma))))
        L = min(max(L, lo), hi)
        L = min(L, pack_len - total)
        lengths.append(L)
        total += L
    return lengths


def pack_lengths(name: str, seed: int | None = None) -> list[int]:
    """Sequence lengths of a workload, in pack order."""
    wl = WORKLOADS[name]
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    if name == "tiny":
        return [4, 2, 3, 7]
    if name == "m130m":
        return _lognormal_fill(rng, 4096, 300, 16, 2048)
    if name in ("m14b_fwd", "m14b", "m14b_small"):
        out = []
        for _ in range(2 if name == "m14b_small" else 8):
            out += _lognormal_fill(rng, 4096, 800, 32, 4096)
        return out
    if name == "longtail":
        out = []
        for _ in range(2):
            short = [int(v) for v in rng.integers(1, 9, size=2000)]
            used = sum(short) + 32768
            bulk = _lognormal_fill(rng, 65536 - used, 800, 32, 4096)
            pack = short + [32768] + bulk
            order = rng.permutation(len(pack))
            out += [pack[i] for i in order]
        return out
    raise KeyError(name)


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    if len(lengths):
        cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64)).astype(np.int32)
    return cu


def bucket_of(L: int) -> int:
    """Right-padding bucket: the smallest of 512..8192 holding L, else L
    rounded up to a multiple of 8192."""
    for b in BUCKETS:
        if L <= b:
            return b
    return ((L + BUCKETS[-1] - 1) // BUCKETS[-1]) * BUCKETS[-1]


def padded_layout(lengths):
    """Each sequence in its own right-padded row of its bucket length.
    Returns (cu_seqlens of the rows, index of each real token in the padded
    token axis)."""
    rows = [bucket_of(L) for L in lengths]
    cu = cu_seqlens_from_lengths(rows)
    idx = np.concatenate([np.arange(L, dtype=np.int64) + int(cu[i]) for i, L in enumerate(lengths)]) \
        if lengths else np.zeros(0, dtype=np.int64)
    return cu, idx


def draw_values(T: int, D: int, N: int, W: int, seed: int, backward: bool = True,
                scan_input: bool = True, params: str = "s4d") -> dict:
    """Seeded float32 values for one pack of T tokens (see module docstring).
    Keys: x, u, delta_raw, z, B, C, dout (activations); A, Dskip, dt_bias,
    conv_w, conv_b (parameters).  params: "s4d" (A = -(n+1), Dskip = 1) or
    "general" (A = -U(0.05, 4), Dskip ~ N(0, 1))."""
    rng = np.random.default_rng(seed + 1_000_003)
    f32 = np.float32
    v = {}
    # parameters first so that they do not depend on T
    if params == "s4d":
        v["A"] = np.tile(-(np.arange(N, dtype=f32) + 1.0), (D, 1)).astype(f32)
        v["Dskip"] = np.ones(D, dtype=f32)
    elif params == "general":
        prng = np.random.default_rng(seed + 2_000_003)
        v["A"] = (-prng.uniform(0.05, 4.0, size=(D, N))).astype(f32)
        v["Dskip"] = prng.standard_normal(D).astype(f32)
    else:
        raise ValueError(f"params must be 's4d' or 'general', got {params!r}")
    dt = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=D))
    v["dt_bias"] = (dt + np.log(-np.expm1(-dt))).astype(f32)
    bound = 1.0 / math.sqrt(W)
    v["conv_w"] = rng.uniform(-bound, bound, size=(D, W)).astype(f32)
    v["conv_b"] = rng.uniform(-bound, bound, size=D).astype(f32)
    v["x"] = rng.standard_normal((T, D), dtype=f32)
    if scan_input:
        v["u"] = rng.standard_normal((T, D), dtype=f32)
    v["delta_raw"] = (0.5 * rng.standard_normal((T, D), dtype=f32)).astype(f32)
    v["z"] = rng.standard_normal((T, D), dtype=f32)
    v["B"] = rng.standard_normal((T, N), dtype=f32)
    v["C"] = rng.standard_normal((T, N), dtype=f32)
    if backward:
        v["dout"] = rng.standard_normal((T, D), dtype=f32)
    return v


def make(name: str, backward: bool | None = None, scan_input: bool = True) -> dict:
    """All inputs of a named workload: lengths, cu_seqlens, T and values."""
    wl = WORKLOADS[name]
    lengths = pack_lengths(name)
    cu = cu_seqlens_from_lengths(lengths)
    T = int(cu[-1])
    vals = draw_values(T, wl.D, wl.N, wl.W, wl.seed,
                       backward=wl.backward if backward is None else backward,
                       scan_input=scan_input)
    return dict(workload=wl, lengths=lengths, cu_seqlens=cu, T=T, **vals)


ACTIVATIONS = ("x", "u", "delta_raw", "z", "B", "C", "dout")


def round_to(a: np.ndarray, dtype: str) -> np.ndarray:
    """Values exactly as a device buffer of `dtype` holds them, returned as
    float32 (every bf16 value is exact in float32); bf16 uses
    round-to-nearest-even, the conversion torch applies."""
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16) \
        .to(torch.float32).numpy()


def rounded(values: dict, dtype: str) -> dict:
    """Round the activations of a draw_values() dict to the I/O dtype; the
    parameters stay float32 (they are float32 on the device too)."""
    return {k: (round_to(v, dtype) if k in ACTIVATIONS else v) for k, v in values.items()}
