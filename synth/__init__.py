"""Seeded synthetic inputs for the head-wise RNN recurrence.

This module is shared by the fp64 oracle and the CUDA path's tests and bench.
It holds no arithmetic of the method itself: only random draws, their
distributions and the storage-format conversion fp32 -> bf16 that the inputs
go through before either side sees them.

Every tensor is drawn from its own PCG64 stream keyed by (seed, tensor id), so
adding a tensor never shifts the values of another.  Values for bf16 runs are
drawn in fp32 and rounded to bf16 (round to nearest, ties to even); both the
oracle and the kernels then receive exactly the same numbers (the oracle widens
them to fp64).

Workloads follow the FlashRNN pages ("FlashRNN: I/O-Aware Optimization of
Traditional RNNs on modern hardware", abstract: LSTM, GRU and sLSTM in a
head-wise form) with the shapes and distributions listed in ``WORKLOADS``.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "TENSOR_IDS", "GATES", "WORKLOADS", "round_bf16", "bf16_bits",
    "make_inputs", "workload_inputs", "make_projection_inputs",
]

# One independent stream per tensor role.
TENSOR_IDS = {"Wx": 1, "R": 2, "b": 3, "dh": 4, "h0": 5, "c0": 6, "n0": 7,
              "m0": 8, "dhT": 9, "dcT": 10, "x": 11, "W": 12, "bW": 13}

# Gates per cell.  Gate-major packing: column g*Dh + j of a G*Dh row is gate g
# of hidden unit j.  LSTM / sLSTM order (i, f, z, o); GRU order (r, z, n).
GATES = {"lstm": 4, "gru": 3, "slstm": 4}

# The five workloads: shapes, dtypes and distributions.
#   bias: "zero"  -> all zeros
#         "forget1" -> +1 on the forget-gate columns (gate 1), 0 elsewhere
#         "normal0.1" -> N(0, 0.1^2) i.i.d. (0.1 is the standard deviation)
#   R ~ U(-1/sqrt(Dh), +1/sqrt(Dh)); Wx ~ N(0, 1); zero initial states.
WORKLOADS = {
    "lstm_f32_1x64_b4_t256": dict(cell="lstm", dtype="f32", NH=1, Dh=64, B=4, T=256,
                                  bias="zero", backward=False),
    "lstm_bf16_12x64_b16_t1024": dict(cell="lstm", dtype="bf16", NH=12, Dh=64, B=16, T=1024,
                                      bias="forget1", backward=False),
    "gru_bf16_6x128_b8_t2048": dict(cell="gru", dtype="bf16", NH=6, Dh=128, B=8, T=2048,
                                    bias="normal0.1", backward=False),
    "slstm_bf16_4x256_b4_t4096": dict(cell="slstm", dtype="bf16", NH=4, Dh=256, B=4, T=4096,
                                      bias="zero", backward=False),
    "lstm_bf16_1x768_b16_t1024_train": dict(cell="lstm", dtype="bf16", NH=1, Dh=768, B=16,
                                            T=1024, bias="forget1", backward=True),
}


def _rng(seed: int, tensor: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), TENSOR_IDS[tensor]])))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 values -> fp32 values exactly representable in bf16 (RNE).

    Inputs are finite draws; NaN handling is not needed here.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of fp32 values that are already bf16-representable."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _cast(x: np.ndarray, dtype: str) -> np.ndarray:
    x = x.astype(np.float32)
    return round_bf16(x) if dtype == "bf16" else x


def make_inputs(cell: str, dtype: str, T: int, B: int, NH: int, Dh: int, *,
                seed: int = 0, bias: str = "zero", r_scale: float | None = None,
                states: str = "zero", backward: bool = False) -> dict:
    """Draw one problem instance.  All arrays are float32 (bf16-valued for bf16).

    Shapes: Wx [T,B,NH,G*Dh], R [NH,Dh,G*Dh], b [NH,G*Dh] (fp32, never rounded),
    h0/c0/n0/m0 [B,NH,Dh] (fp32), dh [T,B,NH,Dh] (input dtype) when backward.
    states: "zero" or "random" (h0,c0 ~ N(0, 0.5^2); sLSTM n0 ~ U(0.5,1.5),
    m0 ~ N(0,1)) to exercise the initial-state paths.
    """
    G = GATES[cell]
    GD = G * Dh
    a = (1.0 / np.sqrt(Dh)) if r_scale is None else float(r_scale)
    out = {"cell": cell, "dtype": dtype, "T": T, "B": B, "NH": NH, "Dh": Dh}
    out["Wx"] = _cast(_rng(seed, "Wx").standard_normal((T, B, NH, GD), dtype=np.float32), dtype)
    out["R"] = _cast(_rng(seed, "R").uniform(-a, a, size=(NH, Dh, GD)).astype(np.float32), dtype)
    if bias == "zero":
        b = np.zeros((NH, GD), np.float32)
    elif bias == "forget1":
        if cell == "gru":
            raise ValueError("forget bias is defined for LSTM-type cells only")
        b = np.zeros((NH, GD), np.float32)
        b[:, Dh:2 * Dh] = 1.0
    elif bias == "normal0.1":
        b = (0.1 * _rng(seed, "b").standard_normal((NH, GD))).astype(np.float32)
    elif bias == "normal":
        b = _rng(seed, "b").standard_normal((NH, GD)).astype(np.float32)
    else:
        raise ValueError(f"unknown bias kind {bias!r}")
    out["b"] = b
    shp = (B, NH, Dh)
    if states == "zero":
        out["h0"] = np.zeros(shp, np.float32)
        out["c0"] = np.zeros(shp, np.float32)
        out["n0"] = np.zeros(shp, np.float32)
        out["m0"] = np.zeros(shp, np.float32)
    elif states == "random":
        out["h0"] = (0.5 * _rng(seed, "h0").standard_normal(shp)).astype(np.float32)
        out["c0"] = (0.5 * _rng(seed, "c0").standard_normal(shp)).astype(np.float32)
        out["n0"] = _rng(seed, "n0").uniform(0.5, 1.5, size=shp).astype(np.float32)
        out["m0"] = _rng(seed, "m0").standard_normal(shp).astype(np.float32)
    else:
        raise ValueError(f"unknown states kind {states!r}")
    if backward:
        out["dh"] = _cast(_rng(seed, "dh").standard_normal((T, B, NH, Dh), dtype=np.float32), dtype)
        out["dhT"] = np.zeros(shp, np.float32)
        out["dcT"] = np.zeros(shp, np.float32)
    return out


def workload_inputs(name: str, *, seed: int = 0, **overrides) -> dict:
    """Inputs for one of the named ``WORKLOADS`` (sizes may be overridden)."""
    w = dict(WORKLOADS[name])
    w.update(overrides)
    return make_inputs(w["cell"], w["dtype"], w["T"], w["B"], w["NH"], w["Dh"], seed=seed,
                       bias=w["bias"], backward=w["backward"], states=w.get("states", "zero"))


def make_projection_inputs(M: int, N: int, K: int, *, seed: int = 0) -> dict:
    """Inputs of the input projection Wx = x W^T + b, rounded to bf16 (x, W).

    x [M, K] ~ N(0, 1) (M = T*B rows of an input sequence), W [N, K] ~
    N(0, 1/K) (so each output has unit variance, like the recurrence's Wx),
    b [N] ~ N(0, 0.1^2) in fp32.
    """
    x = round_bf16(_rng(seed, "x").standard_normal((M, K)).astype(np.float32))
    W = round_bf16((_rng(seed, "W").standard_normal((N, K)) / np.sqrt(max(K, 1))).astype(np.float32))
    b = (0.1 * _rng(seed, "bW").standard_normal(N)).astype(np.float32)
    return {"x": x, "W": W, "b": b}
