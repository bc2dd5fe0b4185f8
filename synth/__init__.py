"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This package draws random numbers only (see ``hc_synth.c``); it holds none of
the read's arithmetic and imports neither the CUDA binding nor the oracle.

Input recipe (one read at geometry (n, d, K), T tokens):

===========  ==========================  =====================  ===========
tensor       shape                       distribution           tensor id
===========  ==========================  =====================  ===========
R            [T][n*d] float32            N(0, 1)                0
P (pending)  [T][n*d] float32            N(0, 0.1)              1
w_norm       [n*d] float32               1 + N(0, 0.05)         2
gate g       [n*d] float32               N(0, 1)                3
W_down       [K][n*d] BF16 (uint16)      N(0, w_std)            4
W_up         [n*d][K] BF16 (uint16)      N(0, w_std)            5
===========  ==========================  =====================  ===========

Activations (R, P) use seed ``s0``; weight set ``j`` (W_down, W_up, w_norm,
gate) uses seed ``s0 + 1 + j``.  ``w_std`` is 0.02 at d=2560, K=320 and 0.015
at d=4096, K=512.

Q2_0 matrix-vector product (rows x cols weights, ncols input columns): the
weights are N(0, 0.02) float32 draws (seed ``s0 + 1 + j`` for copy j, tensor
id 6) quantized to Q2_0 by ``quantize_q2``; the input columns are N(0, 1)
(seed ``s0 + j``, tensor id 7).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hc_synth.c")
LIB = os.path.join(HERE, "libhcsynth.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-pthread"]

TID_R, TID_P, TID_WNORM, TID_GATE, TID_WDOWN, TID_WUP, TID_Q2_W, TID_Q2_X = range(8)


def compile_cmd(out: str = LIB) -> list[str]:
    return ["gcc", *CFLAGS, "-o", out, SRC, "-lm"]


def build(out: str = LIB) -> str:
    subprocess.run(compile_cmd(out), check=True)
    return out


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            build()
        lib = ctypes.CDLL(LIB)
        for name, ptr in (("hc_synth_normal_f32", ctypes.c_void_p),
                          ("hc_synth_normal_bf16", ctypes.c_void_p)):
            f = getattr(lib, name)
            f.restype = None
            f.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_double, ctypes.c_double,
                          ptr, ctypes.c_size_t, ctypes.c_int]
        lib.hc_synth_raw.restype = ctypes.c_uint64
        lib.hc_synth_raw.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.hc_synth_mix64.restype = ctypes.c_uint64
        lib.hc_synth_mix64.argtypes = [ctypes.c_uint64]
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(seed: int, tensor_id: int, mean: float, std: float, shape, out=None) -> np.ndarray:
    """float32 array of N(mean, std) draws (optionally written into ``out``)."""
    a = np.empty(shape, np.float32) if out is None else out
    assert a.dtype == np.float32 and a.flags.c_contiguous
    _load().hc_synth_normal_f32(seed, tensor_id, mean, std, a.ctypes.data, a.size, _threads())
    return a


def normal_bf16(seed: int, tensor_id: int, mean: float, std: float, shape, out=None) -> np.ndarray:
    """uint16 array holding BF16 bits of N(mean, std) draws, rounded to nearest even."""
    a = np.empty(shape, np.uint16) if out is None else out
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    _load().hc_synth_normal_bf16(seed, tensor_id, mean, std, a.ctypes.data, a.size, _threads())
    return a


def raw(key: int, j: int) -> int:
    return int(_load().hc_synth_raw(key, j))


def mix64(z: int) -> int:
    return int(_load().hc_synth_mix64(z))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Geometry:
    n: int
    d: int
    K: int
    w_std: float

    @property
    def N(self) -> int:
        return self.n * self.d


G1 = Geometry(n=4, d=2560, K=320, w_std=0.02)    # the real geometry
G2 = Geometry(n=4, d=4096, K=512, w_std=0.015)   # the scaled-up width


@dataclass
class WeightSet:
    w_norm: np.ndarray  # [N] float32
    gate: np.ndarray    # [N] float32
    W_down: np.ndarray  # [K][N] uint16 (BF16)
    W_up: np.ndarray    # [N][K] uint16 (BF16)


@dataclass
class Activations:
    R: np.ndarray             # [T][N] float32
    P: np.ndarray | None      # [T][N] float32 or None (pending write off)


def weight_set(g: Geometry, j: int = 0, s0: int = 0) -> WeightSet:
    seed = s0 + 1 + j
    return WeightSet(
        w_norm=normal_f32(seed, TID_WNORM, 1.0, 0.05, (g.N,)),
        gate=normal_f32(seed, TID_GATE, 0.0, 1.0, (g.N,)),
        W_down=normal_bf16(seed, TID_WDOWN, 0.0, g.w_std, (g.K, g.N)),
        W_up=normal_bf16(seed, TID_WUP, 0.0, g.w_std, (g.N, g.K)),
    )


@dataclass
class Q8WeightSet:
    """Q8_0 copies of a weight set: per row, blocks of 32 consecutive values
    along the dot-product axis, one IEEE binary16 scale and 32 int8 quants per
    block (weight = scale * q); quants and scales as separate arrays."""
    w_norm: np.ndarray    # [N] float32
    gate: np.ndarray      # [N] float32
    Wd_q: np.ndarray      # [K][N] int8
    Wd_scale: np.ndarray  # [K][N/32] uint16 (binary16 bits)
    Wu_q: np.ndarray      # [N][K] int8
    Wu_scale: np.ndarray  # [N][K/32] uint16 (binary16 bits)


def quantize_q8(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Q8_0 blocks of a [rows][cols] float32 matrix (cols a multiple of 32):
    scale = binary16(max |w| / 127) per block, q = round-to-nearest-even of
    w / scale clamped to [-127, 127] (0 where the scale is 0)."""
    rows, cols = w.shape
    blocks = np.asarray(w, np.float32).reshape(rows, cols // 32, 32)
    scale = (np.abs(blocks).max(axis=2) / np.float32(127)).astype(np.float16)
    s = scale.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s > 0, np.rint(blocks / np.where(s > 0, s, 1)), 0)
    return np.clip(q, -127, 127).astype(np.int8).reshape(rows, cols), scale.view(np.uint16)


def q8_weight_set(g: Geometry, j: int = 0, s0: int = 0) -> Q8WeightSet:
    """Weight set j of ``weight_set`` with its projections drawn in float32
    (the same draws BF16 rounds) and quantized to Q8_0."""
    seed = s0 + 1 + j
    wd_q, wd_s = quantize_q8(normal_f32(seed, TID_WDOWN, 0.0, g.w_std, (g.K, g.N)))
    wu_q, wu_s = quantize_q8(normal_f32(seed, TID_WUP, 0.0, g.w_std, (g.N, g.K)))
    return Q8WeightSet(
        w_norm=normal_f32(seed, TID_WNORM, 1.0, 0.05, (g.N,)),
        gate=normal_f32(seed, TID_GATE, 0.0, 1.0, (g.N,)),
        Wd_q=wd_q, Wd_scale=wd_s, Wu_q=wu_q, Wu_scale=wu_s)


@dataclass
class Q2Matrix:
    """A Q2_0 matrix: per row, blocks of 64 consecutive values, one IEEE
    binary16 scale d and 64 two-bit codes q per block (weight = d * (q - 2)),
    the codes packed four to a byte, least significant bits first."""
    Wq: np.ndarray       # [rows][cols/4] uint8
    Wscale: np.ndarray   # [rows][cols/64] uint16 (binary16 bits)


def pack_q2(codes: np.ndarray) -> np.ndarray:
    """Pack [rows][cols] codes in 0..3 four to a byte: value j of a row at
    bits 2*(j % 4) of byte j // 4."""
    c = np.asarray(codes, np.uint8)
    rows, cols = c.shape
    c = c.reshape(rows, cols // 4, 4)
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def quantize_q2(w: np.ndarray) -> Q2Matrix:
    """Q2_0 blocks of a [rows][cols] float32 matrix (cols a multiple of 64):
    scale = binary16(max |w| / 2) per block, q - 2 = round-to-nearest-even of
    w / scale clamped to [-2, 1] (q = 2 where the scale is 0)."""
    rows, cols = w.shape
    blocks = np.asarray(w, np.float32).reshape(rows, cols // 64, 64)
    scale = (np.abs(blocks).max(axis=2) / np.float32(2)).astype(np.float16)
    s = scale.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s > 0, np.rint(blocks / np.where(s > 0, s, 1)), 0)
    codes = (np.clip(q, -2, 1) + 2).astype(np.uint8).reshape(rows, cols)
    return Q2Matrix(Wq=pack_q2(codes), Wscale=scale.view(np.uint16))


def q2_0_matrix(rows: int, cols: int, j: int = 0, s0: int = 0, w_std: float = 0.02) -> Q2Matrix:
    """Q2_0 copy j of a [rows][cols] projection drawn as N(0, w_std) in
    float32 (seed s0 + 1 + j, tensor id TID_Q2_W)."""
    return quantize_q2(normal_f32(s0 + 1 + j, TID_Q2_W, 0.0, w_std, (rows, cols)))


def q2_0_columns(cols: int, ncols: int, j: int = 0, s0: int = 0) -> np.ndarray:
    """[ncols][cols] float32 input columns, N(0, 1) (seed s0 + j, tensor id
    TID_Q2_X)."""
    return normal_f32(s0 + j, TID_Q2_X, 0.0, 1.0, (ncols, cols))


def activations(g: Geometry, T: int, pending: bool, s0: int = 0) -> Activations:
    R = normal_f32(s0, TID_R, 0.0, 1.0, (T, g.N))
    P = normal_f32(s0, TID_P, 0.0, 0.1, (T, g.N)) if pending else None
    return Activations(R=R, P=P)
