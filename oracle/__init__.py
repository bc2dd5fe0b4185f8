"""FP64 CPU oracle of the hyper-connection read and of the Q2_0 matrix-vector
product (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline / reference arm may import this package.  The CUDA library never
uses it.  ``hc_oracle.cpp`` holds the arithmetic; this module compiles it with
plain ``g++`` and wraps it with ctypes.

The compile flags keep the arithmetic as written: ``-O2`` without fast-math,
and ``-ffp-contract=off`` so that no multiply-add is fused (GCC fuses by
default on aarch64).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hc_oracle.cpp")
LIB = os.path.join(HERE, "libhcoracle.so")

CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def compile_cmd(src: str = SRC, out: str = LIB) -> list[str]:
    return ["g++", *CXXFLAGS, "-o", out, src]


def build(src: str = SRC, out: str = LIB) -> str:
    """Compile the oracle into a shared library and return its path."""
    subprocess.run(compile_cmd(src, out), check=True)
    return out


_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i8p = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


@dataclass
class OracleResult:
    r_out: np.ndarray  # [T][N] float32, R' = fl32(R + P)
    ss: np.ndarray     # [T][n] float64
    rs: np.ndarray     # [T][n] float64
    lo: np.ndarray     # [T][K] float64
    u: np.ndarray      # [T][N] float64
    out: np.ndarray    # [T][N] float64
    mean: np.ndarray   # [T][d] float64


class Oracle:
    """ctypes handle on a compiled oracle library."""

    def __init__(self, path: str = LIB):
        if not os.path.exists(path):
            raise FileNotFoundError(f"oracle library not built: {path} (call oracle.build())")
        self.path = path
        lib = ctypes.CDLL(path)
        lib.hc_oracle_read.restype = ctypes.c_int
        lib.hc_oracle_read.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            _f32p, ctypes.c_void_p, _f32p, _u16p, _u16p, _f32p,
            _f32p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p,
        ]
        lib.hc_oracle_read_q8.restype = ctypes.c_int
        lib.hc_oracle_read_q8.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            _f32p, ctypes.c_void_p, _f32p, _i8p, _u16p, _i8p, _u16p, _f32p,
            _f32p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p,
        ]
        lib.hc_oracle_q2_0_matvec.restype = ctypes.c_int
        lib.hc_oracle_q2_0_matvec.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, _u8p, _u16p, _f32p, _f64p,
        ]
        lib.hc_oracle_half.restype = ctypes.c_double
        lib.hc_oracle_half.argtypes = [ctypes.c_uint16]
        self._lib = lib

    def half(self, h: int) -> float:
        """The value of the IEEE binary16 bit pattern h."""
        return float(self._lib.hc_oracle_half(h))

    def q2_0_matvec(self, Wq, Wscale, x) -> np.ndarray:
        """y [ncols][rows] float64 = W x for Q2_0 weights: Wq [rows][cols/4]
        uint8 (four two-bit codes a byte), Wscale [rows][cols/64] binary16 bits
        (uint16), x [ncols][cols] float32."""
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        rows = Wq.shape[0]
        cols = Wq.shape[1] * 4
        Wscale = np.ascontiguousarray(Wscale, dtype=np.uint16).reshape(rows, cols // 64)
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, cols)
        y = np.empty((x.shape[0], rows))
        rc = self._lib.hc_oracle_q2_0_matvec(rows, cols, x.shape[0], Wq, Wscale, x, y)
        if rc != 0:
            raise ValueError(f"hc_oracle_q2_0_matvec rejected its arguments (rc={rc})")
        return y

    def read_q8(self, n: int, d: int, K: int, R, w_norm, Wd_q, Wd_scale, Wu_q, Wu_scale, gate,
                P=None, eps: float = 1e-6) -> OracleResult:
        """The read over Q8_0 weights: Wd_q [K][n*d] int8 with Wd_scale
        [K][n*d/32] binary16 bits (uint16); Wu_q [n*d][K] int8 with Wu_scale
        [n*d][K/32]."""
        N = n * d
        R = np.ascontiguousarray(R, dtype=np.float32).reshape(-1, N)
        T = R.shape[0]
        w_norm = np.ascontiguousarray(w_norm, dtype=np.float32).reshape(N)
        gate = np.ascontiguousarray(gate, dtype=np.float32).reshape(N)
        Wd_q = np.ascontiguousarray(Wd_q, dtype=np.int8).reshape(K, N)
        Wd_scale = np.ascontiguousarray(Wd_scale, dtype=np.uint16).reshape(K, N // 32)
        Wu_q = np.ascontiguousarray(Wu_q, dtype=np.int8).reshape(N, K)
        Wu_scale = np.ascontiguousarray(Wu_scale, dtype=np.uint16).reshape(N, K // 32)
        if P is not None:
            P = np.ascontiguousarray(P, dtype=np.float32).reshape(T, N)
            p_ptr = P.ctypes.data_as(ctypes.c_void_p)
        else:
            p_ptr = None
        res = OracleResult(
            r_out=np.empty((T, N), np.float32), ss=np.empty((T, n)), rs=np.empty((T, n)),
            lo=np.empty((T, K)), u=np.empty((T, N)), out=np.empty((T, N)),
            mean=np.empty((T, d)),
        )
        rc = self._lib.hc_oracle_read_q8(
            n, d, K, T, float(eps), R, p_ptr, w_norm, Wd_q, Wd_scale, Wu_q, Wu_scale, gate,
            res.r_out, res.ss, res.rs, res.lo, res.u, res.out, res.mean)
        if rc != 0:
            raise ValueError(f"hc_oracle_read_q8 rejected its arguments (rc={rc})")
        return res

    def read(self, n: int, d: int, K: int, R, w_norm, W_down, W_up, gate,
             P=None, eps: float = 1e-6) -> OracleResult:
        """Run the whole read on host arrays.

        R, P: [T][n*d] float32; w_norm, gate: [n*d] float32;
        W_down: [K][n*d] uint16 (BF16 bits); W_up: [n*d][K] uint16.
        """
        N = n * d
        R = np.ascontiguousarray(R, dtype=np.float32).reshape(-1, N)
        T = R.shape[0]
        w_norm = np.ascontiguousarray(w_norm, dtype=np.float32).reshape(N)
        gate = np.ascontiguousarray(gate, dtype=np.float32).reshape(N)
        W_down = np.ascontiguousarray(W_down, dtype=np.uint16).reshape(K, N)
        W_up = np.ascontiguousarray(W_up, dtype=np.uint16).reshape(N, K)
        if P is not None:
            P = np.ascontiguousarray(P, dtype=np.float32).reshape(T, N)
            p_ptr = P.ctypes.data_as(ctypes.c_void_p)
        else:
            p_ptr = None
        res = OracleResult(
            r_out=np.empty((T, N), np.float32), ss=np.empty((T, n)), rs=np.empty((T, n)),
            lo=np.empty((T, K)), u=np.empty((T, N)), out=np.empty((T, N)),
            mean=np.empty((T, d)),
        )
        rc = self._lib.hc_oracle_read(
            n, d, K, T, float(eps), R, p_ptr, w_norm, W_down, W_up, gate,
            res.r_out, res.ss, res.rs, res.lo, res.u, res.out, res.mean)
        if rc != 0:
            raise ValueError(f"hc_oracle_read rejected its arguments (rc={rc})")
        return res


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _default
    if _default is None:
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            build()
        _default = Oracle(LIB)
    return _default
